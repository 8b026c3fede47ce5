"""Seeded synthetic inputs for the KDA chunked forward.

This module only draws random numbers and lays them out. It holds none of the
method's arithmetic (no gate, no norm, no recurrence), so both the fp64 oracle
and the CUDA path can be fed from it without sharing any of the method's code.

The shapes and value distributions follow the KDA forward API described on the
FlashKDA page (discuss.pytorch.kr, section "FlashKDA의 KDA 연산 구조", parameter
table): q, k, g bf16 [B,T,H,K]; v bf16 [B,T,H,V]; beta bf16 [B,T,H] logits;
A_log fp32 [H]; dt_bias fp32 [H,K]; lower_bound scalar in [-5, 0]; state fp32
[N,H,V,K]. The value distributions (q,k,v ~ N(0,1), g ~ 0.1 N(0,1),
A_log ~ 0.01 N(0,1), dt_bias = 0) are the ones the cuLA README quick start uses
(shadowgraph.io mirror of the cuLA README, "KDA (Kimi Delta Attention) -
Blackwell (SM10X)"). Packed variable-length batches use int32 cu_seqlens, as the
same README notes.

Draw order is fixed: sequence lengths (varlen only), q, k, v, g, beta, A_log,
initial_state. Everything is drawn on the CPU from torch.Generator(seed).
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import Optional

import torch

__all__ = ["KDAWorkload", "NAMED", "make_inputs", "named", "seqlens_of"]


@dataclass(frozen=True)
class KDAWorkload:
    """One synthetic KDA forward problem (shapes and distribution knobs)."""

    name: str
    H: int
    K: int
    V: int
    B: int = 1
    T: int = 0                      # per-sequence length when seqlens is None
    seqlens: Optional[tuple] = None  # explicit packed lengths (B must be 1)
    n_varlen: int = 0               # draw this many lengths uniformly ...
    len_lo: int = 0                 # ... from [len_lo, len_hi] inclusive
    len_hi: int = 0
    lower_bound: float = -5.0
    init_state: bool = True         # initial_state ~ 0.1 N(0,1) else None
    g_scale: float = 0.1
    a_log_scale: float = 0.01
    scale: Optional[float] = None   # default K ** -0.5
    extra: dict = field(default_factory=dict)

    @property
    def is_varlen(self) -> bool:
        return self.seqlens is not None or self.n_varlen > 0

    def describe(self) -> str:
        if self.n_varlen:
            shape = (f"{self.n_varlen} seqs len~U[{self.len_lo},{self.len_hi}] "
                     f"packed B=1")
        elif self.seqlens is not None:
            shape = f"{len(self.seqlens)} seqs lens={list(self.seqlens)} packed B=1"
        else:
            shape = f"B={self.B} T={self.T}"
        return (f"{shape} H={self.H} K={self.K} V={self.V} "
                f"lower_bound={self.lower_bound} "
                f"initial_state={'0.1N(0,1)' if self.init_state else 'zeros(None)'}")


# The five reference workloads: shapes and distributions of the KDA forward
# benchmarks (tiny parity case, fixed length, packed varlen, long context,
# many short sequences).
NAMED = {
    "tiny": KDAWorkload("tiny", B=1, T=128, H=2, K=64, V=64, lower_bound=-5.0,
                        init_state=True),
    "fixed": KDAWorkload("fixed", B=2, T=2048, H=32, K=128, V=128,
                         lower_bound=-5.0, init_state=False),
    "varlen": KDAWorkload("varlen", B=1, H=32, K=128, V=128, n_varlen=16,
                          len_lo=64, len_hi=8192, lower_bound=-5.0,
                          init_state=True),
    "long": KDAWorkload("long", B=1, T=65536, H=16, K=128, V=128,
                        lower_bound=-1.0, init_state=False),
    "large_batch": KDAWorkload("large_batch", B=64, T=512, H=64, K=128, V=128,
                               lower_bound=-5.0, init_state=True),
}


def named(name: str) -> KDAWorkload:
    return NAMED[name]


def _randn(gen, shape, scale=1.0):
    x = torch.randn(shape, generator=gen, dtype=torch.float32)
    if scale != 1.0:
        x.mul_(scale)
    return x


def seqlens_of(w: KDAWorkload, seed: int = 0) -> Optional[list]:
    """Sequence lengths of a varlen workload (first draw of the generator)."""
    if w.seqlens is not None:
        return [int(x) for x in w.seqlens]
    if w.n_varlen:
        gen = torch.Generator().manual_seed(seed)
        return [int(x) for x in torch.randint(w.len_lo, w.len_hi + 1,
                                              (w.n_varlen,), generator=gen)]
    return None


def make_inputs(w: KDAWorkload, seed: int = 0) -> dict:
    """Draw the inputs of workload ``w`` on the CPU.

    Returns a dict with bf16 tensors q, k, v, g, beta; fp32 A_log [H],
    dt_bias [H,K], initial_state [N,H,V,K] or None; int32 cu_seqlens [N+1] or
    None; and the scalars lower_bound, scale, B, T, H, K, V, N.
    """
    gen = torch.Generator().manual_seed(seed)
    H, K, V = w.H, w.K, w.V
    cu = None
    if w.is_varlen:
        if w.seqlens is not None:
            lens = [int(x) for x in w.seqlens]
        else:
            lens = [int(x) for x in torch.randint(w.len_lo, w.len_hi + 1,
                                                  (w.n_varlen,), generator=gen)]
        B, T, N = 1, int(sum(lens)), len(lens)
        cu = torch.zeros(N + 1, dtype=torch.int32)
        if N:
            cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    else:
        B, T, N = w.B, w.T, w.B
    bf = torch.bfloat16
    q = _randn(gen, (B, T, H, K)).to(bf)
    k = _randn(gen, (B, T, H, K)).to(bf)
    v = _randn(gen, (B, T, H, V)).to(bf)
    g = _randn(gen, (B, T, H, K), w.g_scale).to(bf)
    beta = _randn(gen, (B, T, H)).to(bf)
    A_log = _randn(gen, (H,), w.a_log_scale)
    dt_bias = torch.zeros(H, K, dtype=torch.float32)
    init = _randn(gen, (N, H, V, K), 0.1) if w.init_state else None
    scale = w.scale if w.scale is not None else K ** -0.5
    return dict(q=q, k=k, v=v, g=g, beta=beta, A_log=A_log, dt_bias=dt_bias,
                initial_state=init, cu_seqlens=cu, lower_bound=float(w.lower_bound),
                scale=float(scale), B=B, T=T, H=H, K=K, V=V, N=N)


def custom(B=1, T=64, H=1, K=64, V=64, lower_bound=-5.0, init_state=True,
           seqlens=None, g_scale=0.1, name="custom") -> KDAWorkload:
    """A workload with explicit shapes (used by parity and edge-case tests)."""
    if seqlens is not None:
        return KDAWorkload(name, B=1, H=H, K=K, V=V, seqlens=tuple(seqlens),
                           lower_bound=lower_bound, init_state=init_state,
                           g_scale=g_scale)
    return KDAWorkload(name, B=B, T=T, H=H, K=K, V=V, lower_bound=lower_bound,
                       init_state=init_state, g_scale=g_scale)
