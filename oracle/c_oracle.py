"""ctypes front end of the plain-C fp64 oracle (oracle/kda_oracle.c).

TEST INFRASTRUCTURE ONLY (tests, the smoke check and the bench's CPU-baseline
leg). Builds the shared object with gcc on first use; computes exactly the
token-by-token definition documented in kda_oracle.c and kda_ref.py, for all
(sequence, head) pairs or for a chosen subset of them.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kda_oracle.c")
_LIB = os.path.join(_HERE, "libkda_oracle.so")
_lock = threading.Lock()
_lib = None

__all__ = ["build", "kda_fwd_c", "default_threads"]


def build(force: bool = False) -> str:
    """Compile kda_oracle.c into oracle/libkda_oracle.so (gcc, portable flags)."""
    with _lock:
        if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
            tmp = _LIB + f".tmp{os.getpid()}"
            subprocess.check_call(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fPIC",
                                   "-shared", "-pthread", "-o", tmp, _SRC, "-lm"])
            os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        P = ctypes.c_void_p
        lib.kda_oracle_fwd.restype = ctypes.c_int
        lib.kda_oracle_fwd.argtypes = [P, P, P, P, P, P, P, ctypes.c_double, ctypes.c_double,
                                       P, P, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                       ctypes.c_int, ctypes.c_int, ctypes.c_int, P,
                                       ctypes.c_int, P, P, P, ctypes.c_double, ctypes.c_int]
        _lib = lib
    return _lib


def default_threads() -> int:
    try:
        return max(1, len(os.sched_getaffinity(0)))
    except AttributeError:  # pragma: no cover
        return max(1, os.cpu_count() or 1)


def _bits16(x):
    """Raw 16-bit patterns of a bf16 torch tensor as a contiguous uint16 array."""
    import torch
    assert x.dtype == torch.bfloat16
    return np.ascontiguousarray(x.detach().cpu().contiguous().view(torch.int16).numpy()).view(np.uint16)


def _f32(x):
    if x is None:
        return None
    import torch
    if isinstance(x, torch.Tensor):
        x = x.detach().cpu().to(torch.float32).numpy()
    return np.ascontiguousarray(x, dtype=np.float32)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def kda_fwd_c(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
              initial_state=None, cu_seqlens=None, pairs=None, eps=1e-6,
              n_threads=None, full_o=True):
    """fp64 oracle over bf16 torch inputs.

    pairs: None (all (sequence, head) pairs) or a list of (seq, head).
    Returns (o, final):
      * full_o=True and pairs None: o float64 [B,T,H,V], final [N,H,V,K];
      * otherwise: o is a list with one float64 [len_s, V] array per pair, and
        final is float64 [n_pairs, V, K].
    """
    B, T, H, K = q.shape
    V = v.shape[-1]
    if cu_seqlens is not None:
        cu = np.ascontiguousarray(np.asarray(cu_seqlens.cpu() if hasattr(cu_seqlens, "cpu")
                                             else cu_seqlens, dtype=np.int32))
        N = cu.size - 1
        lens = np.diff(cu.astype(np.int64))
    else:
        cu = None
        N = B
        lens = np.full(B, T, dtype=np.int64)
    all_pairs = pairs is None
    if all_pairs:
        pr = np.array([(s, h) for s in range(N) for h in range(H)], dtype=np.int32).reshape(-1, 2)
    else:
        pr = np.ascontiguousarray(np.asarray(pairs, dtype=np.int32).reshape(-1, 2))
    n_pairs = pr.shape[0]
    rows = np.zeros(n_pairs, dtype=np.int64)
    if n_pairs:
        rows[1:] = np.cumsum(lens[pr[:-1, 0]])
    total_rows = int(rows[-1] + lens[pr[-1, 0]]) if n_pairs else 0
    o_c = np.zeros((max(total_rows, 1), V), dtype=np.float64)
    fin = np.zeros((max(n_pairs, 1), V, K), dtype=np.float64)
    import torch
    qb, kb, vb, gb, bb = (_bits16(x) for x in (q, k, v, g, beta))
    al = _f32(A_log)
    dt = _f32(dt_bias)
    ini = None if initial_state is None else np.ascontiguousarray(
        initial_state.detach().cpu().to(torch.float64).numpy() if hasattr(initial_state, 'detach')
        else np.asarray(initial_state, np.float64))
    lib = _load()
    rc = lib.kda_oracle_fwd(_ptr(qb), _ptr(kb), _ptr(vb), _ptr(gb), _ptr(bb), _ptr(al), _ptr(dt),
                            float(lower_bound), float(scale), _ptr(ini), _ptr(cu), B, T, H, K, V,
                            N, _ptr(pr), n_pairs, _ptr(rows), _ptr(o_c), _ptr(fin), float(eps),
                            int(n_threads or default_threads()))
    if rc != 0:
        raise RuntimeError(f"kda_oracle_fwd failed with code {rc}")
    starts = np.zeros(N + 1, dtype=np.int64)
    starts[1:] = np.cumsum(lens)
    if all_pairs and full_o:
        o = np.zeros((B, T, H, V))
        for p in range(n_pairs):
            s, h = int(pr[p, 0]), int(pr[p, 1])
            blk = o_c[rows[p]:rows[p] + lens[s]]
            if cu is not None:
                o[0, starts[s]:starts[s + 1], h] = blk
            else:
                o[s, :, h] = blk
        return o, fin[:n_pairs].reshape(N, H, V, K)
    outs = [o_c[rows[p]:rows[p] + lens[int(pr[p, 0])]] for p in range(n_pairs)]
    return outs, fin[:n_pairs]
