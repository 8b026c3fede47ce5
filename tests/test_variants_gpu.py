"""GPU parity of the kda_fwd_ex variants against the fp64 numpy oracle (small shapes).

Variants (include/kda.h): one gate per token and head (g [B,T,H], dt_bias [H]; the
gated delta rule as the oracle reads it), fp32 beta logits, a bf16 state and the
[N,H,K,V] state layout. Inputs are the seeded workload draws plus extra seeded
draws for the variant tensors.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from chunked_gated_delta_02_gb300.workloads import custom, make_inputs
from kda_testlib import TOL_S_REL, assert_parity, rel_l2, to_dev

pytestmark = pytest.mark.gpu

# A bf16 state adds, to the fp32-state bound, the rounding of the stored state: at most 2^-9
# relative per element, about 2^-9 / sqrt(3) = 1.13e-3 in RMS for uniformly spread mantissas.
TOL_S_REL_BF16 = TOL_S_REL + 1.2e-3


def _variant_inputs(w, seed, per_head=False, beta_f32=False, state_bf16=False):
    inp = make_inputs(w, seed=seed)
    gen = torch.Generator().manual_seed(seed + 7)
    B, T, H = inp["q"].shape[:3]
    if per_head:
        inp["g"] = (0.5 * torch.randn(B, T, H, generator=gen)).to(torch.bfloat16)
        inp["dt_bias"] = 0.2 * torch.randn(H, generator=gen)
    else:
        inp["dt_bias"] = 0.1 * torch.randn(inp["dt_bias"].shape, generator=gen)
    if beta_f32:   # logits that bf16 cannot hold exactly
        inp["beta"] = torch.randn(B, T, H, generator=gen) * 1.37
    if state_bf16 and inp["initial_state"] is not None:
        inp["initial_state"] = inp["initial_state"].to(torch.bfloat16)
    return inp


def _oracle(inp):
    from oracle import kda_fwd_ref
    return kda_fwd_ref(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"], inp["dt_bias"],
                       inp["lower_bound"], inp["scale"], inp["initial_state"], inp["cu_seqlens"])


def _run(inp, layout="vk", state_dtype=None):
    import chunked_gated_delta_02_gb300 as kda
    d = to_dev(inp)
    ini = d["initial_state"]
    if ini is not None and layout == "kv":
        ini = ini.transpose(-1, -2).contiguous()
    o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                    d["scale"], ini, True, d["cu_seqlens"], state_layout=layout, state_dtype=state_dtype)
    torch.cuda.synchronize()
    if layout == "kv":
        fs = fs.transpose(-1, -2)
    return o, fs


def _check(inp, what, layout="vk", state_dtype=None, bf16_state=False):
    o, fs = _run(inp, layout, state_dtype)
    ref_o, ref_f = _oracle(inp)
    eo, mo, _ = assert_parity(o, None, ref_o, ref_f, what)
    gf = fs.float().cpu().double().numpy()
    assert np.all(np.isfinite(gf)), f"{what}: non-finite final state"
    es = rel_l2(gf, ref_f)
    tol = TOL_S_REL_BF16 if bf16_state else TOL_S_REL
    assert es <= tol, f"{what}: final_state rel-L2 {es:.3e} (<= {tol})"
    if bf16_state:
        assert fs.dtype == torch.bfloat16
    print(f"{what}: o rel {eo:.2e} maxabs {mo:.2e} state rel {es:.2e}")


@pytest.mark.parametrize("B,T,H,K,V", [(2, 130, 3, 128, 128), (1, 200, 2, 64, 64), (1, 64, 2, 128, 64)])
def test_gate_per_head(B, T, H, K, V):
    w = custom(B=B, T=T, H=H, K=K, V=V, lower_bound=-5.0, init_state=True)
    _check(_variant_inputs(w, seed=T + K, per_head=True), f"per-head gate B{B} T{T} H{H} K{K} V{V}")


def test_gate_per_head_varlen():
    w = custom(H=2, K=64, V=64, seqlens=[0, 1, 63, 64, 65, 150, 7], lower_bound=-2.0)
    _check(_variant_inputs(w, seed=11, per_head=True), "per-head gate varlen")


def test_beta_fp32():
    w = custom(B=2, T=100, H=2, K=128, V=128, lower_bound=-3.0)
    inp = _variant_inputs(w, seed=5, beta_f32=True)
    assert inp["beta"].dtype == torch.float32
    _check(inp, "beta fp32")


@pytest.mark.parametrize("layout", ["vk", "kv"])
def test_state_bf16(layout):
    w = custom(B=2, T=150, H=2, K=128, V=128, lower_bound=-1.0)
    _check(_variant_inputs(w, seed=9, state_bf16=True), f"bf16 state {layout}", layout=layout, bf16_state=True)


@pytest.mark.parametrize("K,V", [(128, 128), (64, 128), (128, 64)])
def test_state_kv_layout(K, V):
    w = custom(B=2, T=90, H=2, K=K, V=V, lower_bound=-5.0)
    _check(_variant_inputs(w, seed=K + V), f"kv layout K{K} V{V}", layout="kv")


def test_bf16_final_state_without_initial_state():
    w = custom(B=1, T=70, H=2, K=64, V=64, init_state=False)
    _check(_variant_inputs(w, seed=3), "bf16 final, no initial", state_dtype=torch.bfloat16, bf16_state=True)


def test_all_variants_together_varlen():
    w = custom(H=3, K=128, V=128, seqlens=[5, 0, 129, 64, 40], lower_bound=-4.0)
    inp = _variant_inputs(w, seed=21, per_head=True, beta_f32=True, state_bf16=True)
    _check(inp, "all variants, varlen", layout="kv", bf16_state=True)


def test_all_variants_wide_slices():
    # 128 sequence-head pairs: the recurrence runs 64-column V slices
    w = custom(B=4, T=100, H=32, K=64, V=64, lower_bound=-5.0)
    inp = _variant_inputs(w, seed=33, per_head=True, beta_f32=True, state_bf16=True)
    _check(inp, "all variants, wide slices", layout="kv", bf16_state=True)


@pytest.mark.parametrize("w", [custom(B=2, T=130, H=3, K=128, V=128, lower_bound=-5.0),
                               custom(H=2, K=64, V=64, seqlens=[0, 1, 63, 64, 65, 150, 7], lower_bound=-1.0)],
                         ids=["fixed-K128", "varlen-K64"])
def test_exp2_poly_option(w):
    import chunked_gated_delta_02_gb300 as kda
    inp = _variant_inputs(w, seed=17)
    d = to_dev(inp)
    o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                    d["scale"], d["initial_state"], True, d["cu_seqlens"], exp2_poly=True)
    torch.cuda.synchronize()
    ref_o, ref_f = _oracle(inp)
    eo, mo, es = assert_parity(o, fs, ref_o, ref_f, "exp2 polynomial")
    print(f"exp2 polynomial: o rel {eo:.2e} maxabs {mo:.2e} state rel {es:.2e}")


def test_exp2_poly_with_per_head_gate():
    w = custom(B=1, T=200, H=2, K=128, V=64, lower_bound=-3.0)
    inp = _variant_inputs(w, seed=19, per_head=True, beta_f32=True)
    import chunked_gated_delta_02_gb300 as kda
    d = to_dev(inp)
    o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                    d["scale"], d["initial_state"], True, d["cu_seqlens"], exp2_poly=True)
    torch.cuda.synchronize()
    ref_o, ref_f = _oracle(inp)
    assert_parity(o, fs, ref_o, ref_f, "exp2 polynomial, per-head gate, fp32 beta")
