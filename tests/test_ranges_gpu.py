"""GPU cases at the edges of the fp16 ranges of the tensor-core operands.

* Keys chosen to make the triangular inverse as large as possible (nearly dependent keys of
  rank 1 plus noise, exactly repeated keys, keys turning in a plane; beta close to 1), as in
  tests/test_ranges.py, run through the kernels: the fp16 hand-off of
  Tb = (I + A)^{-1} diag(beta) and P Tb keeps its range there. With slow decay they match the
  oracle; with no decay at all the operands' precision bounds the error (see below).
* Large values with slow decay that stay inside the fp16 range of the recurrence's operands
  (state, residuals, v) match the oracle.
* Values past that range (|x| > 65504 in the state or in an fp32 initial state) are reported
  through the device status word as KDA_DEVICE_NONFINITE instead of passing silently.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from chunked_gated_delta_02_gb300.workloads import custom, make_inputs
from kda_testlib import check_full, run_gpu

pytestmark = pytest.mark.gpu

KDA_DEVICE_NONFINITE = 3


def _unit(x):
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def _adversarial_keys(kind, B, T, H, K, rng):
    if kind == "rank1+noise":
        base = rng.standard_normal((1, 1, H, K))
        sign = rng.choice([-1.0, 1.0], (B, T, H, 1))
        k = sign * base + 1e-3 * rng.standard_normal((B, T, H, K))
    elif kind == "rank1":
        k = np.broadcast_to(rng.standard_normal((1, 1, H, K)), (B, T, H, K)).copy()
    elif kind == "circle":
        th = 0.5 * np.arange(T)[None, :, None]
        k = np.zeros((B, T, H, K))
        k[..., 0], k[..., 1] = np.cos(th), np.sin(th)
    else:
        raise ValueError(kind)
    return torch.from_numpy(_unit(k)).to(torch.bfloat16)


KINDS = ["rank1+noise", "rank1", "circle"]


def _adversarial_inputs(kind, lb):
    inp = make_inputs(custom(B=1, T=256, H=2, K=128, V=128, lower_bound=lb, init_state=True), seed=51)
    rng = np.random.default_rng(KINDS.index(kind))
    inp["k"] = _adversarial_keys(kind, 1, 256, 2, 128, rng)
    inp["beta"] = torch.full_like(inp["beta"], 8.0)      # beta = sigmoid(8) = 1 - 3.4e-4
    return inp


@pytest.mark.parametrize("kind", KINDS)
def test_adversarial_keys_slow_decay_match_oracle(kind):
    check_full(_adversarial_inputs(kind, -0.1), f"{kind} lb=-0.1")


# Measured precision envelope with no decay at all (lb = 0). Then 1 - beta = 3.4e-4 lies below the
# 2^-11 resolution of the fp16 / tf32 tensor-core operands, so the rounding of A, of Tb and of the
# hand-off M decides the weights (1 - beta)^n of earlier writes along a repeated key. A CPU
# emulation of the kernels' roundings gives the same errors as the GPU (rank1+noise: o 1.07e-2,
# state 2.1e-2; rank1: 9.7e-3, 2.1e-2; circle: 2.9e-3, 4.4e-3). The outputs stay finite and
# bounded; the bounds below are that envelope with some margin, not the parity tolerance.
ENVELOPE_O_REL, ENVELOPE_S_REL = 2e-2, 4e-2


@pytest.mark.parametrize("kind", KINDS)
def test_adversarial_keys_no_decay_stay_in_precision_envelope(kind):
    import chunked_gated_delta_02_gb300 as kda
    from kda_testlib import TOL_O_MAXABS, oracle_full, rel_l2
    kda.device_status()
    inp = _adversarial_inputs(kind, 0.0)
    o, fs = run_gpu(inp)
    ref_o, ref_f = oracle_full(inp)
    go, gf = o.float().cpu().double().numpy(), fs.cpu().double().numpy()
    assert np.isfinite(go).all() and np.isfinite(gf).all()
    eo, es = rel_l2(go, ref_o), rel_l2(gf, ref_f)
    print(f"{kind} lb=0: o rel {eo:.2e} state rel {es:.2e}")
    assert eo <= ENVELOPE_O_REL and float(np.abs(go - ref_o).max()) <= TOL_O_MAXABS
    assert es <= ENVELOPE_S_REL
    assert kda.device_status() == 0


def _growth_inputs(v_value, T=1024):
    """beta = 1, no decay, the same v every token: the state grows to about 2.8 |v| (oracle)."""
    inp = make_inputs(custom(B=1, T=T, H=1, K=128, V=128, lower_bound=0.0, init_state=False), seed=41)
    inp["v"] = torch.full_like(inp["v"], v_value)
    inp["beta"] = torch.full_like(inp["beta"], 20.0)
    return inp


def _check_scaled(inp, data_scale, what):
    """Parity for inputs whose v is data_scale times the workloads' N(0,1): rel-L2 bounds as
    stated, and the max-abs bound (stated for unit-scale data, where it is a few bf16 units of the
    largest outputs) scaled with the data."""
    from kda_testlib import TOL_O_MAXABS, TOL_O_REL, TOL_S_REL, oracle_full, rel_l2
    o, fs = run_gpu(inp)
    ref_o, ref_f = oracle_full(inp)
    go, gf = o.float().cpu().double().numpy(), fs.cpu().double().numpy()
    assert np.isfinite(go).all() and np.isfinite(gf).all(), what
    eo, mo, es = rel_l2(go, ref_o), float(np.abs(go - ref_o).max()), rel_l2(gf, ref_f)
    print(f"{what}: o rel {eo:.2e} max-abs {mo:.2e} (max |o| {np.abs(ref_o).max():.1f}) state rel {es:.2e}")
    assert eo <= TOL_O_REL and mo <= TOL_O_MAXABS * data_scale and es <= TOL_S_REL, what


def test_large_values_inside_fp16_range_match_oracle():
    import chunked_gated_delta_02_gb300 as kda
    kda.device_status()
    _check_scaled(_growth_inputs(1000.0), 1000.0, "state near 2.8e3")
    inp = make_inputs(custom(B=1, T=512, H=2, K=128, V=128, lower_bound=-0.05, init_state=True), seed=42)
    inp["v"] = (inp["v"].float() * 100.0).to(torch.bfloat16)
    _check_scaled(inp, 100.0, "v ~ 100 N(0,1), slow decay")
    assert kda.device_status() == 0


def test_state_past_fp16_range_is_reported():
    """v = 3e4 (inside the fp16 range) drives the state to about 8e4 (past it): the fp16 copy of
    the state overflows, and the call reports KDA_DEVICE_NONFINITE."""
    import chunked_gated_delta_02_gb300 as kda
    from kda_testlib import oracle_full
    kda.device_status()
    inp = _growth_inputs(30000.0)
    ref_o, ref_f = oracle_full(inp)
    assert np.isfinite(ref_f).all() and np.abs(ref_f).max() > 65504.0   # the method itself is fine
    run_gpu(inp)
    assert kda.device_status() == KDA_DEVICE_NONFINITE
    assert kda.device_status() == 0                                     # read and cleared


def test_large_fp32_initial_state_is_reported():
    import chunked_gated_delta_02_gb300 as kda
    kda.device_status()
    inp = make_inputs(custom(B=1, T=100, H=2, K=64, V=64, lower_bound=-1.0, init_state=True), seed=43)
    inp["initial_state"] = inp["initial_state"] * 0.0 + 1.0e5
    run_gpu(inp)
    assert kda.device_status() == KDA_DEVICE_NONFINITE
    # a normal call afterwards is clean
    run_gpu(make_inputs(custom(B=1, T=100, H=2, K=64, V=64, init_state=True), seed=44))
    assert kda.device_status() == 0
