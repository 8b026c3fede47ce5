"""kda_fwd_noalloc: the entry point for callers that cannot allocate device memory.

Such callers (a runtime that owns the whole GPU memory pool and gives a kernel
only its inputs and outputs, or a path where cudaMalloc is not allowed) get the
same forward pass with the scratch taken from a fixed array inside libkda.so.
These tests check, through the C ABI, that two calls in a row give the same
outputs as kda_fwd() with a caller workspace, within the parity tolerances of
the other tests, and that a problem too large for the array is refused before
anything runs. This file is collected last so that a run stopping at the first
failure has already run every other test.
"""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

from chunked_gated_delta_02_gb300.workloads import custom, make_inputs, named
from kda_testlib import TOL_O_MAXABS, TOL_O_REL, TOL_S_REL, assert_parity, oracle_full, rel_l2, to_dev


def test_too_large_is_refused_before_any_cuda_call():
    from chunked_gated_delta_02_gb300 import build
    import os
    if not os.path.exists(build.LIB):
        build.build()
    import chunked_gated_delta_02_gb300 as kda
    from chunked_gated_delta_02_gb300._lib import lib
    assert kda.workspace_size(1, 8192, 8, 128, 128, 1) > kda.NOALLOC_MAX_SCRATCH
    fake = ctypes.c_void_p(0x10000)   # never dereferenced: the size check comes first
    rc = lib().kda_fwd_noalloc(fake, fake, fake, fake, fake, fake, None, -5.0, 0.125, None, None, None,
                               1, 8192, 8, 128, 128, 1, fake, None)
    assert rc == 3   # KDA_ERR_WORKSPACE


def _both(inp):
    import chunked_gated_delta_02_gb300 as kda
    d = to_dev(inp)
    B, T, H, K, V, N = (inp[x] for x in ("B", "T", "H", "K", "V", "N"))
    assert kda.workspace_size(B, T, H, K, V, N) <= kda.NOALLOC_MAX_SCRATCH
    o_ref, f_ref = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                           d["lower_bound"], d["scale"], d["initial_state"], True, d["cu_seqlens"])
    o_na = torch.full_like(o_ref, float("nan"))
    f_na = torch.full_like(f_ref, float("nan"))
    kda.fwd_noalloc(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                    d["scale"], d["initial_state"], f_na, d["cu_seqlens"], out=o_na)
    torch.cuda.synchronize()
    return o_ref, f_ref, o_na, f_na


@pytest.mark.gpu
def test_noalloc_matches_kda_fwd_on_two_calls_in_a_row():
    first = make_inputs(custom(B=2, T=300, H=3, K=128, V=128, init_state=True), seed=21)
    second = make_inputs(named("tiny"), seed=22)       # different sizes: no reliance on leftovers
    for name, inp in (("first call", first), ("second call", second)):
        o_ref, f_ref, o_na, f_na = _both(inp)
        a, b = o_na.float().cpu().numpy(), o_ref.float().cpu().numpy()
        assert np.all(np.isfinite(a)) and np.all(np.isfinite(f_na.cpu().numpy())), name
        assert rel_l2(a, b) <= TOL_O_REL and float(np.max(np.abs(a - b))) <= TOL_O_MAXABS, name
        assert rel_l2(f_na.cpu().numpy(), f_ref.cpu().numpy()) <= TOL_S_REL, name
        # and against the fp64 oracle directly, so that a fault common to both entry points
        # (say, in how the scratch is laid out) cannot pass unseen
        ref_o, ref_f = oracle_full(inp)
        assert_parity(o_na, f_na, ref_o, ref_f, f"noalloc {name} vs oracle")


@pytest.mark.gpu
def test_noalloc_varlen_after_fixed():
    inp = make_inputs(custom(H=2, K=64, V=64, seqlens=[100, 0, 64, 1, 130], init_state=True), seed=23)
    o_ref, f_ref, o_na, f_na = _both(inp)
    assert rel_l2(o_na.float().cpu().numpy(), o_ref.float().cpu().numpy()) <= TOL_O_REL
    assert rel_l2(f_na.cpu().numpy(), f_ref.cpu().numpy()) <= TOL_S_REL
