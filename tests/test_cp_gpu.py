"""GPU parity of intracard context parallelism (segments of a sequence run in parallel).

The segmented recurrence (a local pass with the K x K state transitions, a combine of the
segment start states, a final pass) computes the same forward pass as the plain recurrence:
each case forces a segment count through KDA_CP_SEGMENTS(n) and compares every output with the
fp64 oracle under the usual tolerances. Slow or no decay is used where it matters, since with
the workloads' fast decay the state forgets a segment's start within a chunk or two.
"""
from __future__ import annotations

import numpy as np
import pytest
import torch

from chunked_gated_delta_02_gb300.workloads import custom, make_inputs, named
from kda_testlib import assert_parity, check_all_pairs, oracle_full, to_dev

pytestmark = pytest.mark.gpu


def _run(inp, n_seg, final=True, **kw):
    import chunked_gated_delta_02_gb300 as kda
    d = to_dev(inp)
    o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                    d["scale"], d["initial_state"], final, d["cu_seqlens"], context_parallel=n_seg, **kw)
    torch.cuda.synchronize()
    return o, fs


# (B, T, H, K, V, lower_bound, initial state, segments): chunk-aligned and ragged lengths, uneven
# splits, more segments than chunks (empty segments), both head dimensions, no / slow / fast decay
CASES = [
    (1, 2048, 1, 128, 128, -0.1, True, 2), (1, 2048, 1, 128, 128, -0.1, True, 3),
    (1, 2048, 2, 128, 128, 0.0, True, 4), (2, 1000, 2, 128, 128, 0.0, True, 5),
    (2, 1000, 2, 128, 128, -0.05, False, 3), (1, 700, 2, 64, 64, -0.5, True, 4),
    (1, 640, 2, 64, 128, -0.02, True, 3), (1, 640, 2, 128, 64, -0.02, True, 3),
    (1, 300, 2, 128, 128, 0.0, True, 8), (1, 65, 1, 64, 64, -1.0, True, 3),
    (3, 1500, 3, 128, 128, -5.0, True, 6),
]


@pytest.mark.parametrize("B,T,H,K,V,lb,init,n", CASES)
def test_segments_match_oracle(B, T, H, K, V, lb, init, n):
    import chunked_gated_delta_02_gb300 as kda
    inp = make_inputs(custom(B=B, T=T, H=H, K=K, V=V, lower_bound=lb, init_state=init), seed=B * 100 + T + n)
    assert kda.plan(B, T, H, K, V, B, context_parallel=n) == (n, 64)
    o, fs = _run(inp, n)
    ref_o, ref_f = oracle_full(inp)
    eo, mo, es = assert_parity(o, fs, ref_o, ref_f, f"CP n={n} B{B} T{T} H{H} K{K} V{V} lb{lb}")
    print(f"CP n={n} B{B} T{T} H{H} K{K} V{V} lb{lb}: o rel {eo:.2e} state rel {es:.2e}")
    assert kda.device_status() == 0


def test_segments_agree_with_plain_recurrence():
    inp = make_inputs(custom(B=1, T=3000, H=2, K=128, V=128, lower_bound=-0.02, init_state=True), seed=61)
    o1, f1 = _run(inp, False)
    o2, f2 = _run(inp, 4)
    d = (o1.float() - o2.float()).abs().max().item()
    assert d < 2e-2, d
    assert (f1 - f2).norm().item() / f1.norm().item() < 2e-3


def test_segments_without_final_state_and_in_place():
    import chunked_gated_delta_02_gb300 as kda
    inp = make_inputs(custom(B=2, T=900, H=2, K=128, V=128, lower_bound=-0.05, init_state=True), seed=62)
    ref_o, ref_f = oracle_full(inp)
    o, fs = _run(inp, 3, final=False)
    assert fs is None
    assert_parity(o, None, ref_o, None, "CP without final state")
    d = to_dev(inp)
    st = d["initial_state"].clone()
    o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                    d["scale"], st, True, None, final_state=st, context_parallel=3)
    torch.cuda.synchronize()
    assert fs.data_ptr() == st.data_ptr()
    assert_parity(o, st, ref_o, ref_f, "CP in-place state")


def test_segments_with_state_variants():
    """bf16 state in the [N,H,K,V] layout: segment 0 reads it and the last segment writes it."""
    import chunked_gated_delta_02_gb300 as kda
    from kda_testlib import TOL_S_REL, rel_l2
    inp = make_inputs(custom(B=1, T=1100, H=2, K=128, V=64, lower_bound=-0.05, init_state=True), seed=63)
    inp["initial_state"] = inp["initial_state"].to(torch.bfloat16)
    ref_o, ref_f = oracle_full(inp)
    d = to_dev(inp)
    ini = d["initial_state"].transpose(-1, -2).contiguous()   # [N,H,K,V]
    o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                    d["scale"], ini, True, None, state_layout="kv", context_parallel=4)
    torch.cuda.synchronize()
    assert fs.dtype == torch.bfloat16
    assert_parity(o, None, ref_o, None, "CP bf16 kv state")
    assert rel_l2(fs.float().transpose(-1, -2).cpu().numpy(), ref_f) <= TOL_S_REL + 1.2e-3
    assert kda.device_status() == 0


def test_varlen_ignores_forced_segments():
    import chunked_gated_delta_02_gb300 as kda
    assert kda.plan(1, 3000, 2, 128, 128, 3, varlen=True, context_parallel=4) == (0, 16)
    inp = make_inputs(custom(H=2, K=128, V=128, seqlens=[1000, 0, 2000], init_state=True), seed=64)
    o, fs = _run(inp, 4)
    ref_o, ref_f = oracle_full(inp)
    assert_parity(o, fs, ref_o, ref_f, "varlen with a forced segment count")


def test_segments_in_cuda_graph():
    """The three launches of the segmented recurrence captured in a CUDA graph and replayed give
    the bits of the eager call."""
    import chunked_gated_delta_02_gb300 as kda
    inp = make_inputs(custom(B=1, T=1500, H=2, K=128, V=128, lower_bound=-0.05, init_state=True), seed=65)
    d = to_dev(inp)
    B, T, H, K = d["q"].shape
    V = d["v"].shape[-1]
    ws = torch.empty(kda.workspace_size(B, T, H, K, V, B, False, kda.CP_SEGMENTS(3)), dtype=torch.uint8,
                     device="cuda")
    o = torch.empty(B, T, H, V, dtype=torch.bfloat16, device="cuda")
    fs = torch.empty(B, H, V, K, dtype=torch.float32, device="cuda")

    def call():
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                d["scale"], d["initial_state"], True, None, workspace=ws, out=o, final_state=fs,
                context_parallel=3)

    call()
    torch.cuda.synchronize()
    ref = (o.clone(), fs.clone())
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call()
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call()
    o.zero_()
    fs.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, ref[0]) and torch.equal(fs, ref[1])
    assert kda.device_status() == 0


def test_long_workload_with_segments_all_pairs():
    """The long-context workload (B=1, T=65536, H=16, lower_bound=-1) forced through 4 segments,
    every (sequence, head) against the oracle."""
    import chunked_gated_delta_02_gb300 as kda
    inp = make_inputs(named("long"), seed=0)
    o, fs = _run(inp, 4)
    eo, mo, es = check_all_pairs(inp, o, fs, "long, 4 segments")
    print(f"long with 4 segments: o rel {eo:.2e} maxabs {mo:.2e} state rel {es:.2e} (all pairs)")
    assert kda.device_status() == 0


def test_automatic_plan_takes_segments_for_few_long_sequences():
    """Few heads of one long sequence leave most SMs idle: the library's plan cuts it into
    segments, and the result matches the oracle. Many heads keep the plain recurrence."""
    import chunked_gated_delta_02_gb300 as kda
    n, bv = kda.plan(1, 32768, 2, 128, 128, 1)
    assert n >= 2 and bv == 64, (n, bv)
    assert kda.plan(2, 2048, 32, 128, 128, 2)[0] == 0
    inp = make_inputs(custom(B=1, T=32768, H=2, K=128, V=128, lower_bound=-0.1, init_state=True), seed=66)
    o, fs = _run(inp, None)
    ref_o, ref_f = oracle_full(inp)
    eo, mo, es = assert_parity(o, fs, ref_o, ref_f, f"automatic plan, {n} segments")
    print(f"automatic plan ({n} segments): o rel {eo:.2e} state rel {es:.2e}")
