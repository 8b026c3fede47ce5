"""GPU parity of the CUDA path (through the C ABI) against the fp64 oracle."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from chunked_gated_delta_02_gb300.workloads import custom, make_inputs, named
from kda_testlib import (assert_parity, check_all_pairs, check_full, oracle_full, rel_l2, run_gpu, to_dev)

pytestmark = pytest.mark.gpu


def test_tiny_config():
    eo, mo, es = check_full(make_inputs(named("tiny"), seed=0), "tiny")
    print(f"tiny: o rel {eo:.2e} maxabs {mo:.2e} state rel {es:.2e}")


# Shapes of the reference's end-to-end KDA tests (B-T-H-D: 1-63-1-128, 2-500-3-128,
# 2-1000-3-128, 3-1024-4-128, ...: T need not be a multiple of the chunk) plus
# head dim 64 and the chunk edges T = 1, 64, 65. The recurrence kernel takes 16-column V slices
# when 64-column slices would leave most SMs idle: the small shapes run that way, the last two
# (128 sequence-head pairs x 64-column slices) run with 64-column slices.
SHAPES = [
    (1, 63, 1, 128, 128, -5.0, True), (2, 500, 3, 128, 128, -5.0, False), (2, 1000, 3, 128, 128, -1.0, True),
    (3, 1024, 4, 128, 128, -5.0, True), (1, 1, 2, 64, 64, -5.0, True), (1, 64, 2, 64, 64, -0.1, True),
    (1, 65, 2, 64, 64, -5.0, False), (2, 130, 2, 64, 64, -2.0, True), (1, 200, 2, 64, 128, -5.0, True),
    (1, 200, 2, 128, 64, -0.5, True), (1, 333, 2, 128, 128, 0.0, True),
    (4, 200, 32, 64, 64, -5.0, True), (2, 130, 32, 128, 128, -3.0, True),
]


@pytest.mark.parametrize("B,T,H,K,V,lb,init", SHAPES)
def test_shapes(B, T, H, K, V, lb, init):
    w = custom(B=B, T=T, H=H, K=K, V=V, lower_bound=lb, init_state=init)
    check_full(make_inputs(w, seed=B * 1000 + T), f"B{B}-T{T}-H{H}-K{K}-V{V}-lb{lb}")


@pytest.mark.parametrize("lens", [[0, 1, 63, 64, 65, 200, 0, 7], [500, 3, 1000], [1], [0]])
def test_varlen(lens):
    w = custom(H=3, K=128, V=128, seqlens=lens, init_state=True)
    check_full(make_inputs(w, seed=len(lens)), f"varlen {lens}")


def test_varlen_head_dim_64():
    w = custom(H=2, K=64, V=64, seqlens=[130, 1, 64, 77], init_state=False)
    check_full(make_inputs(w, seed=3), "varlen K=V=64")


def test_initial_state_none_equals_zeros_and_final_optional():
    inp = make_inputs(custom(B=2, T=150, H=2, K=128, V=128, init_state=False), seed=7)
    o1, f1 = run_gpu(inp)
    z = torch.zeros(2, 2, 128, 128, dtype=torch.float32)
    o2, f2 = run_gpu(inp, init=z.cuda())
    o3, f3 = run_gpu(inp, output_final_state=False)
    assert f3 is None
    assert torch.equal(o1, o2) and torch.equal(f1, f2) and torch.equal(o1, o3)


def test_in_place_state_update():
    inp = make_inputs(custom(B=1, T=300, H=2, K=128, V=128, init_state=True), seed=8)
    ref_o, ref_f = oracle_full(inp)
    d = to_dev(inp)
    import chunked_gated_delta_02_gb300 as kda
    st = d["initial_state"].clone()
    o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                    d["scale"], st, True, None, final_state=st)
    torch.cuda.synchronize()
    assert fs.data_ptr() == st.data_ptr()
    assert_parity(o, st, ref_o, ref_f, "in-place state")


def test_split_sequence_carries_state():
    """Running [0,T1) then [T1,T) from the GPU's own final state matches the oracle."""
    inp = make_inputs(custom(B=1, T=400, H=2, K=128, V=128, init_state=True), seed=9)
    ref_o, ref_f = oracle_full(inp)
    cut = 137
    a = {k: (v[:, :cut].contiguous() if k in ("q", "k", "v", "g", "beta") else v) for k, v in inp.items()}
    a["T"] = cut
    oa, fa = run_gpu(a)
    b = {k: (v[:, cut:].contiguous() if k in ("q", "k", "v", "g", "beta") else v) for k, v in inp.items()}
    b["initial_state"] = fa.cpu()
    ob, fb = run_gpu(b)
    assert_parity(torch.cat([oa, ob], 1), fb, ref_o, ref_f, "split at 137")


def test_deterministic():
    inp = make_inputs(custom(B=2, T=257, H=3, K=128, V=128), seed=10)
    o1, f1 = run_gpu(inp)
    o2, f2 = run_gpu(inp)
    assert torch.equal(o1, o2) and torch.equal(f1, f2)


@pytest.mark.parametrize("w", [custom(B=2, T=257, H=3, K=128, V=128, init_state=True),
                               custom(H=2, K=64, V=64, seqlens=[0, 1, 63, 64, 65, 150, 7])],
                         ids=["fixed", "varlen"])
def test_launch_modes_agree(w):
    """The recurrence kernel launched to overlap the prep kernel (no event between them, as in
    kda_fwd) and launched after it (an event between them) give the same bits."""
    import chunked_gated_delta_02_gb300 as kda
    d = to_dev(make_inputs(w, seed=12))
    outs = []
    for mode in ("overlap", "split", "none"):
        ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        events = {"overlap": (ev[0], None, ev[2]), "split": tuple(ev), "none": None}[mode]
        o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                        d["scale"], d["initial_state"], True, d["cu_seqlens"], events=events)
        torch.cuda.synchronize()
        outs.append((o, fs))
    for o, fs in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(fs, outs[0][1])
    assert kda.device_status() == 0


@pytest.mark.parametrize("w", [custom(B=2, T=200, H=3, K=128, V=128, init_state=True),
                               custom(H=2, K=64, V=64, seqlens=[0, 1, 63, 64, 65, 150, 7])],
                         ids=["fixed", "varlen"])
def test_cuda_graph_capture_and_replay(w):
    """The forward captured in a CUDA graph (with a caller workspace; the kernels' overlapped
    launches become graph edges) and replayed gives the same bits as the eager call, also
    after new inputs are copied into the captured buffers."""
    import chunked_gated_delta_02_gb300 as kda
    d = to_dev(make_inputs(w, seed=13))
    d2 = to_dev(make_inputs(w, seed=14))
    B, T, H, K = d["q"].shape
    V = d["v"].shape[-1]
    N = B if d["cu_seqlens"] is None else d["cu_seqlens"].numel() - 1
    ws = torch.empty(max(kda.workspace_size(B, T, H, K, V, N), 1), dtype=torch.uint8, device="cuda")
    o = torch.empty(B, T, H, V, dtype=torch.bfloat16, device="cuda")
    fs = torch.empty(N, H, V, K, dtype=torch.float32, device="cuda")

    def call(x, out=None, final=None):
        return kda.fwd(x["q"], x["k"], x["v"], x["g"], x["beta"], x["A_log"], x["dt_bias"], x["lower_bound"],
                       x["scale"], x["initial_state"], True, x["cu_seqlens"], workspace=ws, out=out,
                       final_state=final)

    ref1 = [t.clone() for t in call(d)]
    ref2 = [t.clone() for t in call(d2)]
    torch.cuda.synchronize()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(d, o, fs)   # warm-up outside the capture
    torch.cuda.current_stream().wait_stream(side)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(d, o, fs)
    o.zero_()
    fs.zero_()
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, ref1[0]) and torch.equal(fs, ref1[1])
    for name in ("q", "k", "v", "g", "beta", "A_log", "dt_bias", "initial_state"):
        if d[name] is not None:
            d[name].copy_(d2[name])
    graph.replay()
    torch.cuda.synchronize()
    assert torch.equal(o, ref2[0]) and torch.equal(fs, ref2[1])
    assert kda.device_status() == 0


def test_prep_stage_matrices():
    """K1 alone: M = [-T diag(b) ; P T diag(b)] against the chunkwise fp64 oracle."""
    import chunked_gated_delta_02_gb300 as kda
    from oracle import chunk_quantities
    for T, K in ((128, 128), (100, 64), (64, 128)):
        inp = make_inputs(custom(B=1, T=T, H=2, K=K, V=K), seed=T + K)
        d = to_dev(inp)
        mats = kda.debug_chunk_matrices(d["q"], d["k"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                                        inp["lower_bound"]).float().cpu().double().numpy()
        for c0 in range(0, T, 64):
            c1 = min(c0 + 64, T)
            L = c1 - c0
            for h in range(2):
                cq = chunk_quantities(inp["q"][0, c0:c1, h], inp["k"][0, c0:c1, h], inp["v"][0, c0:c1, h],
                                      inp["g"][0, c0:c1, h], inp["beta"][0, c0:c1, h], inp["A_log"][h],
                                      inp["dt_bias"][h], inp["lower_bound"])
                Tb = cq["T"] * cq["b"][None, :]
                exp = np.zeros((128, 64))
                exp[:L, :L] = -Tb
                exp[64:64 + L, :L] = cq["P"] @ Tb
                got = mats[c0 // 64, h]
                err = np.max(np.abs(got - exp))
                assert err <= 2e-3 * max(1.0, np.max(np.abs(exp))), f"T={T} K={K} chunk {c0} head {h}: {err}"
                # T (I + A) = I on the valid block: recover T from -Tb and beta
                Tm = -got[:L, :L] / np.where(cq["b"] > 0, cq["b"], 1.0)[None, :]
                assert np.max(np.abs(Tm @ (np.eye(L) + cq["A"]) - np.eye(L))) < 5e-3


def test_bad_cu_seqlens_sets_device_status():
    import chunked_gated_delta_02_gb300 as kda
    inp = make_inputs(custom(H=2, K=64, V=64, seqlens=[40, 30, 50]), seed=11)
    d = to_dev(inp)
    kda.device_status()                     # clear any earlier record
    for bad in ([0, 40, 30, 120], [1, 40, 70, 120], [0, 40, 70, 119]):
        cu = torch.tensor(bad, dtype=torch.int32, device="cuda")
        o = torch.full((1, 120, 2, 64), 7.0, dtype=torch.bfloat16, device="cuda")
        kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], -5.0, 0.125,
                d["initial_state"], True, cu, out=o)
        assert kda.device_status() == 1, bad
        assert bool((o == 7.0).all()), "o written despite a bad cu_seqlens"
    # a good call afterwards works and leaves the status clear
    o, fs = run_gpu(inp)
    assert kda.device_status() == 0


# --- full-size workloads, in the launch configuration the bench times: every (sequence, head)
#     pair of o and of the final state is compared with the oracle, element by element.
@pytest.mark.parametrize("name", ["fixed", "varlen", "long", "large_batch"])
def test_full_size_all_pairs(name):
    inp = make_inputs(named(name), seed=0)
    o, fs = run_gpu(inp)
    eo, mo, es = check_all_pairs(inp, o, fs, name)
    print(f"{name}: o rel {eo:.2e} maxabs {mo:.2e} state rel {es:.2e} (all pairs)")
    import chunked_gated_delta_02_gb300 as kda
    assert kda.device_status() == 0


def test_bounded_wait_timeout_is_reported_and_context_survives():
    """A wait that nothing releases gives up after its bound, records KDA_DEVICE_WAIT_TIMEOUT in
    the device status word (as a pipeline kernel's wait does), and leaves the context usable."""
    import chunked_gated_delta_02_gb300 as kda
    from chunked_gated_delta_02_gb300._lib import lib
    kda.device_status()                     # clear any earlier record
    assert lib().kda_debug_wait_timeout(2_000_000, None) == 0    # about a millisecond of SM clocks
    assert kda.device_status() == 2
    assert kda.device_status() == 0         # read-and-clear
    inp = make_inputs(named("tiny"), seed=0)
    ref_o, ref_f = oracle_full(inp)
    o, fs = run_gpu(inp)
    assert_parity(o, fs, ref_o, ref_f, "after a timeout")
    assert kda.device_status() == 0


GUARD = 4096   # guard bytes before and after each buffer


def _guarded(nbytes, fill):
    """A device buffer of nbytes with GUARD bytes of `fill` on both sides; returns (whole, view)."""
    whole = torch.full((GUARD + nbytes + GUARD,), fill, dtype=torch.uint8, device="cuda")
    return whole, whole[GUARD:GUARD + nbytes]


@pytest.mark.parametrize("w", [custom(B=2, T=300, H=3, K=128, V=128, init_state=True),
                               custom(H=2, K=64, V=64, seqlens=[0, 70, 1, 129], init_state=True)],
                         ids=["fixed", "varlen-K64"])
def test_writes_stay_inside_workspace_and_outputs(w):
    """Canary bytes around the workspace, o and final_state are unchanged by a call that uses
    exactly the workspace size the library asks for."""
    import chunked_gated_delta_02_gb300 as kda
    inp = make_inputs(w, seed=31)
    d = to_dev(inp)
    B, T, H, K, V, N = (inp[x] for x in ("B", "T", "H", "K", "V", "N"))
    need = kda.workspace_size(B, T, H, K, V, N)
    ws_whole, ws = _guarded(need, 0xA5)
    o_whole, o_bytes = _guarded(B * T * H * V * 2, 0x5A)
    f_whole, f_bytes = _guarded(N * H * V * K * 4, 0x3C)
    o = o_bytes.view(torch.bfloat16).view(B, T, H, V)
    fs = f_bytes.view(torch.float32).view(N, H, V, K)
    kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
            d["scale"], d["initial_state"], True, d["cu_seqlens"], workspace=ws, out=o, final_state=fs)
    torch.cuda.synchronize()
    for name, whole, fill in (("workspace", ws_whole, 0xA5), ("o", o_whole, 0x5A), ("final_state", f_whole, 0x3C)):
        assert bool((whole[:GUARD] == fill).all()), f"{name}: bytes before the buffer changed"
        assert bool((whole[-GUARD:] == fill).all()), f"{name}: bytes after the buffer changed"
    ref_o, ref_f = oracle_full(inp)
    assert_parity(o, fs, ref_o, ref_f, "guarded buffers")


def test_deterministic_at_full_size():
    """Repeated calls give the same bits at full size: the prep kernel's hand-off matrices over 16
    runs on the varlen workload (about 38k chunk-head units per run), and the whole forward four
    times on the fixed workload with one reused workspace."""
    import chunked_gated_delta_02_gb300 as kda
    inp = make_inputs(named("varlen"), seed=0)
    d = to_dev(inp)
    ref = None
    for _ in range(16):
        mats = kda.debug_chunk_matrices(d["q"], d["k"], d["g"], d["beta"], d["A_log"], d["dt_bias"],
                                        inp["lower_bound"], d["cu_seqlens"])
        torch.cuda.synchronize()
        if ref is None:
            ref = mats.clone()
        else:
            assert torch.equal(mats, ref), "prep kernel output changed between runs"
    inp = make_inputs(named("fixed"), seed=0)
    d = to_dev(inp)
    B, T, H, K, V, N = (inp[x] for x in ("B", "T", "H", "K", "V", "N"))
    ws = torch.empty(kda.workspace_size(B, T, H, K, V, N), dtype=torch.uint8, device="cuda")
    outs = []
    for _ in range(4):
        o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                        d["scale"], d["initial_state"], True, None, workspace=ws)
        torch.cuda.synchronize()
        outs.append((o, fs))
    for o, fs in outs[1:]:
        assert torch.equal(o, outs[0][0]) and torch.equal(fs, outs[0][1])


def test_varlen_past_the_schedule_bins():
    """A packed batch of more than 8192 chunks (T > 524k tokens) is past the schedule's counting-
    sort bins: the sequences then run in input order instead of longest first. The results are the
    same; every output is compared with the oracle."""
    w = custom(H=1, K=64, V=64, seqlens=[300000, 100, 200000, 30000], init_state=True, lower_bound=-0.2)
    check_full(make_inputs(w, seed=71), "varlen beyond the bins")


# Fixed-length batches with more 64-column (sequence, head, V slice) CTAs than SMs, so that the
# recurrence runs in several waves: short sequences, a ragged last chunk, with and without initial
# states, both head dimensions.
WAVE_SHAPES = [
    (10, 200, 16, 128, 128, -0.5, True), (20, 50, 16, 128, 128, -5.0, True),
    (20, 100, 16, 64, 64, -1.0, False), (12, 129, 16, 128, 64, -0.2, True),
]


@pytest.mark.parametrize("B,T,H,K,V,lb,init", WAVE_SHAPES)
def test_multi_wave_shapes(B, T, H, K, V, lb, init):
    import chunked_gated_delta_02_gb300 as kda
    assert B * H * (V // 64) > 152            # more jobs than the SMs of a GB300
    w = custom(B=B, T=T, H=H, K=K, V=V, lower_bound=lb, init_state=init)
    check_full(make_inputs(w, seed=B * 7 + T), f"multi-wave B{B}-T{T}-H{H}-K{K}-V{V}")
    assert kda.device_status() == 0
