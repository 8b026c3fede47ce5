"""Helpers shared by the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle, element by element.

Tolerances (floating point, bf16 inputs): o rel-L2 <= 5e-3 and max-abs <= 3e-2,
final_state rel-L2 <= 2e-3; rel-L2 = ||x - y||_2 / ||y||_2 over the compared
elements, y the fp64 oracle.
"""
from __future__ import annotations

import numpy as np
import torch

TOL_O_REL = 5e-3
TOL_O_MAXABS = 3e-2
TOL_S_REL = 2e-3


def to_dev(inp: dict, dev="cuda:0") -> dict:
    return {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in inp.items()}


def run_gpu(inp: dict, output_final_state=True, dev="cuda:0", init="given"):
    import chunked_gated_delta_02_gb300 as kda
    d = to_dev(inp, dev)
    ini = d["initial_state"] if init == "given" else init
    o, fs = kda.fwd(d["q"], d["k"], d["v"], d["g"], d["beta"], d["A_log"], d["dt_bias"], d["lower_bound"],
                    d["scale"], ini, output_final_state, d["cu_seqlens"])
    torch.cuda.synchronize()
    return o, fs


def rel_l2(x, y):
    x = np.asarray(x, np.float64)
    y = np.asarray(y, np.float64)
    den = np.linalg.norm(y)
    num = np.linalg.norm(x - y)
    return float(num / den) if den > 0 else float(num)


def oracle_full(inp: dict):
    from oracle import c_oracle
    return c_oracle.kda_fwd_c(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"],
                              inp["dt_bias"], inp["lower_bound"], inp["scale"], inp["initial_state"],
                              inp["cu_seqlens"])


def assert_parity(o_gpu, fs_gpu, ref_o, ref_f, what=""):
    go = o_gpu.float().cpu().double().numpy() if isinstance(o_gpu, torch.Tensor) else o_gpu
    eo = rel_l2(go, ref_o)
    mo = float(np.max(np.abs(go - ref_o))) if np.size(ref_o) else 0.0
    msg = f"{what}: o rel-L2 {eo:.3e} (<= {TOL_O_REL}), max-abs {mo:.3e} (<= {TOL_O_MAXABS})"
    assert np.all(np.isfinite(go)), f"{what}: non-finite o"
    assert eo <= TOL_O_REL and mo <= TOL_O_MAXABS, msg
    es = None
    if fs_gpu is not None:
        gf = fs_gpu.cpu().double().numpy() if isinstance(fs_gpu, torch.Tensor) else fs_gpu
        assert np.all(np.isfinite(gf)), f"{what}: non-finite final_state"
        es = rel_l2(gf, ref_f)
        assert es <= TOL_S_REL, f"{what}: final_state rel-L2 {es:.3e} (<= {TOL_S_REL})"
    return eo, mo, es


def check_full(inp: dict, what=""):
    o, fs = run_gpu(inp)
    ref_o, ref_f = oracle_full(inp)
    return assert_parity(o, fs, ref_o, ref_f, what)


def check_all_pairs(inp, o_gpu, fs_gpu, what="", max_token_heads=1 << 20):
    """Every (sequence, head) of a large workload against the C oracle, element by element.

    The oracle runs on batches of (sequence, head) pairs (at most max_token_heads token-heads, at
    least one pair per host thread) so that host memory stays bounded; the squared errors and
    norms are summed over the batches, so the rel-L2 figures are those of the whole tensors and
    max-abs is the largest error of any element of o."""
    from oracle import c_oracle
    cu = inp["cu_seqlens"]
    N, H = inp["N"], inp["H"]
    lens = [int(cu[i + 1] - cu[i]) for i in range(N)] if cu is not None else [inp["T"]] * N
    threads = c_oracle.default_threads()
    o = o_gpu.float().cpu()
    fs = fs_gpu.cpu().double().numpy()
    pairs = [(s, h) for s in range(N) for h in range(H)]
    num_o = den_o = num_s = den_s = 0.0
    max_abs = 0.0
    i = 0
    while i < len(pairs):
        batch, th = [], 0
        while i < len(pairs) and (len(batch) < threads or th + lens[pairs[i][0]] <= max_token_heads):
            batch.append(pairs[i])
            th += lens[pairs[i][0]]
            i += 1
        ref_o, ref_f = c_oracle.kda_fwd_c(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"],
                                          inp["dt_bias"], inp["lower_bound"], inp["scale"],
                                          inp["initial_state"], cu, pairs=batch, n_threads=threads)
        for j, (s, h) in enumerate(batch):
            g = (o[s, :, h] if cu is None else o[0, int(cu[s]):int(cu[s + 1]), h]).double().numpy()
            r = ref_o[j]
            assert np.all(np.isfinite(g)), f"{what}: non-finite o in (sequence {s}, head {h})"
            d = g - r
            num_o += float(np.sum(d * d))
            den_o += float(np.sum(r * r))
            if d.size:
                max_abs = max(max_abs, float(np.max(np.abs(d))))
            gf = fs[s, h]
            assert np.all(np.isfinite(gf)), f"{what}: non-finite final_state in (sequence {s}, head {h})"
            df = gf - ref_f[j]
            num_s += float(np.sum(df * df))
            den_s += float(np.sum(ref_f[j] * ref_f[j]))
    eo = (num_o / den_o) ** 0.5 if den_o > 0 else num_o ** 0.5
    es = (num_s / den_s) ** 0.5 if den_s > 0 else num_s ** 0.5
    assert eo <= TOL_O_REL and max_abs <= TOL_O_MAXABS, \
        f"{what}: o rel-L2 {eo:.3e} (<= {TOL_O_REL}), max-abs {max_abs:.3e} (<= {TOL_O_MAXABS})"
    assert es <= TOL_S_REL, f"{what}: final_state rel-L2 {es:.3e} (<= {TOL_S_REL})"
    return eo, max_abs, es
