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


def gather_pairs(inp, o_gpu, fs_gpu, pairs):
    """GPU outputs of the chosen (sequence, head) pairs, in the oracle's compact order."""
    cu = inp["cu_seqlens"]
    o = o_gpu.float().cpu()
    outs = []
    for s, h in pairs:
        if cu is None:
            outs.append(o[s, :, h].double().numpy())
        else:
            outs.append(o[0, int(cu[s]):int(cu[s + 1]), h].double().numpy())
    fin = fs_gpu.cpu()[[s for s, _ in pairs], [h for _, h in pairs]].double().numpy()
    return np.concatenate(outs, 0), fin


def check_pairs(inp, o_gpu, fs_gpu, pairs, what=""):
    from oracle import c_oracle
    ref_o, ref_f = c_oracle.kda_fwd_c(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"],
                                      inp["dt_bias"], inp["lower_bound"], inp["scale"],
                                      inp["initial_state"], inp["cu_seqlens"], pairs=pairs)
    go, gf = gather_pairs(inp, o_gpu, fs_gpu, pairs)
    return assert_parity(go, gf, np.concatenate(ref_o, 0), ref_f, what)
