"""The parity helpers themselves (CPU): the all-pairs comparison of the large workloads sees an
error confined to one (sequence, head), one V slice or one token."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from chunked_gated_delta_02_gb300.workloads import custom, make_inputs
from kda_testlib import check_all_pairs, oracle_full


@pytest.mark.parametrize("w", [custom(B=2, T=70, H=3, K=64, V=64, init_state=True),
                               custom(H=2, K=64, V=64, seqlens=[0, 65, 1, 130], init_state=True)],
                         ids=["fixed", "varlen"])
def test_all_pairs_check_sees_a_local_error(w):
    inp = make_inputs(w, seed=5)
    ref_o, ref_f = oracle_full(inp)
    o = torch.from_numpy(ref_o).to(torch.bfloat16)
    fs = torch.from_numpy(ref_f).float()
    # small batches, so that the sums over batches are exercised
    check_all_pairs(inp, o, fs, "exact", max_token_heads=64)
    N, H = inp["N"], inp["H"]
    cu = inp["cu_seqlens"]
    s, h = N - 1, H - 1
    t = (inp["T"] - 1) if cu is None else int(cu[s + 1]) - 1
    bad = o.clone()
    bad[(s if cu is None else 0), t, h, 40] += 0.5          # one element of the last pair
    with pytest.raises(AssertionError, match="max-abs"):
        check_all_pairs(inp, bad, fs, "one element", max_token_heads=64)
    bad_f = fs.clone()
    bad_f[s, h, :, :] *= 1.05                               # the last pair's state, 5 % off
    with pytest.raises(AssertionError, match="final_state"):
        check_all_pairs(inp, o, bad_f, "one state", max_token_heads=64)
    nan_f = fs.clone()
    nan_f[0, 0, 3, 3] = float("nan")
    with pytest.raises(AssertionError, match="non-finite final_state"):
        check_all_pairs(inp, o, nan_f, "nan state", max_token_heads=64)
