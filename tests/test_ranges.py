"""Value ranges that the fp16 hand-off of the prep kernel relies on (CPU, plain numpy).

The prep kernel stores Tb = (I + A)^{-1} diag(beta) and P Tb as fp16 (largest finite
value 65504). With unit keys, beta = sigmoid(.) in (0, 1) and per-channel decays <= 1
between an earlier and a later token of a chunk (KDA chunk form: FlashKDA page,
"Chunkwise" section; A_ij = beta_i sum_k khat_ik khat_jk e^{G_ik - G_jk}, j < i):

  * |P_ij| <= scale by Cauchy-Schwarz, since every decay factor is at most 1;
  * |Tb_ij| <= 1 in every case below: random keys, keys of rank 1, 2 and 8 with beta
    near 1, keys along a circle, with and without decay. This is measured here,
    not proved; the cases are chosen to make the inverse as large as possible
    (nearly dependent keys, beta close to 1, no decay).

So |P Tb| <= 64 scale and fp16 holds both with a wide margin.
"""
from __future__ import annotations

import numpy as np
import pytest

C, K = 64, 128


def _unit(x):
    return x / np.linalg.norm(x, axis=1, keepdims=True)


def _tb(khat, G, beta):
    """Tb = (I + A)^{-1} diag(beta), A strictly lower, from the definition."""
    A = np.einsum("ik,jk->ij", khat * np.exp(G), khat * np.exp(-G))
    A = np.tril(A, -1) * beta[:, None]
    return np.linalg.solve(np.eye(len(beta)) + A, np.diag(beta))


def _decay(rng, lb, shape):
    # log alpha = lb * sigmoid(a), a drawn wide so that both ends of [lb, 0] occur
    return np.cumsum(lb / (1.0 + np.exp(-3.0 * rng.standard_normal(shape))), axis=0)


def _keys(rng, kind):
    if kind == "random":
        return _unit(rng.standard_normal((C, K)))
    if kind == "rank1+noise":
        return _unit(np.outer(rng.choice([-1.0, 1.0], C), rng.standard_normal(K))
                     + 1e-3 * rng.standard_normal((C, K)))
    if kind.startswith("rank"):
        r = int(kind[4:])
        return _unit(rng.standard_normal((C, r)) @ rng.standard_normal((r, K)))
    raise ValueError(kind)


KINDS = ["random", "rank1", "rank2", "rank8", "rank1+noise"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("lb", [0.0, -1.0, -5.0])
def test_tb_entries_within_one(kind, lb):
    rng = np.random.default_rng([KINDS.index(kind), int(-lb)])
    worst = 0.0
    for _ in range(40):
        khat = _keys(rng, kind)
        G = _decay(rng, lb, (C, K)) if lb < 0 else np.zeros((C, K))
        for beta in (1.0 / (1.0 + np.exp(-rng.standard_normal(C))), np.full(C, 0.9999)):
            worst = max(worst, float(np.abs(_tb(khat, G, beta)).max()))
    assert worst <= 1.0 + 1e-9, worst


@pytest.mark.parametrize("step", [0.1, 0.5, 1.0, 2.0, 3.0])
def test_tb_entries_within_one_circle(step):
    # keys turning by a fixed angle in a plane: every pair correlated, no decay, beta near 1
    th = np.arange(C) * step
    khat = np.zeros((C, K))
    khat[:, 0], khat[:, 1] = np.cos(th), np.sin(th)
    tb = _tb(khat, np.zeros((C, K)), np.full(C, 0.9999))
    assert np.abs(tb).max() <= 1.0 + 1e-9


def test_p_entries_within_scale():
    rng = np.random.default_rng(5)
    scale = K ** -0.5
    qhat, khat = _unit(rng.standard_normal((C, K))), _unit(rng.standard_normal((C, K)))
    khat[1::2] = qhat[1::2]                    # some q_i = k_i: the largest possible terms
    G = _decay(rng, -5.0, (C, K))
    P = scale * np.tril(np.einsum("ik,jk->ij", qhat * np.exp(G), khat * np.exp(-G)))
    assert np.abs(P).max() <= scale * (1 + 1e-12)
