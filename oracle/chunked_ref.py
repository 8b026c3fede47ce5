"""fp64 brute-force chunkwise KDA forward (WY form), written independently.

TEST INFRASTRUCTURE ONLY. It pins the token-by-token oracle (the two must agree
to rounding for every chunk size) and defines the per-chunk quantities that the
GPU prep stage hands to the recurrence stage, so that stage can be checked on
its own. It shares no code with kda_ref.py: the gate, sigmoid and norm are
written out again here on purpose.

Chunkwise decomposition of the KDA recurrence (the "chunk intra / recompute wu /
chunk gated delta h / chunk fwd o" stages of the modular KDA forward, cuLA
launch blog, section "Status & Roadmap"; chunk size 64 vs 16 and the
triangular inverse, FlashKDA page, section "Flash Linear Attention과 비교").
Inside one chunk with c tokens and chunk-start state S (K x V):

  G_i      = sum_{j<=i} log alpha_j                      (per channel, inclusive)
  A_ij     = beta_i sum_k k_ik k_jk exp(G_ik - G_jk)     for j < i, else 0
  T        = (I + A)^{-1}                                (unit lower triangular)
  W        = T diag(beta) (K_hat * exp(G))
  U0       = T diag(beta) V
  U        = U0 - W S                                    (the delta-rule residuals)
  P_ij     = sum_k q_ik k_jk exp(G_ik - G_jk)            for j <= i, else 0
  O        = scale ((Q_hat * exp(G)) S + P U)
  S_next   = Diag(exp(G_c)) S + (K_hat * exp(G_c - G))^T U

Every pairwise decay exp(G_i - G_j) is evaluated directly (never as a product
of exp(G_i) and exp(-G_j)), and T is found by forward substitution, so the
result is exact up to rounding for any chunk size.
"""
from __future__ import annotations

import numpy as np

__all__ = ["kda_fwd_chunked", "chunk_quantities", "forward_substitution_inverse"]


def _sig(x):
    x = np.asarray(x, np.float64)
    with np.errstate(over="ignore"):
        return np.where(x >= 0, 1.0 / (1.0 + np.exp(-np.abs(x))),
                        np.exp(-np.abs(x)) / (1.0 + np.exp(-np.abs(x))))


def _f64(x):
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, np.float64)


def forward_substitution_inverse(A):
    """(I + A)^{-1} for strictly lower triangular A, row by row.

    Row i of X = (I + A)^{-1} satisfies X_i = e_i - sum_{j<i} A_ij X_j.
    """
    c = A.shape[0]
    X = np.zeros((c, c))
    for i in range(c):
        X[i, i] = 1.0
        for j in range(i):
            if A[i, j] != 0.0:
                X[i] -= A[i, j] * X[j]
    return X


def chunk_quantities(q, k, v, g, beta, A_log_h, dt_bias_h, lower_bound, eps=1e-6):
    """Per-chunk quantities for ONE (sequence, head) chunk.

    q, k, g: [c, K]; v: [c, V]; beta: [c] logits. Returns a dict with
    G [c,K], qh, kh [c,K], b [c], A [c,c], T [c,c], W [c,K], U0 [c,V], P [c,c],
    gamma [K] = exp(G_last), Kdec [c,K] = kh * exp(G_last - G).
    """
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    c, K = k.shape
    pre = np.exp(float(A_log_h)) * (g + np.asarray(dt_bias_h, np.float64)[None, :])
    la = float(lower_bound) * _sig(pre)                       # [c, K]
    G = np.cumsum(la, axis=0)
    qh = q / np.sqrt((q * q).sum(-1, keepdims=True) + eps)
    kh = k / np.sqrt((k * k).sum(-1, keepdims=True) + eps)
    b = _sig(beta)
    A = np.zeros((c, c))
    P = np.zeros((c, c))
    for i in range(c):
        for j in range(i + 1):
            d = np.exp(G[i] - G[j])                           # exact pairwise decay
            if j < i:
                A[i, j] = b[i] * np.sum(kh[i] * kh[j] * d)
            P[i, j] = np.sum(qh[i] * kh[j] * d)
    T = forward_substitution_inverse(A)
    W = T @ (b[:, None] * kh * np.exp(G))
    U0 = T @ (b[:, None] * v)
    Glast = G[-1] if c else np.zeros(K)
    return dict(G=G, qh=qh, kh=kh, b=b, A=A, T=T, W=W, U0=U0, P=P,
                gamma=np.exp(Glast), Kdec=kh * np.exp(Glast[None, :] - G))


def kda_fwd_chunked(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                    initial_state=None, cu_seqlens=None, chunk=64, eps=1e-6):
    """Chunkwise fp64 KDA forward; same arguments and returns as the token oracle."""
    q, k, v, g, beta = (_f64(x) for x in (q, k, v, g, beta))
    A_log = _f64(A_log)
    B, T, H, K = q.shape
    V = v.shape[-1]
    dt = np.zeros((H, K)) if dt_bias is None else _f64(dt_bias).reshape(H, K)
    if cu_seqlens is None:
        seqs = [(b, 0, T) for b in range(B)]
    else:
        cu = [int(x) for x in np.asarray(cu_seqlens).reshape(-1)]
        seqs = [(0, cu[i], cu[i + 1]) for i in range(len(cu) - 1)]
    N = len(seqs)
    S0 = np.zeros((N, H, V, K)) if initial_state is None else _f64(initial_state)
    o = np.zeros((B, T, H, V))
    final = np.zeros((N, H, V, K))
    for n, (bb, t0, t1) in enumerate(seqs):
        for h in range(H):
            S = S0[n, h].T.copy()                             # K x V
            for c0 in range(t0, t1, chunk):
                c1 = min(c0 + chunk, t1)
                cq = chunk_quantities(q[bb, c0:c1, h], k[bb, c0:c1, h], v[bb, c0:c1, h],
                                      g[bb, c0:c1, h], beta[bb, c0:c1, h], A_log[h], dt[h],
                                      lower_bound, eps)
                U = cq["U0"] - cq["W"] @ S
                O = (cq["qh"] * np.exp(cq["G"])) @ S + cq["P"] @ U
                o[bb, c0:c1, h] = scale * O
                S = cq["gamma"][:, None] * S + cq["Kdec"].T @ U
            final[n, h] = S.T
    return o, final
