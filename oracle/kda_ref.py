"""fp64 token-by-token KDA forward: the plain definition (numpy).

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this module;
only tests/, the smoke check and the bench's CPU-baseline leg do.

What it computes (Kimi Delta Attention, arXiv:2510.26692, the paper the cuLA
overview page cites in section "cuLA 소개"), per sequence s and head h, one
token at a time, in float64 on the exact fp64 widening of the inputs:

    a_k      = exp(A_log[h]) * (g[t,h,k] + dt_bias[h,k])
    log a_k  = lower_bound * sigmoid(a_k)                  (natural log, in [lb, 0])
    q_hat    = q / sqrt(sum q^2 + eps),   k_hat = k / sqrt(sum k^2 + eps)
    beta_t   = sigmoid(beta_logit[t,h])
    S_t      = (I - beta_t k_hat k_hat^T) Diag(alpha_t) S_{t-1} + beta_t k_hat v_t^T
    o_t      = scale * S_t^T q_hat                         (post-update state)

S is K x V. The state tensors are stored [N,H,V,K], i.e. state[s,h,v,k] = S[k,v]
(FlashKDA page, section "FlashKDA의 KDA 연산 구조", initial_state/final_state
rows of the parameter table: shape [B,H,V,K]). The parameter meanings (g is the
pre-activation gate, beta holds logits with the sigmoid applied inside, A_log
[H], dt_bias [H,K], lower_bound in [-5, 0]) come from the same table; q/k L2
normalisation and the beta sigmoid happen inside the operation (same page,
same section: use_qk_l2norm_in_kernel, use_beta_sigmoid_in_kernel). Packed
variable-length input uses int32 cu_seqlens (cuLA README mirror, Quick Start
notes).

Readings where the pages are silent (each is also listed in the design notes):
  * eps of the L2 norm is 1e-6 inside the square root; x = 0 gives x_hat = 0.
  * the decay is applied before the delta-rule write and o_t reads S_t.
  * alpha uses the natural exponential: alpha = exp(lower_bound * sigmoid(a)).
  * with cu_seqlens, B must be 1 and each sequence starts from its own
    initial_state row; a zero-length sequence leaves its state unchanged.
  * sigmoid(+inf) = 1 and sigmoid(-inf) = 0 exactly.
  * the gated delta rule (GDN, named on the cuLA overview and FlashQLA pages
    without its formulas) is read as KDA with one decay per token and head: g
    is [B,T,H] and dt_bias [H], and every channel of the head takes the same
    log alpha = lower_bound * sigmoid(exp(A_log[h]) * (g[t,h] + dt_bias[h])).
    Diag(alpha) is then alpha I.
"""
from __future__ import annotations

import numpy as np

__all__ = ["sigmoid", "gate_log_decay", "l2_normalize", "kda_fwd_ref", "to_f64"]


def to_f64(x) -> np.ndarray:
    """Exact widening of a torch/numpy array (bf16, fp32, ...) to float64."""
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu", torch.float64).numpy()
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def sigmoid(x):
    """Logistic function 1/(1+exp(-x)), evaluated without overflow.

    sigmoid(+inf) = 1 and sigmoid(-inf) = 0 exactly.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.empty_like(x)
    pos = x >= 0
    with np.errstate(over="ignore"):
        out[pos] = 1.0 / (1.0 + np.exp(-x[pos]))
        e = np.exp(x[~pos])
        out[~pos] = e / (1.0 + e)
    return out


def gate_log_decay(g_t, A_log_h, dt_bias_h, lower_bound):
    """Per-channel log decay  lower_bound * sigmoid(exp(A_log) * (g + dt_bias)).

    The in-kernel gate activation with a lower bound (FlashKDA page, parameter
    table rows g / A_log / dt_bias / lower_bound; cuLA quick start arguments
    use_gate_in_kernel, safe_gate, lower_bound). Returns values in
    [lower_bound, 0].
    """
    a = np.exp(A_log_h) * (np.asarray(g_t, np.float64) + dt_bias_h)
    return lower_bound * sigmoid(a)


def l2_normalize(x, eps=1e-6):
    """x / sqrt(sum(x^2) + eps) along the last axis (in-kernel q/k L2 norm)."""
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + eps)


def _sequences(B, T, cu_seqlens):
    """(batch row, start, end) for every sequence."""
    if cu_seqlens is None:
        return [(b, 0, T) for b in range(B)]
    cu = [int(c) for c in np.asarray(cu_seqlens).reshape(-1)]
    return [(0, cu[i], cu[i + 1]) for i in range(len(cu) - 1)]


def kda_fwd_ref(q, k, v, g, beta, A_log, dt_bias, lower_bound, scale,
                initial_state=None, cu_seqlens=None, eps=1e-6, heads=None):
    """Sequential fp64 KDA forward.

    Arguments are arrays (torch or numpy) with the layouts of the module doc:
    q, k, g [B,T,H,K]; v [B,T,H,V]; beta [B,T,H]; A_log [H]; dt_bias [H,K] or
    None; initial_state [N,H,V,K] or None; cu_seqlens [N+1] or None. A gate g
    of shape [B,T,H] (with dt_bias [H] or None) is one decay per token and
    head, the same in every channel.

    Returns (o, final_state): o float64 [B,T,H,V] (rows of heads not in
    ``heads`` are left at zero), final_state float64 [N,H,V,K].
    """
    q, k, v, g, beta = (to_f64(x) for x in (q, k, v, g, beta))
    A_log = to_f64(A_log)
    B, T, H, K = q.shape
    V = v.shape[-1]
    if g.ndim == 3:   # one gate per token and head: the same value in every channel
        g = np.repeat(g[..., None], K, axis=-1)
        dt_bias = None if dt_bias is None else np.repeat(to_f64(dt_bias).reshape(H, 1), K, axis=1)
    dt_bias = np.zeros((H, K)) if dt_bias is None else to_f64(dt_bias).reshape(H, K)
    seqs = _sequences(B, T, cu_seqlens)
    if cu_seqlens is not None and B != 1:
        raise ValueError("cu_seqlens requires B == 1")
    N = len(seqs)
    S0 = np.zeros((N, H, V, K)) if initial_state is None else to_f64(initial_state)
    hs = list(range(H)) if heads is None else list(heads)
    o = np.zeros((B, T, H, V))
    final = np.zeros((N, H, V, K))
    final[:] = S0
    for n, (b, t0, t1) in enumerate(seqs):
        # state for the selected heads: [h, K, V]
        S = np.stack([S0[n, h].T.copy() for h in hs]) if hs else np.zeros((0, K, V))
        ex = np.exp(A_log[hs])[:, None]
        for t in range(t0, t1):
            a = ex * (g[b, t, hs] + dt_bias[hs])                 # [h, K]
            log_alpha = lower_bound * sigmoid(a)
            alpha = np.exp(log_alpha)
            qh = l2_normalize(q[b, t, hs], eps)                  # [h, K]
            kh = l2_normalize(k[b, t, hs], eps)
            bt = sigmoid(beta[b, t, hs])                         # [h]
            S = alpha[:, :, None] * S                            # decay first
            pred = np.einsum("hkv,hk->hv", S, kh)                # S^T k_hat
            S = S + bt[:, None, None] * kh[:, :, None] * (v[b, t, hs] - pred)[:, None, :]
            o[b, t, hs] = scale * np.einsum("hkv,hk->hv", S, qh)
        for i, h in enumerate(hs):
            final[n, h] = S[i].T
    return o, final
