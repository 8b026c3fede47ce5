"""Pins of the fp64 oracle against what the mathematics fixes (CPU only).

Each pin is a function of an implementation ``impl(inp, eps) -> (o, final)``;
the real oracles (numpy token recurrence, plain-C token recurrence) must pass
every pin, and each planted mistake in a CPU copy of the recurrence (see
``_mutant``) must fail at least one of them. The pins:

  * chunked:     an independently written chunkwise (WY) form with exact
                 pairwise decays agrees for chunk sizes 1, 2, 5, 16, 64;
  * frozen:      beta=0 and alpha=1 leave S at S0 and o_t = scale S0^T q_hat
                 (numpy matmul and numpy.linalg.norm);
  * orthonormal: alpha=1, beta=1, orthonormal keys and q_t = k_t give
                 o_t = scale v_t, and the final state recalls every v_j;
  * last write:  the same key written repeatedly keeps only the last value;
  * split:       running [0,T1) then [T1,T) from the carried state equals the
                 whole run; a packed varlen batch equals separate runs;
  * decay only:  beta=0 gives S_T = Diag(prod alpha) S0 with alpha fixed by
                 special gate values (a=0, a=+-inf, a=ln 3, A_log=-inf);
  * scalar:      K=V=1 reduces to a first-order IIR filter (scipy lfilter);
  * golden:      two hand-derived worked examples (tests/golden/).
"""
from __future__ import annotations

import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import kda_fwd_ref, kda_fwd_chunked, forward_substitution_inverse, chunk_quantities
from oracle import c_oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "kda_hand_examples.json")
RNG_SEED = 1234


# --------------------------------------------------------------------------- impls
def impl_numpy(inp, eps):
    return kda_fwd_ref(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"],
                       inp["dt_bias"], inp["lower_bound"], inp["scale"],
                       inp.get("initial_state"), inp.get("cu_seqlens"), eps=eps)


def _exact_bf16(x):
    t = torch.from_numpy(np.asarray(x, np.float64))
    b = t.to(torch.bfloat16)
    ok = (b.to(torch.float64) == t) | (torch.isnan(t) & torch.isnan(b.to(torch.float64)))
    assert bool(ok.all()), "pin input not exactly representable in bf16"
    return b


def _exact_f32(x):
    if x is None:
        return None
    t = torch.from_numpy(np.asarray(x, np.float64))
    f = t.to(torch.float32)
    assert bool((f.to(torch.float64) == t).all()), "pin input not exactly representable in fp32"
    return f


def impl_c(inp, eps):
    cu = inp.get("cu_seqlens")
    return c_oracle.kda_fwd_c(_exact_bf16(inp["q"]), _exact_bf16(inp["k"]), _exact_bf16(inp["v"]),
                              _exact_bf16(inp["g"]), _exact_bf16(inp["beta"]),
                              _exact_f32(inp["A_log"]), _exact_f32(inp["dt_bias"]),
                              inp["lower_bound"], inp["scale"], inp.get("initial_state"),
                              None if cu is None else np.asarray(cu, np.int32), eps=eps, n_threads=2)


IMPLS = {"numpy": impl_numpy, "c": impl_c}


# --------------------------------------------------------------------------- inputs
def _bf(x):
    """Round to bf16 and back (so that both oracles see the same exact values)."""
    return torch.from_numpy(np.asarray(x, np.float64)).to(torch.bfloat16).to(torch.float64).numpy()


def _f32(x):
    return np.asarray(x, np.float32).astype(np.float64)


def rand_inputs(rng, B=1, T=20, H=2, K=6, V=5, lb=-3.0, init=True, seqlens=None, g_scale=0.5):
    if seqlens is not None:
        B, T = 1, int(sum(seqlens))
        cu = np.concatenate([[0], np.cumsum(seqlens)]).astype(np.int32)
        N = len(seqlens)
    else:
        cu = None
        N = B
    return dict(
        q=_bf(rng.standard_normal((B, T, H, K))), k=_bf(rng.standard_normal((B, T, H, K))),
        v=_bf(rng.standard_normal((B, T, H, V))),
        g=_bf(g_scale * rng.standard_normal((B, T, H, K))),
        beta=_bf(rng.standard_normal((B, T, H))), A_log=_f32(0.3 * rng.standard_normal(H)),
        dt_bias=_f32(0.2 * rng.standard_normal((H, K))), lower_bound=lb, scale=K ** -0.5,
        initial_state=_f32(0.5 * rng.standard_normal((N, H, V, K))) if init else None,
        cu_seqlens=cu)


def _close(a, b, rtol=1e-12, atol=1e-12, what=""):
    a = np.asarray(a, np.float64)
    b = np.asarray(b, np.float64)
    assert a.shape == b.shape, f"{what}: shape {a.shape} != {b.shape}"
    err = np.max(np.abs(a - b)) if a.size else 0.0
    lim = atol + rtol * (np.max(np.abs(b)) if b.size else 0.0)
    assert err <= lim, f"{what}: max abs err {err:.3e} > {lim:.3e}"


# --------------------------------------------------------------------------- pins
def pin_chunked(impl):
    rng = np.random.default_rng(RNG_SEED)
    for lb in (-5.0, -1.0, -0.05):
        inp = rand_inputs(rng, B=2, T=37, H=2, K=6, V=5, lb=lb)
        o, f = impl(inp, 1e-6)
        for C in (1, 2, 5, 16, 64):
            oc, fc = kda_fwd_chunked(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"],
                                     inp["A_log"], inp["dt_bias"], lb, inp["scale"],
                                     inp["initial_state"], None, chunk=C)
            _close(o, oc, 1e-10, 1e-12, f"o vs chunked C={C} lb={lb}")
            _close(f, fc, 1e-10, 1e-12, f"final vs chunked C={C} lb={lb}")
    inp = rand_inputs(rng, H=2, K=6, V=5, lb=-2.0, seqlens=[0, 1, 17, 40, 3])
    o, f = impl(inp, 1e-6)
    oc, fc = kda_fwd_chunked(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp["A_log"],
                             inp["dt_bias"], -2.0, inp["scale"], inp["initial_state"],
                             inp["cu_seqlens"], chunk=16)
    _close(o, oc, 1e-10, 1e-12, "varlen o vs chunked")
    _close(f, fc, 1e-10, 1e-12, "varlen final vs chunked")


def pin_frozen(impl):
    rng = np.random.default_rng(RNG_SEED + 1)
    inp = rand_inputs(rng, B=2, T=9, H=3, K=5, V=4)
    inp["lower_bound"] = 0.0
    inp["beta"] = np.full_like(inp["beta"], -np.inf)
    o, f = impl(inp, 1e-6)
    _close(f, inp["initial_state"], 0, 0, "frozen final state")
    q = inp["q"]
    qh = q / np.sqrt(np.linalg.norm(q, axis=-1, keepdims=True) ** 2 + 1e-6)
    for b in range(2):
        for h in range(3):
            exp = inp["scale"] * np.matmul(qh[b, :, h], inp["initial_state"][b, h].T)
            _close(o[b, :, h], exp, 1e-12, 1e-14, "frozen output")


def _orthonormal_keys(rng, K, exact):
    if exact:   # signed permutation of the standard basis: exact in bf16
        perm = rng.permutation(K)
        sign = rng.choice([-1.0, 1.0], K)
        M = np.zeros((K, K))
        M[np.arange(K), perm] = sign
        return M * rng.choice([1.0, 2.0, 0.5], K)[:, None]    # row scales cancel in the norm
    Q, _ = np.linalg.qr(rng.standard_normal((K, K)))
    return Q * rng.uniform(0.5, 2.0, K)[:, None]


def pin_orthonormal(impl, exact=True):
    rng = np.random.default_rng(RNG_SEED + 2)
    K, V = 6, 4
    keys = _orthonormal_keys(rng, K, exact)
    inp = rand_inputs(rng, T=K, H=1, K=K, V=V, lb=0.0)
    inp["k"][0, :, 0] = keys
    inp["q"][0, :, 0] = keys
    inp["beta"] = np.full_like(inp["beta"], np.inf)
    o, f = impl(inp, 0.0)
    _close(o[0, :, 0], inp["scale"] * inp["v"][0, :, 0], 1e-12, 1e-13, "o_t = scale v_t")
    kh = keys / np.linalg.norm(keys, axis=1, keepdims=True)
    S = f[0, 0].T                                          # K x V
    _close(np.matmul(kh, S), inp["v"][0, :, 0], 1e-12, 1e-13, "recall of every v_j")


def pin_last_write(impl):
    rng = np.random.default_rng(RNG_SEED + 3)
    K, V, T = 5, 3, 7
    inp = rand_inputs(rng, T=T, H=1, K=K, V=V, lb=0.0)
    key = np.zeros(K)
    key[2] = -4.0
    inp["k"][0, :, 0] = key
    inp["beta"] = np.full_like(inp["beta"], np.inf)
    o, f = impl(inp, 0.0)
    S = f[0, 0].T
    S0 = inp["initial_state"][0, 0].T
    _close(S[2], inp["v"][0, -1, 0] * -1.0, 1e-13, 1e-14, "last write (k_hat = -e2)")
    others = [i for i in range(K) if i != 2]
    _close(S[others], S0[others], 0, 0, "untouched rows")


def pin_split(impl):
    rng = np.random.default_rng(RNG_SEED + 4)
    inp = rand_inputs(rng, B=1, T=40, H=2, K=6, V=5, lb=-1.5)
    o, f = impl(inp, 1e-6)
    for T1 in (1, 16, 23, 39):
        a = {kk: (vv[:, :T1] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in inp.items()}
        oa, fa = impl(a, 1e-6)
        b = {kk: (vv[:, T1:] if kk in ("q", "k", "v", "g", "beta") else vv) for kk, vv in inp.items()}
        b["initial_state"] = fa
        ob, fb = impl(b, 1e-6)
        _close(fb, f, 1e-12, 1e-13, f"split final T1={T1}")
        _close(np.concatenate([oa, ob], 1), o, 1e-12, 1e-13, f"split o T1={T1}")
    lens = [5, 0, 12, 1, 9]
    pk = rand_inputs(rng, H=2, K=6, V=5, lb=-0.7, seqlens=lens)
    o, f = impl(pk, 1e-6)
    cu = pk["cu_seqlens"]
    for s, L in enumerate(lens):
        one = {kk: (vv[:, cu[s]:cu[s + 1]] if kk in ("q", "k", "v", "g", "beta") else vv)
               for kk, vv in pk.items()}
        one["cu_seqlens"] = None
        one["initial_state"] = pk["initial_state"][s:s + 1]
        os_, fs = impl(one, 1e-6)
        _close(fs, f[s:s + 1], 1e-12, 1e-13, f"varlen final seq {s}")
        _close(os_, o[:, cu[s]:cu[s + 1]], 1e-12, 1e-13, f"varlen o seq {s}")


def pin_decay_only(impl):
    """beta=0: S_T = Diag(prod_t alpha_t) S0 for gate values with known sigmoid."""
    rng = np.random.default_rng(RNG_SEED + 5)
    K, V, T, lb = 6, 3, 5, -1.25
    inp = rand_inputs(rng, T=T, H=2, K=K, V=V, lb=lb)
    inp["beta"] = np.full_like(inp["beta"], -np.inf)
    ln3 = float(np.float32(math.log(3.0)))
    ln2 = float(np.float32(math.log(2.0)))
    inp["A_log"] = np.array([0.0, ln2])
    g = np.zeros_like(inp["g"])
    # head 0: g = 0 with dt_bias = (0, +inf, -inf, ln3, 0, 0)
    inp["dt_bias"] = np.array([[0.0, np.inf, -np.inf, ln3, 0.0, 0.0],
                               [0.0, 0.0, 0.0, 0.0, 0.0, 0.0]])
    # head 1: exp(A_log) = 2, g = ln3 / 2 rounded to bf16 on channel 0, 0 elsewhere
    g[0, :, 1, 0] = _bf(np.full(T, math.log(3.0) / 2))
    inp["g"] = g
    o, f = impl(inp, 1e-6)
    sig = lambda x: 1.0 / (1.0 + math.exp(-x))  # noqa: E731  (scalar special values below)
    a0 = [lb / 2, lb, 0.0, lb * sig(ln3), lb / 2, lb / 2]
    a1 = [lb * sig(math.exp(ln2) * float(g[0, 0, 1, 0]))] + [lb / 2] * (K - 1)
    for h, la in enumerate((a0, a1)):
        decay = np.exp(T * np.array(la))                # alpha^T per channel
        _close(f[0, h], inp["initial_state"][0, h] * decay[None, :], 1e-12, 1e-14,
               f"decay-only head {h}")
    # head 0 channel 3 is 3/4 of lb per step up to the fp32 rounding of ln 3
    assert abs(a0[3] - 0.75 * lb) < 1e-6


def pin_a_log_neg_inf(impl):
    """A_log = -inf -> exp(A_log) = 0 -> a = 0 -> alpha = exp(lb/2) whatever g is."""
    rng = np.random.default_rng(RNG_SEED + 6)
    inp = rand_inputs(rng, T=4, H=1, K=4, V=2, lb=-2.0)
    inp["beta"] = np.full_like(inp["beta"], -np.inf)
    inp["A_log"] = np.array([-np.inf])
    inp["dt_bias"] = np.zeros((1, 4))
    o, f = impl(inp, 1e-6)
    _close(f, inp["initial_state"] * math.exp(4 * -1.0), 1e-12, 1e-14, "A_log=-inf")


def pin_single_step(impl):
    rng = np.random.default_rng(RNG_SEED + 7)
    inp = rand_inputs(rng, T=1, H=1, K=7, V=3, lb=0.0)
    inp["beta"] = np.full_like(inp["beta"], np.inf)
    o, f = impl(inp, 0.0)
    k = inp["k"][0, 0, 0]
    kh = k / np.linalg.norm(k)
    _close(np.matmul(kh, f[0, 0].T), inp["v"][0, 0, 0], 1e-12, 1e-13, "single step recall")


def pin_scalar_iir(impl):
    """K=V=1, k>0, constant alpha and beta: S_t = (1-beta) alpha S_{t-1} + beta v_t."""
    from scipy.signal import lfilter
    rng = np.random.default_rng(RNG_SEED + 8)
    T = 30
    inp = rand_inputs(rng, T=T, H=1, K=1, V=1, lb=-0.5)
    inp["k"] = _bf(np.abs(inp["k"]) + 1.0)
    inp["q"] = _bf(np.abs(inp["q"]) + 1.0)
    inp["g"] = np.zeros_like(inp["g"])
    inp["dt_bias"] = np.zeros((1, 1))
    inp["A_log"] = np.zeros(1)
    inp["beta"] = np.zeros_like(inp["beta"])          # beta = 1/2
    o, f = impl(inp, 0.0)
    alpha, beta = math.exp(-0.25), 0.5
    s0 = inp["initial_state"][0, 0, 0, 0]
    pole = (1 - beta) * alpha
    y, _ = lfilter([beta], [1.0, -pole], inp["v"][0, :, 0, 0], zi=[pole * s0])
    _close(o[0, :, 0, 0], inp["scale"] * y, 1e-12, 1e-14, "scalar IIR output")
    _close(f[0, 0, 0, 0], y[-1], 1e-12, 1e-14, "scalar IIR state")


def pin_golden(impl):
    with open(GOLDEN) as fh:
        ex = json.load(fh)["examples"]
    for e in ex:
        T = len(e["q"])
        fl = lambda a: np.array([[float(x) for x in r] for r in a])  # noqa: E731
        inp = dict(q=fl(e["q"]).reshape(1, T, 1, 2), k=fl(e["k"]).reshape(1, T, 1, 2),
                   v=fl(e["v"]).reshape(1, T, 1, 2), g=fl(e["g"]).reshape(1, T, 1, 2),
                   beta=np.array(e["beta_logit"], float).reshape(1, T, 1),
                   A_log=np.array(e["A_log"], float), dt_bias=fl(e["dt_bias"]),
                   lower_bound=e["lower_bound"], scale=e["scale"],
                   initial_state=None if e["initial_state_VK"] is None
                   else fl(e["initial_state_VK"]).reshape(1, 1, 2, 2), cu_seqlens=None)
        o, f = impl(inp, e["eps"])
        _close(o[0, :, 0], fl(e["o"]), 1e-12, 1e-14, f"golden {e['name']} o")
        _close(f[0, 0], fl(e["final_state_VK"]), 1e-12, 1e-14, f"golden {e['name']} final")


PINS = [pin_chunked, pin_frozen, pin_orthonormal, pin_last_write, pin_split, pin_decay_only,
        pin_a_log_neg_inf, pin_single_step, pin_scalar_iir, pin_golden]


@pytest.mark.parametrize("name", sorted(IMPLS))
@pytest.mark.parametrize("pin", PINS, ids=lambda p: p.__name__)
def test_oracle_pin(name, pin):
    pin(IMPLS[name])


def test_orthonormal_random_rotation_numpy():
    pin_orthonormal(impl_numpy, exact=False)


# --------------------------------------------------------------------------- chunk stage pins
def test_forward_substitution_inverse():
    from scipy.linalg import solve_triangular
    rng = np.random.default_rng(5)
    for c in (1, 2, 16, 64):
        A = np.tril(rng.standard_normal((c, c)) * 0.3, -1)
        T = forward_substitution_inverse(A)
        _close(T @ (np.eye(c) + A), np.eye(c), 1e-11, 1e-11, f"T(I+A)=I c={c}")
        _close(T, solve_triangular(np.eye(c) + A, np.eye(c), lower=True), 1e-11, 1e-11,
               f"solve_triangular c={c}")


def test_chunk_quantities_structure():
    """A is strictly lower, P lower with P_ii = q_hat_i . k_hat_i, T unit lower."""
    rng = np.random.default_rng(6)
    c, K, V = 20, 8, 4
    q, k = rng.standard_normal((c, K)), rng.standard_normal((c, K))
    cq = chunk_quantities(q, k, rng.standard_normal((c, V)), 0.3 * rng.standard_normal((c, K)),
                          rng.standard_normal(c), 0.1, np.zeros(K), -5.0)
    assert np.all(np.triu(cq["A"]) == 0)
    assert np.all(np.triu(cq["P"], 1) == 0)
    _close(np.diag(cq["P"]), np.sum(cq["qh"] * cq["kh"], 1), 1e-13, 1e-14, "P diagonal")
    _close(np.diag(cq["T"]), np.ones(c), 0, 0, "T unit diagonal")
    assert np.all(np.triu(cq["T"], 1) == 0)
    assert np.all(cq["gamma"] <= 1.0) and np.all(cq["Kdec"] ** 2 <= cq["kh"] ** 2 + 1e-15)


# --------------------------------------------------------------------------- mutants
def _mutant(mutation):
    """A CPU copy of the token recurrence with one planted mistake."""

    def sig(x):
        with np.errstate(over="ignore"):
            return np.where(x >= 0, 1 / (1 + np.exp(-np.abs(x))),
                            np.exp(-np.abs(x)) / (1 + np.exp(-np.abs(x))))

    def fwd(inp, eps):
        q, k, v, g, beta = (np.asarray(inp[x], np.float64) for x in ("q", "k", "v", "g", "beta"))
        B, T, H, K = q.shape
        V = v.shape[-1]
        lb, scale = inp["lower_bound"], inp["scale"]
        if mutation == "scale_missing":
            scale = 1.0
        cu = inp.get("cu_seqlens")
        seqs = [(b, 0, T) for b in range(B)] if cu is None else \
            [(0, int(cu[i]), int(cu[i + 1])) for i in range(len(cu) - 1)]
        S0 = np.zeros((len(seqs), H, V, K)) if inp.get("initial_state") is None \
            else np.asarray(inp["initial_state"], np.float64)
        o = np.zeros((B, T, H, V))
        fin = np.zeros((len(seqs), H, V, K))
        for n, (b, t0, t1) in enumerate(seqs):
            for h in range(H):
                S = S0[n, h].T.copy()
                for t in range(t0, t1):
                    ea = inp["A_log"][h] if mutation == "gate_no_exp_Alog" else np.exp(inp["A_log"][h])
                    a = ea * (g[b, t, h] + inp["dt_bias"][h])
                    la = lb * a if mutation == "gate_no_sigmoid" else lb * sig(a)
                    al = np.exp(la)
                    qh = q[b, t, h] / (1.0 if mutation == "q_not_normalized"
                                       else np.sqrt(np.sum(q[b, t, h] ** 2) + eps))
                    kh = k[b, t, h] / (1.0 if mutation == "k_not_normalized"
                                       else np.sqrt(np.sum(k[b, t, h] ** 2) + eps))
                    bt = beta[b, t, h] if mutation == "beta_raw" else sig(beta[b, t, h])
                    if mutation == "decay_on_v":
                        S = S * al[None, :V] if K >= V else S
                    elif mutation not in ("no_decay", "decay_after_write"):
                        S = al[:, None] * S
                    if mutation == "out_before_update":
                        o[b, t, h] = scale * S.T @ qh
                    pred = S.T @ kh
                    delta = (v[b, t, h] + pred) if mutation == "delta_sign" else (v[b, t, h] - pred)
                    S = S + bt * np.outer(kh, delta)
                    if mutation == "decay_after_write":
                        S = al[:, None] * S
                    if mutation != "out_before_update":
                        o[b, t, h] = scale * S.T @ qh
                fin[n, h] = S if mutation == "state_layout_KV" and K == V else S.T
        return o, fin

    return fwd


MUTATIONS = ["out_before_update", "no_decay", "decay_after_write", "decay_on_v", "delta_sign",
             "beta_raw", "k_not_normalized", "q_not_normalized", "gate_no_sigmoid",
             "gate_no_exp_Alog", "scale_missing", "state_layout_KV"]


def test_unmutated_copy_passes_all_pins():
    fwd = _mutant("none")
    for pin in PINS:
        pin(fwd)


@pytest.mark.filterwarnings("ignore::RuntimeWarning")
@pytest.mark.parametrize("mutation", MUTATIONS)
def test_pins_catch_planted_mistake(mutation):
    fwd = _mutant(mutation)
    caught = []
    for pin in PINS:
        try:
            pin(fwd)
        except (AssertionError, ValueError, IndexError):
            caught.append(pin.__name__)
    assert caught, f"no pin catches mutation {mutation}"


# --------------------------------------------------------------------------- per-head gate
# The gated delta rule variant: g [B,T,H] and dt_bias [H], one decay per token and head
# (the oracle's reading of the GDN pages). The numpy oracle takes it directly; these pins tie
# it to closed forms and to a differently ordered scalar-decay recurrence written here.
def _per_head_inputs(rng, B=2, T=23, H=2, K=6, V=5, lb=-2.0, init=True):
    inp = rand_inputs(rng, B=B, T=T, H=H, K=K, V=V, lb=lb, init=init)
    inp["g"] = _bf(0.7 * rng.standard_normal((B, T, H)))
    inp["dt_bias"] = _f32(0.2 * rng.standard_normal(H))
    return inp


def test_per_head_gate_decay_only_closed_form():
    # beta = 0 leaves only the decay. With A_log = 0 and dt_bias = 0 the special gate values
    # g = 0, +huge, -huge give sigmoid = 1/2, 1, 0, i.e. alpha = e^{lb/2}, e^{lb}, 1 exactly, so
    # S_t = (prod alpha) S0 and o_t = scale (prod alpha) S0^T q_hat.
    rng = np.random.default_rng(RNG_SEED + 40)
    B, T, H, K, V, lb = 1, 12, 2, 5, 4, -3.0
    inp = _per_head_inputs(rng, B, T, H, K, V, lb)
    codes = rng.integers(0, 3, size=(B, T, H))
    inp["g"] = np.choose(codes, [0.0, 1e30, -1e30]).astype(np.float64)
    inp["A_log"] = np.zeros(H)
    inp["dt_bias"] = np.zeros(H)
    inp["beta"] = np.full_like(inp["beta"], -np.inf)
    o, f = impl_numpy(inp, 1e-6)
    log_alpha = np.choose(codes, [lb / 2, lb, 0.0])
    cum = np.cumsum(log_alpha, axis=1)                          # [B,T,H]
    q = inp["q"]
    qh = q / np.sqrt(np.linalg.norm(q, axis=-1, keepdims=True) ** 2 + 1e-6)
    for h in range(H):
        S0 = inp["initial_state"][0, h].T                       # K x V
        exp_o = inp["scale"] * np.exp(cum[0, :, h])[:, None] * (qh[0, :, h] @ S0)
        _close(o[0, :, h], exp_o, 1e-12, 1e-14, f"per-head decay-only o, head {h}")
        _close(f[0, h], np.exp(cum[0, -1, h]) * inp["initial_state"][0, h], 1e-12, 1e-14,
               f"per-head decay-only final, head {h}")


def test_per_head_gate_matches_scalar_decay_recurrence():
    # With a scalar decay alpha, Diag(alpha) = alpha I commutes with the projection, so the update
    # may apply it after the delta-rule correction: S_t = alpha_t (S - beta_t k (k^T S)) + beta_t k v^T.
    rng = np.random.default_rng(RNG_SEED + 41)
    B, T, H, K, V, lb = 2, 19, 2, 6, 5, -1.5
    inp = _per_head_inputs(rng, B, T, H, K, V, lb)
    o, f = impl_numpy(inp, 1e-6)
    for b in range(B):
        for h in range(H):
            S = inp["initial_state"][b, h].T.copy()
            for t in range(T):
                a = math.exp(inp["A_log"][h]) * (inp["g"][b, t, h] + inp["dt_bias"][h])
                alpha = math.exp(lb / (1.0 + math.exp(-a)))
                kv = inp["k"][b, t, h]
                kh = kv / math.sqrt(float(kv @ kv) + 1e-6)
                qv = inp["q"][b, t, h]
                qh = qv / math.sqrt(float(qv @ qv) + 1e-6)
                bt = 1.0 / (1.0 + math.exp(-inp["beta"][b, t, h]))
                S = alpha * (S - bt * np.outer(kh, kh @ S)) + bt * np.outer(kh, inp["v"][b, t, h])
                _close(o[b, t, h], inp["scale"] * (qh @ S), 1e-11, 1e-13, f"o b={b} t={t} h={h}")
            _close(f[b, h], S.T, 1e-11, 1e-13, f"final b={b} h={h}")


def test_per_head_gate_equals_channel_broadcast():
    # The per-head gate is the per-channel oracle with g and dt_bias repeated over the channels,
    # cross-checked on the plain-C oracle (exact bf16 / fp32 inputs).
    rng = np.random.default_rng(RNG_SEED + 42)
    inp = _per_head_inputs(rng, B=1, T=17, H=3, K=4, V=3, lb=-4.0)
    o, f = impl_numpy(inp, 1e-6)
    full = dict(inp)
    full["g"] = np.repeat(inp["g"][..., None], 4, axis=-1)
    full["dt_bias"] = np.repeat(inp["dt_bias"][:, None], 4, axis=1)
    oc, fc = impl_c(full, 1e-6)
    _close(o, oc, 1e-12, 1e-14, "per-head o vs broadcast C oracle")
    _close(f, fc, 1e-12, 1e-14, "per-head final vs broadcast C oracle")
