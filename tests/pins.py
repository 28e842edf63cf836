"""Pins for the fp64 oracle: properties that the recurrence itself fixes, independent of any one
implementation of it.

The recurrence (burn-gdn2 0.1.5 docs, "Architecture"):
    S_t = (I - k_t (b_t . k_t)^T) diag(alpha_t) S_{t-1} + k_t (w_t . v_t)^T,   o_t = S_t^T q_t.

Each pin takes a ``run(q, k, v, g, b, w, s0) -> (o, S_T)`` callable (float64 results, layouts as in
the oracle: q, k [B,T,Hk,dk]; g, b [B,T,Hv,dk]; v, w [B,T,Hv,dv]; S [B,Hv,dk,dv]) and returns the
largest violation it saw. The same pins are run against the real oracle (must pass) and against
planted mistakes (each must fail at least one), see test_oracle_mutants.py.
"""
from __future__ import annotations

import json
import math
import os

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _rng(seed):
    return np.random.default_rng(seed)


def unit_rows(rng, shape):
    x = rng.standard_normal(shape)
    return x / np.linalg.norm(x, axis=-1, keepdims=True)


def rand_problem(seed, B=1, T=6, Hk=1, Hv=1, dk=4, dv=3, neg=False, s0=True, decay=True):
    """Generic random fp32-representable problem (all gates in their usual ranges)."""
    r = _rng(seed)
    f = lambda a: np.asarray(a, np.float32).astype(np.float64)
    q = f(unit_rows(r, (B, T, Hk, dk)))
    k = f(unit_rows(r, (B, T, Hk, dk)))
    v = f(r.standard_normal((B, T, Hv, dv)))
    g = f(-np.logaddexp(0, r.standard_normal((B, T, Hv, dk)))) if decay else np.zeros((B, T, Hv, dk))
    b = f((2.0 if neg else 1.0) / (1 + np.exp(-r.standard_normal((B, T, Hv, dk)))))
    w = f(1 / (1 + np.exp(-r.standard_normal((B, T, Hv, dv)))))
    S0 = f(0.3 * r.standard_normal((B, Hv, dk, dv))) if s0 else None
    return q, k, v, g, b, w, S0


def _worse(worst, x):
    """max() that does not swallow NaN (a NaN anywhere is an infinite violation)."""
    x = float(x)
    return float("inf") if x != x else max(worst, x)


def rel(x, ref):
    den = float(np.max(np.abs(ref))) if np.size(ref) else 0.0
    num = float(np.max(np.abs(np.asarray(x) - np.asarray(ref)))) if np.size(ref) else 0.0
    if num != num or den != den:
        return float("inf")
    return num / den if den > 0 else num


def _prefix_states(run, q, k, v, g, b, w, s0):
    """S_t for t = 0..T-1 obtained by running the first t+1 tokens."""
    T = q.shape[1]
    out = []
    for t in range(T):
        sl = lambda a: np.ascontiguousarray(a[:, : t + 1])
        _, sT = run(sl(q), sl(k), sl(v), sl(g), sl(b), sl(w), s0)
        out.append(sT)
    return out


# ----------------------------------------------------------------------------------------------
# 1. retrieval invariant.  With b = 1 and unit k, S_t^T k_t = w_t . v_t for ANY decay. In general
#    (unit k): S_t^T k_t = S'^T((1 - b_t) . k_t) + w_t . v_t with S' = diag(alpha_t) S_{t-1}.
#    Checked in the form that holds for any k (the stored k is unit-norm only to fp32 rounding):
#    S_t^T k_t = S'^T k_t + |k_t|^2 (w_t . v_t - S'^T (b_t . k_t)).

def pin_retrieval(run, seed=1):
    worst = 0.0
    for general in (False, True):
        q, k, v, g, b, w, S0 = rand_problem(seed + general, T=5, dk=5, dv=3, neg=general)
        if not general:
            b = np.ones_like(b)
        states = _prefix_states(run, q, k, v, g, b, w, S0)
        prev = S0 if S0 is not None else np.zeros_like(states[0])
        for t in range(q.shape[1]):
            St = states[t][0, 0]
            kt, gt, bt = k[0, t, 0], g[0, t, 0], b[0, t, 0]
            lhs = St.T @ kt
            Sp = np.exp(gt)[:, None] * prev[0, 0]
            kk = float(kt @ kt)
            rhs = Sp.T @ kt + kk * (w[0, t, 0] * v[0, t, 0] - Sp.T @ (bt * kt))
            worst = _worse(worst, float(np.max(np.abs(lhs - rhs))))
            prev = states[t]
    return worst


# ----------------------------------------------------------------------------------------------
# 2. linear-attention / gated-linear-attention reduction.  With b = 0 the erase vanishes and
#    o_t = S0^T (e^{G_t} . q_t) + sum_{s<=t} (w_s . v_s) sum_c q_t[c] k_s[c] e^{G_t[c] - G_s[c]},
#    G_t = sum_{u<=t} g_u.  Brute force, O(T^2).

def pin_linear_attention(run, seed=2):
    worst = 0.0
    for decay in (False, True):
        q, k, v, g, b, w, S0 = rand_problem(seed, T=7, Hk=1, Hv=2, dk=4, dv=3, decay=decay)
        b = np.zeros_like(b)
        o, sT = run(q, k, v, g, b, w, S0)
        T = q.shape[1]
        for h in range(2):
            G = np.cumsum(g[0, :, h], axis=0)
            for t in range(T):
                ref = S0[0, h].T @ (np.exp(G[t]) * q[0, t, 0])
                for s in range(t + 1):
                    coef = float(np.sum(q[0, t, 0] * k[0, s, 0] * np.exp(G[t] - G[s])))
                    ref = ref + coef * (w[0, s, h] * v[0, s, h])
                worst = _worse(worst, float(np.max(np.abs(o[0, t, h] - ref))))
            Sref = np.exp(G[-1])[:, None] * S0[0, h]
            for s in range(T):
                Sref = Sref + np.outer(k[0, s, 0] * np.exp(G[-1] - G[s]), w[0, s, h] * v[0, s, h])
            worst = _worse(worst, float(np.max(np.abs(sT[0, h] - Sref))))
    return worst


# ----------------------------------------------------------------------------------------------
# 3. scalar gated delta rule.  With b_t = w_t = beta_t (broadcast) and alpha_t a broadcast scalar
#    the recurrence is Gated DeltaNet. Reference written in the usual "memory matrix" convention
#    M in R^{dv x dk}: M_t = alpha_t M_{t-1} (I - beta_t k_t k_t^T) + beta_t v_t k_t^T, o_t = M_t q_t.

def pin_scalar_gated_delta(run, seed=3):
    q, k, v, g, b, w, S0 = rand_problem(seed, T=9, dk=6, dv=5)
    r = _rng(seed + 100)
    T = q.shape[1]
    beta = np.asarray(1 / (1 + np.exp(-r.standard_normal(T))), np.float32).astype(np.float64)
    loga = np.asarray(-np.logaddexp(0, r.standard_normal(T)), np.float32).astype(np.float64)
    b = np.broadcast_to(beta[None, :, None, None], b.shape).copy()
    w = np.broadcast_to(beta[None, :, None, None], w.shape).copy()
    g = np.broadcast_to(loga[None, :, None, None], g.shape).copy()
    o, sT = run(q, k, v, g, b, w, S0)
    Mem = S0[0, 0].T.copy()
    worst = 0.0
    for t in range(T):
        kt, qt, vt = k[0, t, 0], q[0, t, 0], v[0, t, 0]
        Mem = math.exp(loga[t]) * (Mem @ (np.eye(kt.size) - beta[t] * np.outer(kt, kt))) + beta[t] * np.outer(vt, kt)
        worst = _worse(worst, float(np.max(np.abs(o[0, t, 0] - Mem @ qt))))
    worst = _worse(worst, float(np.max(np.abs(sT[0, 0] - Mem.T))))
    return worst


# ----------------------------------------------------------------------------------------------
# 4. standard-basis keys, dyadic values: each state row obeys a scalar recurrence,
#    keyed row i_t:  S[i,:] <- (1 - b_t[i]) alpha_t[i] S[i,:] + w_t . v_t ; other rows r:
#    S[r,:] <- alpha_t[r] S[r,:].  alpha is 0 or 1 (g = -inf or 0) and every other value is dyadic,
#    so the fp64 results must be EXACT.

def pin_standard_basis_exact(run, seed=4):
    r = _rng(seed)
    T, dk, dv = 12, 4, 3
    idx = r.integers(0, dk, T)
    k = np.zeros((1, T, 1, dk))
    k[0, np.arange(T), 0, idx] = 1.0
    k[0, ::3] *= -1.0                                   # a sign flip keeps k unit-norm
    q = r.integers(-4, 5, (1, T, 1, dk)) / 4.0
    v = r.integers(-8, 9, (1, T, 1, dv)) / 8.0
    alpha = r.choice([0.0, 1.0], (1, T, 1, dk), p=[0.25, 0.75])
    g = np.where(alpha == 0.0, -np.inf, 0.0)             # exp(-inf) = 0 and exp(0) = 1 exactly
    b = r.choice([0.5, 1.0, 1.5], (1, T, 1, dk))
    w = r.choice([0.5, 1.0], (1, T, 1, dv))
    S0 = r.integers(-4, 5, (1, 1, dk, dv)) / 8.0
    o, sT = run(q, k, v, g, b, w, S0)
    S = S0[0, 0].copy()
    worst = 0.0
    for t in range(T):
        a = alpha[0, t, 0]
        i = idx[t]
        s = k[0, t, 0, i]                                # +1 or -1
        S = a[:, None] * S
        S[i] = (1.0 - b[0, t, 0, i]) * S[i] + s * (w[0, t, 0] * v[0, t, 0])
        ref = S.T @ q[0, t, 0]
        worst = _worse(worst, float(np.max(np.abs(o[0, t, 0] - ref))))
    worst = _worse(worst, float(np.max(np.abs(sT[0, 0] - S))))
    return worst


# ----------------------------------------------------------------------------------------------
# 5. hand-worked examples (tests/golden/hand_worked.json), derived on paper from the recurrence.

def pin_hand_worked(run):
    with open(os.path.join(GOLDEN, "hand_worked.json")) as f:
        cases = json.load(f)["cases"]
    worst = 0.0
    for c in cases:
        arr = lambda key: np.asarray(np.asarray(c[key], np.float32), np.float64)
        q, k, v, g, b, w = (arr(x) for x in ("q", "k", "v", "g", "b", "w"))
        S0 = arr("S0") if c.get("S0") is not None else None
        o, sT = run(q, k, v, g, b, w, S0)
        worst = _worse(_worse(worst, rel(o, np.asarray(c["o"]))), rel(sT, np.asarray(c["S_T"])))
    return worst


# ----------------------------------------------------------------------------------------------
# 6. grouped heads: value head h reads key head h // (Hv / Hk); equal to running with q, k repeated
#    per value head.

def pin_gqa_grouping(run, seed=6):
    q, k, v, g, b, w, S0 = rand_problem(seed, B=2, T=5, Hk=2, Hv=6, dk=3, dv=2)
    o, sT = run(q, k, v, g, b, w, S0)
    rep = lambda a: np.ascontiguousarray(np.repeat(a, 3, axis=2))
    o2, sT2 = run(rep(q), rep(k), v, g, b, w, S0)
    return _worse(_worse(0.0, np.max(np.abs(o - o2))), np.max(np.abs(sT - sT2)))


ALL_PINS = {
    "retrieval": pin_retrieval,
    "linear_attention": pin_linear_attention,
    "scalar_gated_delta": pin_scalar_gated_delta,
    "standard_basis_exact": pin_standard_basis_exact,
    "hand_worked": pin_hand_worked,
    "gqa_grouping": pin_gqa_grouping,
}

# tolerance per pin (fp64 arithmetic; the standard-basis case is exact)
PIN_TOL = {
    "retrieval": 1e-12,
    "linear_attention": 1e-12,
    "scalar_gated_delta": 1e-12,
    "standard_basis_exact": 0.0,
    "hand_worked": 2e-6,   # inputs are float32 roundings of the paper values (0.6, 0.8, ln 0.5)
    "gqa_grouping": 0.0,
}
