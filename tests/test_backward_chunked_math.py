"""The algebra of the chunked backward (reverse mode of the chunked WY form of the burn-gdn2 0.1.5
docs, "chunked WY decomposition (training)") restated in fp64 NumPy and checked against the
oracle's autograd gradients of the per-token recurrence: the chains over chunks (dU, dS), the
per-chunk products (dK^, dQ_bar, dW, dM, dT, dA), and the pair terms with each factor
e^{G_t - G_s} of tokens in different 8-token blocks split at a block edge into two factors <= 1.
This pins the derivation the GPU kernels follow, independently of them (it shares no code with
the CUDA path and uses the oracle only as the reference)."""
import numpy as np
import pytest

from oracle import backward as oback

C = 32      # chunk
BLK = 8     # token block of the pair terms


def _inv_unit_lower(A):
    return np.linalg.inv(np.eye(A.shape[0]) + A)


def _pair_terms(G, k, beta, q, dA, dM):
    """X, Y, Z, V of one chunk (all [C][d]) with the block-edge split; G is the cumulative log-decay."""
    Cn, d = G.shape
    X, Y, Z, V = (np.zeros((Cn, d)) for _ in range(4))
    nb = Cn // BLK
    for bt in range(nb):  # X_t = sum_{s<t} dA_ts k_s e^{G_t-G_s}, Y_t = sum_{s<=t} dM_ts k_s e^{G_t-G_s}
        t0 = BLK * bt
        ts = range(t0, t0 + BLK)
        if bt > 0:  # earlier blocks through r = t0
            ks = k[:t0] * np.exp(G[t0] - G[:t0])            # e^{G_r - G_s} <= 1
            for t in ts:
                et = np.exp(G[t] - G[t0])                   # e^{G_t - G_r} <= 1
                X[t] += et * (dA[t, :t0, None] * ks).sum(0)
                Y[t] += et * (dM[t, :t0, None] * ks).sum(0)
        for t in ts:  # the same block, pair by pair
            for s in range(t0, t + 1):
                e = np.exp(G[t] - G[s])
                if s < t:
                    X[t] += dA[t, s] * k[s] * e
                Y[t] += dM[t, s] * k[s] * e
    for bs in range(nb):  # Z_s = sum_{u>s} dA_us b_u k_u e^{G_u-G_s}, V_s = sum_{u>=s} dM_us q_u e^{G_u-G_s}
        s0 = BLK * bs
        r = s0 + BLK - 1
        ss = range(s0, s0 + BLK)
        if bs < nb - 1:  # later blocks through r = the block's last token
            bu = beta[r + 1:] * np.exp(G[r + 1:] - G[r])    # e^{G_u - G_r} <= 1
            qu = q[r + 1:] * np.exp(G[r + 1:] - G[r])
            for s in ss:
                es = np.exp(G[r] - G[s])                    # e^{G_r - G_s} <= 1
                Z[s] += es * (dA[r + 1:, s, None] * bu).sum(0)
                V[s] += es * (dM[r + 1:, s, None] * qu).sum(0)
        for s in ss:
            for u in range(s, s0 + BLK):
                e = np.exp(G[u] - G[s])
                if u > s:
                    Z[s] += dA[u, s] * beta[u] * e
                V[s] += dM[u, s] * q[u] * e
    return X, Y, Z, V


def chunked_gradients(q, k, v, g, b, w, s0, do, ds_t, scale=1.0):
    """Gradients of sum(o . do) + sum(S_T . ds_t) by the chunked reverse mode; shapes as the oracle's."""
    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    NC = (T + C - 1) // C
    pad = NC * C - T
    P = lambda x: np.concatenate([x, np.zeros((B, pad) + x.shape[2:])], axis=1) if pad else x
    q, k, v, g, b, w, do = (P(np.asarray(x, np.float64)) for x in (q, k, v, g, b, w, do))
    out = {n: np.zeros_like(x) for n, x in (("dv", v), ("dg", g), ("db", b), ("dw", w))}
    dq_v = np.zeros((B, NC * C, Hv, dk))
    dk_v = np.zeros((B, NC * C, Hv, dk))
    ds0 = np.zeros((B, Hv, dk, dv))
    grp = Hv // Hk
    for bi in range(B):
        for hv in range(Hv):
            hk = hv // grp
            S = np.zeros((dk, dv)) if s0 is None else np.asarray(s0[bi, hv], np.float64).copy()
            fac, Ss, Us = [], [], []
            for n in range(NC):  # forward chain, keeping the factors, S_n and U_n
                sl = slice(n * C, (n + 1) * C)
                qq, kk, gg, bb = q[bi, sl, hk], k[bi, sl, hk], g[bi, sl, hv], b[bi, sl, hv]
                G = np.cumsum(gg, axis=0)
                Gl = G[-1]
                beta = bb * kk
                E = np.exp(G[:, None, :] - G[None, :, :])            # [t][s][c]; used for s <= t only
                low = np.tril(np.ones((C, C)))
                A = np.tril(np.einsum("tc,sc,tsc->ts", beta, kk, np.where(low[:, :, None] > 0, E, 0)), -1)
                M = np.einsum("tc,sc,tsc->ts", qq, kk, np.where(low[:, :, None] > 0, E, 0))
                Tm = _inv_unit_lower(A)
                Kb = beta * np.exp(G)
                Qb = qq * np.exp(G)
                Kh = kk * np.exp(Gl - G)
                U0 = w[bi, sl, hv] * v[bi, sl, hv]
                W = Tm @ Kb
                U = Tm @ U0 - W @ S
                fac.append((G, Gl, beta, Kb, Qb, Kh, M, Tm, W, U0, qq, kk, bb))
                Ss.append(S.copy())
                Us.append(U)
                S = np.exp(Gl)[:, None] * S + Kh.T @ U
            dS = np.zeros((dk, dv)) if ds_t is None else np.asarray(ds_t[bi, hv], np.float64).copy()
            for n in reversed(range(NC)):  # backward chain and the per-chunk gradients
                sl = slice(n * C, (n + 1) * C)
                G, Gl, beta, Kb, Qb, Kh, M, Tm, W, U0, qq, kk, bb = fac[n]
                S, U = Ss[n], Us[n]
                dOt = scale * do[bi, sl, hv]
                dSp = dS
                dU = M.T @ dOt + Kh @ dSp
                dS = np.exp(Gl)[:, None] * dSp + Qb.T @ dOt - W.T @ dU
                dQb = dOt @ S.T
                dW = -dU @ S.T
                dKh = U @ dSp.T
                dgam = (dSp * S).sum(1)
                dM = np.tril(dOt @ U.T)
                dT = dU @ U0.T + dW @ Kb.T
                dU0 = Tm.T @ dU
                dKb = Tm.T @ dW
                dA = -np.tril(Tm.T @ dT @ Tm.T, -1)
                X, Y, Z, V = _pair_terms(G, kk, beta, qq, dA, dM)
                eG, eH = np.exp(G), np.exp(Gl - G)
                dbeta = dKb * eG + X
                dq_v[bi, sl, hv] = dQb * eG + Y
                dk_v[bi, sl, hv] = dKh * eH + Z + V + dbeta * bb
                out["db"][bi, sl, hv] = dbeta * kk
                dG = dQb * qq * eG + dKb * Kb - dKh * kk * eH + beta * X + qq * Y - kk * (Z + V)
                dGl = (dKh * kk * eH).sum(0) + dgam * np.exp(Gl)
                out["dg"][bi, sl, hv] = np.cumsum(dG[::-1], axis=0)[::-1] + dGl
                out["dv"][bi, sl, hv] = w[bi, sl, hv] * dU0
                out["dw"][bi, sl, hv] = v[bi, sl, hv] * dU0
            ds0[bi, hv] = dS
    res = {n: x[:, :T] for n, x in out.items()}
    res["dq"] = dq_v.reshape(B, NC * C, Hk, grp, dk).sum(3)[:, :T]
    res["dk"] = dk_v.reshape(B, NC * C, Hk, grp, dk).sum(3)[:, :T]
    res["ds0"] = ds0
    return res


@pytest.mark.parametrize("T,Hk,Hv,with_state", [(70, 1, 2, True), (64, 2, 2, False), (19, 1, 1, True)])
def test_chunked_backward_algebra_matches_the_oracle(T, Hk, Hv, with_state):
    rng = np.random.default_rng(T + 10 * Hv)
    B, d = 1, 16
    q = rng.standard_normal((B, T, Hk, d)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, Hk, d)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, d))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, Hv, d))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv, d))))
    w = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv, d))))
    s0 = 0.1 * rng.standard_normal((B, Hv, d, d)) if with_state else None
    ds_t = 0.1 * rng.standard_normal((B, Hv, d, d)) if with_state else None
    do = rng.standard_normal((B, T, Hv, d))
    ref = oback.gradients(q, k, v, g, b, w, s0, do, ds_t, scale=0.5)
    got = chunked_gradients(q, k, v, g, b, w, s0, do, ds_t, scale=0.5)
    for name in ("dq", "dk", "dv", "dg", "db", "dw", "ds0"):
        r = np.asarray(ref[name])
        e = np.abs(got[name] - r).max() / max(np.abs(r).max(), 1e-300)
        assert e < 1e-10, (name, e)


def test_chunked_backward_algebra_catches_a_dropped_pair_term():
    """A plausible slip (the V term left out of dk) must not pass the comparison above."""
    rng = np.random.default_rng(3)
    B, T, H, d = 1, 40, 1, 16
    q = rng.standard_normal((B, T, H, d)); q /= np.linalg.norm(q, axis=-1, keepdims=True)
    k = rng.standard_normal((B, T, H, d)); k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v, do = rng.standard_normal((B, T, H, d)), rng.standard_normal((B, T, H, d))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, H, d))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H, d))))
    w = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, H, d))))
    ref = oback.gradients(q, k, v, g, b, w, None, do, None)
    global _pair_terms
    orig = _pair_terms
    try:
        _pair_terms = lambda *a: (lambda X, Y, Z, V: (X, Y, Z, 0.0 * V))(*orig(*a))
        bad = chunked_gradients(q, k, v, g, b, w, None, do, None)
    finally:
        _pair_terms = orig
    e = np.abs(bad["dk"] - ref["dk"]).max() / np.abs(ref["dk"]).max()
    assert e > 1e-3
