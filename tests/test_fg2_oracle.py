"""Pins of the FG^2-GDN oracle (CPU only): reductions and identities that hold independently of it."""
import numpy as np
import pytest

import oracle
from oracle.fg2 import fg2_recurrent
from oracle import max_rel_err

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")


def _inputs(rng, B=2, T=13, Hk=1, Hv=2, d=8):
    """Values chosen so that every product the transform forms is exact in float32 (the GDN-2 oracle
    reads float32 inputs): sqrt(beta) = m / 64, k on a 2^-10 grid."""
    f32 = lambda a: a.astype(np.float32).astype(np.float64)
    q = f32(rng.standard_normal((B, T, Hk, d)))
    k = np.round(rng.standard_normal((B, T, Hk, d)) / np.sqrt(d) * 1024) / 1024
    v = f32(rng.standard_normal((B, T, Hv, d)))
    g = f32(-np.log1p(np.exp(rng.standard_normal((B, T, Hv, d)))))
    root = rng.integers(8, 65, (B, T, Hv, d)) / 64.0
    beta = root * root
    s0 = f32(0.1 * rng.standard_normal((B, Hv, d, d)))
    return q, k, v, g, beta, s0


def _expand(x, Hv):
    """per-key-head tensor -> per-value-head (contiguous groups)"""
    Hk = x.shape[2]
    return np.repeat(x, Hv // Hk, axis=2)


def test_beta_one_is_the_delta_rule():
    """beta = 1: S_t = (I - k k^T) Diag(alpha) S + k v^T, the GDN-2 recurrence with b = w = 1."""
    rng = np.random.default_rng(1)
    q, k, v, g, beta, s0 = _inputs(rng)
    ones = np.ones_like(beta)
    o, s = fg2_recurrent(q, k, v, g, ones, s0)
    o_ref, s_ref = oracle.run(q, k, v, g, ones, ones, s0, form="recurrent")
    assert max_rel_err(o, o_ref) < 1e-12 and max_rel_err(s, s_ref) < 1e-12


def test_retrieval_of_the_scaled_value():
    """No decay and a unit scaled key: the updated state maps k~_t to v~_t exactly."""
    rng = np.random.default_rng(2)
    B, T, H, d = 1, 9, 1, 6
    beta = rng.uniform(0.2, 1.0, (B, T, H, d))
    k = rng.standard_normal((B, T, H, d))
    k /= np.linalg.norm(np.sqrt(beta) * k, axis=-1, keepdims=True)   # |sqrt(beta) . k| = 1
    v = rng.standard_normal((B, T, H, d))
    g = np.zeros((B, T, H, d))
    S = np.zeros((d, d))
    for t in range(T):   # chain one token at a time through the oracle
        kt = np.sqrt(beta[:, t:t + 1]) * k[:, t:t + 1]
        o, s = fg2_recurrent(kt, k[:, t:t + 1], v[:, t:t + 1], g[:, t:t + 1], beta[:, t:t + 1], S[None, None])
        S = s[0, 0]
        assert np.allclose(o[0, 0, 0], np.sqrt(beta[0, t, 0]) * v[0, t, 0], rtol=0, atol=1e-12)


def test_gdn2_core_with_transformed_inputs():
    """k <- sqrt(beta) . k, b <- 1, w <- sqrt(beta) on the GDN-2 core gives FG^2-GDN (grouped heads)."""
    rng = np.random.default_rng(3)
    q, k, v, g, beta, s0 = _inputs(rng, Hk=2, Hv=4)
    o, s = fg2_recurrent(q, k, v, g, beta, s0, scale=0.7)
    qx, kx = _expand(q, 4), _expand(k, 4)
    root = np.sqrt(beta)
    for form in ("recurrent", "chunked"):
        o_ref, s_ref = oracle.run(qx, root * kx, v, g, np.ones_like(beta), root, s0, form=form, C=4, scale=0.7)
        assert max_rel_err(o, o_ref) < 1e-12 and max_rel_err(s, s_ref) < 1e-12


@pytest.mark.parametrize("mistake", ["rate_on_key_only", "rate_without_root"])
def test_planted_mistakes_are_rejected(mistake):
    rng = np.random.default_rng(4)
    q, k, v, g, beta, s0 = _inputs(rng, Hk=1, Hv=2)
    o, s = fg2_recurrent(q, k, v, g, beta, s0)
    qx, kx = _expand(q, 2), _expand(k, 2)
    ones = np.ones_like(beta)
    if mistake == "rate_on_key_only":
        args = (qx, np.sqrt(beta) * kx, v, g, ones, ones)
    else:
        args = (qx, beta * kx, v, g, ones, beta)
    o_bad, s_bad = oracle.run(*args, s0, form="recurrent")
    assert max_rel_err(o_bad, o) > 1e-3
