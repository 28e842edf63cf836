"""Pins of the gradient oracle (CPU only): its forward against the C oracle, and every gradient
against central finite differences of the same functional."""
import numpy as np
import pytest

import oracle
from oracle import backward, max_rel_err


def _inputs(rng, B=1, T=5, Hk=1, Hv=2, dk=4, dv=3):
    q = rng.standard_normal((B, T, Hk, dk))
    k = rng.standard_normal((B, T, Hk, dk))
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((B, T, Hv, dv))
    g = -np.log1p(np.exp(rng.standard_normal((B, T, Hv, dk))))
    b = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv, dk))))
    w = 1.0 / (1.0 + np.exp(-rng.standard_normal((B, T, Hv, dv))))
    s0 = 0.3 * rng.standard_normal((B, Hv, dk, dv))
    return [x.astype(np.float32).astype(np.float64) for x in (q, k, v, g, b, w, s0)]


def test_forward_matches_the_c_oracle():
    import torch

    rng = np.random.default_rng(0)
    q, k, v, g, b, w, s0 = _inputs(rng, B=2, T=9, Hk=2, Hv=4, dk=8, dv=6)
    o, s = backward.forward_torch(*(torch.tensor(x) for x in (q, k, v, g, b, w, s0)), scale=0.5)
    o_ref, s_ref = oracle.run(q, k, v, g, b, w, s0, scale=0.5)
    assert max_rel_err(o.numpy(), o_ref) < 1e-12 and max_rel_err(s.numpy(), s_ref) < 1e-12


@pytest.mark.parametrize("with_ds", [False, True])
def test_gradients_against_finite_differences(with_ds):
    rng = np.random.default_rng(1 + with_ds)
    xs = _inputs(rng)
    B, T, Hv, dv = xs[2].shape
    dk = xs[0].shape[3]
    do = rng.standard_normal((B, T, Hv, dv))
    ds_t = rng.standard_normal((B, Hv, dk, dv)) if with_ds else None
    gr = backward.gradients(*xs, do, ds_t, scale=0.8)

    def functional(vals):
        import torch

        o, s = backward.forward_torch(*(torch.tensor(x) for x in vals), scale=0.8)
        f = float((o.numpy() * do).sum())
        return f + (float((s.numpy() * ds_t).sum()) if ds_t is not None else 0.0)

    h = 1e-6
    for idx, name in enumerate(("dq", "dk", "dv", "dg", "db", "dw", "ds0")):
        x = xs[idx]
        fd = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            i = it.multi_index
            up = [a.copy() for a in xs]
            dn = [a.copy() for a in xs]
            up[idx][i] += h
            dn[idx][i] -= h
            fd[i] = (functional(up) - functional(dn)) / (2 * h)
        assert max_rel_err(gr[name], fd) < 1e-6, name


def test_grouped_heads_sum_key_gradients():
    """dq, dk of a key head are the sums over its value heads (compare with the ungrouped problem
    where every value head has its own copy of q and k)."""
    rng = np.random.default_rng(3)
    q, k, v, g, b, w, s0 = _inputs(rng, B=1, T=4, Hk=1, Hv=3, dk=4, dv=2)
    do = rng.standard_normal(v.shape)
    gr = backward.gradients(q, k, v, g, b, w, s0, do)
    qx, kx = np.repeat(q, 3, axis=2), np.repeat(k, 3, axis=2)
    gx = backward.gradients(qx, kx, v, g, b, w, s0, do)
    assert np.allclose(gr["dq"][:, :, 0], gx["dq"].sum(axis=2), atol=1e-12)
    assert np.allclose(gr["dk"][:, :, 0], gx["dk"].sum(axis=2), atol=1e-12)
    for n in ("dv", "dg", "db", "dw", "ds0"):
        assert np.allclose(gr[n], gx[n], atol=1e-12)
