"""Pins of the prologue / epilogue oracle (CPU only): closed forms, special cases and invariants."""
import numpy as np
import pytest

from oracle import mixer


def test_conv_identity_and_shift():
    rng = np.random.default_rng(0)
    x = rng.standard_normal((2, 9, 5))
    eye = np.zeros((5, 4))
    eye[:, 3] = 1.0                                       # tap on the current token
    y, st = mixer.short_conv(x, eye)
    assert np.array_equal(y, x)
    assert np.array_equal(st, x[:, -3:])
    shift = np.zeros((5, 4))
    shift[:, 1] = 1.0                                     # the token two steps back
    y, _ = mixer.short_conv(x, shift)
    assert np.array_equal(y[:, 2:], x[:, :-2]) and np.all(y[:, :2] == 0)


def test_conv_brute_force_small():
    """y_t = sum_j W[c, j] x_{t-3+j} written out by hand for one channel and a carried state."""
    x = np.array([[[1.0], [2.0], [3.0]]])                 # B=1, T=3, C=1
    st = np.array([[[10.0], [20.0], [30.0]]])             # x_{-3}, x_{-2}, x_{-1}
    W = np.array([[1.0, 0.1, 0.01, 0.001]])
    y, new = mixer.short_conv(x, W, st)
    expect = [10 * 1 + 20 * 0.1 + 30 * 0.01 + 1 * 0.001,
              20 * 1 + 30 * 0.1 + 1 * 0.01 + 2 * 0.001,
              30 * 1 + 1 * 0.1 + 2 * 0.01 + 3 * 0.001]
    assert np.allclose(y[0, :, 0], expect, rtol=0, atol=1e-12)
    assert np.array_equal(new[0, :, 0], [1.0, 2.0, 3.0])


@pytest.mark.parametrize("split", [1, 2, 3, 7])
def test_conv_state_chaining(split):
    """Two calls with the carried state equal one call (also when a call is shorter than 3 tokens)."""
    rng = np.random.default_rng(1)
    x = rng.standard_normal((2, 10, 6))
    W = rng.standard_normal((6, 4))
    st0 = rng.standard_normal((2, 3, 6))
    y, st = mixer.short_conv(x, W, st0)
    y1, s1 = mixer.short_conv(x[:, :split], W, st0)
    y2, s2 = mixer.short_conv(x[:, split:], W, s1)
    assert np.allclose(np.concatenate([y1, y2], axis=1), y, rtol=0, atol=1e-12)
    assert np.array_equal(s2, st)


def test_l2_norm_unit_and_scale_invariant():
    rng = np.random.default_rng(2)
    x = rng.standard_normal((3, 4, 2, 16)) * 5
    n = mixer.l2_norm(x)
    assert np.allclose(np.linalg.norm(n, axis=-1), 1.0, atol=1e-7)
    assert np.allclose(mixer.l2_norm(3.0 * x), n, atol=1e-7)
    assert np.array_equal(mixer.l2_norm(np.zeros(4)), np.zeros(4))


def test_gate_activations_closed_forms():
    a = np.array([-40.0, -1.0, 0.0, 1.0, 40.0])
    assert np.isclose(mixer.softplus(0.0), np.log(2.0))
    assert np.isclose(mixer.sigmoid(0.0), 0.5)
    assert np.allclose(mixer.softplus(a) - mixer.softplus(-a), a)          # softplus(a) - softplus(-a) = a
    assert np.allclose(mixer.sigmoid(a) + mixer.sigmoid(-a), 1.0)
    rng = np.random.default_rng(3)
    shp = (1, 3, 2, 8)
    xs = [rng.standard_normal(shp) for _ in range(3)]
    ws = [np.zeros((16, 4)) for _ in range(3)]
    ag, ab, aw = (rng.standard_normal(shp) for _ in range(3))
    _, _, _, g, b, w, _ = mixer.prologue(*xs, *ws, ag, ab, aw)
    _, _, _, g2, b2, w2, _ = mixer.prologue(*xs, *ws, ag, ab, aw, neg_eigval=True)
    assert np.all(g <= 0) and np.all((b > 0) & (b < 1)) and np.all((w > 0) & (w < 1))
    assert np.allclose(b2, 2 * b) and np.array_equal(g2, g) and np.array_equal(w2, w)


def test_epilogue_special_cases():
    d = 8
    weight = np.linspace(0.5, 2.0, d)
    c = 3.0
    o = np.full((1, 1, 1, d), c)
    z = np.full((1, 1, 1, d), 2.0)
    y = mixer.epilogue(o, z, weight)
    silu2 = 2.0 / (1.0 + np.exp(-2.0))
    assert np.allclose(y[0, 0, 0], c / np.sqrt(c * c + 1e-5) * weight * silu2, rtol=1e-12)
    assert np.array_equal(mixer.epilogue(o, np.zeros_like(z), weight), np.zeros_like(o))   # silu(0) = 0
    # with weight 1 and a constant gate g, the output's RMS over d_v is |silu(g)| * rms/sqrt(rms^2 + eps)
    rng = np.random.default_rng(4)
    o = rng.standard_normal((2, 3, 2, d))
    y = mixer.epilogue(o, np.full_like(o, 5.0), np.ones(d), eps=0.0)
    assert np.allclose(np.sqrt(np.mean(y * y, axis=-1)), 5.0 / (1.0 + np.exp(-5.0)), rtol=1e-12)
