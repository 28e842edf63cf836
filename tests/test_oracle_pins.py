"""The fp64 oracle against what the recurrence itself fixes (CPU only).

Pins (tests/pins.py): retrieval invariant, linear-attention reduction, scalar gated-delta-rule
reduction, exact standard-basis-key cases, hand-worked examples, grouped-head mapping. Plus the
oracle's three forms (recurrent, literal, chunked) agreeing with each other, linearity in (v, S0),
independence of value columns, state chaining, empty input, a full reset (alpha = 0) and scale.
"""
import numpy as np
import pytest

import oracle
from tests import pins

FORMS = [("recurrent", None), ("literal", None), ("chunked", 1), ("chunked", 3), ("chunked", 4),
         ("chunked", 64)]


def runner(form, C):
    def run(q, k, v, g, b, w, s0):
        return oracle.run(q, k, v, g, b, w, s0, form=form, C=C or 64, nthreads=2)
    return run


@pytest.mark.parametrize("form,C", FORMS)
@pytest.mark.parametrize("pin", sorted(pins.ALL_PINS))
def test_pin(form, C, pin):
    err = pins.ALL_PINS[pin](runner(form, C))
    assert err <= pins.PIN_TOL[pin], f"{pin} violated by oracle form {form}/C={C}: {err:.3e}"


@pytest.mark.parametrize("T,C", [(1, 64), (37, 8), (64, 64), (65, 64), (130, 16), (29, 1), (29, 2)])
def test_forms_agree(T, C):
    q, k, v, g, b, w, S0 = pins.rand_problem(11 + T, B=2, T=T, Hk=2, Hv=4, dk=8, dv=6, neg=True)
    o_r, s_r = oracle.run(q, k, v, g, b, w, S0, form="recurrent")
    o_l, s_l = oracle.run(q, k, v, g, b, w, S0, form="literal")
    o_c, s_c = oracle.run(q, k, v, g, b, w, S0, form="chunked", C=C)
    for x, ref in ((o_l, o_r), (s_l, s_r), (o_c, o_r), (s_c, s_r)):
        assert pins.rel(x, ref) < 1e-12


def test_forms_agree_full_width():
    """d_k = d_v = 128, C = 64, two chunks and a ragged tail, with the workload distributions."""
    import synth

    wl = synth.WORKLOADS["train_bf16"].with_(B=1, Hk=1, Hv=1, T=150)
    inp = synth.make_inputs(wl)
    o_r, s_r = oracle.run_inputs(inp, form="recurrent")
    o_c, s_c = oracle.run_inputs(inp, form="chunked", C=64)
    assert pins.rel(o_c, o_r) < 1e-11 and pins.rel(s_c, s_r) < 1e-11


def test_linearity_in_values_and_state():
    q, k, v1, g, b, w, S1 = pins.rand_problem(21, T=9, dk=5, dv=4)
    _, _, v2, _, _, _, S2 = pins.rand_problem(22, T=9, dk=5, dv=4)
    # values on a 2^-10 grid so that 2 v1 - 3 v2 is exact in the oracle's fp32 input type
    v1, v2 = np.round(v1 * 1024) / 1024, np.round(v2 * 1024) / 1024
    for form in ("recurrent", "chunked"):
        o1, s1 = oracle.run(q, k, v1, g, b, w, S1, form=form, C=4)
        o2, s2 = oracle.run(q, k, v2, g, b, w, S2, form=form, C=4)
        o3, s3 = oracle.run(q, k, 2.0 * v1 - 3.0 * v2, g, b, w, 2.0 * S1 - 3.0 * S2, form=form, C=4)
        assert pins.rel(o3, 2.0 * o1 - 3.0 * o2) < 1e-12
        assert pins.rel(s3, 2.0 * s1 - 3.0 * s2) < 1e-12


def test_value_columns_independent():
    q, k, v, g, b, w, S0 = pins.rand_problem(23, T=11, dk=5, dv=4)
    o, s = oracle.run(q, k, v, g, b, w, S0)
    v2 = v.copy()
    v2[..., 2] += 1.0
    o2, s2 = oracle.run(q, k, v2, g, b, w, S0)
    keep = [0, 1, 3]
    assert np.array_equal(o[..., keep], o2[..., keep]) and np.array_equal(s[..., keep], s2[..., keep])
    assert not np.allclose(o[..., 2], o2[..., 2])


@pytest.mark.parametrize("form", ["recurrent", "literal", "chunked"])
def test_state_chaining(form):
    q, k, v, g, b, w, S0 = pins.rand_problem(24, B=2, T=23, Hk=1, Hv=2, dk=6, dv=5)
    o, s = oracle.run(q, k, v, g, b, w, S0, form=form, C=4)
    cut = 10
    a = lambda x: np.ascontiguousarray(x[:, :cut])
    z = lambda x: np.ascontiguousarray(x[:, cut:])
    o1, s1 = oracle.run(a(q), a(k), a(v), a(g), a(b), a(w), S0, form=form, C=4)
    o2, s2 = oracle.run(z(q), z(k), z(v), z(g), z(b), z(w), s1, form=form, C=4)
    assert pins.rel(np.concatenate([o1, o2], axis=1), o) < 1e-12 and pins.rel(s2, s) < 1e-12


@pytest.mark.parametrize("form", ["recurrent", "literal", "chunked"])
def test_empty_sequence(form):
    q, k, v, g, b, w, S0 = pins.rand_problem(25, T=0, dk=3, dv=2)
    o, s = oracle.run(q, k, v, g, b, w, S0, form=form)
    assert o.shape[1] == 0 and np.array_equal(s, S0)


@pytest.mark.parametrize("form", ["recurrent", "literal", "chunked"])
def test_full_reset_forgets_the_past(form):
    """alpha_t = 0 on every key channel erases all memory: later outputs ignore earlier tokens."""
    q, k, v, g, b, w, S0 = pins.rand_problem(26, T=12, dk=4, dv=3)
    t = 5
    g[:, t] = -np.inf
    o, s = oracle.run(q, k, v, g, b, w, S0, form=form, C=4)
    q2, k2, v2, g2, b2, w2, _ = pins.rand_problem(27, T=12, dk=4, dv=3)
    for x, y in ((q, q2), (k, k2), (v, v2), (b, b2), (w, w2)):
        y[:, t:] = x[:, t:]
    g2[:, t:] = g[:, t:]
    o2, s2 = oracle.run(q2, k2, v2, g2, b2, w2, None, form=form, C=4)
    assert pins.rel(o2[:, t:], o[:, t:]) < 1e-13 and pins.rel(s2, s) < 1e-13
    if form != "chunked":
        assert np.array_equal(o2[:, t:], o[:, t:])


def test_scale_multiplies_output_only():
    q, k, v, g, b, w, S0 = pins.rand_problem(28, T=7, dk=4, dv=3)
    o1, s1 = oracle.run(q, k, v, g, b, w, S0)
    o2, s2 = oracle.run(q, k, v, g, b, w, S0, scale=0.125)
    assert np.allclose(o2, 0.125 * o1, rtol=1e-15, atol=0) and np.array_equal(s1, s2)


def test_bad_arguments_rejected():
    q, k, v, g, b, w, S0 = pins.rand_problem(29, B=1, T=3, Hk=2, Hv=3, dk=2, dv=2)
    with pytest.raises(RuntimeError):
        oracle.run(q, k, v, g, b, w, S0)          # H_v not a multiple of H_k
