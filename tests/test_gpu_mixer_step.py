"""The one-launch decode step of the whole mixer (gdn2_mixer_decode_step) against the fp64 oracles
chained token by token (mixer.prologue with T = 1 -> oracle.run -> mixer.epilogue), and against the
separate GPU entry points (gdn2_mixer_prologue -> gdn2_recurrent_step -> gdn2_mixer_epilogue)."""
import numpy as np
import pytest

import oracle
import synth
from oracle import mixer
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import gated_deltanet_mixer_gdn2_gb300 as mod

    return mod


def _problem(rng, B, N, Hk, Hv, dk, dv, dtype):
    r = lambda *s: synth.round_to(rng.standard_normal(s), dtype).astype(np.float64)
    xs = (r(B, N, Hk, dk), r(B, N, Hk, dk), r(B, N, Hv, dv))
    ws = tuple(0.5 * rng.standard_normal((n, 4)).astype(np.float32).astype(np.float64)
               for n in (Hk * dk, Hk * dk, Hv * dv))
    gates = (r(B, N, Hv, dk), r(B, N, Hv, dk), r(B, N, Hv, dv))
    conv_states = tuple(rng.standard_normal((B, 3, n)).astype(np.float32).astype(np.float64)
                        for n in (Hk * dk, Hk * dk, Hv * dv))
    s0 = (0.02 * rng.standard_normal((B, Hv, dk, dv))).astype(np.float32).astype(np.float64)
    z = r(B, N, Hv, dv)
    wt = rng.uniform(0.5, 1.5, dv).astype(np.float32).astype(np.float64)
    return xs, ws, gates, conv_states, s0, z, wt


def _f32dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _chained(g, dtype, B, N, Hk, Hv, dk, dv, neg, carry, seed):
    """N fused steps against the fp64 oracles chained token by token; carry = False passes no conv
    states (every token's conv sees zeros before it)."""
    import torch

    rng = np.random.default_rng(seed)
    scale = 0.7
    xs, ws, gates, cst, s0, z, wt = _problem(rng, B, N, Hk, Hv, dk, dv, dtype)
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a, dtype=np.float32), dtype, "cuda")
    conv_d = [_f32dev(w) for w in ws]
    cst_d = [_f32dev(s) for s in cst] if carry else [None, None, None]
    st_d = _f32dev(s0)
    w_d = _f32dev(wt)
    ys = []
    for t in range(N):
        tok = lambda a: dev(a[:, t])
        y = torch.empty_like(tok(z))
        g.gdn2_mixer_decode_step(*(tok(x) for x in xs), *conv_d, *(tok(a) for a in gates), st_d, tok(z), w_d, y,
                                 states=tuple(cst_d), neg_eigval=neg, scale=scale)
        ys.append(y)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    # the oracles, token by token, carrying the conv states and the core state
    S, cs, y_ref = s0, cst if carry else (None, None, None), []
    for t in range(N):
        sl = lambda a: a[:, t:t + 1]
        q, k, v, gg, b, w, ns = mixer.prologue(*(sl(x) for x in xs), *ws, *(sl(a) for a in gates), states=cs,
                                               neg_eigval=neg)
        if carry:
            cs = ns
        o, S = oracle.run(q, k, v, gg, b, w, S, scale=scale)
        y_ref.append(mixer.epilogue(o, sl(z), wt)[:, 0])
    tol = H.tol_for(dtype)
    print(H.check("y", H.to_np(torch.stack(ys, dim=1)), np.stack(y_ref, axis=1), tol),
          H.check("core state", st_d.cpu().numpy(), S, tol, head_axis=1))
    if carry:
        for got, want in zip(cst_d, cs):
            assert np.array_equal(got.cpu().numpy().astype(np.float64), want)  # conv states hold copies of samples


# groups of 1 to 8 value heads per key head run as thread-block clusters (one CTA per value head);
# larger groups (12) as one CTA per key head
@pytest.mark.parametrize("dtype,dk,dv,Hk,Hv,neg", [("bf16", 128, 128, 2, 4, False), ("bf16", 64, 64, 1, 3, True),
                                                   ("f32", 128, 64, 2, 2, False), ("f32", 64, 128, 1, 2, True),
                                                   ("f32", 64, 64, 1, 8, False), ("bf16", 64, 128, 1, 12, False)])
def test_decode_step_against_chained_oracles(g, dtype, dk, dv, Hk, Hv, neg):
    _chained(g, dtype, 3, 6, Hk, Hv, dk, dv, neg, True, dk + dv + Hv)


# the persistent form (d_k = d_v = 128, at least four value heads per SM): groups of 3, 12 and 1 value
# heads per key head, with and without carried conv states
@pytest.mark.parametrize("dtype,B,Hk,Hv,neg,carry", [("bf16", 16, 16, 48, False, True), ("f32", 14, 4, 48, True, True),
                                                     ("bf16", 20, 38, 38, False, False)])
def test_decode_step_persistent_against_chained_oracles(g, dtype, B, Hk, Hv, neg, carry):
    _chained(g, dtype, B, 3, Hk, Hv, 128, 128, neg, carry, B + Hk + Hv)


def test_decode_step_matches_separate_entry_points(g):
    """The fused step and the three separate launches on the same bf16 inputs (64 x 48 heads, the decode
    workload's shape): the fused step keeps q, k, v, the gates and o in fp32 where the separate path
    stores them in bf16, so the two agree to bf16 rounding."""
    import torch

    rng = np.random.default_rng(5)
    B, Hk, Hv, d = 64, 16, 48, 128
    xs, ws, gates, cst, s0, z, wt = _problem(rng, B, 1, Hk, Hv, d, d, "bf16")
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a, dtype=np.float32), "bf16", "cuda")
    x_d = [dev(x) for x in xs]
    a_d = [dev(a) for a in gates]
    conv_d = [_f32dev(w) for w in ws]
    # fused
    cst1 = [_f32dev(s) for s in cst]
    st1 = _f32dev(s0)
    y1 = torch.empty_like(dev(z[:, 0]))
    g.gdn2_mixer_decode_step(*(x[:, 0] for x in x_d), *conv_d, *(a[:, 0] for a in a_d), st1, dev(z[:, 0]),
                             _f32dev(wt), y1, states=cst1)
    # separate: prologue (T = 1) -> recurrent step -> epilogue
    cst2 = [_f32dev(s) for s in cst]
    st2 = _f32dev(s0)
    outs = [torch.empty_like(x_d[0]), torch.empty_like(x_d[1]), torch.empty_like(x_d[2]),
            torch.empty_like(a_d[0]), torch.empty_like(a_d[1]), torch.empty_like(a_d[2])]
    g.gdn2_mixer_prologue(*x_d, *conv_d, *a_d, *outs, states=cst2)
    o2 = g.recurrent_step(*(t[:, 0] for t in outs), st2)
    y2 = torch.empty_like(o2)
    g.gdn2_mixer_epilogue(o2[:, None], dev(z[:, 0])[:, None], _f32dev(wt), y2[:, None])
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    assert oracle.max_rel_err(H.to_np(y1), H.to_np(y2)) < H.BF16_TOL
    assert oracle.max_rel_err(st1.cpu().numpy(), st2.cpu().numpy()) < H.BF16_TOL
    for a, b in zip(cst1, cst2):
        assert torch.equal(a, b)
