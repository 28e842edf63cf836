"""The fused mixer prologue and epilogue (GPU) against their fp64 oracle (oracle/mixer.py), conv
state chaining across calls, and the whole mixer (prologue -> chunked core -> epilogue) against the
oracles chained the same way."""
import numpy as np
import pytest

import oracle
import synth
from oracle import max_rel_err, mixer
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import gated_deltanet_mixer_gdn2_gb300 as mod

    return mod


def _raw(rng, B, T, Hk, Hv, dk, dv, dtype):
    r = lambda *s: synth.round_to(rng.standard_normal(s), dtype).astype(np.float64)
    xs = (r(B, T, Hk, dk), r(B, T, Hk, dk), r(B, T, Hv, dv))
    ws = tuple(0.5 * rng.standard_normal((n, 4)).astype(np.float32).astype(np.float64)
               for n in (Hk * dk, Hk * dk, Hv * dv))
    gates = (r(B, T, Hv, dk), r(B, T, Hv, dk), r(B, T, Hv, dv))
    states = tuple(rng.standard_normal((B, 3, n)).astype(np.float32).astype(np.float64)
                   for n in (Hk * dk, Hk * dk, Hv * dv))
    return xs, ws, gates, states


def _dev(a, dtype):
    return synth.to_torch(np.ascontiguousarray(a, dtype=np.float32), dtype, "cuda")


def _f32dev(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def _run_prologue(g, xs, ws, gates, states, dtype, neg, t0=0, t1=None):
    import torch

    sl = lambda a: a[:, t0:t1]
    xd = [_dev(sl(x), dtype) for x in xs]
    gd = [_dev(sl(a), dtype) for a in gates]
    outs = [torch.empty_like(xd[0]), torch.empty_like(xd[1]), torch.empty_like(xd[2]),
            torch.empty_like(gd[0]), torch.empty_like(gd[1]), torch.empty_like(gd[2])]
    g.gdn2_mixer_prologue(*xd, *(_f32dev(w) for w in ws), *gd, *outs, states=states, neg_eigval=neg)
    return outs


@pytest.mark.parametrize("dtype,d,neg", [("bf16", 128, False), ("bf16", 128, True), ("f32", 64, False),
                                         ("bf16", 256, False), ("f32", 16, True), ("bf16", 32, False)])
def test_prologue_parity(g, dtype, d, neg):
    import torch

    rng = np.random.default_rng(7 + d)
    B, T, Hk, Hv = 2, 70, 2, 4
    xs, ws, gates, states = _raw(rng, B, T, Hk, Hv, d, d, dtype)
    st_dev = [_f32dev(s) for s in states]
    outs = _run_prologue(g, xs, ws, gates, st_dev, dtype, neg)
    torch.cuda.synchronize()
    ref = mixer.prologue(*xs, *ws, *gates, states=states, neg_eigval=neg)
    tol = 1e-2 if dtype == "bf16" else 1e-5
    for name, got, want in zip("qkvgbw", outs, ref[:6]):
        e = max_rel_err(H.to_np(got), want)
        assert e < tol, (name, e)
    for got, want in zip(st_dev, ref[6]):
        assert np.array_equal(got.cpu().numpy().astype(np.float64), want)   # copies of stored samples


@pytest.mark.parametrize("B,T", [(3, 2), (1, 129), (2, 256)])
def test_prologue_tile_edges(g, B, T):
    """The conv works on 128-token tiles with a 3-sample halo: sequences shorter than the halo, one
    token past a tile, and whole tiles across several batch rows."""
    import torch

    rng = np.random.default_rng(100 + T)
    Hk, Hv, d = 1, 2, 128
    xs, ws, gates, states = _raw(rng, B, T, Hk, Hv, d, d, "bf16")
    outs = _run_prologue(g, xs, ws, gates, [_f32dev(s) for s in states], "bf16", False)
    torch.cuda.synchronize()
    ref = mixer.prologue(*xs, *ws, *gates, states=states)
    for name, got, want in zip("qkvgbw", outs, ref[:6]):
        assert max_rel_err(H.to_np(got), want) < 1e-2, (name, T)


def test_prologue_state_chaining_is_exact(g):
    """One call over 70 tokens equals calls over 33, 1 and 36 tokens that carry the conv state."""
    import torch

    rng = np.random.default_rng(11)
    B, T, Hk, Hv, d = 2, 70, 1, 2, 128
    xs, ws, gates, states = _raw(rng, B, T, Hk, Hv, d, d, "bf16")
    full = _run_prologue(g, xs, ws, gates, [_f32dev(s) for s in states], "bf16", False)
    st = [_f32dev(s) for s in states]
    parts = [_run_prologue(g, xs, ws, gates, st, "bf16", False, a, b) for a, b in ((0, 33), (33, 34), (34, 70))]
    torch.cuda.synchronize()
    for i in range(6):
        joined = torch.cat([p[i] for p in parts], dim=1)
        assert torch.equal(joined, full[i]), "qkvgbw"[i]


@pytest.mark.parametrize("dtype,d", [("bf16", 128), ("f32", 32)])
def test_epilogue_parity(g, dtype, d):
    import torch

    rng = np.random.default_rng(13)
    B, T, Hv = 2, 37, 3
    o = synth.round_to(rng.standard_normal((B, T, Hv, d)), dtype).astype(np.float64)
    z = synth.round_to(rng.standard_normal((B, T, Hv, d)), dtype).astype(np.float64)
    wt = rng.uniform(0.5, 1.5, d).astype(np.float32).astype(np.float64)
    y = torch.empty_like(_dev(o, dtype))
    g.gdn2_mixer_epilogue(_dev(o, dtype), _dev(z, dtype), _f32dev(wt), y)
    torch.cuda.synchronize()
    e = max_rel_err(H.to_np(y), mixer.epilogue(o, z, wt))
    assert e < (1e-2 if dtype == "bf16" else 1e-5), e


def test_whole_mixer_against_chained_oracles(g):
    """prologue -> gdn2_chunk_fwd -> epilogue on the GPU against mixer.prologue -> oracle.run ->
    mixer.epilogue (the core oracle reads the GPU prologue's stored outputs)."""
    import torch

    rng = np.random.default_rng(17)
    B, T, Hk, Hv, d = 1, 150, 2, 4, 128
    xs, ws, gates, _ = _raw(rng, B, T, Hk, Hv, d, d, "bf16")
    q, k, v, gg, b, w = _run_prologue(g, xs, ws, gates, None, "bf16", False)
    o, st = g.chunk_fwd(q, k, v, gg, b, w, None)
    z = synth.round_to(rng.standard_normal((B, T, Hv, d)), "bf16").astype(np.float64)
    wt = rng.uniform(0.5, 1.5, d).astype(np.float32).astype(np.float64)
    y = torch.empty_like(o)
    g.gdn2_mixer_epilogue(o, _dev(z, "bf16"), _f32dev(wt), y)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    stored = [H.to_np(t) for t in (q, k, v, gg, b, w)]
    ref_pro = mixer.prologue(*xs, *ws, *gates)
    for name, got, want in zip("qkvgbw", stored, ref_pro[:6]):
        assert max_rel_err(got, want) < 1e-2, name
    o_ref, _ = oracle.run(*stored, None)
    y_ref = mixer.epilogue(o_ref, z, wt)
    assert max_rel_err(H.to_np(o), o_ref) < H.BF16_TOL
    assert max_rel_err(H.to_np(y), y_ref) < H.BF16_TOL
