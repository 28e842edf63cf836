"""Gradients of the core on the GPU against the fp64 autograd oracle (oracle/backward.py): the
chunked path (gdn2_backward) and the per-token recurrent path (gdn2_backward_recurrent), bf16 and
fp32 token tensors, grouped heads, a ragged last chunk, an initial state and an upstream
final-state gradient; at lengths the oracle cannot reach, the two paths against each other."""
import dataclasses

import numpy as np
import pytest

import synth
from oracle import backward as oback
from oracle import max_rel_err
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

TOL = {"bf16": 2e-2, "f32": 1e-4}


@pytest.fixture(scope="module")
def g():
    import gated_deltanet_mixer_gdn2_gb300 as mod

    return mod


@pytest.mark.parametrize("recurrent", [False, True], ids=["chunked", "recurrent"])
@pytest.mark.parametrize("dtype,T,with_ds", [("bf16", 77, True), ("f32", 45, False), ("f32", 64, True), ("f32", 5, True)])
def test_backward_parity(g, dtype, T, with_ds, recurrent):
    import torch

    wl = synth.Workload("bwd", B=2, T=T, Hk=1, Hv=2, dk=128, dv=128, dtype=dtype, seed=21 + T, s0_std=0.02)
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(5)
    d_o = synth.round_to(rng.standard_normal((2, T, 2, 128)), dtype).astype(np.float64)
    ds_t = (0.1 * rng.standard_normal((2, 2, 128, 128))).astype(np.float32).astype(np.float64) if with_ds else None
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a), dtype, "cuda")
    ts = [dev(getattr(inp, n)) for n in ("q", "k", "v", "g", "b", "w")]
    s0 = H.state_to_device(inp.s0)
    dsd = H.state_to_device(ds_t) if with_ds else None
    outs = g.backward(*ts, dev(d_o), s0, dsd, recurrent=recurrent)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    ref = oback.gradients(inp.q, inp.k, inp.v, inp.g, inp.b, inp.w, inp.s0, d_o, ds_t)
    for name, got in zip(("dq", "dk", "dv", "dg", "db", "dw", "ds0"), outs):
        e = max_rel_err(H.to_np(got), ref[name])
        assert e < TOL[dtype], (name, e)


def test_backward_empty_sequence_passes_the_state_gradient(g):
    import torch

    x = torch.zeros((1, 0, 1, 128), dtype=torch.bfloat16, device="cuda")
    ds = torch.randn((1, 1, 128, 128), device="cuda")
    ds0 = torch.empty_like(ds)
    g.gdn2_backward(x, x, x, x, x, x, x, x, x, x, x, x, x, None, ds, ds0)
    torch.cuda.synchronize()
    assert torch.equal(ds0, ds)


@pytest.mark.parametrize("T,Hk,Hv", [(2050, 1, 2), (700, 2, 4)])
def test_backward_chunked_matches_recurrent_on_long_sequences(g, T, Hk, Hv):
    """Two fp32 computations of the same gradients that share no arithmetic: they agree to the
    rounding of fp32 sums over thousands of tokens."""
    import torch

    wl = synth.Workload("bwd-long", B=1, T=T, Hk=Hk, Hv=Hv, dk=128, dv=128, dtype="f32", seed=3 + T, s0_std=0.02)
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(T)
    d_o = rng.standard_normal((1, T, Hv, 128)).astype(np.float32)
    ds_t = (0.1 * rng.standard_normal((1, Hv, 128, 128))).astype(np.float32)
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a), "f32", "cuda")
    ts = [dev(getattr(inp, n)) for n in ("q", "k", "v", "g", "b", "w")]
    s0, dsd = H.state_to_device(inp.s0), H.state_to_device(ds_t)
    a = g.backward(*ts, dev(d_o), s0, dsd)
    r = g.backward(*ts, dev(d_o), s0, dsd, recurrent=True)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    for name, x, y in zip(("dq", "dk", "dv", "dg", "db", "dw", "ds0"), a, r):
        assert torch.isfinite(x).all(), name
        e = max_rel_err(H.to_np(x), H.to_np(y).astype(np.float64))
        assert e < 1e-3, (name, e)


@pytest.mark.parametrize("decay", ["strong", "none", "reset", "bursts"])
def test_backward_extreme_decays(g, decay):
    """Gates far from the synthetic recipe: log-decays near -3 per token (products of the pair factors
    underflow inside a 32-token chunk), no decay at all (every factor is 1), full resets (alpha = 0,
    g = -inf, at random positions and on whole tokens) and runs of g = -20."""
    import torch

    T = 70
    rng = np.random.default_rng(11)
    if decay in ("reset", "bursts"):
        wl = synth.Workload("bwd-decay", B=1, T=T, Hk=1, Hv=2, dk=128, dv=128, dtype="f32", seed=7, s0_std=0.02,
                            decay=decay)
        inp = synth.make_inputs(wl)
    else:
        wl = synth.Workload("bwd-decay", B=1, T=T, Hk=1, Hv=2, dk=128, dv=128, dtype="f32", seed=7, s0_std=0.02)
        inp = synth.make_inputs(wl)
        if decay == "strong":
            gg = -np.log1p(np.exp(rng.normal(3.0, 1.0, inp.g.shape)))
        else:
            gg = np.zeros(inp.g.shape)
        inp = dataclasses.replace(inp, g=gg.astype(np.float32).astype(np.float64))
    d_o = rng.standard_normal((1, T, 2, 128)).astype(np.float32).astype(np.float64)
    ds_t = (0.1 * rng.standard_normal((1, 2, 128, 128))).astype(np.float32).astype(np.float64)
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a), "f32", "cuda")
    ts = [dev(getattr(inp, n)) for n in ("q", "k", "v", "g", "b", "w")]
    outs = g.backward(*ts, dev(d_o), H.state_to_device(inp.s0), H.state_to_device(ds_t))
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    ref = oback.gradients(inp.q, inp.k, inp.v, inp.g, inp.b, inp.w, inp.s0, d_o, ds_t)
    for name, got in zip(("dq", "dk", "dv", "dg", "db", "dw", "ds0"), outs):
        x = H.to_np(got)
        assert np.isfinite(x).all(), name
        e = max_rel_err(x, ref[name])
        assert e < TOL["f32"], (name, e)


@pytest.mark.parametrize("decay", ["standard", "strong", "bursts", "reset"])
@pytest.mark.parametrize("T,Hk,Hv", [(150, 1, 2), (130, 2, 4)])
def test_backward_bf16_decay_domain(g, decay, T, Hk, Hv):
    """The bf16 path (tensor cores, 64-token chunks) over the decay domain: standard gates take the
    anchored pair terms on the tensor cores, strong decay (a chunk spans ~200 in log-decay) and
    whole-token resets take the exact CUDA-core pair terms, bursts of g = -20 mix both kinds of chunk
    in one call; grouped heads, a ragged last chunk, an initial state and dS_T."""
    import torch

    wl = synth.Workload("bwd-bf16", B=2, T=T, Hk=Hk, Hv=Hv, dk=128, dv=128, dtype="bf16", seed=40 + T, s0_std=0.02,
                        decay=decay)
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(T + Hv)
    d_o = synth.round_to(rng.standard_normal((2, T, Hv, 128)), "bf16").astype(np.float64)
    ds_t = (0.1 * rng.standard_normal((2, Hv, 128, 128))).astype(np.float32).astype(np.float64)
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a), "bf16", "cuda")
    ts = [dev(getattr(inp, n)) for n in ("q", "k", "v", "g", "b", "w")]
    outs = g.backward(*ts, dev(d_o), H.state_to_device(inp.s0), H.state_to_device(ds_t))
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    ref = oback.gradients(inp.q, inp.k, inp.v, inp.g, inp.b, inp.w, inp.s0, d_o, ds_t)
    for name, got in zip(("dq", "dk", "dv", "dg", "db", "dw", "ds0"), outs):
        x = H.to_np(got)
        assert np.isfinite(x).all(), name
        e = max_rel_err(x, ref[name])
        print(f"{name}: {e:.2e}")
        assert e < TOL["bf16"], (name, e)


@pytest.mark.parametrize("T,Hk,Hv", [(1, 1, 1), (64, 2, 2), (65, 1, 3), (200, 3, 3)])
def test_backward_bf16_edge_lengths(g, T, Hk, Hv):
    """The bf16 path at a single token, exactly one chunk, one chunk and one token, and ungrouped heads
    (H_k = H_v, the key-head sum over one value head), against the oracle."""
    import torch

    wl = synth.Workload("bwd-edge", B=2, T=T, Hk=Hk, Hv=Hv, dk=128, dv=128, dtype="bf16", seed=60 + T + Hv,
                        s0_std=0.02)
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(T)
    d_o = synth.round_to(rng.standard_normal((2, T, Hv, 128)), "bf16").astype(np.float64)
    ds_t = (0.1 * rng.standard_normal((2, Hv, 128, 128))).astype(np.float32).astype(np.float64)
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a), "bf16", "cuda")
    ts = [dev(getattr(inp, n)) for n in ("q", "k", "v", "g", "b", "w")]
    outs = g.backward(*ts, dev(d_o), H.state_to_device(inp.s0), H.state_to_device(ds_t), scale=0.5)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    ref = oback.gradients(inp.q, inp.k, inp.v, inp.g, inp.b, inp.w, inp.s0, d_o, ds_t, scale=0.5)
    for name, got in zip(("dq", "dk", "dv", "dg", "db", "dw", "ds0"), outs):
        x = H.to_np(got)
        assert np.isfinite(x).all(), name
        e = max_rel_err(x, ref[name])
        assert e < TOL["bf16"], (name, e)


@pytest.mark.parametrize("dk,dv,decay", [(64, 64, "standard"), (64, 128, "standard"), (128, 64, "standard"),
                                         (64, 64, "strong")])
def test_backward_bf16_head_dim_64(g, dk, dv, decay):
    """head_dim 64 (the pages' quick-start size) on the tensor-core backward: the 64-wide channels or
    columns read as zero-padded 128; grouped heads, a ragged last chunk, an initial state and dS_T."""
    import torch

    T, Hk, Hv = 100, 1, 2
    wl = synth.Workload("bwd-hd64", B=2, T=T, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype="bf16", seed=70 + dk + dv,
                        s0_std=0.02, decay=decay)
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(dk * dv)
    d_o = synth.round_to(rng.standard_normal((2, T, Hv, dv)), "bf16").astype(np.float64)
    ds_t = (0.1 * rng.standard_normal((2, Hv, dk, dv))).astype(np.float32).astype(np.float64)
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a), "bf16", "cuda")
    ts = [dev(getattr(inp, n)) for n in ("q", "k", "v", "g", "b", "w")]
    outs = g.backward(*ts, dev(d_o), H.state_to_device(inp.s0), H.state_to_device(ds_t))
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    ref = oback.gradients(inp.q, inp.k, inp.v, inp.g, inp.b, inp.w, inp.s0, d_o, ds_t)
    for name, got in zip(("dq", "dk", "dv", "dg", "db", "dw", "ds0"), outs):
        x = H.to_np(got)
        assert x.shape == ref[name].shape, name
        assert np.isfinite(x).all(), name
        e = max_rel_err(x, ref[name])
        assert e < TOL["bf16"], (name, e)


def test_backward_chunked_matches_recurrent_at_the_bench_shape(g):
    """The bench workload's shapes (B 2, T 32768, H_k 16, H_v 32, bf16 tensors): the chunked path against
    the per-token recurrent path, two fp32 computations that share no arithmetic; errors are normwise
    over each whole output, computed on the device."""
    import torch

    B, T, Hk, Hv, d = 2, 32768, 16, 32, 128
    gen = torch.Generator(device="cuda")
    gen.manual_seed(2024)
    rnd = lambda *s: torch.randn(s, generator=gen, device="cuda")
    bf = torch.bfloat16
    q = torch.nn.functional.normalize(rnd(B, T, Hk, d), dim=-1).to(bf)
    k = torch.nn.functional.normalize(rnd(B, T, Hk, d), dim=-1).to(bf)
    v, d_o = rnd(B, T, Hv, d).to(bf), rnd(B, T, Hv, d).to(bf)
    gg = (-torch.nn.functional.softplus(rnd(B, T, Hv, d))).to(bf)
    bb = torch.sigmoid(rnd(B, T, Hv, d)).to(bf)
    ww = torch.sigmoid(rnd(B, T, Hv, d)).to(bf)
    s0 = 0.02 * rnd(B, Hv, d, d)
    ds_t = 0.1 * rnd(B, Hv, d, d)
    a = g.backward(q, k, v, gg, bb, ww, d_o, s0, ds_t)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    r = g.backward(q, k, v, gg, bb, ww, d_o, s0, ds_t, recurrent=True)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    for name, x, y in zip(("dq", "dk", "dv", "dg", "db", "dw", "ds0"), a, r):
        x, y = x.float(), y.float()
        assert torch.isfinite(x).all(), name
        e = ((x - y).abs().max() / y.abs().max()).item()
        print(f"{name}: {e:.2e}")
        assert e < 1e-2, (name, e)


def test_backward_in_a_cuda_graph(g):
    """The chunked backward, captured in a CUDA graph on a side stream of the caller's and replayed,
    gives the same gradients as the eager call."""
    import torch

    T = 100
    wl = synth.Workload("bwd-graph", B=1, T=T, Hk=1, Hv=2, dk=128, dv=128, dtype="bf16", seed=9, s0_std=0.02)
    inp = synth.make_inputs(wl)
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a), "bf16", "cuda")
    ts = [dev(getattr(inp, n)) for n in ("q", "k", "v", "g", "b", "w")]
    d_o = dev(np.random.default_rng(1).standard_normal((1, T, 2, 128)))
    s0 = H.state_to_device(inp.s0)
    eager = g.backward(*ts, d_o, s0)
    torch.cuda.synchronize()
    outs = [torch.empty_like(t) for t in ts]
    ds0 = torch.empty_like(s0)
    ws = torch.empty(g.lib.gdn2_backward_workspace_size(1, T, 1, 2, 128, 128, g.GDN2_BF16), dtype=torch.uint8,
                     device="cuda")
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(stream):  # warm-up outside the capture
        g.gdn2_backward(*ts, d_o, *outs, s0, None, ds0, workspace=ws, stream=stream)
    torch.cuda.current_stream().wait_stream(stream)
    torch.cuda.synchronize()
    for o in outs:
        o.zero_()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        g.gdn2_backward(*ts, d_o, *outs, s0, None, ds0, workspace=ws, stream=torch.cuda.current_stream())
    graph.replay()
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    for name, x, y in zip(("dq", "dk", "dv", "dg", "db", "dw", "ds0"), (*outs, ds0), eager):
        assert torch.equal(x, y), name


_CANARY = 4096  # elements of sentinel after each gradient output


@pytest.mark.parametrize("T,dk,dv", [(77, 128, 128), (130, 64, 128), (64, 128, 64)])
def test_backward_writes_stay_in_bounds(g, T, dk, dv):
    """The tensor-core backward writes dq, dk, db, dg, dv and dw through tensor maps clipped at T and at
    d_k / d_v: canary elements after every gradient and after dS0 stay untouched (ragged last chunk,
    64-wide channels or columns), and the gradients match the oracle."""
    import torch

    wl = synth.Workload("bwd", B=2, T=T, Hk=1, Hv=2, dk=dk, dv=dv, dtype="bf16", seed=90 + T, s0_std=0.02)
    inp = synth.make_inputs(wl)
    rng = np.random.default_rng(T)
    d_o = synth.round_to(rng.standard_normal((2, T, 2, dv)), "bf16").astype(np.float64)
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a), "bf16", "cuda")
    ts = [dev(getattr(inp, n)) for n in ("q", "k", "v", "g", "b", "w")]

    def canary(shape, dtype):
        n = int(np.prod(shape))
        buf = torch.full((n + _CANARY,), -7.0, dtype=dtype, device="cuda")
        return buf, buf[:n].view(shape)

    bf = torch.bfloat16
    shapes = {"dq": (2, T, 1, dk), "dk": (2, T, 1, dk), "dv": (2, T, 2, dv), "dg": (2, T, 2, dk),
              "db": (2, T, 2, dk), "dw": (2, T, 2, dv)}
    bufs = {name: canary(shp, bf) for name, shp in shapes.items()}
    ds0_buf, ds0 = canary((2, 2, dk, dv), torch.float32)
    g.gdn2_backward(*ts, dev(d_o), *(bufs[n][1] for n in ("dq", "dk", "dv", "dg", "db", "dw")),
                    H.state_to_device(inp.s0), None, ds0)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    for name, (buf, t) in list(bufs.items()) + [("ds0", (ds0_buf, ds0))]:
        assert bool((buf[t.numel():] == -7.0).all()), f"{name} canary overwritten"
    ref = oback.gradients(inp.q, inp.k, inp.v, inp.g, inp.b, inp.w, inp.s0, d_o, None)
    for name in ("dq", "dk", "dv", "dg", "db", "dw"):
        e = max_rel_err(H.to_np(bufs[name][1]), ref[name])
        assert e < TOL["bf16"], (name, e)
    assert max_rel_err(ds0.cpu().numpy(), ref["ds0"]) < TOL["bf16"]
