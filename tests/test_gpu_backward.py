"""Gradients of the core on the GPU (gdn2_backward) against the fp64 autograd oracle
(oracle/backward.py): bf16 and fp32 token tensors, grouped heads, a ragged tail of the 32-token
recompute stretches, an initial state and an upstream final-state gradient."""
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


@pytest.mark.parametrize("dtype,T,with_ds", [("bf16", 77, True), ("f32", 45, False)])
def test_backward_parity(g, dtype, T, with_ds):
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
    outs = g.backward(*ts, dev(d_o), s0, dsd)
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
