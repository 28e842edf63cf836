"""GPU parity over the whole decay domain alpha in [0, 1] (burn-gdn2 docs, "Architecture": the
per-channel decay diag(alpha_t)), against the fp64 oracle on the same seeded inputs.

Decay recipes (synth.DECAYS): "strong" (g = -softplus(N(3,1)), a 64-token chunk spans ~195 in
log-decay), "bursts" (runs of 8 tokens at g = -20 in a few channels: chunks with and without a run),
"reset" (g = -inf, alpha = 0, at random (token, channel) positions and on whole tokens in the middle
of chunks). Tolerances as everywhere: 1e-4 for fp32 token inputs, 2e-2 for bf16, normwise per tensor
and per head.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu

UNIT_BYTES = 66048  # one (chunk, value head) unit of the tensor-core path's workspace


@pytest.fixture(scope="module")
def g():
    import gated_deltanet_mixer_gdn2_gb300 as mod

    mod.gdn2_set_wait_limit(-1)
    return mod


def _tc_run(g, inp, wl):
    """Tensor-core chunked forward with a workspace of our own; returns o, S_T and the number of
    units the exact kernel formed (the int32 after the units, documented in gdn2.h)."""
    import torch

    q, k, v, gg, b, w = H.upload(inp, 0, wl.T)
    s0 = H.state_to_device(inp.s0)
    need = g.gdn2_chunk_fwd_workspace_size(wl.B, wl.T, wl.Hk, wl.Hv, 128, 128, 64, g.GDN2_BF16, "tcgen05")
    ws = torch.empty(need, dtype=torch.uint8, device="cuda")
    o = torch.empty_like(v)
    sT = torch.empty((wl.B, wl.Hv, 128, 128), dtype=torch.float32, device="cuda")
    g.gdn2_chunk_fwd(q, k, v, gg, b, w, o, s0, sT, workspace=ws, path="tcgen05")
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    units = -(-wl.T // 64) * wl.B * wl.Hv
    n_exact = int(ws[units * UNIT_BYTES:units * UNIT_BYTES + 4].view(torch.int32).item())
    return H.to_np(o), sT.cpu().numpy(), n_exact, units


@pytest.mark.parametrize("decay", ["standard", "strong", "bursts", "reset"])
def test_tc_decay_domain(g, decay):
    wl = synth.Workload("t", B=2, T=300, Hk=1, Hv=2, dk=128, dv=128, dtype="bf16", seed=31, s0_std=0.02,
                        decay=decay)
    inp = synth.make_inputs(wl)
    o, sT, n_exact, units = _tc_run(g, inp, wl)
    o_ref, s_ref = oracle.run_inputs(inp)
    print(H.check("o", o, o_ref, H.BF16_TOL), "|", H.check("state", sT, s_ref, H.BF16_TOL, head_axis=1),
          f"| exact units {n_exact} of {units}")
    # which kernel formed the units: the anchored one for standard decays, the exact one for the
    # chunks whose log-decay spans more than the anchored operands hold
    if decay == "standard":
        assert n_exact == 0
    elif decay in ("strong", "reset"):
        assert n_exact == units
    else:
        assert 0 < n_exact < units


def test_tc_strong_decay_long(g):
    """2048 tokens, 4 value heads over 2 key heads, b in (0, 2), every chunk on the exact kernel."""
    wl = synth.Workload("t", B=1, T=2048, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", seed=32, s0_std=0.02,
                        neg_eigval=True, decay="strong")
    inp = synth.make_inputs(wl)
    o, sT, n_exact, units = _tc_run(g, inp, wl)
    o_ref, s_ref = oracle.run_inputs(inp)
    H.check("o", o, o_ref, H.BF16_TOL)
    H.check("state", sT, s_ref, H.BF16_TOL, head_axis=1)
    assert n_exact == units


def test_tc_reset_forgets_initial_state(g):
    """A whole-token reset (g = -inf on every channel) inside the first chunk: after it the output does
    not depend on S0 at all, exactly as the recurrence says."""
    wl = synth.Workload("t", B=1, T=128, Hk=1, Hv=1, dk=128, dv=128, dtype="bf16", seed=33, s0_std=0.5)
    inp = synth.make_inputs(wl)
    inp.g[:, 40] = -np.inf
    o1, s1, _, _ = _tc_run(g, inp, wl)
    inp2 = synth.Inputs(inp.dtype, inp.q, inp.k, inp.v, inp.g, inp.b, inp.w, inp.s0 * 0.0)
    o2, s2, _, _ = _tc_run(g, inp2, wl)
    assert np.array_equal(o1[:, 40:], o2[:, 40:])
    assert np.array_equal(s1, s2)
    o_ref, s_ref = oracle.run_inputs(inp)
    H.check("o", o1, o_ref, H.BF16_TOL)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("decay", ["strong", "bursts", "reset"])
@pytest.mark.parametrize("C,d", [(16, 64), (32, 128), (64, 64)])
def test_simt_decay_domain(g, dtype, decay, C, d):
    wl = synth.Workload("t", B=1, T=200, Hk=1, Hv=2, dk=d, dv=d, C=C, dtype=dtype, seed=34 + C, s0_std=0.02,
                        decay=decay)
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, C=C, path="simt")
    o_ref, s_ref = oracle.run_inputs(inp)
    tol = H.tol_for(dtype)
    print(H.check("o", o, o_ref, tol), "|", H.check("state", st.cpu().numpy(), s_ref, tol, head_axis=1))


@pytest.mark.parametrize("decay", ["strong", "reset"])
def test_decode_decay_domain(g, decay):
    wl = synth.Workload("t", B=3, T=0, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", seed=35, s0_std=0.02,
                        decode_steps=40, decay=decay)
    inp = synth.make_inputs(wl)
    st = H.state_to_device(inp.s0)
    o = H.run_decode(g, inp, st, 0, wl.decode_steps)
    o_ref, s_ref = oracle.run_inputs(inp)
    H.check("o", o, o_ref, H.BF16_TOL)
    H.check("state", st.cpu().numpy(), s_ref, H.BF16_TOL, head_axis=1)
