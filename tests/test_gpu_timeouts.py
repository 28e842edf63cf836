"""Bounded waits give up with a status, not a hang, on the backward, the streaming decode kernel and
the persistent fused decode step: with a zero wait budget each call reports GDN2_ERR_TIMEOUT through
the device status word and returns, the device stays usable, and the same path with the default
budget is then correct against the oracle (the chunked forward's case is in test_gpu_parity.py)."""
import numpy as np
import pytest

import synth
from tests import gpu_helpers as H
from tests.test_gpu_backward import test_backward_parity as _backward_parity
from tests.test_gpu_decode_variants import test_streaming_kernel_tokens_and_state_types as _stream_parity
from tests.test_gpu_mixer_step import _chained as _mixer_step_chained

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import gated_deltanet_mixer_gdn2_gb300 as mod

    mod.gdn2_set_wait_limit(-1)
    return mod


def _times_out(g, call):
    g.gdn2_set_wait_limit(0)
    try:
        call()
        assert g.gdn2_last_device_status() == g.GDN2_ERR_TIMEOUT
    finally:
        g.gdn2_set_wait_limit(-1)
    assert g.gdn2_last_device_status() == g.GDN2_OK  # the status word was read and cleared


def _dev(a, dtype):
    return synth.to_torch(np.ascontiguousarray(a), dtype, "cuda")


def test_backward_timeout_then_correct(g):
    import torch

    wl = synth.Workload("t", B=1, T=130, Hk=1, Hv=2, dk=128, dv=128, dtype="bf16", seed=3, s0_std=0.02)
    inp = synth.make_inputs(wl)
    ts = [_dev(getattr(inp, n), "bf16") for n in ("q", "k", "v", "g", "b", "w")]
    d_o = _dev(np.random.default_rng(3).standard_normal((1, 130, 2, 128)), "bf16")
    _times_out(g, lambda: (g.backward(*ts, d_o, H.state_to_device(inp.s0), None), torch.cuda.synchronize()))
    _backward_parity(g, "bf16", 77, True, False)


@pytest.mark.parametrize("N", [1, 4])
def test_streaming_decode_timeout_then_correct(g, N):
    """160 x 4 = 640 heads: the streaming kernel (one token, or four with the state held between them)."""
    import torch

    wl = synth.Workload("t", B=160, T=N, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", seed=80 + N, s0_std=0.02)
    inp = synth.make_inputs(wl)
    q, k, v, gg, b, w = (_dev(getattr(inp, n), "bf16") for n in ("q", "k", "v", "g", "b", "w"))
    st = H.state_to_device(inp.s0)
    o = torch.empty_like(v)
    _times_out(g, lambda: (g.gdn2_recurrent_update(q, k, v, gg, b, w, st, o), torch.cuda.synchronize()))
    _stream_parity(g, N, "f32", "bf16")


def test_fused_step_timeout_then_correct(g):
    """16 x 48 value heads: the persistent ring form of the fused decode step."""
    import torch

    B, Hk, Hv, d = 16, 16, 48, 128
    rng = np.random.default_rng(9)
    r = lambda *s: _dev(rng.standard_normal(s), "bf16")
    f32 = lambda *s: torch.from_numpy(rng.standard_normal(s).astype(np.float32)).cuda()
    xq, xk, xv = r(B, Hk, d), r(B, Hk, d), r(B, Hv, d)
    ag, ab, aw, z = r(B, Hv, d), r(B, Hv, d), r(B, Hv, d), r(B, Hv, d)
    cw = [0.5 * f32(n, 4) for n in (Hk * d, Hk * d, Hv * d)]
    cs = [f32(B, 3, n) for n in (Hk * d, Hk * d, Hv * d)]
    st = 0.02 * f32(B, Hv, d, d)
    y = torch.empty_like(z)
    _times_out(g, lambda: (g.gdn2_mixer_decode_step(xq, xk, xv, *cw, ag, ab, aw, st, z, torch.ones(d, device="cuda"),
                                                    y, states=tuple(cs)), torch.cuda.synchronize()))
    _mixer_step_chained(g, "bf16", B, 2, Hk, Hv, d, d, False, True, 11)
