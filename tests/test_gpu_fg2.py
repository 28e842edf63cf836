"""FG^2-GDN on the GDN-2 core (GPU): gdn2_fg2_inputs writes the transformed inputs, then the chunked
forward and the multi-token recurrent update run unchanged; both are compared with the FG^2-GDN
oracle (oracle/fg2.py), which follows the FG^2 update directly. The erase gate b of the synthetic
workload serves as the per-channel rate beta (in (0, 1), one per value head and key channel)."""
import numpy as np
import pytest

import synth
from oracle import max_rel_err
from oracle.fg2 import fg2_recurrent
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import gated_deltanet_mixer_gdn2_gb300 as mod

    return mod


@pytest.mark.parametrize("T", [200])
def test_fg2_chunked_and_decode(g, T):
    import torch

    wl = synth.Workload("fg2", B=2, T=T, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", seed=5, s0_std=0.02,
                        decode_steps=8)
    inp = synth.make_inputs(wl, T=T + 8)
    beta = inp.b                                    # stored bf16 values in (0, 1)
    dev = "cuda"
    to = lambda a: synth.to_torch(np.ascontiguousarray(a), "bf16", dev)
    q, k, v, gg, bt = (to(x) for x in (inp.q, inp.k, inp.v, inp.g, beta))

    q2, k2, b2, w2 = g.fg2_inputs(q, k, bt)
    torch.cuda.synchronize()
    # the transform itself: q copied per value head, b = 1, w = sqrt(beta), k~ = sqrt(beta) . k
    qx = np.repeat(inp.q, 2, axis=2)
    kx = np.repeat(inp.k, 2, axis=2)
    assert np.array_equal(H.to_np(q2), qx)
    assert np.array_equal(H.to_np(b2), np.ones_like(beta))
    root = np.sqrt(beta)
    assert np.max(np.abs(H.to_np(w2) - root)) <= 2.0 ** -8 * np.max(root)
    assert np.max(np.abs(H.to_np(k2) - root * kx)) <= 2.0 ** -8 * np.max(np.abs(kx))

    # chunked forward over the first T tokens, then 8 decode tokens (N = 8 in one update call)
    s0 = H.state_to_device(inp.s0)
    sl = lambda t, a, b: t[:, a:b].contiguous()
    o, st = g.chunk_fwd(sl(q2, 0, T), sl(k2, 0, T), sl(v, 0, T), sl(gg, 0, T), sl(b2, 0, T), sl(w2, 0, T), s0)
    o_dec = torch.empty_like(sl(v, T, T + 8))
    g.gdn2_recurrent_update(sl(q2, T, T + 8), sl(k2, T, T + 8), sl(v, T, T + 8), sl(gg, T, T + 8),
                            sl(b2, T, T + 8), sl(w2, T, T + 8), st, o_dec)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK

    o_ref, s_ref = fg2_recurrent(inp.q, inp.k, inp.v, inp.g, beta, inp.s0)
    e_o = max_rel_err(H.to_np(o), o_ref[:, :T])
    e_d = max_rel_err(H.to_np(o_dec), o_ref[:, T:])
    e_s = max_rel_err(st.cpu().numpy(), s_ref)
    assert e_o < H.BF16_TOL and e_d < H.BF16_TOL and e_s < H.BF16_TOL, (e_o, e_d, e_s)


def test_fg2_argument_errors(g):
    import torch

    x = torch.zeros((1, 4, 1, 12), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.Gdn2Error):
        g.fg2_inputs(x, x, x)                       # d % 8
    y = torch.zeros((1, 4, 3, 16), dtype=torch.bfloat16, device="cuda")
    z = torch.zeros((1, 4, 4, 16), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(g.Gdn2Error):
        g.fg2_inputs(y, y, z)                       # H_v % H_k
