"""The host-streaming chunked forward equals one device call on the same inputs (segments chain the
state exactly, so the results agree to rounding of the segment boundaries)."""
import numpy as np
import pytest

import synth
from oracle import max_rel_err
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("T,segment_tokens", [(1000, 192), (3000, 1024)])
def test_segments_match_one_call(T, segment_tokens):
    import torch

    import gated_deltanet_mixer_gdn2_gb300 as g
    from gated_deltanet_mixer_gdn2_gb300.host_stream import chunk_fwd_from_host

    wl = synth.Workload("hs", B=2, T=T, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", seed=3, s0_std=0.02)
    inp = synth.make_inputs(wl)
    host = [synth.to_torch(np.ascontiguousarray(getattr(inp, n)), "bf16", "cpu").pin_memory()
            for n in ("q", "k", "v", "g", "b", "w")]
    o_h = torch.empty((2, T, 4, 128), dtype=torch.bfloat16).pin_memory()
    s0 = H.state_to_device(inp.s0)
    # (1000, 192): 6 segments, the last one ragged; (3000, 1024): 512, 1024, 952, 512 (ramp + ragged middle)
    st = chunk_fwd_from_host(*host, o_h, s0, segment_tokens=segment_tokens)
    torch.cuda.synchronize()
    o_ref, s_ref = g.chunk_fwd(*(t.cuda() for t in host), s0)
    torch.cuda.synchronize()
    assert max_rel_err(o_h.float().numpy(), H.to_np(o_ref)) < 1e-2
    assert max_rel_err(st.cpu().numpy(), s_ref.cpu().numpy()) < 1e-2
