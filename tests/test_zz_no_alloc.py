"""gdn2_chunk_fwd_noalloc against gdn2_chunk_fwd (GPU).

Some callers cannot allocate device memory (their host framework owns the allocator, or their
serving loop must not call cudaMalloc / cudaFree, which can block or synchronise the device), so
the library offers a chunked forward that uses its own fixed 32 MiB device array instead of a
caller workspace. This test calls that entry point directly through the C ABI, twice in a row with
different problems, and checks each result against the workspace entry point on the same inputs
and against the fp64 oracle (same tolerance as the parity tests). It lives in a file of its own that
pytest collects last.
"""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


def _noalloc(g, q, k, v, gg, b, w, o, s0, sT, C):
    B, T, Hk, dk = q.shape
    Hv, dv = v.shape[2], v.shape[3]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    import torch

    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return g.lib.gdn2_chunk_fwd_noalloc(p(q), p(k), p(v), p(gg), p(b), p(w), p(s0), p(sT), p(o), B, T, Hk, Hv, dk,
                                        dv, C, 1.0, g._dtype_code(q), stream)


@pytest.mark.parametrize("first,second", [("bf16", "bf16"), ("f32", "bf16")])
def test_noalloc_matches_workspace_entry_point(first, second):
    import torch

    import gated_deltanet_mixer_gdn2_gb300 as g

    shapes = {"bf16": [dict(B=2, T=1500, Hk=2, Hv=4, dk=128, dv=128, C=64, seed=21, s0_std=0.02),
                       dict(B=1, T=2000, Hk=4, Hv=8, dk=128, dv=128, C=64, seed=22, s0_std=0.0)],
              "f32": [dict(B=1, T=300, Hk=2, Hv=4, dk=64, dv=64, C=32, seed=23, s0_std=0.02)]}
    for call, dtype in enumerate((first, second)):
        kw = shapes[dtype][min(call, len(shapes[dtype]) - 1)]
        wl = synth.Workload("noalloc", dtype=dtype, **kw)
        inp = synth.make_inputs(wl)
        q, k, v, gg, b, w = H.upload(inp, 0, wl.T)
        s0 = H.state_to_device(inp.s0)
        o_ref = torch.empty_like(v)
        s_ref = torch.empty((wl.B, wl.Hv, wl.dk, wl.dv), dtype=torch.float32, device="cuda")
        g.gdn2_chunk_fwd(q, k, v, gg, b, w, o_ref, s0, s_ref, C=wl.C)
        o = torch.full_like(v, float("nan"))
        sT = torch.full_like(s_ref, float("nan"))
        st = _noalloc(g, q, k, v, gg, b, w, o, s0, sT, wl.C)
        assert st == g.GDN2_OK, g.status_string(st)
        torch.cuda.synchronize()
        assert g.gdn2_last_device_status() == g.GDN2_OK
        tol = H.tol_for(dtype)
        assert oracle.max_rel_err(H.to_np(o), H.to_np(o_ref)) <= tol
        assert oracle.max_rel_err(sT.cpu().numpy(), s_ref.cpu().numpy()) <= tol
        assert np.isfinite(H.to_np(o)).all()
        o_or, s_or = oracle.run_inputs(inp)
        H.check("o (no-alloc) vs oracle", H.to_np(o), o_or, tol)
        H.check("state (no-alloc) vs oracle", sT.cpu().numpy(), s_or, tol, head_axis=1)


def test_noalloc_rejects_problems_beyond_its_array():
    import torch

    import gated_deltanet_mixer_gdn2_gb300 as g

    x = torch.empty(16, dtype=torch.bfloat16, device="cuda")
    p = ctypes.c_void_p(x.data_ptr())
    # 2 x 32768 tokens, 32 value heads: 2.9 GB of workspace, far beyond 32 MiB
    st = g.lib.gdn2_chunk_fwd_noalloc(p, p, p, p, p, p, None, None, p, 2, 32768, 16, 32, 128, 128, 64, 1.0,
                                      g.GDN2_BF16, None)
    assert st == g.GDN2_ERR_WORKSPACE
