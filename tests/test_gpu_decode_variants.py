"""gdn2_recurrent_update against the fp64 oracle: several tokens per call, a slot map into a state
pool (with inactive rows), and bf16 state storage, on both the register and the streaming decode
kernels. Tolerances as in the parity tests (max normwise relative error 2e-2 for bf16 tokens)."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import gated_deltanet_mixer_gdn2_gb300 as mod

    return mod


def _dev(inp, names=("q", "k", "v", "g", "b", "w")):
    return tuple(synth.to_torch(np.ascontiguousarray(getattr(inp, n)), inp.dtype, "cuda") for n in names)


def _err(x, ref):
    return oracle.max_rel_err(x, ref)


@pytest.mark.parametrize("N", [1, 3, 8])
@pytest.mark.parametrize("dk,dv", [(128, 128), (64, 32)])
def test_multi_token_update(g, N, dk, dv):
    import torch

    wl = synth.Workload("t", B=2, T=N, Hk=2, Hv=4, dk=dk, dv=dv, seed=40 + N, s0_std=0.02)
    inp = synth.make_inputs(wl)
    q, k, v, gg, b, w = _dev(inp)
    st = H.state_to_device(inp.s0)
    o = torch.full_like(v, float("nan"))
    g.gdn2_recurrent_update(q, k, v, gg, b, w, st, o)
    torch.cuda.synchronize()
    o_ref, s_ref = oracle.run_inputs(inp)
    assert _err(H.to_np(o), o_ref) < H.BF16_TOL
    assert _err(st.cpu().numpy(), s_ref) < H.BF16_TOL


def test_multi_token_equals_repeated_steps(g):
    import torch

    wl = synth.Workload("t", B=3, T=5, Hk=1, Hv=2, dk=128, dv=128, seed=47, s0_std=0.02)
    inp = synth.make_inputs(wl)
    q, k, v, gg, b, w = _dev(inp)
    s1 = H.state_to_device(inp.s0)
    s2 = s1.clone()
    o1 = torch.empty_like(v)
    g.gdn2_recurrent_update(q, k, v, gg, b, w, s1, o1)
    o2 = H.run_decode(g, inp, s2, 0, wl.T)
    torch.cuda.synchronize()
    assert _err(H.to_np(o1), o2) < 1e-2
    assert _err(s1.cpu().numpy(), s2.cpu().numpy()) < 1e-5


@pytest.mark.parametrize("B,Hv,state_dt,N", [(4, 2, "f32", 1), (16, 48, "f32", 1), (16, 48, "bf16", 1), (4, 2, "bf16", 1),
                                              (16, 48, "f32", 3), (16, 48, "bf16", 4)])
def test_slot_map_and_inactive_rows(g, B, Hv, state_dt, N):
    """B * H_v = 768 heads takes the streaming kernel (one token, or several with the slot of an
    inactive head refilled at once); 8 heads the register kernel."""
    import torch

    wl = synth.Workload("t", B=B, T=N, Hk=Hv // 2 if Hv > 1 else 1, Hv=Hv, dk=128, dv=128, seed=50 + B + N,
                        s0_std=0.02)
    inp = synth.make_inputs(wl)
    n_slots = B + 3
    rng = np.random.default_rng(B)
    pool = (0.02 * rng.standard_normal((n_slots, Hv, 128, 128))).astype(np.float32)
    if state_dt == "bf16":
        pool = synth.round_to(pool.astype(np.float64), "bf16")
    slot_of = rng.permutation(n_slots)[:B].astype(np.int32)
    slot_of[1] = -1             # inactive
    slot_of[-1] = n_slots + 5   # out of range: inactive too
    q, k, v, gg, b, w = _dev(inp)
    tdt = torch.bfloat16 if state_dt == "bf16" else torch.float32
    pool_d = torch.from_numpy(pool).to("cuda").to(tdt)
    before = pool_d.clone()
    slots = torch.from_numpy(slot_of).to("cuda")
    o = torch.full_like(v, float("nan"))
    g.gdn2_recurrent_update(q, k, v, gg, b, w, pool_d, o, slots)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    o_np = H.to_np(o)
    after = pool_d.float().cpu().numpy()
    active = [i for i in range(B) if 0 <= slot_of[i] < n_slots]
    tol = H.BF16_TOL
    for i in active:
        sub = synth.Inputs(inp.dtype, *(np.ascontiguousarray(getattr(inp, n)[i:i + 1]) for n in ("q", "k", "v", "g", "b", "w")),
                           s0=pool[slot_of[i]][None])
        o_ref, s_ref = oracle.run_inputs(sub)
        assert _err(o_np[i:i + 1], o_ref) < tol
        assert _err(after[slot_of[i]], s_ref[0]) < tol
    for i in range(B):
        if i not in active:
            assert np.isnan(o_np[i]).all(), "inactive rows must not be written"
    untouched = sorted(set(range(n_slots)) - {int(slot_of[i]) for i in active})
    assert torch.equal(pool_d[untouched], before[untouched])


@pytest.mark.parametrize("B", [2, 16])
def test_bf16_state_many_steps(g, B):
    """64 successive single-token updates with the state stored in bf16, against the fp64 oracle
    whose state stays exact (starting from the same bf16 initial values)."""
    import torch

    wl = synth.Workload("t", B=B, T=64, Hk=16, Hv=48, dk=128, dv=128, seed=60 + B, s0_std=0.02)
    inp = synth.make_inputs(wl)
    inp.s0 = synth.round_to(inp.s0.astype(np.float64), "bf16")
    st = torch.from_numpy(inp.s0).to("cuda").to(torch.bfloat16)
    outs = []
    for t in range(wl.T):
        tok = [synth.to_torch(np.ascontiguousarray(getattr(inp, n)[:, t:t + 1]), "bf16", "cuda")
               for n in ("q", "k", "v", "g", "b", "w")]
        o = torch.empty_like(tok[2])
        g.gdn2_recurrent_update(*tok, st, o)
        outs.append(o)
    torch.cuda.synchronize()
    o_gpu = H.to_np(torch.cat(outs, dim=1))
    for bi, hv in [(0, 0), (B - 1, 47), (B // 2, 13)]:
        sub = inp.heads(bi, hv, wl.Hk, wl.Hv)
        o_ref, s_ref = oracle.run_inputs(sub)
        assert _err(o_gpu[bi:bi + 1, :, hv:hv + 1], o_ref) < H.BF16_TOL
        assert _err(st[bi, hv].float().cpu().numpy(), s_ref[0, 0]) < H.BF16_TOL


@pytest.mark.parametrize("N,state_dt,tok_dt", [(2, "f32", "bf16"), (4, "f32", "bf16"), (4, "bf16", "bf16"),
                                               (3, "bf16", "f32"), (4, "f32", "f32"), (5, "f32", "bf16")])
def test_streaming_kernel_tokens_and_state_types(g, N, state_dt, tok_dt):
    """160 x 4 = 640 heads: the streaming kernel (several tokens per call with the state held between
    them, up to 4; N = 5 takes the register kernel), fp32 or bf16 state, fp32 or bf16 tokens, against
    the oracle on every head."""
    import torch

    wl = synth.Workload("t", B=160, T=N, Hk=2, Hv=4, dk=128, dv=128, dtype=tok_dt, seed=70 + N, s0_std=0.02)
    inp = synth.make_inputs(wl)
    if state_dt == "bf16":
        inp.s0 = synth.round_to(inp.s0.astype(np.float64), "bf16")
    q, k, v, gg, b, w = _dev(inp)
    st = H.state_to_device(inp.s0)
    if state_dt == "bf16":
        st = st.to(torch.bfloat16)
    o = torch.full_like(v, float("nan"))
    g.gdn2_recurrent_update(q, k, v, gg, b, w, st, o)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    o_ref, s_ref = oracle.run_inputs(inp)
    tol = H.BF16_TOL if (tok_dt == "bf16" or state_dt == "bf16") else H.F32_TOL
    H.check("o", H.to_np(o), o_ref, tol)
    H.check("state", st.float().cpu().numpy(), s_ref, tol, head_axis=1)
