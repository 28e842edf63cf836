"""GPU parity: the CUDA path (through the C ABI binding) against the fp64 oracle on the same seeded
inputs. Tolerances (max normwise relative error, max|x - ref| / max|ref|, for o and for the final
state separately): 1e-4 for fp32 token inputs, 2e-2 for bf16 token inputs."""
import numpy as np
import pytest

import oracle
import synth
from tests import gpu_helpers as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def g():
    import gated_deltanet_mixer_gdn2_gb300 as mod

    mod.gdn2_set_wait_limit(-1)
    return mod


def _check(name, got, ref, tol):
    """Normwise max relative error over the tensor and over each (batch, head) slice (token tensors
    [B, T, H, d] and states [B, H, d_k, d_v]), with the elementwise error in the report."""
    got = np.asarray(got)
    axis = 1 if name.startswith(("state", "S")) else 2
    print(H.check(name, got, ref, tol, head_axis=axis if got.ndim == 4 else None))
    return oracle.max_rel_err(got, ref)


# ---------------------------------------------------------------------------------------------
# decode step

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("dk,dv,Hk,Hv", [(128, 128, 2, 4), (64, 64, 1, 3), (32, 48, 2, 2), (16, 256, 1, 2),
                                         (128, 16, 1, 1)])
def test_decode_small(g, dtype, dk, dv, Hk, Hv):
    wl = synth.Workload("t", B=3, T=0, Hk=Hk, Hv=Hv, dk=dk, dv=dv, dtype=dtype, seed=7, s0_std=0.02,
                        decode_steps=9)
    inp = synth.make_inputs(wl)
    st = H.state_to_device(inp.s0)
    o = H.run_decode(g, inp, st, 0, 9, scale=0.5)
    o_ref, s_ref = oracle.run_inputs(inp, scale=0.5)
    tol = H.tol_for(dtype)
    _check("o", o, o_ref, tol)
    _check("state", st.cpu().numpy(), s_ref, tol)


def test_decode_b64_256_steps(g):
    """The 64-sequence, 48-value-head decode workload, all 256 steps; every head against the oracle."""
    wl = synth.WORKLOADS["decode_b64"]
    inp = synth.make_inputs(wl)
    st = H.state_to_device(inp.s0)
    o = H.run_decode(g, inp, st, 0, wl.decode_steps)
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("o", o, o_ref, H.BF16_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.BF16_TOL)


def test_decode_batch_zero_is_noop(g):
    import torch

    e = torch.empty((0, 1, 128), dtype=torch.bfloat16, device="cuda")
    s = torch.empty((0, 1, 128, 128), dtype=torch.float32, device="cuda")
    g.gdn2_recurrent_step(e, e, e, e, e, e, s, e)


# ---------------------------------------------------------------------------------------------
# chunked forward, SIMT path (fp32 inputs, and any shape)

def test_chunk_tiny_f32(g):
    wl = synth.WORKLOADS["tiny_f32"]
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, C=wl.C)
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("o", o, o_ref, H.F32_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.F32_TOL)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("T,C,dk,dv,Hk,Hv", [(1, 64, 64, 64, 1, 1), (37, 16, 32, 48, 1, 2), (100, 32, 128, 128, 2, 4),
                                             (130, 64, 128, 64, 1, 3), (64, 64, 16, 16, 2, 2)])
def test_chunk_simt_shapes(g, dtype, T, C, dk, dv, Hk, Hv):
    wl = synth.Workload("t", B=2, T=T, Hk=Hk, Hv=Hv, dk=dk, dv=dv, C=C, dtype=dtype, seed=T + dk, s0_std=0.02,
                        neg_eigval=(T % 2 == 1))
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, C=C, path="simt")
    o_ref, s_ref = oracle.run_inputs(inp)
    tol = H.tol_for(dtype)
    _check("o", o, o_ref, tol)
    _check("state", st.cpu().numpy(), s_ref, tol)


# ---------------------------------------------------------------------------------------------
# chunked forward, tensor-core path

@pytest.mark.parametrize("T,Hk,Hv,s0", [(64, 1, 1, False), (1, 1, 1, True), (100, 1, 2, True), (200, 2, 2, False),
                                        (191, 1, 3, True)])
def test_chunk_tc_small(g, T, Hk, Hv, s0):
    wl = synth.Workload("t", B=2, T=T, Hk=Hk, Hv=Hv, dk=128, dv=128, dtype="bf16", seed=11 + T,
                        s0_std=0.02 if s0 else 0.0)
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, path="tcgen05")
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("o", o, o_ref, H.BF16_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.BF16_TOL)


def test_chunk_tc_train_bf16(g):
    """4 x 2048 tokens, 8 heads, S0 ~ N(0, 0.02^2): every head checked."""
    wl = synth.WORKLOADS["train_bf16"]
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp)
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("o", o, o_ref, H.BF16_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.BF16_TOL)


def test_chunk_tc_long_negeig(g):
    """1 x 8192 tokens, 16 heads, b in (0, 2): every head checked."""
    wl = synth.WORKLOADS["long_negeig_bf16"]
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp)
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("o", o, o_ref, H.BF16_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.BF16_TOL)


def test_prefill32k_then_decode(g):
    """2 x 32768-token prefill (16 key / 32 value heads), then 64 decode steps from its final state;
    the oracle runs the same 32832 tokens straight through, and every head is checked."""
    wl = synth.WORKLOADS["prefill32k_decode"]
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, t0=0, t1=wl.T)
    od = H.run_decode(g, inp, st, wl.T, wl.T + wl.decode_steps)
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("prefill o", o, o_ref[:, :wl.T], H.BF16_TOL)
    _check("decode o", od, o_ref[:, wl.T:], H.BF16_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.BF16_TOL)


def test_chunk_paths_agree(g):
    wl = synth.Workload("t", B=1, T=300, Hk=2, Hv=4, dk=128, dv=128, dtype="bf16", seed=5, s0_std=0.02)
    inp = synth.make_inputs(wl)
    o1, s1 = H.run_chunk(g, inp, path="simt")
    o2, s2 = H.run_chunk(g, inp, path="tcgen05")
    assert oracle.max_rel_err(o2, o1) < H.BF16_TOL
    assert oracle.max_rel_err(s2.cpu().numpy(), s1.cpu().numpy()) < H.BF16_TOL


@pytest.mark.parametrize("path", ["tcgen05", "simt"])
def test_chunk_state_chaining(g, path):
    """chunk(T) equals chunk(T1) -> final state -> chunk(T - T1)."""
    wl = synth.Workload("t", B=1, T=320, Hk=1, Hv=2, dk=128, dv=128, dtype="bf16", seed=9, s0_std=0.02)
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, path=path)
    o1, s1 = H.run_chunk(g, inp, path=path, t0=0, t1=128)
    o2, s2 = H.run_chunk(g, inp, path=path, t0=128, t1=320, s0=s1.cpu().numpy())
    assert oracle.max_rel_err(np.concatenate([o1, o2], axis=1), o) < 1e-2
    assert oracle.max_rel_err(s2.cpu().numpy(), st.cpu().numpy()) < 1e-2


def test_chunk_then_step_matches_longer_chunk(g):
    wl = synth.Workload("t", B=2, T=129, Hk=1, Hv=2, dk=128, dv=128, dtype="bf16", seed=3)
    inp = synth.make_inputs(wl)
    o_full, s_full = H.run_chunk(g, inp)
    o_pre, s = H.run_chunk(g, inp, t0=0, t1=128)
    od = H.run_decode(g, inp, s, 128, 129)
    assert oracle.max_rel_err(od, o_full[:, 128:]) < H.BF16_TOL
    assert oracle.max_rel_err(s.cpu().numpy(), s_full.cpu().numpy()) < H.BF16_TOL


def test_chunk_state_aliasing(g):
    """initial_state and final_state may be the same buffer."""
    import torch

    wl = synth.Workload("t", B=1, T=96, Hk=1, Hv=2, dk=128, dv=128, dtype="bf16", seed=4, s0_std=0.02)
    inp = synth.make_inputs(wl)
    o_ref, s_ref = oracle.run_inputs(inp)
    q, k, v, gg, b, w = H.upload(inp, 0, wl.T)
    st = H.state_to_device(inp.s0)
    o = torch.empty_like(v)
    g.gdn2_chunk_fwd(q, k, v, gg, b, w, o, st, st)
    torch.cuda.synchronize()
    _check("o", H.to_np(o), o_ref, H.BF16_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.BF16_TOL)


def test_chunk_empty_sequence(g):
    import torch

    s0 = torch.randn(1, 2, 128, 128, device="cuda")
    fs = torch.full_like(s0, float("nan"))
    e = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda")
    g.gdn2_chunk_fwd(e, e, e, e, e, e, e, s0, fs)
    torch.cuda.synchronize()
    assert torch.equal(fs, s0)
    g.gdn2_chunk_fwd(e, e, e, e, e, e, e, None, fs)
    torch.cuda.synchronize()
    assert torch.count_nonzero(fs).item() == 0


def test_wait_timeout_is_reported_and_recoverable(g):
    """A zero wait budget makes every guarded wait give up at once: the call reports a timeout
    through the device status word, the device stays usable, and the next call is correct."""
    wl = synth.Workload("t", B=1, T=130, Hk=1, Hv=1, dk=128, dv=128, dtype="bf16", seed=2)
    inp = synth.make_inputs(wl)
    q, k, v, gg, b, w = H.upload(inp, 0, wl.T)
    g.gdn2_set_wait_limit(0)
    try:
        g.chunk_fwd(q, k, v, gg, b, w, None, path="tcgen05")
        assert g.gdn2_last_device_status() == g.GDN2_ERR_TIMEOUT
    finally:
        g.gdn2_set_wait_limit(-1)
    assert g.gdn2_last_device_status() == g.GDN2_OK
    o, st = H.run_chunk(g, inp, path="tcgen05")
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("o", o, o_ref, H.BF16_TOL)


# ---------------------------------------------------------------------------------------------
# bounds: canary regions right after every output buffer

_CANARY = 4096  # elements of sentinel after each output


def _with_canary(shape, dtype, fill):
    """A contiguous tensor of `shape` that is the head of a larger buffer whose tail holds `fill`."""
    import torch

    n = int(np.prod(shape))
    buf = torch.full((n + _CANARY,), fill, dtype=dtype, device="cuda")
    return buf, buf[:n].view(shape)


@pytest.mark.parametrize("path,dtype,T,C", [("tcgen05", "bf16", 37, 64), ("tcgen05", "bf16", 130, 64),
                                            ("simt", "f32", 37, 64), ("simt", "bf16", 70, 32),
                                            ("simt", "f32", 5, 16)])
def test_chunk_writes_stay_in_bounds(g, path, dtype, T, C):
    """Ragged T (the last chunk padded) and T < C: o and final_state are followed by canary elements,
    which the call must leave untouched; the results still match the oracle."""
    import torch

    d = 128 if path == "tcgen05" else 64
    wl = synth.Workload("t", B=2, T=T, Hk=1, Hv=2, dk=d, dv=d, C=C, dtype=dtype, seed=40 + T, s0_std=0.02)
    inp = synth.make_inputs(wl)
    q, k, v, gg, b, w = H.upload(inp, 0, T)
    s0 = H.state_to_device(inp.s0)
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    obuf, o = _with_canary(tuple(v.shape), tdt, -7.0)
    sbuf, sT = _with_canary((2, 2, d, d), torch.float32, -7.0)
    g.gdn2_chunk_fwd(q, k, v, gg, b, w, o, s0, sT, C=C, path=path)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    assert bool((obuf[o.numel():] == -7.0).all()), "o canary overwritten"
    assert bool((sbuf[sT.numel():] == -7.0).all()), "final_state canary overwritten"
    o_ref, s_ref = oracle.run_inputs(inp)
    tol = H.tol_for(dtype)
    _check("o", H.to_np(o), o_ref, tol)
    _check("state", sT.cpu().numpy(), s_ref, tol)


@pytest.mark.parametrize("B,Hk,Hv", [(3, 1, 2), (160, 2, 4)])
def test_decode_writes_stay_in_bounds(g, B, Hk, Hv):
    """The decode step updates the state in place and writes o: canaries after both stay untouched
    (the second shape has enough heads for the streaming kernel)."""
    import torch

    wl = synth.Workload("t", B=B, T=0, Hk=Hk, Hv=Hv, dk=128, dv=128, dtype="bf16", seed=41, s0_std=0.02,
                        decode_steps=2)
    inp = synth.make_inputs(wl)
    sbuf, st = _with_canary((B, Hv, 128, 128), torch.float32, -7.0)
    st.copy_(H.state_to_device(inp.s0))
    outs = []
    for t in range(2):
        q, k, v, gg, b, w = H.upload_token(inp, t)
        obuf, o = _with_canary((B, Hv, 128), torch.bfloat16, -7.0)
        g.gdn2_recurrent_step(q, k, v, gg, b, w, st, o)
        torch.cuda.synchronize()
        assert bool((obuf[o.numel():] == -7.0).all()), "o canary overwritten"
        outs.append(o)
    assert g.gdn2_last_device_status() == g.GDN2_OK
    assert bool((sbuf[st.numel():] == -7.0).all()), "state canary overwritten"
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("o", H.to_np(torch.stack(outs, dim=1)), o_ref, H.BF16_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.BF16_TOL)


# ---------------------------------------------------------------------------------------------
# value dimensions other than d_k (expand_v): the tensor-core path runs d_v / 64 state CTAs per head

@pytest.mark.parametrize("dv,Hk,Hv,T", [(256, 1, 2, 200), (64, 2, 2, 130), (192, 1, 3, 64), (512, 1, 1, 70)])
def test_chunk_tc_value_dims(g, dv, Hk, Hv, T):
    wl = synth.Workload("t", B=2, T=T, Hk=Hk, Hv=Hv, dk=128, dv=dv, dtype="bf16", seed=50 + dv, s0_std=0.02)
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, path="tcgen05")
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("o", o, o_ref, H.BF16_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.BF16_TOL)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_chunk_simt_value_dim_256(g, dtype):
    wl = synth.Workload("t", B=1, T=150, Hk=1, Hv=2, dk=64, dv=256, C=32, dtype=dtype, seed=57, s0_std=0.02)
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, C=32, path="simt")
    o_ref, s_ref = oracle.run_inputs(inp)
    tol = H.tol_for(dtype)
    _check("o", o, o_ref, tol)
    _check("state", st.cpu().numpy(), s_ref, tol)


@pytest.mark.parametrize("dv,decay,s0", [(64, "standard", True), (128, "standard", False), (64, "reset", True)])
def test_chunk_tc_head_dim_64(g, dv, decay, s0):
    """head_dim 64 (the burn-gdn2 Quick start's shape) on the tensor-core path: d_k = 64 runs as
    d_k = 128 with zero channels; ragged T, grouped heads, an initial state and the exact kernel."""
    wl = synth.Workload("t", B=2, T=170, Hk=1, Hv=2, dk=64, dv=dv, dtype="bf16", seed=60 + dv,
                        s0_std=0.02 if s0 else 0.0, decay=decay)
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, path="tcgen05")
    o_ref, s_ref = oracle.run_inputs(inp)
    _check("o", o, o_ref, H.BF16_TOL)
    _check("state", st.cpu().numpy(), s_ref, H.BF16_TOL)
