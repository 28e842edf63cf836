"""Exact and scaled GPU checks.

* Decode with standard-basis keys and dyadic values: every product and sum the recurrence forms is
  exact in fp32, so the GPU state and outputs must equal the fp64 reference bit for bit. Each state
  row then obeys a scalar recurrence (keyed row i: S[i,:] <- (1 - b[i]) alpha[i] S[i,:] + k_i w.v;
  others: S[r,:] <- alpha[r] S[r,:]); a transposed gate axis or a misplaced factor shows at once.
* The tensor-core chunked path with scale != 1 against the oracle (the output read-out applies it).
"""
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


# (batch, tokens per call, d, state dtype): 12 heads take the register kernel, 640 heads the streaming
# kernel (one token, or several with the state held between them). With a bf16 state the erase gate
# is 1, so every stored state value keeps few significant bits and rounds to bf16 exactly.
@pytest.mark.parametrize("B,N,d,state_dt", [(3, 24, 128, "f32"), (3, 24, 64, "f32"), (160, 1, 128, "f32"),
                                            (160, 4, 128, "f32"), (160, 1, 128, "bf16"), (160, 4, 128, "bf16"),
                                            (3, 4, 128, "bf16")])
def test_decode_standard_basis_is_bit_exact(g, B, N, d, state_dt):
    import torch

    rng = np.random.default_rng(40 + d + B + N)
    Hk, Hv = 2, 4
    idx = rng.integers(0, d, (B, N, Hk))
    k = np.zeros((B, N, Hk, d))
    for bi in range(B):
        for t in range(N):
            for h in range(Hk):
                k[bi, t, h, idx[bi, t, h]] = -1.0 if (t % 3 == 0) else 1.0
    q = rng.integers(-4, 5, (B, N, Hk, d)) / 4.0
    v = rng.integers(-8, 9, (B, N, Hv, d)) / 8.0
    alpha = rng.choice([0.0, 1.0], (B, N, Hv, d), p=[0.2, 0.8])
    gg = np.where(alpha == 0.0, -np.inf, 0.0)
    b = rng.choice([0.5, 1.0, 1.5], (B, N, Hv, d)) if state_dt == "f32" else np.ones((B, N, Hv, d))
    w = rng.choice([0.5, 1.0], (B, N, Hv, d))
    s0 = rng.integers(-4, 5, (B, Hv, d, d)) / 8.0
    # fp64 reference of the same recurrence (values stay dyadic with few bits: exact)
    S = s0.copy()
    o_ref = np.zeros((B, N, Hv, d))
    for t in range(N):
        for bi in range(B):
            for h in range(Hv):
                hk = h * Hk // Hv
                Sp = alpha[bi, t, h][:, None] * S[bi, h]
                r = Sp.T @ (b[bi, t, h] * k[bi, t, hk])
                S[bi, h] = Sp + np.outer(k[bi, t, hk], w[bi, t, h] * v[bi, t, h] - r)
                o_ref[bi, t, h] = S[bi, h].T @ q[bi, t, hk]
    dev = lambda a: synth.to_torch(np.ascontiguousarray(a, dtype=np.float32), "bf16", "cuda")
    st = torch.from_numpy(s0.astype(np.float32)).cuda()
    if state_dt == "bf16":
        st = st.to(torch.bfloat16)
    o = torch.empty((B, N, Hv, d), dtype=torch.float32, device="cuda")
    ts = [dev(x) for x in (q, k, v, gg, b, w)]
    # fp32 tokens keep the outputs exact too (bf16 outputs would round them)
    ts32 = [t.float() for t in ts]
    g.gdn2_recurrent_update(*ts32, st, o)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    assert np.array_equal(st.float().cpu().numpy().astype(np.float64), S)
    assert np.array_equal(o.cpu().numpy().astype(np.float64), o_ref)


@pytest.mark.parametrize("scale", [0.25, 1.7])
def test_chunk_tc_scale(g, scale):
    wl = synth.Workload("sc", B=1, T=150, Hk=1, Hv=2, dk=128, dv=128, dtype="bf16", seed=33, s0_std=0.02)
    inp = synth.make_inputs(wl)
    o, st = H.run_chunk(g, inp, path="tcgen05", scale=scale)
    o_ref, s_ref = oracle.run_inputs(inp, scale=scale)
    assert oracle.max_rel_err(o, o_ref) < H.BF16_TOL
    assert oracle.max_rel_err(st.cpu().numpy(), s_ref) < H.BF16_TOL
