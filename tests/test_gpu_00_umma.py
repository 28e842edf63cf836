"""tcgen05 operand layouts: one M=128 product per layout combination the chunked kernels use, with
shared-memory operands staged by TMA (128-byte swizzle) and by ordinary stores with the same
swizzle, and A operands held in tensor memory, against numpy.
Values are small multiples of 1/8, so every product and sum is exact in fp32."""
import numpy as np
import pytest

pytestmark = pytest.mark.gpu

# (A storage is [rows][cols] = M x K (K-major) or K x M (MN-major); B likewise with N)
CASES = {
    0: dict(M=128, N=64, K=128, a_mn=False, b_mn=False),
    1: dict(M=128, N=64, K=64, a_mn=True, b_mn=False),
    2: dict(M=128, N=64, K=128, a_mn=True, b_mn=True),
    3: dict(M=128, N=64, K=64, a_mn=False, b_mn=True),
    4: dict(M=128, N=64, K=128, a_mn=False, b_mn=False, neg=True),
    # A read from tensor memory (row-major M x K storage, written with tcgen05.st)
    5: dict(M=128, N=64, K=64, a_mn=False, b_mn=False),
    6: dict(M=128, N=128, K=64, a_mn=False, b_mn=True),
    7: dict(M=128, N=128, K=128, a_mn=False, b_mn=False),
}


@pytest.mark.parametrize("soft", [0, 1])
@pytest.mark.parametrize("case", sorted(CASES))
def test_umma_layout(case, soft):
    import torch

    import gated_deltanet_mixer_gdn2_gb300 as g

    c = CASES[case]
    rng = np.random.default_rng(100 + case)
    A = rng.integers(-8, 9, (c["M"], c["K"])) / 8.0     # math operand, M x K
    B = rng.integers(-8, 9, (c["K"], c["N"])) / 8.0     # math operand, K x N
    a_st = A.T if c["a_mn"] else A                      # MN-major stores K rows of M
    b_st = B if c["b_mn"] else B.T                      # K-major stores N rows of K
    dev = torch.device("cuda")
    at = torch.tensor(np.ascontiguousarray(a_st), dtype=torch.bfloat16, device=dev)
    bt = torch.tensor(np.ascontiguousarray(b_st), dtype=torch.bfloat16, device=dev)
    d = torch.full((128, c["N"]), float("nan"), dtype=torch.float32, device=dev)
    g.gdn2_selftest_umma(case, soft, at, bt, d)
    torch.cuda.synchronize()
    assert g.gdn2_last_device_status() == g.GDN2_OK
    ref = -(A @ B) if c.get("neg") else A @ B
    got = d.cpu().numpy()
    assert np.array_equal(got, ref), f"case {case} soft {soft}: max err {np.nanmax(np.abs(got - ref))}"
