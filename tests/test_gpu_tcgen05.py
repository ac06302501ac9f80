"""The fifth-generation tensor-core building block (edge0_tc_gemm_f16) against a
plain fp32 product of the same fp16 operands: shared-memory descriptors,
instruction descriptor, TMEM allocation and read-out, several K chunks."""
import pytest
import torch

from int4_routed_expert_prerouter_gb300 import binding

pytestmark = pytest.mark.gpu
DEV = "cuda:0"


@pytest.fixture(scope="module", autouse=True)
def _built():
    import __graft_entry__
    __graft_entry__.build()


@pytest.mark.parametrize("M,N,K", [(128, 16, 64), (128, 64, 128), (256, 128, 320), (384, 256, 2048)])
def test_tc_gemm_matches_fp32_product(M, N, K):
    g = torch.Generator().manual_seed(M * 7 + N * 3 + K)
    A = (torch.randn(M, K, generator=g) * 0.5).half()
    B = (torch.randn(N, K, generator=g) * 0.5).half()
    D = binding.tc_gemm_f16(A.to(DEV), B.to(DEV)).cpu()
    ref = A.double() @ B.double().T
    err = (D.double() - ref).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item() + 1e-6, f"max|diff| {err:.3e}"


def test_tc_gemm_structure():
    # one nonzero per row of A and of B: D is a permutation-like pattern that
    # exposes a swapped row, column or K-step at once
    M, N, K = 128, 32, 64
    A = torch.zeros(M, K, dtype=torch.float16)
    B = torch.zeros(N, K, dtype=torch.float16)
    for i in range(M):
        A[i, (i * 5) % K] = float(i % 7 + 1)
    for j in range(N):
        B[j, (j * 3) % K] = 1.0
    D = binding.tc_gemm_f16(A.to(DEV), B.to(DEV)).cpu()
    assert torch.equal(D, (A.float() @ B.float().T))


def test_tc_gemm_rejects_bad_shapes():
    lib = binding.lib()
    x = torch.zeros(128 * 64, dtype=torch.float16, device=DEV)
    d = torch.zeros(128 * 16, dtype=torch.float32, device=DEV)
    st = torch.zeros(1, dtype=torch.int32, device=DEV)
    P = binding._ptr
    assert lib.edge0_tc_gemm_f16(P(x), P(x), P(d), 100, 16, 64, P(st), None) == binding.EDGE0_EINVAL
    assert lib.edge0_tc_gemm_f16(P(x), P(x), P(d), 128, 24, 64, P(st), None) == binding.EDGE0_EINVAL
    assert lib.edge0_tc_gemm_f16(P(x), P(x), P(d), 128, 16, 32, P(st), None) == binding.EDGE0_EINVAL
