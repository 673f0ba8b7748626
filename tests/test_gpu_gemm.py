"""The tcgen05/TMA projection engine alone: C = A·B for every operand major-ness,
ragged in every dimension, against a float64 product of the same bf16 values."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kd(cuda_device):
    from sparse_teacher_kl_gb300.build import build_library
    build_library()
    import sparse_teacher_kl_gb300 as kd
    return kd


def _case(M, N, K, a_mn, b_mn, seed, dev):
    g = torch.Generator().manual_seed(seed)
    A = torch.randn((K, M) if a_mn else (M, K), generator=g).to(torch.bfloat16)
    B = torch.randn((K, N) if b_mn else (N, K), generator=g).to(torch.bfloat16)
    Am = A.double().T if a_mn else A.double()           # [M, K]
    Bm = B.double() if b_mn else B.double().T           # [K, N]
    return A.to(dev), B.to(dev), Am @ Bm


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (0, 1), (1, 1), (1, 0)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (296, 520, 200), (64, 16, 8), (1000, 264, 1096), (640, 704, 320)])
def test_gemm_matches_float64(kd, cuda_device, a_mn, b_mn, M, N, K):
    A, B, ref = _case(M, N, K, a_mn, b_mn, seed=M * 7 + N + K, dev=cuda_device)
    C, ws = kd.gemm_bf16(A, B, M, N, K, a_mn, b_mn)
    torch.cuda.synchronize()
    assert kd.device_error(ws)[0] == 0
    err = (C.double().cpu() - ref).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item() * max(1.0, K / 64)


@pytest.mark.parametrize("M,N,K", [
    (256, 512, 128),    # reductions up to 2048 deep: staged blocks added by TMA reduce-adds
    (296, 520, 200),    # the same, ragged rows and columns (clipped by the tensor map)
    (1000, 264, 1096),
    (600, 264, 2112),   # deeper: each thread adds its own row with vector reductions
])
def test_gemm_accumulates(kd, cuda_device, M, N, K):
    A, B, ref = _case(M, N, K, 1, 1, seed=3 + K, dev=cuda_device)
    C0 = torch.randn((M, N), generator=torch.Generator().manual_seed(4))
    C = C0.clone().to(cuda_device)
    kd.gemm_bf16(A, B, M, N, K, 1, 1, C=C)
    torch.cuda.synchronize()
    err = (C.double().cpu() - (ref + C0.double())).abs().max().item()
    assert err <= 1e-5 * ref.abs().max().item() * max(1.0, K / 64) + 1e-5
