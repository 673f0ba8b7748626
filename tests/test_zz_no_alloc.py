"""kd_fused_kl_fwd_static, the forward pass for callers that cannot allocate
device memory (framework plugins whose allocator owns all device memory, and
paths that cannot take the synchronisation cudaMalloc may cause): it uses a
scratch array compiled into the library instead of a caller workspace.

Checked through the C ABI against kd_fused_kl_fwd with its own workspace, on
two calls in a row with different inputs (the shared array keeps the previous
call's contents), within the forward tolerances of the other parity tests.
This file is collected last on purpose.
"""
import pytest
import torch

pytestmark = pytest.mark.gpu

LOSS_RTOL = 1e-3
ROW_TOL = 1e-3


@pytest.fixture(scope="module")
def kd(cuda_device):
    from sparse_teacher_kl_gb300.build import build_library
    build_library()
    import sparse_teacher_kl_gb300 as kd
    return kd


def _inputs(seed, N, d, V, K, dev, masked):
    from synth import Workload, make_inputs
    w = Workload("noalloc", 1, N, d, V, K, 128, "zipf", 0.9 if masked else 1.0, seed)
    H, W, ids, tlog, mask = make_inputs(w, dev)
    return H, W, ids, tlog, mask


def _call_static(kd, H, W, ids, tlog, mask, chunk):
    N, d = H.shape
    V, K = W.shape[0], ids.shape[1]
    loss = torch.full((1,), float("nan"), device=H.device)
    lse = torch.full((N,), float("nan"), device=H.device)
    kl = torch.full((N,), float("nan"), device=H.device)
    st = kd._abi.kd_fused_kl_fwd_static(H.data_ptr(), W.data_ptr(), ids.data_ptr(), tlog.data_ptr(),
                                        None if mask is None else mask.data_ptr(), N, d, V, K, chunk, 1.0,
                                        loss.data_ptr(), lse.data_ptr(), kl.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream)
    return st, loss, lse, kl


def _call_regular(kd, H, W, ids, tlog, mask, chunk):
    N = H.shape[0]
    kl = torch.empty((N,), device=H.device)
    loss, lse, ws = kd.fused_kl_forward(H, W, ids, tlog, mask, chunk, 1.0, kl_out=kl)
    return loss, lse, kl


def _close(a, b, tol):
    return float((a - b).abs().max()) <= tol * float(b.abs().max())


def test_static_scratch_forward_matches_workspace_forward(kd, cuda_device):
    dev = cuda_device
    cases = [(11, 384, 256, 4096, 16, 128, False), (12, 300, 520, 2560, 64, 256, True)]
    for seed, N, d, V, K, chunk, masked in cases:           # two calls in a row
        H, W, ids, tlog, mask = _inputs(seed, N, d, V, K, dev, masked)
        need = kd._abi.kd_fused_kl_workspace(N, d, V, K, chunk)
        assert need <= kd._abi.KD_STATIC_SCRATCH_BYTES
        st, loss_s, lse_s, kl_s = _call_static(kd, H, W, ids, tlog, mask, chunk)
        assert st == 0, kd._abi.status_string(st)
        loss_r, lse_r, kl_r = _call_regular(kd, H, W, ids, tlog, mask, chunk)
        torch.cuda.synchronize()
        assert abs(loss_s.item() - loss_r.item()) <= LOSS_RTOL * abs(loss_r.item())
        assert _close(lse_s, lse_r, ROW_TOL)
        assert _close(kl_s, kl_r, ROW_TOL)


def test_static_scratch_rejects_problems_beyond_its_size(kd, cuda_device):
    dev = cuda_device
    N, d, V, K, chunk = 4096, 64, 201088, 100, 4096
    assert kd._abi.kd_fused_kl_workspace(N, d, V, K, chunk) > kd._abi.KD_STATIC_SCRATCH_BYTES
    H = torch.zeros((N, d), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((V, d), dtype=torch.bfloat16, device=dev)
    ids = torch.zeros((N, K), dtype=torch.int32, device=dev)
    tlog = torch.zeros((N, K), device=dev)
    st, loss, _, _ = _call_static(kd, H, W, ids, tlog, None, chunk)
    torch.cuda.synchronize()
    assert st == kd._abi.KD_ERR_WORKSPACE
    assert torch.isnan(loss).all()          # nothing was launched
