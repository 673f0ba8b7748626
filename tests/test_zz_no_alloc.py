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


def test_static_scratch_call_allocates_no_device_memory(kd, cuda_device):
    """After a first call (which looks up the array's address), further calls change
    neither the device's free memory nor torch's allocator: nothing is allocated."""
    dev = cuda_device
    H, W, ids, tlog, mask = _inputs(13, 512, 256, 4096, 16, dev, True)
    N, d = H.shape
    V, K = W.shape[0], ids.shape[1]
    loss = torch.empty((1,), device=dev)
    lse = torch.empty((N,), device=dev)
    stream = torch.cuda.current_stream().cuda_stream

    def call():
        return kd._abi.kd_fused_kl_fwd_static(H.data_ptr(), W.data_ptr(), ids.data_ptr(), tlog.data_ptr(),
                                              mask.data_ptr(), N, d, V, K, 128, 1.0, loss.data_ptr(),
                                              lse.data_ptr(), None, stream)

    assert call() == 0
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info(dev)
    alloc0 = torch.cuda.memory_allocated(dev)
    for _ in range(3):
        assert call() == 0
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info(dev)
    assert free1 == free0
    assert torch.cuda.memory_allocated(dev) == alloc0
    assert torch.isfinite(loss).all()


def test_static_scratch_error_word_is_readable(kd, cuda_device):
    """A device-side condition of the static variant (a teacher id out of range) lands in
    the array's error word, which kd_get_device_error reads and clears given NULL."""
    import ctypes
    dev = cuda_device
    H, W, ids, tlog, _ = _inputs(14, 256, 128, 2048, 16, dev, False)
    ids = ids.clone()
    ids[201, 5] = W.shape[0]    # out of range: recorded, never used as an address
    st, loss, _, _ = _call_static(kd, H, W, ids, tlog, None, 128)
    assert st == 0
    stream = torch.cuda.current_stream().cuda_stream
    detail = ctypes.c_int64(-1)
    assert kd._abi.kd_get_device_error(None, stream, ctypes.byref(detail)) == kd._abi.KD_ERR_DEVICE
    assert detail.value == 201
    assert kd._abi.kd_get_device_error(None, stream, ctypes.byref(detail)) == 0   # reading clears it
    # the next call starts from a clean control block and matches the workspace forward
    H2, W2, ids2, tlog2, mask2 = _inputs(15, 256, 128, 2048, 16, dev, True)
    st, loss_s, lse_s, kl_s = _call_static(kd, H2, W2, ids2, tlog2, mask2, 128)
    assert st == 0
    loss_r, lse_r, kl_r = _call_regular(kd, H2, W2, ids2, tlog2, mask2, 128)
    torch.cuda.synchronize()
    assert abs(loss_s.item() - loss_r.item()) <= LOSS_RTOL * abs(loss_r.item())
    assert _close(lse_s, lse_r, ROW_TOL)
    assert kd._abi.kd_get_device_error(None, stream, ctypes.byref(detail)) == 0
