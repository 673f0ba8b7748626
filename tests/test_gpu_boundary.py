"""The boundary on a GPU: argument errors leave outputs untouched, the bounded
waits give up with KD_ERR_TIMEOUT instead of hanging, and the context survives."""
import pytest
import torch

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kd(cuda_device):
    from sparse_teacher_kl_gb300.build import build_library
    build_library()
    import sparse_teacher_kl_gb300 as kd
    return kd


def test_wait_gives_up_and_reports_timeout(kd, cuda_device):
    ws = kd.workspace(kd._abi.kd_gemm_workspace(), cuda_device)
    st = kd._abi.kd_check_wait_timeout(ws.data_ptr(), ws.numel(), 20_000_000, torch.cuda.current_stream().cuda_stream)
    assert st == 0
    status, detail = kd.device_error(ws)
    assert status == kd._abi.KD_ERR_TIMEOUT and detail == 0x7E57
    # the context is still usable
    x = torch.ones(1024, device=cuda_device)
    assert float((x * 2).sum().item()) == 2048.0
    assert kd.device_error(ws)[0] == 0


def test_invalid_calls_do_not_touch_outputs(kd, cuda_device):
    dev = cuda_device
    X = torch.randn((4, 256), device=dev).to(torch.bfloat16)
    ids = torch.full((4, 8), -7, dtype=torch.int32, device=dev)
    vals = torch.full((4, 8), 3.0, device=dev)
    ws = kd.workspace(256, dev)
    s = torch.cuda.current_stream().cuda_stream
    assert kd._abi.kd_topk_cache(X.data_ptr(), 4, 256, 256, 300, ids.data_ptr(), vals.data_ptr(), None,
                                 None, ws.data_ptr(), 256, s) == kd._abi.KD_ERR_INVALID_ARG
    assert kd._abi.kd_topk_cache(X.data_ptr() + 2, 4, 256, 256, 8, ids.data_ptr(), vals.data_ptr(), None,
                                 None, ws.data_ptr(), 256, s) == kd._abi.KD_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert torch.all(ids == -7) and torch.all(vals == 3.0)
    with pytest.raises(kd.KDError):
        kd.topk_cache(X, 257)


def test_workspace_too_small_is_rejected(kd, cuda_device):
    dev = cuda_device
    H = torch.zeros((128, 64), dtype=torch.bfloat16, device=dev)
    W = torch.zeros((512, 64), dtype=torch.bfloat16, device=dev)
    ids = torch.zeros((128, 4), dtype=torch.int32, device=dev)
    tl = torch.zeros((128, 4), device=dev)
    need = kd._abi.kd_fused_kl_workspace(128, 64, 512, 4, 128)
    ws = kd.workspace(need - 256, dev)
    with pytest.raises(kd.KDError) as e:
        kd.fused_kl_forward(H, W, ids, tl, None, 128, 1.0, ws=ws)
    assert e.value.status == kd._abi.KD_ERR_WORKSPACE
