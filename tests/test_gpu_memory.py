"""Peak device memory of one fused fwd+bwd grows with the chunk, not with N x V.

The fused formulation keeps only one chunk's logits gradient (bf16 [chunk, V]) and
per-chunk partials, so the memory a call needs beyond its inputs and outputs is the
workspace, sized by the chunk; a dense formulation would add N x V fp32 grids
([ART] paragraph on the three loss formulations; [EPO] "Adónde se va la memoria").
Measured with the caching allocator's peak, around calls that allocate their
workspace, outputs and gradients themselves.
"""
import pytest
import torch

from synth import Workload, make_inputs

pytestmark = pytest.mark.gpu

D, V, K = 512, 32000, 16


@pytest.fixture(scope="module")
def kd(cuda_device):
    from sparse_teacher_kl_gb300.build import build_library
    build_library()
    import sparse_teacher_kl_gb300 as kd
    return kd


def _peak(kd, dev, N, chunk):
    """Bytes allocated at the peak of one fwd+bwd beyond the inputs, and the workspace size."""
    w = Workload("mem", 1, N, D, V, K, chunk, "zipf", 1.0, 4242)
    H, W, ids, tlog, mask = make_inputs(w, device=dev)
    g = torch.ones((1,), dtype=torch.float32, device=dev)
    torch.cuda.synchronize(dev)
    torch.cuda.empty_cache()
    base = torch.cuda.memory_allocated(dev)
    torch.cuda.reset_peak_memory_stats(dev)
    loss, lse, ws = kd.fused_kl_forward(H, W, ids, tlog, mask, chunk=chunk)
    grad_H, grad_W = kd.fused_kl_backward(H, W, ids, tlog, mask, lse, g, chunk=chunk, ws=ws)
    torch.cuda.synchronize(dev)
    assert torch.isfinite(loss).all()
    peak = torch.cuda.max_memory_allocated(dev) - base
    nws = ws.numel()
    del loss, lse, ws, grad_H, grad_W, H, W, ids, tlog
    return peak, nws


def test_peak_grows_with_chunk_not_with_tokens(kd, cuda_device):
    outputs = V * D * 4  # grad_W fp32; grad_H, lse and loss are O(N d)
    # fixed N, growing chunk: the growth is the workspace's, about chunk x V x 2 bytes
    p = {c: _peak(kd, cuda_device, 8192, c) for c in (512, 1024, 2048)}
    for c in (512, 1024, 2048):
        peak, nws = p[c]
        assert nws >= c * V * 2
        assert peak <= nws + outputs + 8192 * D * 2 + (16 << 20)
    assert p[2048][0] - p[512][0] >= 0.9 * (2048 - 512) * V * 2
    # fixed chunk, 4x the tokens: the growth is O(N (d + K)), far below one N x V grid
    small, _ = _peak(kd, cuda_device, 4096, 1024)
    large, _ = _peak(kd, cuda_device, 16384, 1024)
    grid = (16384 - 4096) * V * 4
    assert large - small <= (16384 - 4096) * (D * 2 + 64) + (4 << 20)
    assert large - small < 0.01 * grid
