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


def _peak(kd, dev, N, chunk, d=D, v=V, k=K, teacher="zipf", p_valid=1.0):
    """Bytes allocated at the peak of one fwd+bwd beyond the inputs, and the workspace size."""
    w = Workload("mem", 1, N, d, v, k, chunk, teacher, p_valid, 4242)
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


def test_headline_shape_peak_grows_with_chunk_not_tokens(kd, cuda_device):
    """The pages' headline shape (d = 2880, V = 201088, K = 100, 2 % padding): going from chunk 4096
    to 8192 adds the workspace's growth to the peak (4096 more rows of bf16 dZ, V x 2 bytes each, plus
    their logsumexp partials and split buffers), and four times the positions at chunk 8192 adds only
    the O(N d) outputs, far below one N x V grid ([EPO] "Adónde se va la memoria": the dense teacher
    tensor alone is 4 x 201,088 x 32,768 values)."""
    hd, hv, hk = 2880, 201088, 100
    kw = dict(d=hd, v=hv, k=hk, teacher="peaked_flat", p_valid=0.98)
    N = 4 * 32768
    p4, ws4 = _peak(kd, cuda_device, N, 4096, **kw)
    p8, ws8 = _peak(kd, cuda_device, N, 8192, **kw)
    assert ws8 - ws4 >= 4096 * hv * 2
    assert abs((p8 - p4) - (ws8 - ws4)) <= (64 << 20)
    # fixed chunk, a quarter of the positions: the peaks differ by the O(N d) outputs and O(N) rows
    q8, _ = _peak(kd, cuda_device, N // 4, 8192, **kw)
    dN = N - N // 4
    assert p8 - q8 <= dN * (hd * 2 + 64) + (64 << 20)
    assert p8 - q8 < 0.01 * dN * hv * 4
    # the whole call beyond its inputs at the headline shape, next to the dense grids
    assert p8 < 16e9 < 0.05 * N * hv * (2 + 4 * 5)
