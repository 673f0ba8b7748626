"""kd_fused_kl_fwd / kd_fused_kl_bwd against the float64 oracle on identical bf16 inputs.

Tolerances: loss within 1e-3 relative; each gradient tensor max|err| <= 2e-2 *
max|ref|; per-position KL and logsumexp within 1e-3 * max|ref| (fp32 accumulation
over d, fp32 online logsumexp over V).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from synth import WORKLOADS, Workload, bf16_bits, make_inputs

pytestmark = pytest.mark.gpu

LOSS_RTOL = 1e-3
GRAD_TOL = 2e-2
ROW_TOL = 1e-3


@pytest.fixture(scope="module")
def kd(cuda_device):
    from sparse_teacher_kl_gb300.build import build_library
    build_library()
    import sparse_teacher_kl_gb300 as kd
    return kd


def run_gpu(kd, dev, H, W, ids, tlog, mask, chunk, tau=1.0, grad=1.0, grad_H_fp32=True, want_bwd=True):
    Hd, Wd, idd, tld = (t.to(dev).contiguous() for t in (H, W, ids, tlog))
    md = None if mask is None else mask.to(dev).contiguous()
    N = Hd.shape[0]
    kl = torch.empty(N, dtype=torch.float32, device=dev)
    loss, lse, ws = kd.fused_kl_forward(Hd, Wd, idd, tld, md, chunk, tau, kl_out=kl)
    out = dict(loss=loss, lse=lse, kl=kl)
    if want_bwd:
        g = torch.full((1,), grad, dtype=torch.float32, device=dev)
        gH, gW = kd.fused_kl_backward(Hd, Wd, idd, tld, md, lse, g, chunk, tau, ws=ws, grad_H_fp32=grad_H_fp32)
        out.update(grad_H=gH, grad_W=gW)
    torch.cuda.synchronize()
    st, detail = kd.device_error(ws)
    assert st == 0, f"device error {st} detail {detail}"
    return out


def maxrel(got, ref):
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.max(np.abs(got - ref)) / max(np.max(np.abs(ref)), 1e-30))


def compare_full(out, ref, check_grads=True):
    assert abs(float(out["loss"].item()) - ref.loss) <= LOSS_RTOL * abs(ref.loss), (out["loss"].item(), ref.loss)
    assert maxrel(out["kl"].cpu().numpy(), ref.kl) <= ROW_TOL
    assert maxrel(out["lse"].cpu().numpy(), ref.lse) <= ROW_TOL
    if check_grads:
        assert maxrel(out["grad_H"].double().cpu().numpy(), ref.grad_H) <= GRAD_TOL
        assert maxrel(out["grad_W"].double().cpu().numpy(), ref.grad_W) <= GRAD_TOL


def _host(w, **kw):
    return make_inputs(w, "cpu", **kw)


@pytest.mark.parametrize("tau", [1.0, 2.0])
@pytest.mark.parametrize("masked", [False, True])
def test_tiny_full(kd, cuda_device, tau, masked):
    w = WORKLOADS["tiny"]
    H, W, ids, tlog, _ = _host(w)
    mask = None
    if masked:
        mask = (torch.rand(w.N, generator=torch.Generator().manual_seed(2)) < 0.7).to(torch.uint8)
    out = run_gpu(kd, cuda_device, H, W, ids, tlog, mask, chunk=128, tau=tau, grad=0.75)
    ref = oracle.dense_kl(bf16_bits(H), bf16_bits(W), ids.numpy(), tlog.numpy(),
                          None if mask is None else mask.numpy(), tau, grad_loss=0.75)
    compare_full(out, ref)
    if masked:
        assert torch.all(out["grad_H"].cpu()[mask == 0] == 0)


def test_grad_H_bf16_output(kd, cuda_device):
    w = WORKLOADS["tiny"]
    H, W, ids, tlog, _ = _host(w)
    out = run_gpu(kd, cuda_device, H, W, ids, tlog, None, chunk=128, grad_H_fp32=False)
    assert out["grad_H"].dtype == torch.bfloat16
    ref = oracle.dense_kl(bf16_bits(H), bf16_bits(W), ids.numpy(), tlog.numpy(), None)
    compare_full(out, ref)


@pytest.mark.parametrize("N,d,V,K,chunk", [
    (300, 72, 1000, 5, 128),      # ragged chunks (128, 128, 44), K-tail in d, vocab tail
    (257, 136, 1001, 33, 256),    # V not a multiple of 8 (padded dZ rows), 2 chunks, 1-row tail
    (128, 64, 256, 256, 128),     # K = V: the sparse teacher is the whole vocabulary
    (640, 520, 2560, 64, 384),    # several tiles in every direction
    (512, 192, 3000, 20, 256),    # CTA pairs, d = 3 k-blocks: the last stage's depth-2 box half past d
    (600, 320, 2100, 10, 256),    # CTA pairs over 5 k-blocks, then a single-CTA 88-row chunk
    (200, 64, 1500, 300, 128),    # K = 300: the prologue sorts 16 entries per lane
    (130, 64, 1024, 1024, 128),   # K = V = 1024 (the largest K): 32 entries per lane
])
def test_ragged_shapes(kd, cuda_device, N, d, V, K, chunk):
    w = Workload("ragged", 1, N, d, V, K, chunk, "normal3", 0.9, 4242 + N)
    H, W, ids, tlog, mask = _host(w)
    out = run_gpu(kd, cuda_device, H, W, ids, tlog, mask, chunk=chunk)
    ref = oracle.dense_kl(bf16_bits(H), bf16_bits(W), ids.numpy(), tlog.numpy(), mask.numpy())
    compare_full(out, ref)


def test_chunk_size_invariance(kd, cuda_device):
    w = Workload("inv", 1, 1024, 256, 5000, 20, 1024, "zipf", 1.0, 77)
    H, W, ids, tlog, _ = _host(w)
    res = [run_gpu(kd, cuda_device, H, W, ids, tlog, None, chunk=c) for c in (128, 384, 1024)]
    for r in res[1:]:
        assert abs(r["loss"].item() - res[0]["loss"].item()) <= 1e-5 * abs(res[0]["loss"].item())
        assert maxrel(r["grad_W"].cpu().numpy(), res[0]["grad_W"].cpu().numpy()) <= 1e-5


def test_small_workload_reduced_rows(kd, cuda_device):
    """The small LM shape (d=2048, V=32000, K=100, Zipf teacher, 5% padding) on 512 positions, 2 chunks."""
    w = WORKLOADS["small"]
    H, W, ids, tlog, mask = _host(w, rows=512)
    out = run_gpu(kd, cuda_device, H, W, ids, tlog, mask, chunk=256)
    ref = oracle.dense_kl(bf16_bits(H), bf16_bits(W), ids.numpy(), tlog.numpy(), mask.numpy())
    compare_full(out, ref)


def test_kl_zero_construction(kd, cuda_device):
    """Student softmax on the cached ids equals the teacher's, negligible mass elsewhere: KL = 0.

    H = I (d = N) makes z_t = W[:, t] exactly; all values are bf16-representable.
    """
    N, V, K = 128, 4096, 16
    g = torch.Generator().manual_seed(9)
    ids = torch.stack([torch.randperm(V, generator=g)[:K] for _ in range(N)]).to(torch.int32)
    tlog = torch.sort(torch.randn((N, K), generator=g) * 3, dim=1, descending=True)[0]
    tlog = tlog.to(torch.bfloat16).float()
    shift = (torch.randn(N, generator=g) * 2).to(torch.bfloat16).float()
    H = torch.eye(N, dtype=torch.bfloat16)
    W = torch.full((V, N), -9984.0)
    for t in range(N):
        W[ids[t].long(), t] = (tlog[t] + shift[t]).to(torch.bfloat16).float()
    W = W.to(torch.bfloat16)
    tl = (W.float().T.gather(1, ids.long()) - shift[:, None]).contiguous()   # teacher logits the student realises
    out = run_gpu(kd, cuda_device, H, W, ids, tl, None, chunk=128)
    assert out["kl"].abs().max().item() <= 1e-4
    assert abs(out["loss"].item()) <= 1e-4
    assert out["grad_H"].abs().max().item() <= 1e-4


def test_zero_valid_positions(kd, cuda_device):
    w = WORKLOADS["tiny"]
    H, W, ids, tlog, _ = _host(w)
    mask = torch.zeros(w.N, dtype=torch.uint8)
    out = run_gpu(kd, cuda_device, H, W, ids, tlog, mask, chunk=128)
    assert out["loss"].item() == 0.0
    assert torch.all(out["grad_H"] == 0) and torch.all(out["grad_W"] == 0)


def test_grad_W_accumulates(kd, cuda_device):
    w = WORKLOADS["tiny"]
    H, W, ids, tlog, _ = _host(w)
    dev = cuda_device
    Hd, Wd, idd, tld = (t.to(dev) for t in (H, W, ids, tlog))
    loss, lse, ws = kd.fused_kl_forward(Hd, Wd, idd, tld, None, 128)
    g = torch.ones(1, device=dev)
    _, gW1 = kd.fused_kl_backward(Hd, Wd, idd, tld, None, lse, g, 128, ws=ws)
    base = torch.randn(gW1.shape, device=dev)
    _, gW2 = kd.fused_kl_backward(Hd, Wd, idd, tld, None, lse, g, 128, ws=ws, grad_W=base.clone())
    torch.cuda.synchronize()
    assert torch.allclose(gW2, gW1 + base, atol=1e-6, rtol=0)


def test_bad_teacher_id_is_reported(kd, cuda_device):
    w = WORKLOADS["tiny"]
    H, W, ids, tlog, _ = _host(w)
    ids = ids.clone()
    ids[77, 3] = w.V            # out of range: recorded, never used as an address
    dev = cuda_device
    loss, lse, ws = kd.fused_kl_forward(H.to(dev), W.to(dev), ids.to(dev), tlog.to(dev), None, 128)
    st, detail = kd.device_error(ws)
    assert st == kd._abi.KD_ERR_DEVICE and detail == 77
    assert kd.device_error(ws)[0] == 0      # reading clears it


def test_autograd_function(kd, cuda_device):
    w = WORKLOADS["tiny"]
    H, W, ids, tlog, _ = _host(w)
    dev = cuda_device
    Hd = H.to(dev).requires_grad_(True)
    Wd = W.to(dev).requires_grad_(True)
    loss = kd.fused_kl(Hd, Wd, ids.to(dev), tlog.to(dev), None, chunk=128)
    (2.0 * loss).backward()
    ref = oracle.dense_kl(bf16_bits(H), bf16_bits(W), ids.numpy(), tlog.numpy(), None, grad_loss=2.0)
    assert abs(loss.item() - ref.loss) <= LOSS_RTOL * ref.loss
    assert Hd.grad.dtype == torch.bfloat16 and Wd.grad.dtype == torch.bfloat16
    assert maxrel(Hd.grad.double().cpu().numpy(), ref.grad_H) <= GRAD_TOL
    assert maxrel(Wd.grad.double().cpu().numpy(), ref.grad_W) <= GRAD_TOL


# ----------------------------------------------------------------------------
# Full-size workloads: the GPU runs the whole shape; the oracle checks a seeded
# subset S of positions spread over every chunk.  Forward: per-position KL and
# logsumexp on S, and the loss against the fp64 mean of the GPU's own per-position
# KL.  Backward: a second run with the mask restricted to S, whose gradients the
# oracle computes from the S rows alone (grad_H on S, grad_W on sampled vocab rows).

def _subset(N, chunk, n=96, seed=0):
    rng = np.random.default_rng(seed)
    starts = np.arange(0, N, chunk)
    edge = np.concatenate([starts, np.minimum(starts + chunk - 1, N - 1)])
    rows = np.unique(np.concatenate([edge, rng.choice(N, n, replace=False)]))
    return rows


@pytest.mark.parametrize("name", ["small", "mid", "gptoss", "headline"])
def test_full_workload_masked_subset(kd, cuda_device, name):
    w = WORKLOADS[name]
    dev = cuda_device
    H, W, ids, tlog, mask = make_inputs(w, dev)
    N = w.N
    out = run_gpu(kd, dev, H, W, ids, tlog, mask, chunk=w.chunk, want_bwd=False)
    kl = out["kl"].double().cpu().numpy()
    valid = np.ones(N, bool) if mask is None else mask.cpu().numpy().astype(bool)
    assert np.all(np.isfinite(kl)) and np.all(kl >= -1e-3)
    assert abs(out["loss"].item() - kl[valid].mean()) <= 1e-5 * abs(kl[valid].mean())

    S = _subset(N, w.chunk, seed=w.seed)
    S = S[valid[S]]
    St = torch.as_tensor(S, device=dev)
    Hs, ids_s, tl_s = bf16_bits(H[St]), ids[St].cpu().numpy(), tlog[St].cpu().numpy()
    Wb = bf16_bits(W)
    rng = np.random.default_rng(1)
    vrows = np.unique(np.concatenate([ids_s.ravel()[:2000], rng.choice(w.V, 512, replace=False), [0, w.V - 1]]))
    ref = oracle.fused_chunked_kl(Hs, Wb, ids_s, tl_s, None, 1.0, chunk=len(S), vtile=8192, vocab_rows=vrows)
    assert maxrel(out["lse"].cpu().numpy()[S], ref.lse) <= ROW_TOL
    assert maxrel(kl[S], ref.kl) <= ROW_TOL

    mask_s = torch.zeros(N, dtype=torch.uint8, device=dev)
    mask_s[St] = 1
    out2 = run_gpu(kd, dev, H, W, ids, tlog, mask_s, chunk=w.chunk)
    assert abs(out2["loss"].item() - ref.loss) <= LOSS_RTOL * abs(ref.loss)
    gH = out2["grad_H"]
    assert maxrel(gH[St].double().cpu().numpy(), ref.grad_H) <= GRAD_TOL
    others = torch.ones(N, dtype=torch.bool, device=dev)
    others[St] = False
    assert torch.all(gH[others] == 0)
    gW = out2["grad_W"][torch.as_tensor(vrows, device=dev)].double().cpu().numpy()
    assert maxrel(gW, ref.grad_W) <= GRAD_TOL


# ----------------------------------------------------------------------------
# Forward-chunked mode: the forward keeps each chunk's logits (bf16), the backward
# reads them instead of recomputing.  Checked against the oracle's forward-chunked
# formulation (which keeps float64 logits) with the same tolerances, and against
# the fused path's own forward (same arithmetic, so equal up to launch order).

def run_chunked(kd, dev, H, W, ids, tlog, mask, chunk, tau=1.0, grad=1.0):
    Hd, Wd, idd, tld = (t.to(dev).contiguous() for t in (H, W, ids, tlog))
    md = None if mask is None else mask.to(dev).contiguous()
    kl = torch.empty(Hd.shape[0], dtype=torch.float32, device=dev)
    loss, lse, ws, z = kd.chunked_kl_forward(Hd, Wd, idd, tld, md, chunk, tau, kl_out=kl)
    g = torch.full((1,), grad, dtype=torch.float32, device=dev)
    gH, gW = kd.chunked_kl_backward(Hd, Wd, idd, tld, md, lse, g, z, chunk, tau, ws=ws, grad_H_fp32=True)
    torch.cuda.synchronize()
    assert kd.device_error(ws)[0] == 0
    return dict(loss=loss, lse=lse, kl=kl, grad_H=gH, grad_W=gW, z=z)


@pytest.mark.parametrize("N,d,V,K,chunk,tau", [
    (128, 256, 4096, 16, 128, 1.0),
    (300, 72, 1000, 5, 128, 1.0),
    (257, 136, 1001, 33, 256, 2.0),
])
def test_forward_chunked_matches_oracle(kd, cuda_device, N, d, V, K, chunk, tau):
    w = Workload("fc", 1, N, d, V, K, chunk, "normal3", 0.9, 777 + N)
    H, W, ids, tlog, mask = _host(w)
    out = run_chunked(kd, cuda_device, H, W, ids, tlog, mask, chunk, tau, grad=0.5)
    ref = oracle.forward_chunked_kl(bf16_bits(H), bf16_bits(W), ids.numpy(), tlog.numpy(), mask.numpy(), tau,
                                    chunk=chunk, grad_loss=0.5)
    compare_full(out, ref)
    fused = run_gpu(kd, cuda_device, H, W, ids, tlog, mask, chunk=chunk, tau=tau, want_bwd=False)
    assert abs(out["loss"].item() - fused["loss"].item()) <= 1e-6 * abs(fused["loss"].item())
    # the kept logits are H W^T rounded to bf16, in the blocked layout
    nvb = (V + 63) // 64
    zb = out["z"].view(torch.int16).view(nvb, N, 64).permute(1, 0, 2).reshape(N, nvb * 64)[:, :V]
    zg = zb.contiguous().view(torch.bfloat16).double().cpu().numpy()
    zr = oracle.bf16_to_f64(bf16_bits(H)) @ oracle.bf16_to_f64(bf16_bits(W)).T
    assert np.max(np.abs(zg - zr) / (np.abs(zr) + 1e-3)) <= 2.0 ** -7
