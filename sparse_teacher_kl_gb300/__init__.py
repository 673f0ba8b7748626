"""Fused chunked KL distillation against an offline top-K teacher cache, on GB300.

PyTorch supplies device memory and the current stream; every step of the path
runs in the CUDA kernels of ``libkdkl.so`` (see ``include/kdkl.h``).

    from sparse_teacher_kl_gb300 import topk_cache, fused_kl
    ids, vals = topk_cache(teacher_logits_bf16, K=100)          # offline cache
    loss = fused_kl(H, W, ids, vals, mask, chunk=4096)          # drop-in KL term
    loss.backward()                                             # recompute per chunk
"""
from __future__ import annotations

import ctypes
from typing import Optional

import torch

from . import _abi
from ._abi import KDError, KD_MAX_K

__all__ = [
    "topk_cache",
    "teacher_topk",
    "fused_kl",
    "fused_kl_forward",
    "fused_kl_backward",
    "chunked_kl_forward",
    "chunked_kl_backward",
    "gemm_bf16",
    "cache_write",
    "cache_info",
    "cache_read",
    "CacheReader",
    "device_error",
    "Profile",
    "KDError",
    "KD_MAX_K",
    "workspace",
]


def _ptr(t: Optional[torch.Tensor]) -> Optional[int]:
    return None if t is None else t.data_ptr()


def _stream(device) -> int:
    return torch.cuda.current_stream(device).cuda_stream


def workspace(nbytes: int, device) -> torch.Tensor:
    """A 256-byte aligned uint8 device buffer of at least ``nbytes`` (zeroed control block)."""
    buf = torch.zeros(int(nbytes) + 256, dtype=torch.uint8, device=device)
    off = (-buf.data_ptr()) % 256
    return buf[off:off + int(nbytes)]


def _require_cuda(*ts):
    for t in ts:
        if t is not None and not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors")
        if t is not None and not t.is_contiguous():
            raise ValueError("all tensors must be contiguous")


def topk_cache(logits: torch.Tensor, K: int, ws: Optional[torch.Tensor] = None, with_lse: bool = False,
               with_dropped: bool = False):
    """Top-K teacher cache of a dense bf16 [N, V] logits tensor: (ids int32 [N, K], vals fp32 [N, K]), then,
    when asked, the full-row logsumexp [N] (``with_lse``) and the teacher probability outside the K kept
    logits [N] (``with_dropped``), both computed by the kernel in the same pass."""
    _require_cuda(logits)
    if logits.dtype != torch.bfloat16 or logits.dim() != 2:
        raise ValueError("logits must be a 2-D bf16 tensor")
    N, V = logits.shape
    dev = logits.device
    ids = torch.empty((N, K), dtype=torch.int32, device=dev)
    vals = torch.empty((N, K), dtype=torch.float32, device=dev)
    if ws is None:
        ws = workspace(_abi.kd_topk_cache_workspace(N, V, K), dev)
    lse = torch.empty((N,), dtype=torch.float32, device=dev) if with_lse else None
    dropped = torch.empty((N,), dtype=torch.float32, device=dev) if with_dropped else None
    st = _abi.kd_topk_cache(_ptr(logits), N, V, logits.stride(0), K, _ptr(ids), _ptr(vals), _ptr(lse), _ptr(dropped),
                            _ptr(ws), ws.numel(), _stream(dev))
    _abi.check(st, "kd_topk_cache")
    return (ids, vals) + ((lse,) if with_lse else ()) + ((dropped,) if with_dropped else ())


def teacher_topk(Ht: torch.Tensor, Wt: torch.Tensor, K: int, chunk: int = 1024, with_lse: bool = False,
                 with_dropped: bool = False, ws: Optional[torch.Tensor] = None):
    """Top-K cache straight from teacher hidden states Ht [N, dt] and LM-head Wt [V, dt] (bf16): the
    teacher logits exist only one chunk at a time (see kd_teacher_topk).  Returns as topk_cache."""
    _require_cuda(Ht, Wt)
    N, dt = Ht.shape
    V = Wt.shape[0]
    dev = Ht.device
    ids = torch.empty((N, K), dtype=torch.int32, device=dev)
    vals = torch.empty((N, K), dtype=torch.float32, device=dev)
    lse = torch.empty((N,), dtype=torch.float32, device=dev) if with_lse else None
    dropped = torch.empty((N,), dtype=torch.float32, device=dev) if with_dropped else None
    if ws is None:
        ws = workspace(_abi.kd_teacher_topk_workspace(N, dt, V, K, chunk), dev)
    st = _abi.kd_teacher_topk(_ptr(Ht), _ptr(Wt), N, dt, V, K, chunk, _ptr(ids), _ptr(vals), _ptr(lse), _ptr(dropped),
                              _ptr(ws), ws.numel(), _stream(dev))
    _abi.check(st, "kd_teacher_topk")
    return (ids, vals) + ((lse,) if with_lse else ()) + ((dropped,) if with_dropped else ())


def fused_kl_forward(H, W, ids, tlog, mask=None, chunk=4096, tau=1.0, ws=None, kl_out=None):
    """kd_fused_kl_fwd: returns (loss [1] fp32, lse [N] fp32, ws)."""
    _require_cuda(H, W, ids, tlog, mask)
    N, d = H.shape
    V = W.shape[0]
    K = ids.shape[1]
    if ws is None:
        ws = workspace(_abi.kd_fused_kl_workspace(N, d, V, K, chunk), H.device)
    loss = torch.empty((1,), dtype=torch.float32, device=H.device)
    lse = torch.empty((N,), dtype=torch.float32, device=H.device)
    st = _abi.kd_fused_kl_fwd(_ptr(H), _ptr(W), _ptr(ids), _ptr(tlog), _ptr(mask), N, d, V, K, chunk, float(tau),
                              _ptr(loss), _ptr(lse), _ptr(kl_out), _ptr(ws), ws.numel(), _stream(H.device))
    _abi.check(st, "kd_fused_kl_fwd")
    return loss, lse, ws


def fused_kl_backward(H, W, ids, tlog, mask, lse, grad_loss, chunk=4096, tau=1.0, ws=None, grad_H=None,
                      grad_W=None, grad_H_fp32=False):
    """kd_fused_kl_bwd: returns (grad_H [N, d] bf16 or fp32, grad_W [V, d] fp32 accumulated)."""
    _require_cuda(H, W, ids, tlog, mask, lse, grad_loss)
    N, d = H.shape
    V = W.shape[0]
    K = ids.shape[1]
    if ws is None:
        ws = workspace(_abi.kd_fused_kl_workspace(N, d, V, K, chunk), H.device)
    if grad_H is None:
        grad_H = torch.empty((N, d), dtype=torch.float32 if grad_H_fp32 else torch.bfloat16, device=H.device)
    if grad_W is None:
        grad_W = torch.zeros((V, d), dtype=torch.float32, device=H.device)
    st = _abi.kd_fused_kl_bwd(_ptr(H), _ptr(W), _ptr(ids), _ptr(tlog), _ptr(mask), N, d, V, K, chunk, float(tau),
                              _ptr(lse), _ptr(grad_loss), _ptr(grad_H), 1 if grad_H.dtype == torch.float32 else 0,
                              _ptr(grad_W), _ptr(ws), ws.numel(), _stream(H.device))
    _abi.check(st, "kd_fused_kl_bwd")
    return grad_H, grad_W


def chunked_kl_forward(H, W, ids, tlog, mask=None, chunk=4096, tau=1.0, ws=None, kl_out=None, z_store=None):
    """kd_chunked_kl_fwd (forward-chunked mode): returns (loss, lse, ws, z_store); z_store keeps the logits."""
    _require_cuda(H, W, ids, tlog, mask)
    N, d = H.shape
    V = W.shape[0]
    K = ids.shape[1]
    if ws is None:
        ws = workspace(_abi.kd_fused_kl_workspace(N, d, V, K, chunk), H.device)
    zb = _abi.kd_chunked_kl_logits_bytes(N, V)
    if z_store is None:
        z_store = torch.empty((zb,), dtype=torch.uint8, device=H.device)
    loss = torch.empty((1,), dtype=torch.float32, device=H.device)
    lse = torch.empty((N,), dtype=torch.float32, device=H.device)
    st = _abi.kd_chunked_kl_fwd(_ptr(H), _ptr(W), _ptr(ids), _ptr(tlog), _ptr(mask), N, d, V, K, chunk, float(tau),
                                _ptr(loss), _ptr(lse), _ptr(kl_out), _ptr(z_store), z_store.numel(), _ptr(ws),
                                ws.numel(), _stream(H.device))
    _abi.check(st, "kd_chunked_kl_fwd")
    return loss, lse, ws, z_store


def chunked_kl_backward(H, W, ids, tlog, mask, lse, grad_loss, z_store, chunk=4096, tau=1.0, ws=None, grad_H=None,
                        grad_W=None, grad_H_fp32=False):
    """kd_chunked_kl_bwd: gradients from the logits kept by chunked_kl_forward (no recompute)."""
    _require_cuda(H, W, ids, tlog, mask, lse, grad_loss, z_store)
    N, d = H.shape
    V = W.shape[0]
    K = ids.shape[1]
    if ws is None:
        ws = workspace(_abi.kd_fused_kl_workspace(N, d, V, K, chunk), H.device)
    if grad_H is None:
        grad_H = torch.empty((N, d), dtype=torch.float32 if grad_H_fp32 else torch.bfloat16, device=H.device)
    if grad_W is None:
        grad_W = torch.zeros((V, d), dtype=torch.float32, device=H.device)
    st = _abi.kd_chunked_kl_bwd(_ptr(H), _ptr(W), _ptr(ids), _ptr(tlog), _ptr(mask), N, d, V, K, chunk, float(tau),
                                _ptr(lse), _ptr(grad_loss), _ptr(z_store), z_store.numel(), _ptr(grad_H),
                                1 if grad_H.dtype == torch.float32 else 0, _ptr(grad_W), _ptr(ws), ws.numel(),
                                _stream(H.device))
    _abi.check(st, "kd_chunked_kl_bwd")
    return grad_H, grad_W


class _FusedKL(torch.autograd.Function):
    @staticmethod
    def forward(ctx, H, W, ids, tlog, mask, chunk, tau):
        loss, lse, ws = fused_kl_forward(H, W, ids, tlog, mask, chunk, tau)
        ctx.save_for_backward(H, W, ids, tlog, lse)
        ctx.mask = mask
        ctx.chunk, ctx.tau, ctx.ws = chunk, tau, ws
        return loss[0]

    @staticmethod
    def backward(ctx, grad_out):
        H, W, ids, tlog, lse = ctx.saved_tensors
        g = grad_out.reshape(1).to(torch.float32).contiguous()
        grad_H, grad_W = fused_kl_backward(H, W, ids, tlog, ctx.mask, lse, g, ctx.chunk, ctx.tau, ws=ctx.ws)
        return grad_H.to(H.dtype), grad_W.to(W.dtype), None, None, None, None, None


def fused_kl(H, W, ids, tlog, mask=None, chunk=4096, tau=1.0):
    """Differentiable fused chunked KL(p_teacher || q_student) token mean (scalar tensor)."""
    return _FusedKL.apply(H, W, ids, tlog, mask, int(chunk), float(tau))


def gemm_bf16(A, B, M, N, K, a_mn_major=False, b_mn_major=False, C=None):
    """The projection engine on its own: C[M, N] fp32 = A·B (see kd_gemm_bf16)."""
    _require_cuda(A, B)
    if C is None:
        C = torch.empty((M, N), dtype=torch.float32, device=A.device)
        acc = 0
    else:
        acc = 1
    ws = workspace(_abi.kd_gemm_workspace(), A.device)
    st = _abi.kd_gemm_bf16(_ptr(A), _ptr(B), _ptr(C), M, N, K, int(a_mn_major), int(b_mn_major), acc, _ptr(ws),
                           ws.numel(), _stream(A.device))
    _abi.check(st, "kd_gemm_bf16")
    return C, ws


def device_error(ws: torch.Tensor):
    """(status, detail) of a workspace's device error word; synchronises the current stream."""
    detail = ctypes.c_int64(0)
    st = _abi.kd_get_device_error(_ptr(ws), _stream(ws.device), ctypes.byref(detail))
    return st, detail.value


# ---------------------------------------------------------------- disk cache

def _host_c(t, dtype):
    t = torch.as_tensor(t)
    if t.is_cuda:
        t = t.cpu()
    return t.to(dtype).contiguous()


def cache_write(path: str, ids, vals, V: int, lse=None, row0: int = 0, bf16: bool = False):
    """Write a top-K cache shard (host copies of ids [N, K] int32, vals [N, K] fp32, lse [N] or None)."""
    ids = _host_c(ids, torch.int32)
    vals = _host_c(vals, torch.float32)
    N, K = ids.shape
    lse_t = None if lse is None else _host_c(lse, torch.float32)
    st = _abi.kd_cache_write(str(path).encode(), ids.data_ptr(), vals.data_ptr(), _ptr(lse_t), N, K, int(V),
                             int(row0), int(bool(bf16)))
    _abi.check(st, "kd_cache_write")


def cache_info(path: str) -> dict:
    N, K, V, row0, bf, hl = (ctypes.c_int64(), ctypes.c_int(), ctypes.c_int64(), ctypes.c_int64(), ctypes.c_int(),
                             ctypes.c_int())
    st = _abi.kd_cache_info(str(path).encode(), ctypes.byref(N), ctypes.byref(K), ctypes.byref(V), ctypes.byref(row0),
                            ctypes.byref(bf), ctypes.byref(hl))
    _abi.check(st, "kd_cache_info")
    return dict(N=N.value, K=K.value, V=V.value, row0=row0.value, bf16=bool(bf.value), has_lse=bool(hl.value))


def cache_read(path: str, first: int = 0, count: Optional[int] = None, with_lse: bool = False, pin: bool = False):
    """Read positions [first, first + count) of a shard into (pinned, if asked) host tensors."""
    info = cache_info(path)
    if count is None:
        count = info["N"] - first
    K = info["K"]
    ids = torch.empty((count, K), dtype=torch.int32, pin_memory=pin)
    vals = torch.empty((count, K), dtype=torch.float32, pin_memory=pin)
    lse = torch.empty((count,), dtype=torch.float32, pin_memory=pin) if with_lse else None
    st = _abi.kd_cache_read(str(path).encode(), int(first), int(count), ids.data_ptr(), vals.data_ptr(), _ptr(lse))
    _abi.check(st, "kd_cache_read")
    return (ids, vals, lse) if with_lse else (ids, vals)


class CacheReader:
    """Iterate a shard in batches of consecutive positions; the next batch is read from disk on a
    background thread (native) while the current one is in use.  Yields (ids, vals) host tensors."""

    def __init__(self, path: str, rows_per_batch: int, pin: bool = False):
        self.info = cache_info(path)
        self.rows = int(rows_per_batch)
        self.pin = pin
        self._h = ctypes.c_void_p()
        _abi.check(_abi.kd_cache_reader_open(str(path).encode(), self.rows, ctypes.byref(self._h)),
                   "kd_cache_reader_open")

    def __iter__(self):
        K = self.info["K"]
        while True:
            ids = torch.empty((self.rows, K), dtype=torch.int32, pin_memory=self.pin)
            vals = torch.empty((self.rows, K), dtype=torch.float32, pin_memory=self.pin)
            n = ctypes.c_int64(0)
            _abi.check(_abi.kd_cache_reader_next(self._h, ids.data_ptr(), vals.data_ptr(), ctypes.byref(n)),
                       "kd_cache_reader_next")
            if n.value == 0:
                return
            yield ids[:n.value], vals[:n.value]

    def close(self):
        if self._h:
            _abi.kd_cache_reader_close(self._h)
            self._h = ctypes.c_void_p()

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()
        return False

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class Profile:
    """Per-launch CUDA-event timing of the library's kernels while the context is open."""

    def __init__(self, capacity: int = 4096):
        self.capacity = capacity
        self.records = []

    def __enter__(self):
        _abi.check(_abi.kd_profile_begin(self.capacity), "kd_profile_begin")
        return self

    def __exit__(self, *exc):
        _abi.kd_profile_end()
        n = self.capacity
        names = (ctypes.c_char_p * n)()
        ms = (ctypes.c_float * n)()
        got = _abi.kd_profile_read(names, ms, n)
        if got < 0:
            raise KDError(-got, "kd_profile_read")
        self.records = [(names[i].decode(), ms[i]) for i in range(min(got, n))]
        return False

    def summary(self):
        out = {}
        for name, t in self.records:
            c, tot = out.get(name, (0, 0.0))
            out[name] = (c + 1, tot + t)
        return out
