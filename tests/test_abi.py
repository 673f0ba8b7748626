"""The C-ABI library builds, loads and exports what include/kdkl.h declares;
host-side argument checks reject bad calls before any CUDA work (no GPU needed)."""
import ctypes
import os
import subprocess

import pytest

from sparse_teacher_kl_gb300 import _abi
from sparse_teacher_kl_gb300.build import build_library, LIB


@pytest.fixture(scope="module")
def lib():
    build_library()
    return _abi.load()


def test_header_names_are_exported(lib):
    names = _abi.header_functions()
    assert {"kd_topk_cache", "kd_fused_kl_fwd", "kd_fused_kl_bwd", "kd_fused_kl_workspace",
            "kd_topk_cache_workspace", "kd_get_device_error", "kd_status_string"} <= set(names)
    out = subprocess.run(["nm", "-D", "--defined-only", LIB], capture_output=True, text=True, check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if " T " in ln}
    missing = [n for n in names if n not in exported]
    assert not missing, f"declared but not exported: {missing}"
    extra = sorted(n for n in exported if n.startswith("kd_") and n not in names)
    assert not extra, f"exported but not declared: {extra}"
    for n in names:
        assert hasattr(lib, n)


def test_status_strings(lib):
    assert _abi.status_string(0) == "KD_OK"
    assert _abi.status_string(1) == "KD_ERR_INVALID_ARG"
    assert _abi.status_string(5) == "KD_ERR_TIMEOUT"
    assert _abi.status_string(99) == "KD_ERR_UNKNOWN"
    assert lib.kd_version() >= 100


def test_workspace_queries_scale_with_chunk_not_sequence(lib):
    small = lib.kd_fused_kl_workspace(32768, 2880, 201088, 100, 1024)
    big_chunk = lib.kd_fused_kl_workspace(32768, 2880, 201088, 100, 4096)
    long_seq = lib.kd_fused_kl_workspace(131072, 2880, 201088, 100, 1024)
    assert big_chunk > 3 * small
    # only O(N) per-token floats grow with the sequence
    assert long_seq - small == pytest.approx((131072 - 32768) * 4, abs=1024)
    assert lib.kd_topk_cache_workspace(8192, 151936, 100) >= 256
    assert lib.kd_fused_kl_workspace(0, 1, 1, 1, 1) == 0


P = 1 << 20  # a fake, 256-aligned "device address"; never dereferenced on these paths


@pytest.mark.parametrize("args", [
    dict(N=0), dict(V=0), dict(K=0), dict(K=2000), dict(K=300, V=200), dict(ld=100, V=200),
    dict(ld=203, V=200), dict(ptr=None), dict(ptr=P + 2),
])
def test_topk_rejects_bad_arguments(lib, args):
    a = dict(N=4, V=256, ld=256, K=8, ptr=P)
    a.update(args)
    st = lib.kd_topk_cache(a["ptr"], a["N"], a["V"], a["ld"], a["K"], P, P, None, None, P, 4096, None)
    assert st == _abi.KD_ERR_INVALID_ARG


def test_topk_rejects_bad_workspace(lib):
    assert lib.kd_topk_cache(P, 4, 256, 256, 8, P, P, None, None, None, 4096, None) == _abi.KD_ERR_WORKSPACE
    assert lib.kd_topk_cache(P, 4, 256, 256, 8, P, P, None, None, P + 16, 4096, None) == _abi.KD_ERR_WORKSPACE
    assert lib.kd_topk_cache(P, 4, 256, 256, 8, P, P, None, None, P, 16, None) == _abi.KD_ERR_WORKSPACE
    assert lib.kd_topk_cache(P, 4, 256, 256, 8, P, P, P + 2, None, P, 4096, None) == _abi.KD_ERR_INVALID_ARG
    assert lib.kd_topk_cache(P, 4, 256, 256, 8, P, P, None, P + 2, P, 4096, None) == _abi.KD_ERR_INVALID_ARG


def _fwd(lib, **kw):
    a = dict(H=P, W=P, ids=P, tlog=P, mask=None, N=256, d=64, V=1000, K=8, chunk=128, tau=1.0,
             loss=P, lse=P, kl=None, ws=P, wsb=1 << 30)
    a.update(kw)
    return lib.kd_fused_kl_fwd(a["H"], a["W"], a["ids"], a["tlog"], a["mask"], a["N"], a["d"], a["V"], a["K"],
                               a["chunk"], a["tau"], a["loss"], a["lse"], a["kl"], a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw", [
    dict(N=0), dict(d=60), dict(d=0), dict(K=0), dict(K=1025), dict(K=2000, V=1000), dict(chunk=100),
    dict(chunk=0), dict(tau=0.0), dict(tau=-1.0), dict(tau=float("inf")), dict(tau=float("nan")),
    dict(H=None), dict(W=None), dict(ids=None), dict(tlog=None), dict(H=P + 8), dict(loss=None),
    dict(lse=None),
])
def test_fused_fwd_rejects_bad_arguments(lib, kw):
    assert _fwd(lib, **kw) == _abi.KD_ERR_INVALID_ARG


def test_fused_fwd_rejects_bad_workspace(lib):
    need = lib.kd_fused_kl_workspace(256, 64, 1000, 8, 128)
    assert _fwd(lib, wsb=need - 1) == _abi.KD_ERR_WORKSPACE
    assert _fwd(lib, ws=None) == _abi.KD_ERR_WORKSPACE
    assert _fwd(lib, ws=P + 64) == _abi.KD_ERR_WORKSPACE


def test_fused_bwd_rejects_bad_arguments(lib):
    f = lib.kd_fused_kl_bwd
    ok = (P, P, P, P, None, 256, 64, 1000, 8, 128, 1.0, P, P, P, 0, P, P, 1 << 30, None)
    for i, bad in [(11, None), (12, None), (13, None), (15, None), (13, P + 4), (5, -1), (10, 0.0)]:
        a = list(ok)
        a[i] = bad
        assert f(*a) == _abi.KD_ERR_INVALID_ARG, i


def test_gemm_rejects_bad_arguments(lib):
    ws = lib.kd_gemm_workspace()
    assert lib.kd_gemm_bf16(P, P, P, 0, 8, 8, 0, 0, 0, P, ws, None) == _abi.KD_ERR_INVALID_ARG
    assert lib.kd_gemm_bf16(P, P, P, 8, 6, 8, 0, 0, 0, P, ws, None) == _abi.KD_ERR_INVALID_ARG
    assert lib.kd_gemm_bf16(P, P, P, 8, 8, 12, 0, 0, 0, P, ws, None) == _abi.KD_ERR_INVALID_ARG
    assert lib.kd_gemm_bf16(P, P, P, 12, 8, 8, 1, 0, 0, P, ws, None) == _abi.KD_ERR_INVALID_ARG
    assert lib.kd_gemm_bf16(P, P, P, 8, 8, 8, 0, 0, 0, None, ws, None) == _abi.KD_ERR_WORKSPACE


def test_python_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_abi, "_lib", None)
    monkeypatch.setattr(_abi, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        _abi.load()
