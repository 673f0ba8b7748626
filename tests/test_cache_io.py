"""The on-disk teacher cache (native C++ host code, no GPU): exact round trips in
fp32 and bf16, row-range reads, the streaming reader, and detection of corrupt,
truncated or foreign files."""
import os

import numpy as np
import pytest
import torch

import sparse_teacher_kl_gb300 as kd
from sparse_teacher_kl_gb300 import _abi
from sparse_teacher_kl_gb300.build import build_library


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build_library()
    _abi.load()


def _cache(N=37, K=5, V=1000, seed=0, bf16_exact=True):
    g = torch.Generator().manual_seed(seed)
    ids = torch.stack([torch.randperm(V, generator=g)[:K] for _ in range(N)]).to(torch.int32)
    vals = torch.sort(torch.randn((N, K), generator=g) * 3, dim=1, descending=True)[0]
    if bf16_exact:
        vals = vals.to(torch.bfloat16).float()
    lse = torch.randn(N, generator=g) + 10
    return ids, vals, lse


@pytest.mark.parametrize("bf16", [False, True])
def test_round_trip(tmp_path, bf16):
    ids, vals, lse = _cache()
    p = tmp_path / "shard0.kdtopk"
    kd.cache_write(p, ids, vals, V=1000, lse=lse, row0=4096, bf16=bf16)
    info = kd.cache_info(p)
    assert info == dict(N=37, K=5, V=1000, row0=4096, bf16=bf16, has_lse=True)
    assert _abi.kd_cache_verify(str(p).encode()) == 0
    rid, rval, rlse = kd.cache_read(p, with_lse=True)
    assert torch.equal(rid, ids) and torch.equal(rval, vals) and torch.equal(rlse, lse)
    size = os.path.getsize(p)
    assert size == 64 + 37 * 5 * 4 + 37 * 5 * (2 if bf16 else 4) + 37 * 4


def test_bf16_storage_rounds_to_nearest_even(tmp_path):
    ids, vals, _ = _cache(bf16_exact=False)
    p = tmp_path / "s.kdtopk"
    kd.cache_write(p, ids, vals, V=1000, bf16=True)
    _, rval = kd.cache_read(p)
    assert torch.equal(rval, vals.to(torch.bfloat16).float())


def test_row_ranges_and_reader(tmp_path):
    ids, vals, _ = _cache(N=1000, K=7)
    p = tmp_path / "s.kdtopk"
    kd.cache_write(p, ids, vals, V=1000)
    rid, rval = kd.cache_read(p, 123, 456)
    assert torch.equal(rid, ids[123:579]) and torch.equal(rval, vals[123:579])
    got_i, got_v = [], []
    with kd.CacheReader(p, 128) as r:
        for bi, bv in r:
            got_i.append(bi.clone())
            got_v.append(bv.clone())
    assert [len(x) for x in got_i] == [128] * 7 + [104]
    assert torch.equal(torch.cat(got_i), ids) and torch.equal(torch.cat(got_v), vals)


def test_empty_shard(tmp_path):
    p = tmp_path / "e.kdtopk"
    kd.cache_write(p, torch.zeros((0, 4), dtype=torch.int32), torch.zeros((0, 4)), V=10)
    assert kd.cache_info(p)["N"] == 0
    with kd.CacheReader(p, 8) as r:
        assert list(r) == []


def test_corruption_and_truncation_are_detected(tmp_path):
    ids, vals, lse = _cache()
    p = tmp_path / "c.kdtopk"
    kd.cache_write(p, ids, vals, V=1000, lse=lse)
    raw = bytearray(p.read_bytes())
    raw[64 + 10] ^= 0x40                                   # flip a bit in the ids
    bad = tmp_path / "bad.kdtopk"
    bad.write_bytes(bytes(raw))
    assert _abi.kd_cache_verify(str(bad).encode()) == _abi.KD_ERR_IO
    short = tmp_path / "short.kdtopk"
    short.write_bytes(p.read_bytes()[:-3])
    with pytest.raises(kd.KDError) as e:
        kd.cache_info(short)
    assert e.value.status == _abi.KD_ERR_IO
    foreign = tmp_path / "foreign.bin"
    foreign.write_bytes(b"\0" * 200)
    with pytest.raises(kd.KDError) as e:
        kd.cache_info(foreign)
    assert e.value.status == _abi.KD_ERR_UNSUPPORTED
    with pytest.raises(kd.KDError):
        kd.cache_read(p, 30, 10)                            # past the end
    with pytest.raises(kd.KDError) as e:
        kd.cache_info(tmp_path / "missing.kdtopk")
    assert e.value.status == _abi.KD_ERR_IO


def test_write_rejects_bad_arguments(tmp_path):
    ids, vals, _ = _cache()
    with pytest.raises(kd.KDError):
        kd.cache_write(tmp_path / "x", ids, vals, V=3)        # V < K
    assert _abi.kd_cache_write(None, None, None, None, 1, 1, 1, 0, 0) == _abi.KD_ERR_INVALID_ARG
    with pytest.raises(kd.KDError) as e:
        kd.cache_write(tmp_path / "no_such_dir" / "x", ids, vals, V=1000)
    assert e.value.status == _abi.KD_ERR_IO
