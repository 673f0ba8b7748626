"""kd_topk_cache against the oracle's full sort: ids and values bit-exact."""
import numpy as np
import pytest
import torch

import oracle
from synth import WORKLOADS, bf16_bits, make_dense_teacher_logits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def kd(cuda_device):
    from sparse_teacher_kl_gb300.build import build_library
    build_library()
    import sparse_teacher_kl_gb300 as kd
    return kd


def _check(kd, X_host, K, dev, rows=None, ld=None):
    """Run the GPU on X_host (bf16 [N, V], optionally inside a wider [N, ld] buffer); compare rows."""
    N, V = X_host.shape
    if ld is None and V % 8 != 0:
        ld = (V + 7) // 8 * 8
    if ld is not None and ld != V:
        buf = torch.zeros((N, ld), dtype=torch.bfloat16)
        buf[:, :V] = X_host
        Xd = buf.to(dev)[:, :V]
    else:
        Xd = X_host.to(dev)
    ids = torch.empty((N, K), dtype=torch.int32, device=dev)
    vals = torch.empty((N, K), dtype=torch.float32, device=dev)
    ws = kd.workspace(kd._abi.kd_topk_cache_workspace(N, V, K), dev)
    lse = torch.empty((N,), dtype=torch.float32, device=dev)
    dropped = torch.empty((N,), dtype=torch.float32, device=dev)
    st = kd._abi.kd_topk_cache(Xd.data_ptr(), N, V, Xd.stride(0), K, ids.data_ptr(), vals.data_ptr(),
                               lse.data_ptr(), dropped.data_ptr(), ws.data_ptr(), ws.numel(),
                               torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert kd.device_error(ws) == (0, 0)
    rows = np.arange(N) if rows is None else np.asarray(rows)
    bits = bf16_bits(X_host[torch.as_tensor(rows)])
    ref_lse = oracle.teacher_logsumexp(bits)
    got_lse = lse.cpu().numpy()[rows].astype(np.float64)
    fin = np.isfinite(ref_lse)
    assert np.array_equal(np.isfinite(got_lse), fin)
    lse_tol = 1e-5 * max(1.0, np.max(np.abs(ref_lse[fin]), initial=1.0))
    assert np.max(np.abs(got_lse[fin] - ref_lse[fin]), initial=0.0) <= lse_tol
    # dropped mass 1 - sum_k exp(v_k - lse): d/d(lse) is at most 1, plus fp32 rounding of the sum
    ref_drop = oracle.dropped_mass(bits, K)
    got_drop = dropped.cpu().numpy()[rows].astype(np.float64)
    assert np.max(np.abs(got_drop[fin] - ref_drop[fin]), initial=0.0) <= lse_tol + 1e-5
    rid, rval = oracle.topk_cache(bits, K)
    gid = ids.cpu().numpy()[rows]
    gval = vals.cpu().numpy()[rows]
    assert np.array_equal(gid, rid), f"ids differ in {np.sum(np.any(gid != rid, axis=1))} rows"
    assert np.array_equal(gval.view(np.uint32), rval.view(np.uint32)), "values differ"


@pytest.mark.parametrize("N,V,K", [(64, 4096, 16), (33, 1000, 100), (8, 40000, 1024), (5, 8, 8), (3, 17, 1)])
def test_topk_random(kd, cuda_device, N, V, K):
    X = make_dense_teacher_logits(N, V, seed=N + V + K)
    _check(kd, X, K, cuda_device)


@pytest.mark.parametrize("N,V,K", [(700, 4097, 100), (650, 12289, 7), (610, 20483, 256), (400, 33333, 100),
                                   (257, 9000, 128), (333, 16411, 129)])
def test_topk_rows_of_many_steps(kd, cuda_device, N, V, K):
    """Rows of 17 to 131 warp steps with a ragged end, K on both sides of the boundary
    between the two buffer sizes and at the streaming path's limit."""
    X = make_dense_teacher_logits(N, V, seed=N * 7 + K)
    _check(kd, X, K, cuda_device)


# Resident row warps of the streaming path: one block of 15 (K <= 128) or 12 (K <= 256)
# per SM, 152 SMs; the cases below give every warp at least three rows.
@pytest.mark.parametrize("N,V,K", [(7000, 4097, 100), (5600, 6151, 256), (7001, 2053, 16), (6900, 3001, 7)])
def test_topk_many_rows_per_warp(kd, cuda_device, N, V, K):
    """Each warp streams several rows, its copies running on into the next row while it
    sorts the current one."""
    X = make_dense_teacher_logits(N, V, seed=N * 3 + K)
    _check(kd, X, K, cuda_device)


def _reselected(ws):
    """Rows the last top-K call on this workspace selected a second time (control block word 2)."""
    return int(ws[8:12].view(torch.int32).item())


def test_topk_speculative_start_misses(kd, cuda_device):
    """Rows whose first 4096 values sit far above the rest, so that the start extrapolated from
    them lies above the row's K-th value and the row is selected a second time, among rows of a
    few distinct values, rows with infinities, and rows whose scale and offset jump: every row
    exact against the oracle, and the control block's count shows that second selections ran."""
    g = torch.Generator().manual_seed(9)
    N, V = 3000, 30000
    X = torch.randn((N, V), generator=g)
    X = X * 10.0 ** (torch.rand((N, 1), generator=g) * 6 - 3) + torch.randint(-50, 51, (N, 1), generator=g).float()
    X[0::5, :4096] += 6.0 * X[0::5].std(dim=1, keepdim=True)    # the prefix far above the rest
    X[1::7] = torch.randint(-3, 4, (len(range(1, N, 7)), V), generator=g).float()  # few distinct values
    X[2::11, ::97] = float("inf")
    X[3::13, ::5] = float("-inf")
    X = X.to(torch.bfloat16)
    Xd = X.to(cuda_device)
    bits = bf16_bits(X)
    for K in (16, 100, 200):
        ws = kd.workspace(kd._abi.kd_topk_cache_workspace(N, V, K), cuda_device)
        ids, vals = kd.topk_cache(Xd, K, ws=ws)
        torch.cuda.synchronize()
        assert kd.device_error(ws) == (0, 0)
        rid, rval = oracle.topk_cache(bits, K)
        assert np.array_equal(ids.cpu().numpy(), rid), K
        assert np.array_equal(vals.cpu().numpy().view(np.uint32), rval.view(np.uint32)), K
        assert _reselected(ws) > 0, K


def test_topk_ties_and_signed_zero(kd, cuda_device):
    g = torch.Generator().manual_seed(1)
    N, V = 12, 20000
    X = (torch.round(torch.randn((N, V), generator=g) * 2) / 2)
    X[0] = 0.0                                   # all equal: lowest ids win
    X[1, ::2] = -0.0                             # -0 == +0
    X[2] = torch.linspace(-3, 3, V)              # ascending: every element enters the buffer
    X[3] = torch.linspace(3, -3, V)              # descending
    X[4, :] = float("-inf"); X[4, 5000:5003] = 1.0
    X[5] = torch.round(torch.randn(V, generator=g)) * 0 + 7.0
    X[5, 19990:] = 8.0                           # best values at the very end
    X = X.to(torch.bfloat16)
    for K in (1, 100, 1024):
        _check(kd, X, K, cuda_device)


def test_topk_strided_rows(kd, cuda_device):
    X = make_dense_teacher_logits(20, 1001, seed=5)
    _check(kd, X, 50, cuda_device, ld=1008)


def test_topk_small_workload(kd, cuda_device):
    w = WORKLOADS["small"]
    X = make_dense_teacher_logits(256, w.V, seed=w.seed)
    _check(kd, X, w.K, cuda_device)


def _oracle_rows_parallel(bits, K, block=256):
    """oracle.topk_cache and oracle.teacher_logsumexp over every row of a large host array, in
    row blocks on a pool of spawned workers (the oracle is a per-row sort; spawned, not
    forked, because this process already holds a CUDA context)."""
    import multiprocessing as mp
    import os
    from functools import partial
    N = bits.shape[0]
    blocks = [bits[i:i + block] for i in range(0, N, block)]
    workers = max(1, min(len(os.sched_getaffinity(0)), 32))
    with mp.get_context("spawn").Pool(workers) as pool:
        tk = pool.map(partial(oracle.topk_cache, K=K), blocks)
        lse = pool.map(oracle.teacher_logsumexp, blocks)
    return (np.concatenate([t[0] for t in tk]), np.concatenate([t[1] for t in tk]), np.concatenate(lse))


def test_topk_mid_workload_every_row(kd, cuda_device):
    """The 8192 x 151936 dense teacher logits N(0, 2), K = 100: three launches (one with the row
    logsumexp), every row of each compared with the oracle: ids and value bits exact, logsumexp
    within 1e-5 of its magnitude.  Three launches so that a fault that strikes about once per
    launch (a race between a ring refill and a read, say) cannot pass unseen."""
    w = WORKLOADS["mid"]
    dev = cuda_device
    X = make_dense_teacher_logits(w.N, w.V, seed=w.seed, device=dev)
    ws = kd.workspace(kd._abi.kd_topk_cache_workspace(w.N, w.V, w.K), dev)
    outs = []
    lse = torch.empty((w.N,), dtype=torch.float32, device=dev)
    for run in range(3):
        ids = torch.empty((w.N, w.K), dtype=torch.int32, device=dev)
        vals = torch.empty((w.N, w.K), dtype=torch.float32, device=dev)
        st = kd._abi.kd_topk_cache(X.data_ptr(), w.N, w.V, w.V, w.K, ids.data_ptr(), vals.data_ptr(),
                                   lse.data_ptr() if run == 1 else None, None, ws.data_ptr(), ws.numel(),
                                   torch.cuda.current_stream().cuda_stream)
        assert st == 0
        outs.append((ids, vals))
    torch.cuda.synchronize()
    assert kd.device_error(ws) == (0, 0)
    bits = bf16_bits(X)
    del X
    rid, rval, rlse = _oracle_rows_parallel(bits, w.K)
    for run, (ids, vals) in enumerate(outs):
        gid, gval = ids.cpu().numpy(), vals.cpu().numpy()
        bad = np.flatnonzero(np.any(gid != rid, axis=1) | np.any(gval.view(np.uint32) != rval.view(np.uint32), axis=1))
        assert bad.size == 0, f"launch {run}: {bad.size} rows differ, first {bad[:8].tolist()}"
    glse = lse.cpu().numpy().astype(np.float64)
    assert np.max(np.abs(glse - rlse)) <= 1e-5 * np.max(np.abs(rlse))


def test_topk_nan_rows(kd, cuda_device):
    """Rows holding NaNs of both signs and several payloads among ordinary values and
    infinities, ordered as the IEEE 754 totalOrder with the two zeros equal: positive NaNs
    above +inf, negative NaNs below -inf."""
    g = torch.Generator().manual_seed(31)
    N, V = 40, 6000
    X = torch.randn((N, V), generator=g).to(torch.bfloat16)
    b = X.view(torch.int16)
    pos_nan = [0x7FC0, 0x7F81, 0x7FFF, 0x7FA5]
    neg_nan = [0xFFC0 - 0x10000, 0xFF81 - 0x10000, 0xFFFF - 0x10000]
    for r in range(N):
        cols = torch.randperm(V, generator=g)[: 3 + (r % 9) * 17]
        for j, c in enumerate(cols.tolist()):
            if r % 5 == 4:
                b[r, c] = neg_nan[j % 3]                      # only negative NaNs in this row
            else:
                b[r, c] = (pos_nan + neg_nan)[j % 7]
        if r % 3 == 0:
            b[r, (r * 37) % V] = 0x7F80                        # +inf
            b[r, (r * 53) % V] = 0xFF80 - 0x10000              # -inf
    b[N - 1, :] = 0x7FC0                                       # a row of one NaN pattern: lowest ids
    for K in (1, 100, 300):
        _check_ids_and_bits(kd, X, K, cuda_device)


def _check_ids_and_bits(kd, X_host, K, dev):
    """As _check for rows whose logsumexp is not a number: ids and value bits only."""
    N, V = X_host.shape
    Xd = X_host.to(dev)
    ids = torch.empty((N, K), dtype=torch.int32, device=dev)
    vals = torch.empty((N, K), dtype=torch.float32, device=dev)
    ws = kd.workspace(kd._abi.kd_topk_cache_workspace(N, V, K), dev)
    st = kd._abi.kd_topk_cache(Xd.data_ptr(), N, V, V, K, ids.data_ptr(), vals.data_ptr(), None, None,
                               ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream)
    assert st == 0
    torch.cuda.synchronize()
    assert kd.device_error(ws) == (0, 0)
    rid, rval = oracle.topk_cache(bf16_bits(X_host), K)
    gid, gval = ids.cpu().numpy(), vals.cpu().numpy()
    assert np.array_equal(gid, rid), f"K={K}: ids differ in rows {np.flatnonzero(np.any(gid != rid, axis=1))[:8]}"
    assert np.array_equal(gval.view(np.uint32), rval.view(np.uint32)), f"K={K}: value bits differ"


def test_topk_dropped_mass(kd, cuda_device):
    """The mass outside the cache, from the cached values and the row logsumexp, against the oracle;
    zero (up to rounding) when K = V."""
    X = make_dense_teacher_logits(16, 2048, seed=3, std=3.0)
    Xd = X.to(cuda_device)
    for K in (16, 200, 1024):
        ids, vals, dropped = kd.topk_cache(Xd, K, with_dropped=True)
        got = dropped.double().cpu().numpy()
        ref = oracle.dropped_mass(bf16_bits(X), K)
        assert np.max(np.abs(got - ref)) <= 1e-5
    assert np.all(ref >= -1e-12)


@pytest.mark.parametrize("N,dt,chunk,V,K", [
    (300, 64, 128, 5000, 37),    # one row tile per chunk: single-CTA tiles
    (300, 192, 256, 5000, 37),   # CTA pairs, 3 k-blocks, then a 44-row single-CTA chunk
    (700, 320, 384, 5000, 37),   # CTA pairs over 3 row tiles (the pair's phantom tile stores nothing)
    (600, 200, 256, 5000, 37),   # dt not a multiple of 64: a ragged last k-block
    (300, 192, 256, 12000, 37),  # 47 column tiles >= K: rows start from their tile maxima (ragged last tile)
    (520, 64, 256, 20000, 64),   # the same over 79 tiles, three chunks
    (300, 64, 128, 5123, 37),    # a last tile of 3 columns: the tile sums skip the columns past V
    (300, 64, 128, 5000, 300),   # K > 256: the block selection computes the row logsumexp itself
])
def test_teacher_topk_exact_integer_logits(kd, cuda_device, N, dt, chunk, V, K):
    """Small-integer teacher hidden states and weights make every logit an integer that fp32 holds
    exactly, rounded once to bf16, so the fused projection + top-K must match the oracle's cache of
    the logits bit for bit (with many ties, broken by the lower id)."""
    g = torch.Generator().manual_seed(21 + dt)
    Ht = torch.randint(-2, 3, (N, dt), generator=g).to(torch.bfloat16)
    Wt = torch.randint(-2, 3, (V, dt), generator=g).to(torch.bfloat16)
    ids, vals, lse, dropped = kd.teacher_topk(Ht.to(cuda_device), Wt.to(cuda_device), K, chunk=chunk,
                                              with_lse=True, with_dropped=True)
    torch.cuda.synchronize()
    zbits = oracle.teacher_logits_bf16(bf16_bits(Ht), bf16_bits(Wt))
    rid, rval = oracle.topk_cache(zbits, K)
    assert np.array_equal(ids.cpu().numpy(), rid)
    assert np.array_equal(vals.cpu().numpy().view(np.uint32), rval.view(np.uint32))
    ref_lse = oracle.teacher_logsumexp(zbits)
    lse_tol = 1e-5 * np.max(np.abs(ref_lse))
    assert np.max(np.abs(lse.cpu().numpy() - ref_lse)) <= lse_tol
    ref_drop = oracle.dropped_mass(zbits, K)
    assert np.max(np.abs(dropped.cpu().numpy() - ref_drop)) <= lse_tol + 1e-5


@pytest.mark.parametrize("N,dt,chunk,V", [(260, 200, 128, 3001), (520, 256, 256, 3001), (400, 128, 256, 16411)])
def test_teacher_topk_random_is_a_valid_topk(kd, cuda_device, N, dt, chunk, V):
    """Random teacher inputs: the kept values are the logits rounded to bf16 (within one bf16 step of the
    float64 product) and no logit left out exceeds the smallest kept one by more than that rounding."""
    g = torch.Generator().manual_seed(22)
    K = 50
    Ht = torch.randn((N, dt), generator=g).to(torch.bfloat16)
    Wt = (torch.randn((V, dt), generator=g) / 14).to(torch.bfloat16)
    ids, vals = kd.teacher_topk(Ht.to(cuda_device), Wt.to(cuda_device), K, chunk=chunk)
    torch.cuda.synchronize()
    z = oracle.bf16_to_f64(bf16_bits(Ht)) @ oracle.bf16_to_f64(bf16_bits(Wt)).T
    ids, vals = ids.cpu().numpy(), vals.cpu().numpy().astype(np.float64)
    for r in range(N):
        sel = ids[r]
        assert len(set(sel.tolist())) == K and np.all(np.diff(vals[r]) <= 0)
        ulp = 2.0 ** (np.floor(np.log2(np.maximum(np.abs(z[r, sel]), 1e-30))) - 7)
        assert np.all(np.abs(vals[r] - z[r, sel]) <= ulp)
        rest = np.ones(V, bool)
        rest[sel] = False
        assert z[r, rest].max() <= vals[r].min() + 2 * ulp.max()
