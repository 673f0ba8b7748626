"""Pins of the float64 oracle against facts that do not come from the oracle itself.

Each pin is chosen so that a plausible slip in the oracle (a dropped term, a
wrong sign, a transposed operand, a wrong normaliser or temperature) fails at
least one of them; ``test_oracle_mutants.py`` plants such slips and checks that.
"""
import json
import math
import os

import numpy as np
import pytest
import scipy.special
import torch

import oracle
from oracle import dense_kl, forward_chunked_kl, fused_chunked_kl, sparse_teacher, topk_cache

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def rand_problem(N=37, d=16, V=300, K=7, seed=0, mask_p=0.8, scale=1.0):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, d)) * scale
    W = rng.standard_normal((V, d)) / math.sqrt(d) * scale
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(N)]).astype(np.int32)
    tlog = np.sort(rng.standard_normal((N, K)) * 2.0, axis=1)[:, ::-1].copy()
    mask = (rng.random(N) < mask_p).astype(np.uint8) if mask_p < 1 else None
    return H, W, ids, tlog, mask


def relerr(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.max(np.abs(a - b)) / max(np.max(np.abs(b)), 1e-300))


# P1: the three formulations are equal (the fused-loss paragraph calls them
# mathematically equivalent), for chunk sizes that do and do not divide N and
# vocabulary tiles with a ragged tail.
@pytest.mark.parametrize("chunk,vtile", [(1, 256), (5, 64), (16, 7), (37, 300), (64, 1000)])
@pytest.mark.parametrize("tau", [1.0, 1.7])
def test_formulations_agree(chunk, vtile, tau):
    H, W, ids, tlog, mask = rand_problem()
    a = dense_kl(H, W, ids, tlog, mask, tau, grad_loss=0.7)
    b = forward_chunked_kl(H, W, ids, tlog, mask, tau, chunk=chunk, grad_loss=0.7)
    c = fused_chunked_kl(H, W, ids, tlog, mask, tau, chunk=chunk, vtile=vtile, grad_loss=0.7)
    for r in (b, c):
        assert abs(r.loss - a.loss) <= 1e-12 * abs(a.loss)
        assert relerr(r.kl, a.kl) <= 1e-12
        assert relerr(r.lse, a.lse) <= 1e-12
        assert relerr(r.grad_H, a.grad_H) <= 1e-12
        assert relerr(r.grad_W, a.grad_W) <= 1e-12


def test_lse_is_library_logsumexp():
    H, W, ids, tlog, mask = rand_problem(scale=3.0)
    r = fused_chunked_kl(H, W, ids, tlog, mask, 1.3, chunk=8, vtile=50, want_grads=False)
    ref = scipy.special.logsumexp(H @ W.T / 1.3, axis=1)
    assert relerr(r.lse, ref) <= 1e-13


# P2: Gibbs' inequality, KL >= 0 per position, for any student.
def test_kl_nonnegative():
    for seed in range(5):
        H, W, ids, tlog, mask = rand_problem(seed=seed, scale=2.5)
        r = dense_kl(H, W, ids, tlog, mask, want_grads=False)
        assert np.all(r.kl >= -1e-12)
        assert r.loss >= 0


# P3: KL = 0 when the student's softmax restricted to the cached ids equals the
# teacher's and the student puts negligible mass elsewhere.  H = I makes the
# student logits of position t equal to column t of W.
def test_kl_zero_construction():
    N, V, K = 24, 200, 9
    rng = np.random.default_rng(3)
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(N)]).astype(np.int32)
    tlog = np.sort(rng.standard_normal((N, K)) * 3, axis=1)[:, ::-1].copy()
    shift = rng.standard_normal(N) * 5
    H = np.eye(N)
    W = np.full((V, N), -1.0e4)
    for t in range(N):
        W[ids[t], t] = tlog[t] + shift[t]
    for f in (dense_kl, fused_chunked_kl):
        r = f(H, W, ids, tlog, None)
        assert np.max(np.abs(r.kl)) <= 1e-12
        assert np.max(np.abs(r.grad_H)) <= 1e-12


# P4: each row of dL/dz sums to 0 (sum q = sum p = 1).
def test_dz_rows_sum_to_zero():
    H, W, ids, tlog, mask = rand_problem(scale=2.0)
    r = dense_kl(H, W, ids, tlog, mask, want_dz=True)
    row_sums = r.dz.sum(axis=1)
    assert np.max(np.abs(row_sums)) <= 1e-15 * max(1.0, np.max(np.abs(r.dz)) * r.dz.shape[1])
    # and the gradients are the dz contracted through the projection
    assert relerr(r.grad_H, r.dz @ W) <= 1e-12


# P5: central finite differences of the loss agree with the hand-written
# gradients (this pins signs, the 1/N_valid, the 1/tau and the operand order).
@pytest.mark.parametrize("tau", [1.0, 2.0])
def test_finite_differences(tau):
    N, d, V, K = 4, 8, 32, 4
    H, W, ids, tlog, _ = rand_problem(N, d, V, K, seed=11)
    mask = np.array([1, 0, 1, 1], dtype=np.uint8)
    r = dense_kl(H, W, ids, tlog, mask, tau, grad_loss=1.0)
    eps = 1e-6

    def L(H_, W_):
        return dense_kl(H_, W_, ids, tlog, mask, tau, want_grads=False).loss

    num_H = np.zeros_like(H)
    for i in range(N):
        for j in range(d):
            Hp = H.copy(); Hp[i, j] += eps
            Hm = H.copy(); Hm[i, j] -= eps
            num_H[i, j] = (L(Hp, W) - L(Hm, W)) / (2 * eps)
    num_W = np.zeros_like(W)
    for i in range(V):
        for j in range(d):
            Wp = W.copy(); Wp[i, j] += eps
            Wm = W.copy(); Wm[i, j] -= eps
            num_W[i, j] = (L(H, Wp) - L(H, Wm)) / (2 * eps)
    assert relerr(r.grad_H, num_H) <= 1e-6
    assert relerr(r.grad_W, num_W) <= 1e-6
    assert np.all(r.grad_H[1] == 0)


# P7: with K = V the sparse teacher is the full teacher, and the loss is the
# library's full-vocabulary KL (torch.nn.functional.kl_div, float64).
def test_k_equals_v_is_full_kl():
    N, d, V = 16, 12, 64
    rng = np.random.default_rng(5)
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d))
    ids = np.stack([rng.permutation(V) for _ in range(N)]).astype(np.int32)
    tlog = rng.standard_normal((N, V)) * 2
    r = fused_chunked_kl(H, W, ids, tlog, None, chunk=5, vtile=24)
    teacher_full = np.empty((N, V))
    teacher_full[np.arange(N)[:, None], ids] = tlog
    logq = torch.log_softmax(torch.tensor(H @ W.T, dtype=torch.float64), dim=1)
    logp = torch.log_softmax(torch.tensor(teacher_full, dtype=torch.float64), dim=1)
    ref = torch.nn.functional.kl_div(logq, logp, reduction="batchmean", log_target=True).item()
    assert abs(r.loss - ref) <= 1e-12 * abs(ref)


# Hand-worked example with rational probabilities (tests/golden).
def test_golden_worked_example():
    with open(os.path.join(GOLDEN, "worked_example_v4.json")) as f:
        g = json.load(f)
    inp, exp = g["inputs"], g["expected"]
    H = np.array(inp["H"]); W = np.array(inp["W"])
    ids = np.array(inp["ids"], dtype=np.int32); tlog = np.array(inp["tlog"])
    for f in (lambda: dense_kl(H, W, ids, tlog),
              lambda: forward_chunked_kl(H, W, ids, tlog, chunk=1),
              lambda: fused_chunked_kl(H, W, ids, tlog, chunk=1, vtile=3)):
        r = f()
        assert abs(r.loss - exp["loss"]) <= 1e-14
        assert np.allclose(r.lse, exp["lse"], rtol=0, atol=1e-14)
        assert np.allclose(r.grad_H, exp["grad_H"], rtol=0, atol=1e-14)
        assert np.allclose(r.grad_W[:, 0], exp["grad_W_col0"], rtol=0, atol=1e-14)
        assert np.all(r.grad_W[:, 1:] == 0)


# Temperature: KL at tau on (H, t) equals KL at tau = 1 on (H/tau, t/tau), and
# grad_H scales by 1/tau (exact in float64 for tau = 2).
def test_temperature_identity():
    H, W, ids, tlog, mask = rand_problem(seed=9)
    a = fused_chunked_kl(H, W, ids, tlog, mask, tau=2.0, chunk=10, vtile=77)
    b = dense_kl(H / 2.0, W, ids, tlog / 2.0, mask, tau=1.0)
    assert abs(a.loss - b.loss) <= 1e-12 * abs(b.loss)
    assert relerr(a.grad_H, b.grad_H / 2.0) <= 1e-12
    assert relerr(a.grad_W, b.grad_W) <= 1e-12


# Reduction and mask (reading R5/R6): loss is the mean over valid positions,
# padding rows get zero gradient; no valid position gives 0 everywhere.
def test_mask_semantics():
    H, W, ids, tlog, _ = rand_problem(seed=4)
    mask = np.zeros(H.shape[0], dtype=np.uint8)
    mask[[0, 3, 5]] = 1
    r = dense_kl(H, W, ids, tlog, mask)
    assert abs(r.loss - r.kl[[0, 3, 5]].mean()) <= 1e-14
    assert np.all(r.grad_H[mask == 0] == 0)
    sub = dense_kl(H[[0, 3, 5]], W, ids[[0, 3, 5]], tlog[[0, 3, 5]], None)
    assert relerr(r.grad_W, sub.grad_W) <= 1e-12
    z = fused_chunked_kl(H, W, ids, tlog, np.zeros_like(mask), chunk=8)
    assert z.loss == 0.0 and np.all(z.grad_H == 0) and np.all(z.grad_W == 0)


def test_sparse_teacher_is_softmax():
    t = np.array([[2.0, 1.0, -np.inf, 0.5]])
    p, logp, negent = sparse_teacher(t, 1.0)
    ref = scipy.special.softmax(t, axis=1)
    assert np.allclose(p, ref, rtol=1e-15, atol=0)
    assert p[0, 2] == 0.0
    assert abs(negent[0] - np.sum(ref[0, [0, 1, 3]] * np.log(ref[0, [0, 1, 3]]))) <= 1e-15


def test_vocab_rows_subset():
    H, W, ids, tlog, mask = rand_problem(seed=2)
    full = fused_chunked_kl(H, W, ids, tlog, mask, chunk=9, vtile=64)
    rows = [0, 5, 17, 299, 123]
    part = fused_chunked_kl(H, W, ids, tlog, mask, chunk=9, vtile=64, vocab_rows=rows)
    assert relerr(part.grad_W, full.grad_W[rows]) <= 1e-13


# P8: top-K against a brute-force Python sort, on rows with heavy ties and
# signed zeros.
def _bf16_bits_of(x):
    return torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_topk_bruteforce_with_ties():
    rng = np.random.default_rng(7)
    N, V = 12, 500
    x = np.round(rng.standard_normal((N, V)) * 2) / 2          # many exact ties
    x[0, :] = 0.0
    x[1, ::3] = -0.0                                         # -0 == +0
    x[2, :] = np.linspace(-3, 3, V)
    x[3, 100:] = -np.inf
    bits = _bf16_bits_of(x)
    vals = oracle.bf16_to_f64(bits)
    for K in (1, 5, 64, V):
        ids, out = topk_cache(bits, K)
        for r in range(N):
            order = sorted(range(V), key=lambda i: (-vals[r, i], i))[:K]
            assert list(ids[r]) == order
            assert np.array_equal(out[r], vals[r, order].astype(np.float32))
    ids, _ = topk_cache(bits, 7)
    assert list(ids[0]) == list(range(7))                     # all equal: lowest ids


# NaN reading (the pages never mention NaN): IEEE 754 totalOrder with the two zeros
# equal.  The expected order below is written out by hand from the standard's
# description (+NaN above +inf, larger payload further out; -NaN below -inf, larger
# payload further down), not computed.
NAN_ROW_BITS = [0x3F80,   # 0: 1.0
                0x7FC0,   # 1: +NaN, payload 0x40
                0xFF80,   # 2: -inf
                0xFFC0,   # 3: -NaN, payload 0x40
                0x7F80,   # 4: +inf
                0x0000,   # 5: +0
                0x8000,   # 6: -0 (equal to +0: the lower id first)
                0x7F81,   # 7: +NaN, payload 0x01
                0xC000,   # 8: -2.0
                0xFF81]   # 9: -NaN, payload 0x01
NAN_ROW_ORDER = [1, 7, 4, 0, 5, 6, 8, 2, 9, 3]


def nan_order_pin(topk_fn) -> bool:
    bits = np.array([NAN_ROW_BITS], dtype=np.uint16)
    ok = True
    for K in (1, 4, 10):
        ids, vals = topk_fn(bits, K)
        ok &= list(ids[0]) == NAN_ROW_ORDER[:K]
        # values are the input bits widened, payloads kept
        ok &= list(vals[0].view(np.uint32) >> 16) == [NAN_ROW_BITS[i] for i in NAN_ROW_ORDER[:K]]
    return bool(ok)


def test_topk_nan_order_by_hand():
    assert nan_order_pin(topk_cache)


def test_bf16_widening_is_exact():
    x = np.array([1.0, -2.5, 3.140625, 65280.0, 1e-38, -0.0], dtype=np.float32)
    bits = _bf16_bits_of(x)
    y = oracle.bf16_to_f64(bits)
    assert np.array_equal(y, torch.tensor(x).to(torch.bfloat16).double().numpy())


# The teacher's full-row logsumexp (tail-mass diagnostic) is the library logsumexp;
# the dropped mass is 0 with K = V, in [0, 1) otherwise, and shrinks as K grows.
def test_teacher_logsumexp_and_dropped_mass():
    rng = np.random.default_rng(8)
    x = rng.standard_normal((6, 300)) * 3
    bits = _bf16_bits_of(x)
    vals = oracle.bf16_to_f64(bits)
    assert np.allclose(oracle.teacher_logsumexp(bits), scipy.special.logsumexp(vals, axis=1), rtol=1e-14, atol=0)
    assert np.max(np.abs(oracle.dropped_mass(bits, 300))) <= 1e-13
    d10, d50 = oracle.dropped_mass(bits, 10), oracle.dropped_mass(bits, 50)
    assert np.all((d10 > 0) & (d10 < 1)) and np.all(d50 < d10)
    # by hand: top-1 of [0, ln 3] keeps 3/4 of the mass
    b = _bf16_bits_of(np.array([[0.0, np.log(3.0)]]))
    v = oracle.bf16_to_f64(b)[0]
    assert abs(oracle.dropped_mass(b, 1)[0] - np.exp(v[0]) / (np.exp(v[0]) + np.exp(v[1]))) <= 1e-15


# The teacher-logit rounding of the fused cache builder is torch's own fp32 -> bf16
# conversion (round to nearest even) applied to the product.
def test_teacher_logits_bf16_rounding():
    rng = np.random.default_rng(12)
    Ht = _bf16_bits_of(rng.standard_normal((9, 24)))
    Wt = _bf16_bits_of(rng.standard_normal((40, 24)))
    got = oracle.teacher_logits_bf16(Ht, Wt)
    z = oracle.bf16_to_f64(Ht) @ oracle.bf16_to_f64(Wt).T
    ref = torch.tensor(z, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)
