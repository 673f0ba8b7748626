"""Top-K teacher cache extraction, by a full per-row sort.

TEST INFRASTRUCTURE (see the package docstring).

[ART] offline-cache paragraph, [DAI] "As duas inovações" item 1 and [EPO] "Los
dos cambios propuestos": the teacher is run once and only its K highest logits
per position (the most probable tokens) are kept, together with their token ids.

Readings: the cache holds the raw logits (not log-probabilities), widened
exactly from bf16 to fp32; it is ordered by value, highest first; equal values
are ordered by ascending token id, and the cut at K keeps the lowest ids;
-0.0 and +0.0 are equal.  The pages never mention NaN; a NaN logit takes its
place in the IEEE 754 totalOrder predicate (the ordering the standard defines
for every bit pattern): positive NaNs above +inf, negative NaNs below -inf,
and among NaNs of one sign the larger payload further from zero.  The only
departure from totalOrder is the one above: the two zeros are equal.
"""
from __future__ import annotations

import numpy as np

from .kl import bf16_to_f64


def rank_keys(bits_row: np.ndarray):
    """(class, within) of each bf16 element: an element ranks above another when its
    pair is larger.  class 2 = positive NaN, 1 = a number (infinities included),
    0 = negative NaN; within a number's class its value (-0.0 == +0.0); within a NaN
    class the payload (the 7 mantissa bits), negated for negative NaNs, which
    totalOrder orders further below -inf the larger their payload."""
    b = np.asarray(bits_row).astype(np.int64)
    is_nan = ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)
    negative = (b & 0x8000) != 0
    cls = np.where(is_nan, np.where(negative, 0, 2), 1)
    payload = (b & 0x007F).astype(np.float64)
    with np.errstate(invalid="ignore"):
        value = bf16_to_f64(b.astype(np.uint16))
    within = np.where(is_nan, np.where(negative, -payload, payload), value)
    return cls, within


def widen_bits(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns to fp32 with every bit kept (NaN payloads included)."""
    return (np.asarray(bits).astype(np.uint32) << np.uint32(16)).view(np.float32)


def topk_cache(bits: np.ndarray, K: int):
    """Per row of a bf16 [N, V] logits array (raw uint16 bits): ids int32 [N, K], logits fp32 [N, K].

    A stable lexicographic sort on (rank descending, id ascending) per row, then the first K.
    """
    bits = np.asarray(bits)
    assert bits.dtype == np.uint16 and bits.ndim == 2
    N, V = bits.shape
    if not (1 <= K <= V):
        raise ValueError("K must be in [1, V]")
    ids = np.empty((N, K), dtype=np.int32)
    vals = np.empty((N, K), dtype=np.float32)
    col = np.arange(V)
    for r in range(N):
        cls, within = rank_keys(bits[r])
        order = np.lexsort((col, -within, -cls))[:K]   # keys: -class, then -within, then id
        ids[r] = order
        vals[r] = widen_bits(bits[r, order])
    return ids, vals


def teacher_logsumexp(bits: np.ndarray) -> np.ndarray:
    """log sum_v exp(t_v) of each row of dense bf16 teacher logits [N, V], in float64.

    [ART] paragraph on the top-K limitation: keeping only the top K logits drops the
    teacher's tail; with the full-row logsumexp the dropped probability is
    1 - sum_k exp(t_k - logsumexp).  Rows of all -inf give -inf.
    """
    x = bf16_to_f64(np.asarray(bits))
    m = np.max(x, axis=1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    with np.errstate(divide="ignore"):
        return m_safe + np.log(np.sum(np.exp(x - m_safe[:, None]), axis=1))


def dropped_mass(bits: np.ndarray, K: int) -> np.ndarray:
    """Teacher probability (softmax over the full row) outside the row's top-K logits."""
    lse = teacher_logsumexp(bits)
    _, vals = topk_cache(bits, K)
    return 1.0 - np.sum(np.exp(vals.astype(np.float64) - lse[:, None]), axis=1)


def teacher_logits_bf16(Ht_bits: np.ndarray, Wt_bits: np.ndarray) -> np.ndarray:
    """Teacher logits Ht Wt^T from bf16 inputs, as the bf16 bit patterns a bf16 teacher emits.

    The product is taken in float64 and rounded to the nearest bf16 (ties to even)
    through float32; when every product and partial sum is exact (small integer
    inputs) this is the exact logit.  [ART] paragraph on the first fix: the
    teacher's single pass produces the logits the cache is taken from.
    """
    z = bf16_to_f64(Ht_bits) @ bf16_to_f64(Wt_bits).T
    f = z.astype(np.float32).view(np.uint32).astype(np.uint64)
    rounded = (f + 0x7FFF + ((f >> 16) & 1)) >> 16
    return rounded.astype(np.uint16)
