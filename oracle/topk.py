"""Top-K teacher cache extraction, by a full per-row sort.

TEST INFRASTRUCTURE (see the package docstring).

[ART] offline-cache paragraph, [DAI] "As duas inovações" item 1 and [EPO] "Los
dos cambios propuestos": the teacher is run once and only its K highest logits
per position (the most probable tokens) are kept, together with their token ids.

Readings: the cache holds the raw logits (not log-probabilities), widened
exactly from bf16 to fp32; it is ordered by value, highest first; equal values
are ordered by ascending token id, and the cut at K keeps the lowest ids;
-0.0 and +0.0 are equal.
"""
from __future__ import annotations

import numpy as np

from .kl import bf16_to_f64


def topk_cache(bits: np.ndarray, K: int):
    """Per row of a bf16 [N, V] logits array (raw uint16 bits): ids int32 [N, K], logits fp32 [N, K].

    A stable lexicographic sort on (-value, id) per row, then the first K.
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
        v = bf16_to_f64(bits[r])
        order = np.lexsort((col, -v))[:K]          # primary key: -value; secondary: id
        ids[r] = order
        vals[r] = v[order].astype(np.float32)
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
