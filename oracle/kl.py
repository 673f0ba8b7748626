"""KL(p_teacher || q_student) against a sparse top-K teacher, three ways, in float64.

TEST INFRASTRUCTURE (see the package docstring): plain, slow and meant to be
checked by eye against the pages.  All arithmetic is numpy float64; the student
inputs arrive as the raw bf16 bit patterns the GPU path consumes, widened
exactly.

What the pages fix ([ART], paragraph on the second fix; [DAI] "As duas
inovações"; [EPO] "Adónde se va la memoria"):
  * the teacher is kept as its K cached logits per position (the offline cache);
  * the student side is a log-probability over the whole vocabulary, obtained by
    projecting hidden states through the output (LM-head) matrix;
  * the loss is a KL divergence between the two; three formulations of it are
    called mathematically equivalent: dense, forward-chunked and fused chunked;
  * the fused one projects one chunk of positions at a time, folds it into a
    running accumulator and discards it; its backward recomputes each chunk.

Readings where the pages are silent (each the plainest one the rest supports):
  R1  forward KL(p_T || q_S): the student is trained to match the teacher, and
      with a top-K teacher the reverse direction is infinite.
  R2  outside its K cached ids the teacher has probability 0 (logit -inf), so
      p_T is the softmax of the K cached logits; this is the only fill that makes
      the dense and sparse formulations equal.
  R3  q_S is normalised over the full vocabulary (log-softmax of all V logits).
  R4  temperature tau divides both teacher and student logits; no tau^2 factor.
  R5  the loss is the mean of KL over valid (mask = 1) positions; with no valid
      position the loss and all gradients are 0.
  R6  mask is uint8 per position, 1 = valid, 0 = padding; padding contributes
      nothing and gets a zero gradient.
  R7  chunks run over the flattened B*T positions.
  R8  H and W are bf16; everything here is float64 on those exact values.
  R11 ids within a row are distinct (a top-K list always is).
  R14 grad_W is a gradient to be accumulated; grad_H is per position; the
      teacher cache is a constant and gets no gradient.
"""
from __future__ import annotations

import dataclasses
from typing import Optional, Sequence

import numpy as np

F64 = np.float64


@dataclasses.dataclass
class OracleResult:
    loss: float
    kl: np.ndarray          # [N] per-position KL (padding rows included, unmasked value)
    lse: np.ndarray         # [N] log-sum-exp of the student logits z = H W^T / tau
    grad_H: Optional[np.ndarray] = None   # [N, d]
    grad_W: Optional[np.ndarray] = None   # [V, d] (or [len(vocab_rows), d])
    dz: Optional[np.ndarray] = None       # [N, V] dL/dz (dense formulation only)
    n_valid: int = 0


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns (uint16) exactly: bf16 is the top half of an fp32."""
    b = np.ascontiguousarray(bits).astype(np.uint32) << np.uint32(16)
    return b.view(np.float32).astype(F64)


def _as_f64(x) -> np.ndarray:
    x = np.asarray(x)
    if x.dtype == np.uint16:
        return bf16_to_f64(x)
    return x.astype(F64)


def _lse_rows(x: np.ndarray) -> np.ndarray:
    """log(sum(exp(x))) along the last axis, with the max pulled out."""
    m = np.max(x, axis=-1)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    s = np.sum(np.exp(x - m_safe[..., None]), axis=-1)
    return m_safe + np.log(s)


def sparse_teacher(tlog: np.ndarray, tau: float = 1.0):
    """p_T over the K cached logits and its negative entropy sum_k p_k log p_k.

    [ART] offline-cache paragraph and [DAI] "As duas inovações": only the top-K
    teacher logits per position are kept; [ART] fused-loss paragraph: the
    teacher stays sparse.  Reading R2: p_T = softmax(t / tau) over those K
    entries; the mass outside them is dropped.  0 log 0 is taken as 0.
    """
    t = _as_f64(tlog) / tau
    logp = t - _lse_rows(t)[:, None]
    p = np.exp(logp)
    negent = np.sum(np.where(p > 0, p * np.where(p > 0, logp, 0.0), 0.0), axis=1)
    return p, logp, negent


def _masks(mask, N):
    m = np.ones(N, dtype=F64) if mask is None else (np.asarray(mask) != 0).astype(F64)
    n_valid = int(m.sum())
    return m, n_valid


def dense_kl(H, W, ids, tlog, mask=None, tau: float = 1.0, grad_loss: float = 1.0,
             want_grads: bool = True, want_dz: bool = False) -> OracleResult:
    """Formulation 1, dense KL ([ART] fused-loss paragraph, first formulation).

    The cached top-K teacher logits are spread onto a full-vocabulary grid
    (-inf off the cached ids, reading R2) and compared with the equally dense
    student log-probability grid; both [N, V] grids are materialised.
    Gradients are written out by hand: with z = H W^T / tau,
        dKL_t / dz_t = q_t - p_t          (softmax Jacobian, reading R1/R3)
        dL / dz_t    = grad_loss * mask_t / N_valid * (q_t - p_t)
        grad_H = (dL/dz / tau) W,   grad_W = (dL/dz / tau)^T H.
    """
    H = _as_f64(H)
    W = _as_f64(W)
    ids = np.asarray(ids).astype(np.int64)
    N, V = H.shape[0], W.shape[0]
    m, n_valid = _masks(mask, N)

    z = (H @ W.T) / tau                                  # [N, V] student logits
    lse = _lse_rows(z)
    logq = z - lse[:, None]                              # dense student log-prob grid

    tgrid = np.full((N, V), -np.inf)                     # dense teacher grid
    rows = np.arange(N)[:, None]
    tgrid[rows, ids] = _as_f64(tlog) / tau
    logp = tgrid - _lse_rows(tgrid)[:, None]
    p = np.exp(logp)                                     # 0 off the cached ids

    kl = np.sum(np.where(p > 0, p * (np.where(p > 0, logp, 0.0) - logq), 0.0), axis=1)
    loss = float(np.sum(kl * m) / n_valid) if n_valid > 0 else 0.0

    res = OracleResult(loss=loss, kl=kl, lse=lse, n_valid=n_valid)
    if want_grads or want_dz:
        scale = (grad_loss / n_valid) if n_valid > 0 else 0.0
        dz = (np.exp(logq) - p) * (m * scale)[:, None]   # dL/dz
        if want_grads:
            res.grad_H = (dz / tau) @ W
            res.grad_W = (dz / tau).T @ H
        if want_dz:
            res.dz = dz
    return res


def forward_chunked_kl(H, W, ids, tlog, mask=None, tau: float = 1.0, chunk: int = 1024,
                       grad_loss: float = 1.0, want_grads: bool = True) -> OracleResult:
    """Formulation 2, forward-chunked KL ([ART] fused-loss paragraph, second formulation).

    The teacher stays sparse; the loss is computed one slice of positions at a
    time, and each slice's full student logits are kept for the backward pass
    (so memory still grows with the sequence).  Per slice and position:
        lse_t = logsumexp_v z_t,v
        G_t   = sum_k p_t,k z_t,id_k            (student logits at the cached ids)
        KL_t  = sum_k p_t,k log p_t,k - G_t + lse_t
    which is sum_k p_k (log p_k - log q_id_k) regrouped.
    """
    H = _as_f64(H)
    W = _as_f64(W)
    ids = np.asarray(ids).astype(np.int64)
    N, d = H.shape
    V = W.shape[0]
    m, n_valid = _masks(mask, N)
    p, _, negent = sparse_teacher(tlog, tau)

    stored = []
    kl = np.empty(N)
    lse = np.empty(N)
    for c0 in range(0, N, chunk):
        c1 = min(N, c0 + chunk)
        zc = (H[c0:c1] @ W.T) / tau                      # kept for backward
        stored.append(zc)
        lse[c0:c1] = _lse_rows(zc)
        G = np.sum(p[c0:c1] * np.take_along_axis(zc, ids[c0:c1], axis=1), axis=1)
        kl[c0:c1] = negent[c0:c1] - G + lse[c0:c1]
    loss = float(np.sum(kl * m) / n_valid) if n_valid > 0 else 0.0
    res = OracleResult(loss=loss, kl=kl, lse=lse, n_valid=n_valid)
    if want_grads:
        scale = (grad_loss / n_valid) if n_valid > 0 else 0.0
        gH = np.zeros((N, d))
        gW = np.zeros((V, d))
        for i, c0 in enumerate(range(0, N, chunk)):
            c1 = min(N, c0 + chunk)
            dz = np.exp(stored[i] - lse[c0:c1, None])    # q from the stored logits
            np.put_along_axis(dz, ids[c0:c1],
                              np.take_along_axis(dz, ids[c0:c1], axis=1) - p[c0:c1], axis=1)
            dz *= (m[c0:c1] * scale)[:, None]
            gH[c0:c1] = (dz / tau) @ W
            gW += (dz / tau).T @ H[c0:c1]
        res.grad_H, res.grad_W = gH, gW
    return res


def fused_chunked_kl(H, W, ids, tlog, mask=None, tau: float = 1.0, chunk: int = 1024,
                     vtile: int = 256, grad_loss: float = 1.0, want_grads: bool = True,
                     vocab_rows: Optional[Sequence[int]] = None) -> OracleResult:
    """Formulation 3, fused chunked KL ([ART] fused-loss paragraph, third formulation;
    [DAI] "As duas inovações", item 2).

    The output projection sits inside the loss loop: for each chunk of positions
    and each tile of the vocabulary, the logits tile z = H_c W_tile^T / tau is
    formed, folded into running per-position accumulators and dropped:
        m <- max(m, max z);  s <- s e^(m_old - m) + sum e^(z - m)   (online logsumexp)
        G <- G + sum over cached ids inside the tile of p_k z_id_k
    so the [chunk, V] logits never exist at once.  The backward pass recomputes
    every tile from H and W:
        dz = (e^(z - lse) - p on the cached ids) * grad_loss * mask / N_valid
        grad_H_c += dz W_tile / tau,   grad_W_tile += dz^T H_c / tau.
    ``vocab_rows`` limits the returned grad_W to those vocabulary rows.
    """
    H = _as_f64(H)
    W = _as_f64(W)
    ids = np.asarray(ids).astype(np.int64)
    N, d = H.shape
    V = W.shape[0]
    m, n_valid = _masks(mask, N)
    p, _, negent = sparse_teacher(tlog, tau)

    lse = np.empty(N)
    kl = np.empty(N)
    for c0 in range(0, N, chunk):
        c1 = min(N, c0 + chunk)
        n = c1 - c0
        run_m = np.full(n, -np.inf)
        run_s = np.zeros(n)
        G = np.zeros(n)
        for v0 in range(0, V, vtile):
            v1 = min(V, v0 + vtile)
            zt = (H[c0:c1] @ W[v0:v1].T) / tau
            new_m = np.maximum(run_m, zt.max(axis=1))
            run_s = run_s * np.exp(run_m - new_m) + np.sum(np.exp(zt - new_m[:, None]), axis=1)
            run_m = new_m
            inside = (ids[c0:c1] >= v0) & (ids[c0:c1] < v1)
            r, k = np.nonzero(inside)
            np.add.at(G, r, p[c0:c1][r, k] * zt[r, ids[c0:c1][r, k] - v0])
        lse[c0:c1] = run_m + np.log(run_s)
        kl[c0:c1] = negent[c0:c1] - G + lse[c0:c1]
    loss = float(np.sum(kl * m) / n_valid) if n_valid > 0 else 0.0
    res = OracleResult(loss=loss, kl=kl, lse=lse, n_valid=n_valid)
    if not want_grads:
        return res

    scale = (grad_loss / n_valid) if n_valid > 0 else 0.0
    gH = np.zeros((N, d))
    vr = np.arange(V) if vocab_rows is None else np.asarray(vocab_rows, dtype=np.int64)
    pos_in_vr = np.full(V, -1, dtype=np.int64)
    pos_in_vr[vr] = np.arange(len(vr))
    gW = np.zeros((len(vr), d))
    for c0 in range(0, N, chunk):
        c1 = min(N, c0 + chunk)
        rowscale = m[c0:c1] * scale
        for v0 in range(0, V, vtile):
            v1 = min(V, v0 + vtile)
            zt = (H[c0:c1] @ W[v0:v1].T) / tau             # recomputed, never stored
            dz = np.exp(zt - lse[c0:c1, None])
            inside = (ids[c0:c1] >= v0) & (ids[c0:c1] < v1)
            r, k = np.nonzero(inside)
            np.add.at(dz, (r, ids[c0:c1][r, k] - v0), -p[c0:c1][r, k])
            dz *= rowscale[:, None]
            gH[c0:c1] += (dz / tau) @ W[v0:v1]
            sel = pos_in_vr[v0:v1]
            keep = sel >= 0
            if keep.any():
                gW[sel[keep]] += (dz[:, keep] / tau).T @ H[c0:c1]
    res.grad_H, res.grad_W = gH, gW
    return res
