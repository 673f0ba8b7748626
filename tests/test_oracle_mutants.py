"""Plant plausible slips in copies of the oracle and check that a pin catches each.

A mutant is the oracle source with one textual edit, loaded as a throw-away
module on the CPU; the real oracle is never modified.
"""
import json
import math
import os
import sys
import types

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
KL_SRC = open(os.path.join(ROOT, "oracle", "kl.py")).read()
TOPK_SRC = open(os.path.join(ROOT, "oracle", "topk.py")).read()
GOLDEN = os.path.join(ROOT, "tests", "golden", "worked_example_v4.json")


def _load(src, name):
    mod = types.ModuleType(name)
    mod.__dict__["__name__"] = name
    sys.modules[name] = mod          # dataclasses look their module up here
    exec(compile(src, name, "exec"), mod.__dict__)
    return mod


def _problem(N=9, d=6, V=40, K=5, seed=0):
    rng = np.random.default_rng(seed)
    H = rng.standard_normal((N, d))
    W = rng.standard_normal((V, d)) / math.sqrt(d)
    ids = np.stack([rng.choice(V, K, replace=False) for _ in range(N)]).astype(np.int32)
    tlog = np.sort(rng.standard_normal((N, K)) * 2, axis=1)[:, ::-1].copy()
    mask = np.ones(N, dtype=np.uint8); mask[[1, N - 1]] = 0
    return H, W, ids, tlog, mask


def pin_golden(m):
    g = json.load(open(GOLDEN))
    i, e = g["inputs"], g["expected"]
    args = (np.array(i["H"]), np.array(i["W"]), np.array(i["ids"]), np.array(i["tlog"]))
    for r in (m.dense_kl(*args), m.forward_chunked_kl(*args, chunk=1), m.fused_chunked_kl(*args, chunk=1, vtile=3)):
        if abs(r.loss - e["loss"]) > 1e-12 or not np.allclose(r.grad_H, e["grad_H"], atol=1e-12):
            return False
    return True


def pin_fd(m, tau):
    H, W, ids, tlog, mask = _problem(4, 3, 12, 3, seed=1)
    r = m.dense_kl(H, W, ids, tlog, mask, tau)
    eps = 1e-6
    L = lambda H_, W_: m.dense_kl(H_, W_, ids, tlog, mask, tau, want_grads=False).loss
    for (i, j) in [(0, 0), (2, 1), (3, 2)]:
        Hp, Hm = H.copy(), H.copy(); Hp[i, j] += eps; Hm[i, j] -= eps
        if abs((L(Hp, W) - L(Hm, W)) / (2 * eps) - r.grad_H[i, j]) > 1e-6:
            return False
    for (i, j) in [(0, 0), (5, 1), (11, 2), (int(ids[0, 0]), 1)]:
        Wp, Wm = W.copy(), W.copy(); Wp[i, j] += eps; Wm[i, j] -= eps
        if abs((L(H, Wp) - L(H, Wm)) / (2 * eps) - r.grad_W[i, j]) > 1e-6:
            return False
    return True


def pin_formulations(m):
    H, W, ids, tlog, mask = _problem()
    a = m.dense_kl(H, W, ids, tlog, mask)
    for r in (m.forward_chunked_kl(H, W, ids, tlog, mask, chunk=4),
              m.fused_chunked_kl(H, W, ids, tlog, mask, chunk=4, vtile=16)):
        if abs(r.loss - a.loss) > 1e-12 * abs(a.loss):
            return False
        if np.max(np.abs(r.grad_W - a.grad_W)) > 1e-12 * np.max(np.abs(a.grad_W)):
            return False
    return True


def pin_mask(m):
    H, W, ids, tlog, mask = _problem()
    r = m.dense_kl(H, W, ids, tlog, mask)
    return abs(r.loss - r.kl[mask == 1].mean()) <= 1e-14


def all_kl_pins(m):
    return pin_golden(m) and pin_fd(m, 1.0) and pin_fd(m, 2.0) and pin_formulations(m) and pin_mask(m)


KL_MUTANTS = [
    ("dz sign", "dz = (np.exp(logq) - p)", "dz = (p - np.exp(logq))"),
    ("tau on grad_W", "res.grad_W = (dz / tau).T @ H", "res.grad_W = (dz * tau).T @ H"),
    ("teacher not normalised", "logp = tgrid - _lse_rows(tgrid)[:, None]", "logp = tgrid"),
    ("student not normalised", "logq = z - lse[:, None]", "logq = z"),
    ("online lse without rescale", "run_s = run_s * np.exp(run_m - new_m) +", "run_s = run_s +"),
    ("entropy term dropped", "kl[c0:c1] = negent[c0:c1] - G + lse[c0:c1]\n    loss = float(np.sum(kl * m) / n_valid) if n_valid > 0 else 0.0\n    res = OracleResult(loss=loss, kl=kl, lse=lse, n_valid=n_valid)\n    if not want_grads",
     "kl[c0:c1] = - G + lse[c0:c1]\n    loss = float(np.sum(kl * m) / n_valid) if n_valid > 0 else 0.0\n    res = OracleResult(loss=loss, kl=kl, lse=lse, n_valid=n_valid)\n    if not want_grads"),
    ("mean ignores mask", "loss = float(np.sum(kl * m) / n_valid) if n_valid > 0 else 0.0\n\n    res", "loss = float(np.mean(kl))\n\n    res"),
    ("operands transposed in grad_H", "gH[c0:c1] += (dz / tau) @ W[v0:v1]", "gH[c0:c1] += (dz / tau) @ W[v0:v1][::-1]"),
]


def test_real_oracle_passes_all_pins():
    assert all_kl_pins(_load(KL_SRC, "oracle_kl_copy"))


@pytest.mark.parametrize("name,old,new", KL_MUTANTS, ids=[m[0] for m in KL_MUTANTS])
def test_kl_mutant_is_caught(name, old, new):
    assert KL_SRC.count(old) == 1, f"mutation anchor not unique: {name}"
    mutant = _load(KL_SRC.replace(old, new), "oracle_kl_mutant")
    with np.errstate(all="ignore"):
        assert not all_kl_pins(mutant), f"no pin caught mutant: {name}"


def _topk_mutant(old, new):
    assert TOPK_SRC.count(old) == 1, f"mutation anchor not unique: {old}"
    kl_mod = _load(KL_SRC, "oracle_kl_for_topk_mutant")
    src = TOPK_SRC.replace(old, new).replace("from .kl import bf16_to_f64", "")
    mut = _load(src, "oracle_topk_mutant")
    mut.bf16_to_f64 = kl_mod.bf16_to_f64
    return mut, kl_mod


# Slips in the NaN reading: NaN ranked by its numeric comparison (last, the behaviour of a
# plain sort on values), the payload order of negative NaNs not reversed, and values
# re-rounded through float64 (a signalling NaN comes back quieted).
TOPK_NAN_MUTANTS = [
    ("nan_class_dropped", "np.lexsort((col, -within, -cls))", "np.lexsort((col, -within, 0 * cls))"),
    ("negative_payload_not_reversed", "np.where(negative, -payload, payload)", "payload"),
    ("values_through_float64", "vals[r] = widen_bits(bits[r, order])",
     "vals[r] = bf16_to_f64(bits[r, order]).astype(np.float32)"),
]


@pytest.mark.parametrize("name,old,new", TOPK_NAN_MUTANTS, ids=[m[0] for m in TOPK_NAN_MUTANTS])
def test_topk_nan_mutant_is_caught(name, old, new):
    from test_oracle_pins import nan_order_pin
    mut, _ = _topk_mutant(old, new)
    with np.errstate(all="ignore"):
        assert not nan_order_pin(mut.topk_cache), f"no pin caught mutant: {name}"


def test_topk_tie_mutant_is_caught():
    mut, kl_mod = _topk_mutant("np.lexsort((col, -within, -cls))", "np.lexsort((-col, -within, -cls))")
    rng = np.random.default_rng(0)
    import torch
    x = np.round(rng.standard_normal((4, 64)) * 2) / 2
    bits = torch.tensor(x, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    ids, _ = mut.topk_cache(bits, 10)
    vals = kl_mod.bf16_to_f64(bits)
    brute = [sorted(range(64), key=lambda i: (-vals[r, i], i))[:10] for r in range(4)]
    assert any(list(ids[r]) != brute[r] for r in range(4))
