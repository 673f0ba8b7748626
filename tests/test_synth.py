"""The seeded input generators draw what the workload recipes state."""
import math

import torch

from synth import WORKLOADS, make_inputs, make_dense_teacher_logits
from synth.workloads import _teacher_logits


def test_tiny_inputs_shapes_and_seeding():
    w = WORKLOADS["tiny"]
    H, W, ids, tlog, mask = make_inputs(w)
    assert H.shape == (128, 256) and H.dtype == torch.bfloat16
    assert W.shape == (4096, 256) and W.dtype == torch.bfloat16
    assert ids.shape == (128, 16) and ids.dtype == torch.int32
    assert tlog.shape == (128, 16) and tlog.dtype == torch.float32
    assert mask is None
    assert int(ids.min()) >= 0 and int(ids.max()) < 4096
    s, _ = torch.sort(ids, dim=1)
    assert bool((s[:, 1:] != s[:, :-1]).all())
    assert bool((tlog[:, 1:] <= tlog[:, :-1]).all())
    H2, W2, ids2, tlog2, _ = make_inputs(w)
    assert torch.equal(H.view(torch.int16), H2.view(torch.int16)) and torch.equal(ids, ids2)
    assert abs(float(W.float().std()) - 1 / math.sqrt(256)) < 0.002
    assert abs(float(tlog.std()) - math.sqrt(3)) < 0.2


def test_small_mask_rate():
    w = WORKLOADS["small"]
    _, _, _, _, mask = make_inputs(w, rows=4096)
    assert mask.dtype == torch.uint8 and abs(float(mask.float().mean()) - 0.95) < 0.02


def test_peaked_margin():
    g = torch.Generator().manual_seed(3)
    t = _teacher_logits("peaked_flat", 2000, 100, g, "cpu")
    margin = t[:, 0] - t[:, 1]
    peaked = margin >= 6
    assert 0.4 < float(peaked.float().mean()) < 0.6
    assert bool((t[:, 1:] <= t[:, :-1]).all())


def test_dense_teacher_logits():
    x = make_dense_teacher_logits(4, 1000, seed=5)
    assert x.dtype == torch.bfloat16 and x.shape == (4, 1000)
    assert abs(float(x.float().std()) - math.sqrt(2)) < 0.1
