"""The five synthetic workloads and their seeded generators.

Shapes follow the distillation example of "Efficient Knowledge Distillation for
LLMs: Offline Top-K Logits and a Fused Chunked KL Loss" (gpt-oss-120b vocabulary
of 201,088 tokens, 32K sequence, batch 4, a top-100 cache per position) plus
three smaller shapes of the same structure.  N(mu, x) below means variance x.

Every tensor is drawn with a ``torch.Generator`` seeded from the workload seed
(1000 + workload index, plus a per-tensor offset), on the device the caller
names: the CPU generator for the small cases the oracle runs in full, the CUDA
generator for the large ones (the oracle then reads back the rows it checks).
Both sides of a comparison always consume the same bytes.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional

import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    T: int
    d: int
    V: int
    K: int
    chunk: int
    teacher: str          # "normal3" | "zipf" | "peaked_flat"
    p_valid: float        # 1.0 = no padding mask
    seed: int

    @property
    def N(self) -> int:
        return self.B * self.T

    def flops_executed(self) -> float:
        """Forward projection + recompute + two gradient GEMMs: 8*d*V per token."""
        return 8.0 * self.N * self.d * self.V

    def flops_useful(self) -> float:
        """Without the backward recompute: 6*d*V per token."""
        return 6.0 * self.N * self.d * self.V


WORKLOADS = {
    "tiny": Workload("tiny", 1, 128, 256, 4096, 16, 128, "normal3", 1.0, 1000),
    "small": Workload("small", 2, 4096, 2048, 32000, 100, 1024, "zipf", 0.95, 1001),
    "mid": Workload("mid", 1, 8192, 4096, 151936, 100, 2048, "peaked_flat", 1.0, 1002),
    "gptoss": Workload("gptoss", 1, 32768, 2880, 201088, 100, 4096, "zipf", 1.0, 1003),
    "headline": Workload("headline", 4, 32768, 2880, 201088, 100, 8192, "peaked_flat", 0.98, 1004),
}


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _distinct_ids(N: int, K: int, V: int, g: torch.Generator, device) -> torch.Tensor:
    """K distinct uniform ids in [0, V) per row, by redrawing rows that repeat an id.

    The ids stay in draw order (not sorted), the way a cache of "the K most
    probable tokens" pairs each id with its logit.
    """
    if K * K > V:
        # dense case (K close to V): the first K of a random permutation per row
        keys = torch.rand((N, V), generator=g, device=device)
        return torch.argsort(keys, dim=1)[:, :K].to(torch.int32).contiguous()
    ids = torch.randint(0, V, (N, K), generator=g, device=device, dtype=torch.int64)
    if K > 1:
        for _ in range(1000):
            s, _ = torch.sort(ids, dim=1)
            bad = (s[:, 1:] == s[:, :-1]).any(dim=1)
            nbad = int(bad.sum())
            if nbad == 0:
                break
            ids[bad] = torch.randint(0, V, (nbad, K), generator=g, device=device, dtype=torch.int64)
        else:
            raise RuntimeError("could not draw distinct ids")
    return ids.to(torch.int32)


def _teacher_logits(kind: str, N: int, K: int, g: torch.Generator, device) -> torch.Tensor:
    """fp32 [N, K] teacher logits, sorted descending along K."""
    if kind == "normal3":
        t = torch.randn((N, K), generator=g, device=device) * math.sqrt(3.0)
    elif kind == "zipf":
        r = torch.arange(1, K + 1, device=device, dtype=torch.float32)
        t = 8.0 - 1.5 * torch.log(r)[None, :] + torch.randn((N, K), generator=g, device=device) * math.sqrt(0.5)
    elif kind == "peaked_flat":
        flat = torch.randn((N, K), generator=g, device=device)
        flat, _ = torch.sort(flat, dim=1, descending=True)
        peaked_rows = torch.rand((N,), generator=g, device=device) < 0.5
        bump = torch.randn((N,), generator=g, device=device).abs()
        t = flat.clone()
        if K > 1:
            # top-1 margin >= 6: t1 <- t2 + 6 + |N(0,1)| on the peaked rows
            t[:, 0] = torch.where(peaked_rows, flat[:, 1] + 6.0 + bump, flat[:, 0])
    else:
        raise ValueError(kind)
    t, _ = torch.sort(t.float(), dim=1, descending=True)
    return t.contiguous()


def make_inputs(w: Workload, device="cpu", rows: Optional[int] = None, materialise_mask: bool = False):
    """Draw (H, W, ids, tlog, mask) for workload ``w`` on ``device``.

    H  : bf16 [N, d], N(0, 1)           W    : bf16 [V, d], N(0, 1/d)
    ids: int32 [N, K], distinct per row tlog : fp32 [N, K], sorted descending
    mask: uint8 [N] (1 = valid) or None when every position is valid (unless
    ``materialise_mask``).  ``rows`` overrides N (B*T) for reduced tests.
    """
    N = w.N if rows is None else rows
    gH = _gen(device, w.seed * 16 + 1)
    gW = _gen(device, w.seed * 16 + 2)
    gI = _gen(device, w.seed * 16 + 3)
    gT = _gen(device, w.seed * 16 + 4)
    gM = _gen(device, w.seed * 16 + 5)
    H = torch.randn((N, w.d), generator=gH, device=device, dtype=torch.float32).to(torch.bfloat16)
    W = (torch.randn((w.V, w.d), generator=gW, device=device, dtype=torch.float32)
         * (1.0 / math.sqrt(w.d))).to(torch.bfloat16)
    ids = _distinct_ids(N, w.K, w.V, gI, device)
    tlog = _teacher_logits(w.teacher, N, w.K, gT, device)
    if w.p_valid < 1.0:
        mask = (torch.rand((N,), generator=gM, device=device) < w.p_valid).to(torch.uint8)
    elif materialise_mask:
        mask = torch.ones((N,), dtype=torch.uint8, device=device)
    else:
        mask = None
    return H, W, ids, tlog, mask


def make_dense_teacher_logits(N: int, V: int, seed: int, device="cpu", std: float = math.sqrt(2.0)) -> torch.Tensor:
    """Dense bf16 teacher logits [N, V] ~ N(0, 2) for the top-K cache extraction."""
    g = _gen(device, seed * 16 + 7)
    out = torch.empty((N, V), dtype=torch.bfloat16, device=device)
    step = max(1, (1 << 26) // max(V, 1))
    for r0 in range(0, N, step):
        r1 = min(N, r0 + step)
        out[r0:r1] = (torch.randn((r1 - r0, V), generator=g, device=device) * std).to(torch.bfloat16)
    return out


def bf16_bits(x: torch.Tensor):
    """The raw uint16 bit patterns of a bf16 tensor, as a host numpy array."""
    import numpy as np
    assert x.dtype == torch.bfloat16
    return x.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)
