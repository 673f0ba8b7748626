"""Float64 CPU oracle for the top-K teacher cache and the fused chunked KL loss.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
legs of ``bench.py`` (``cpu_baseline`` and ``--impl reference``) may import
this package.  The product package ``sparse_teacher_kl_gb300`` never imports it,
and the two share no code: no kernels, helpers, constants or pre/post-processing.

Every function cites the page passage it restates.  Page keys used throughout:

  [ART]  aiexpert.news article "Making knowledge distillation cheap enough to
         run in production": its paragraphs on the offline top-K cache, on the
         three loss formulations (dense, forward-chunked, fused chunked) and on
         the top-K limitation.
  [DAI]  dailyai.com.br, "Efficient Knowledge Distillation" launch report,
         sections "As duas inovações" and "O problema da distilação em larga escala".
  [EPO]  epoka.news, "Dos cambios de sistema que abaratan la destilación de
         conocimiento", sections "Adónde se va la memoria" and "Los dos cambios
         propuestos".
  [TIC]  aiexpert.news ticker on the same publication.
"""
from .kl import (
    bf16_to_f64,
    sparse_teacher,
    dense_kl,
    forward_chunked_kl,
    fused_chunked_kl,
    OracleResult,
)
from .topk import topk_cache, teacher_logsumexp, dropped_mass, teacher_logits_bf16

__all__ = [
    "bf16_to_f64",
    "sparse_teacher",
    "dense_kl",
    "forward_chunked_kl",
    "fused_chunked_kl",
    "OracleResult",
    "topk_cache",
    "teacher_logsumexp",
    "dropped_mass",
    "teacher_logits_bf16",
]
