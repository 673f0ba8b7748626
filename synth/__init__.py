"""Seeded synthetic inputs shared by the oracle tests, the GPU parity tests and the bench.

This package holds no arithmetic of the method itself: it only draws random
student hidden states, LM-head weights, teacher top-K caches, padding masks and
dense teacher logits with the shapes and distributions of the five workloads.
"""
from .workloads import WORKLOADS, Workload, make_inputs, make_dense_teacher_logits, bf16_bits

__all__ = ["WORKLOADS", "Workload", "make_inputs", "make_dense_teacher_logits", "bf16_bits"]
