"""Fused, chunked top-K KL distillation loss over the LM head, for B300 (sm_103a).

The compute path is libkdtopk.so (hand-written tcgen05 / TMA kernels behind a
C ABI, include/kdtopk.h); ``lm_head_top_tma_b300.api`` marshals torch tensors
into it, and ``lm_head_top_tma_b300.dp`` runs it token-parallel across
processes.  ``lm_head_top_tma_b300.inputs`` draws the seeded synthetic
workloads.  Importing the package loads nothing; the library is loaded on
first use and its absence is an error, never a fallback.
"""

__all__ = ["api", "dp", "inputs"]
