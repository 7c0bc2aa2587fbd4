"""fp64 CPU oracle for the teacher-cache builder (top-K selection + softmax).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU legs of ``bench.py`` may import this module; the library never calls it.

What is computed (the offline step of the pipeline the pages describe:
thorstenmeyerai.com "Making Knowledge Distillation Cheap Enough to Run at
Scale", pipeline steps "Infer once" and "Select top-K"; aimodeling.com "The
Hidden Memory Bottleneck in LLM Distillation", "First cut": the teacher's
top-100 probabilities are cached for every token).  For teacher logits
Z[T, V]:

    order_t  = ids sorted by logit descending, equal logits by ascending id
    idx_t    = order_t[:K]
    lse_t    = log sum_j exp(z_tj)            (max-shifted; -inf terms add 0)
    p_tk     = exp(z_{t, idx_tk} - lse_t)     (so sum_k p_tk <= 1)

Readings where the pages are silent: temperature 1; the cache holds
probabilities (fp32) in rank order; ties go to the lower id.

Pinned by ``tests/test_cache_oracle.py`` (closed forms, invariants, brute
force against ``topk_cache_naive``, torch.topk's values).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["topk_cache_oracle", "topk_cache_naive"]


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):
        import torch

        a = a.detach().to("cpu").to(torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def topk_cache_oracle(Z, K: int):
    """idx [T,K] int32, p [T,K] fp64, lse [T] fp64 for logits Z [T,V] (any float dtype)."""
    Z = _f64(Z)
    T, V = Z.shape
    idx = np.empty((T, K), dtype=np.int32)
    p = np.empty((T, K))
    lse = np.empty(T)
    ids = np.arange(V)
    for t in range(T):
        z = Z[t]
        order = np.lexsort((ids, -z))        # last key primary: -z ascending, then id ascending
        idx[t] = order[:K]
        m = z.max()
        lse[t] = m + math.log(np.exp(z[np.isfinite(z)] - m).sum()) if np.isfinite(m) else -math.inf
        p[t] = np.exp(z[idx[t]] - lse[t])
    return {"idx": idx, "p": p, "lse": lse}


def topk_cache_naive(Z, K: int):
    """Pure-Python selection for tiny inputs: K times take the largest remaining
    logit, the first (lowest id) of equal ones; lse by an explicit sum."""
    rows = _f64(Z).tolist()
    out_i, out_p, out_l = [], [], []
    for z in rows:
        taken = [False] * len(z)
        sel = []
        for _ in range(K):
            best = -1
            for j, v in enumerate(z):
                if not taken[j] and (best < 0 or v > z[best]):
                    best = j
            taken[best] = True
            sel.append(best)
        m = max(z)
        lse = m + math.log(sum(math.exp(v - m) for v in z if v != -math.inf))
        out_i.append(sel)
        out_l.append(lse)
        out_p.append([math.exp(z[j] - lse) for j in sel])
    return {"idx": np.array(out_i, dtype=np.int32), "p": np.array(out_p), "lse": np.array(out_l)}
