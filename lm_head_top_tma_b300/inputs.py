"""Seeded synthetic inputs for the fused, chunked top-K KL distillation loss.

This module is the one thing the CUDA path, its tests, the benchmark and the
fp64 CPU oracle share.  It holds none of the loss arithmetic: it only draws
student hidden states H[T,d], LM-head weights W[V,d] (both bf16) and an offline
teacher cache (idx[T,K] int32, p[T,K] fp32) with the shapes and value
distributions of the workloads below.

Workloads (sizes from the pages' own settings: a ~3.2B student head with the
Llama-3 vocabulary, long-context 32K recovery, a 201,088-token vocabulary
head, and the output-head-only 4K..256K scaling benchmark):

* ``tiny``     T 256, d 256, V 4096, K 16, chunk 64.  H, W ~ N(0, 0.02^2) with H
  scaled by 50; ids: K distinct uniform ids per row; p = softmax of N(0, 2^2)
  logits over the K ids, times a row mass M_t ~ U(0.8, 1.0).  Seed 0.
* ``head3b``   T 8192, d 3072, V 128256, K 100, chunk 1024.  Seed 1.
* ``longctx``  T 32768, d 3072, V 128256, K 100, chunk 2048.  Seed 2.
* ``bigvocab`` T 131072, d 2880, V 201088, K 100, chunk 2048.  Seed 3.
* ``sweep``    d 4096, V 128256, K 100, chunk 4096, T in 4K..256K.
  Seed 5 + log2(T / 4096).

For every workload but ``tiny``: H ~ N(0, 1) and W ~ N(0, 0.02^2), rounded to
bf16; ids are K distinct draws (without replacement, in draw order) from a
Zipf(s = 1.1) law over vocabulary rank, mapped rank -> id by a seeded
permutation; p = softmax of K N(0, 3^2) logits sorted in descending order
(the first-drawn id gets the largest probability), times M_t ~ U(0.85, 0.99).
The cache keeps ids in rank (draw) order, not id order, as a top-K cache
written by an offline teacher pass would.

H and W come from a seeded ``torch.Generator`` on the requested device, so a
CUDA-generated pair differs from a CPU-generated one with the same seed; a test
that compares the two sides generates once and copies.  The cache is drawn on
the host with NumPy's PCG64.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, replace

import numpy as np

__all__ = ["Workload", "WORKLOADS", "sweep_workload", "get_workload",
           "make_cache", "make_hw", "make_inputs", "make_teacher_logits"]


@dataclass(frozen=True)
class Workload:
    name: str
    T: int
    d: int
    V: int
    K: int
    chunk: int
    seed: int
    kind: str  # "uniform" (tiny) or "zipf"

    def with_T(self, T: int) -> "Workload":
        return replace(self, T=int(T))


WORKLOADS = {
    "tiny": Workload("tiny", 256, 256, 4096, 16, 64, 0, "uniform"),
    "head3b": Workload("head3b", 8192, 3072, 128256, 100, 1024, 1, "zipf"),
    "longctx": Workload("longctx", 32768, 3072, 128256, 100, 2048, 2, "zipf"),
    "bigvocab": Workload("bigvocab", 131072, 2880, 201088, 100, 2048, 3, "zipf"),
}

SWEEP_T = (4096, 8192, 16384, 32768, 65536, 131072, 262144)


def sweep_workload(T: int) -> Workload:
    """Output-head-only scaling point at sequence length T."""
    return Workload(f"sweep{T}", int(T), 4096, 128256, 100, 4096,
                    5 + int(round(math.log2(T / 4096))), "zipf")


def get_workload(name: str) -> Workload:
    if name in WORKLOADS:
        return WORKLOADS[name]
    if name.startswith("sweep"):
        return sweep_workload(int(name[5:]))
    raise KeyError(name)


# ----------------------------------------------------------------------------
# teacher cache
# ----------------------------------------------------------------------------

def _first_k_distinct(cand: np.ndarray, K: int):
    """For each row of ``cand`` keep the first K distinct values in order.

    Returns (rows_ok mask, [n_ok, K] array of the kept values)."""
    order = np.argsort(cand, axis=1, kind="stable")
    s = np.take_along_axis(cand, order, axis=1)
    first_sorted = np.ones(s.shape, dtype=bool)
    first_sorted[:, 1:] = s[:, 1:] != s[:, :-1]
    first = np.empty_like(first_sorted)
    np.put_along_axis(first, order, first_sorted, axis=1)
    cnt = np.cumsum(first, axis=1)
    ok = cnt[:, -1] >= K
    take = first & (cnt <= K)
    kept = cand[ok][take[ok]].reshape(-1, K)
    return ok, kept


def _draw_ids(rng: np.random.Generator, T: int, V: int, K: int, kind: str,
              zipf_s: float = 1.1, block: int = 8192) -> np.ndarray:
    if K > V:
        raise ValueError("K must not exceed V")
    if kind == "uniform":
        sampler = lambda n, m: rng.integers(0, V, size=(n, m), dtype=np.int64)
        perm = None
    elif kind == "zipf":
        w = np.arange(1, V + 1, dtype=np.float64) ** (-zipf_s)
        cdf = np.cumsum(w)
        cdf /= cdf[-1]
        perm = rng.permutation(V).astype(np.int64)

        def sampler(n, m):
            u = rng.random(size=(n, m))
            r = np.searchsorted(cdf, u, side="right")
            return np.minimum(r, V - 1)
    else:
        raise ValueError(kind)
    out = np.empty((T, K), dtype=np.int64)
    for t0 in range(0, T, block):
        n = min(block, T - t0)
        pending = np.arange(n)
        m = max(2 * K, 8) if kind == "uniform" else 4 * K + 64
        while pending.size:
            cand = sampler(pending.size, m)
            ok, kept = _first_k_distinct(cand, K)
            out[t0 + pending[ok]] = kept
            pending = pending[~ok]
            m *= 2
            if K == V and kind == "zipf":
                m = max(m, 64 * V)
    if perm is not None:
        out = perm[out]
    return out.astype(np.int32)


def _draw_probs(rng: np.random.Generator, T: int, K: int, kind: str) -> np.ndarray:
    if kind == "uniform":
        logits = rng.normal(0.0, 2.0, size=(T, K))
        mass = rng.uniform(0.8, 1.0, size=(T, 1))
    else:
        logits = -np.sort(-rng.normal(0.0, 3.0, size=(T, K)), axis=1)
        mass = rng.uniform(0.85, 0.99, size=(T, 1))
    logits -= logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    probs = e / e.sum(axis=1, keepdims=True)
    return (probs * mass).astype(np.float32)


def make_cache(T: int, V: int, K: int, kind: str, seed: int):
    """Offline top-K teacher cache: (idx [T,K] int32, p [T,K] float32)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    idx = _draw_ids(rng, T, V, K, kind)
    p = _draw_probs(rng, T, K, kind)
    return np.ascontiguousarray(idx), np.ascontiguousarray(p)


# ----------------------------------------------------------------------------
# student hidden states and LM-head weights
# ----------------------------------------------------------------------------

def make_hw(T: int, d: int, V: int, kind: str, seed: int, device="cpu",
            block: int = 16384):
    """H [T,d] and W [V,d] as bf16 torch tensors on ``device``."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    h_scale = 0.02 * 50.0 if kind == "uniform" else 1.0

    def draw(rows, scale):
        out = torch.empty(rows, d, dtype=torch.bfloat16, device=device)
        for r0 in range(0, rows, block):
            n = min(block, rows - r0)
            x = torch.randn(n, d, generator=g, device=device, dtype=torch.float32)
            out[r0:r0 + n] = (x * scale).to(torch.bfloat16)
        return out

    H = draw(T, h_scale)
    W = draw(V, 0.02)
    return H, W


def make_inputs(workload, device="cpu", T: int | None = None, seed: int | None = None):
    """All inputs of one workload: dict with H, W (torch bf16 on ``device``),
    idx, p (NumPy on the host) and the workload record."""
    wl = get_workload(workload) if isinstance(workload, str) else workload
    if T is not None:
        wl = wl.with_T(T)
    if seed is not None:
        wl = replace(wl, seed=int(seed))
    H, W = make_hw(wl.T, wl.d, wl.V, wl.kind, wl.seed, device=device)
    idx, p = make_cache(wl.T, wl.V, wl.K, wl.kind, wl.seed)
    return {"H": H, "W": W, "idx": idx, "p": p, "workload": wl}


# ----------------------------------------------------------------------------
# teacher logits (input of the cache builder)
# ----------------------------------------------------------------------------

def make_teacher_logits(T: int, V: int, seed: int, device="cpu", dtype="bf16",
                        zipf_s: float = 1.1, noise: float = 2.0, block: int = 4096):
    """Synthetic teacher logits Z [T,V] on ``device``: a Zipf-shaped prior over
    a seeded vocabulary ranking plus per-token Gaussian noise,
    z_tj = -s log(1 + rank(j)) + noise * N(0, 1), rounded to ``dtype``
    ("bf16" or "fp32").  The top-K ids of such rows follow the same
    rank-permuted Zipf law as ``make_cache``'s ids; bf16 rounding leaves many
    exactly equal logits, so the builder's tie order is exercised."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    perm = torch.randperm(V, generator=g, device=device)
    prior = torch.empty(V, dtype=torch.float32, device=device)
    prior[perm] = -zipf_s * torch.log1p(torch.arange(V, dtype=torch.float32, device=device))
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    out = torch.empty(T, V, dtype=tdt, device=device)
    for r0 in range(0, T, block):
        n = min(block, T - r0)
        x = torch.randn(n, V, generator=g, device=device, dtype=torch.float32)
        out[r0:r0 + n] = (prior[None, :] + noise * x).to(tdt)
    return out
