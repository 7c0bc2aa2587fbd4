"""fp64 CPU oracle for the fused, chunked top-K KL distillation loss.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference legs of ``bench.py`` may import this module.  The
library under ``lm_head_top_tma_b300/`` never calls it and shares no code with
it; the two meet only at the seeded inputs of ``lm_head_top_tma_b300.inputs``.

Source pages: "Efficient Knowledge Distillation for LLMs: Offline Top-K Logits
and a Fused Chunked KL Loss" (arXiv 2608.03796) as summarised by
legiblepapers.com ("Efficient Knowledge Distillation for Large Models"),
aimodeling.com ("The Hidden Memory Bottleneck in LLM Distillation") and
thorstenmeyerai.com ("Making Knowledge Distillation Cheap Enough to Run at
Scale").

What is computed.  For student hidden states H[T,d], LM-head weights W[V,d]
and a teacher cache of top-K ids idx[T,K] with probabilities p[T,K]:

    z_t    = H_t W^T                                 student logits
    lse_t  = log sum_j exp(z_tj)                     (max-shifted)
    L_t    = sum_k p_tk (log p_tk - (z_{t,idx_tk} - lse_t)),   0 log 0 := 0
    L      = sum_t L_t                               (sum, no 1/T)
    M_t    = sum_k p_tk                              teacher mass on the top-K
    G_t    = M_t softmax(z_t) - sum_k p_tk e_{idx_tk}
    dH     = G W ,   dW = G^T H

The loss is the forward KL from the teacher's top-K distribution to the
student's softmax, restricted to the top-K support; G is its exact logit
gradient.  That gradient is the one the legiblepapers summary states in FAQ Q5
(a dense M-times-softmax term minus the sparse teacher correction at the top-K
positions), and the chunking over the sequence (aimodeling "Second cut";
thorstenmeyerai "Fuse and chunk") changes only where the work happens, not the
result (thorstenmeyerai "Quality and Generality Need Testing": the dense,
forward-chunked and fused losses are mathematically equivalent).  This oracle
therefore writes the plain definition out, blocked over rows only to bound
host memory.

Readings where the pages are silent (each is stated again in the design
notes):  reduction is a sum over tokens; temperature 1; a duplicate id in a
row contributes once per occurrence; p = 0 entries contribute nothing; a row
whose ids are not all in [0, V) contributes nothing (L_t = 0, G_t = 0);
a row with M_t = 0 has L_t = 0 and G_t = 0.

Every function here is pinned by ``tests/test_oracle.py`` (finite differences,
torch cross-entropy and KL-divergence autograd special cases, closed forms and
invariants, and brute force against ``kd_oracle_naive``).
"""
from __future__ import annotations

import math

import numpy as np

__all__ = ["kd_oracle", "kd_oracle_rows", "kd_oracle_dW_rows", "kd_oracle_naive", "valid_rows"]


def _f64(a) -> np.ndarray:
    """Widen a NumPy array or a torch tensor (bf16/fp32 included) to fp64."""
    if hasattr(a, "detach"):
        a = a.detach().to("cpu")
        import torch  # local: only when a torch tensor is handed in

        a = a.to(torch.float64).numpy()
    return np.asarray(a, dtype=np.float64)


def valid_rows(idx: np.ndarray, V: int) -> np.ndarray:
    """Rows whose ids all lie in [0, V)."""
    idx = np.asarray(idx)
    return np.all((idx >= 0) & (idx < V), axis=1)


def kd_oracle(H, W, idx, p, want_grads: bool = True, rows_per_block: int = 256):
    """fp64 loss, per-row loss, lse and (optionally) dH, dW.

    H [T,d], W [V,d] (any float dtype, widened to fp64); idx [T,K] integer
    ids; p [T,K] non-negative probabilities.  Returns a dict with ``loss``
    (float), ``loss_rows`` [T], ``lse`` [T] and, if ``want_grads``, ``dH``
    [T,d] and ``dW`` [V,d].
    """
    Wd = _f64(W)
    idx = np.asarray(idx).astype(np.int64)
    pd = _f64(p)
    T, K = idx.shape
    V, d = Wd.shape
    ok = valid_rows(idx, V)
    lse = np.zeros(T)
    loss_rows = np.zeros(T)
    dH = np.zeros((T, d)) if want_grads else None
    dW = np.zeros((V, d)) if want_grads else None
    for t0 in range(0, T, rows_per_block):
        t1 = min(T, t0 + rows_per_block)
        Hb = _f64(H[t0:t1])
        z = Hb @ Wd.T                                        # [B, V]
        zmax = z.max(axis=1)
        lse_b = zmax + np.log(np.exp(z - zmax[:, None]).sum(axis=1))
        lse[t0:t1] = lse_b
        ib = idx[t0:t1]
        pb = pd[t0:t1]
        okb = ok[t0:t1]
        ib_safe = np.where(okb[:, None], ib, 0)
        zk = np.take_along_axis(z, ib_safe, axis=1)          # [B, K]
        log_q = zk - lse_b[:, None]                          # log softmax at the ids
        with np.errstate(divide="ignore", invalid="ignore"):
            terms = np.where(pb > 0, pb * (np.log(np.where(pb > 0, pb, 1.0)) - log_q), 0.0)
        lrow = terms.sum(axis=1)
        loss_rows[t0:t1] = np.where(okb, lrow, 0.0)
        if want_grads:
            M = pb.sum(axis=1)
            G = M[:, None] * np.exp(z - lse_b[:, None])      # M_t softmax(z_t)
            rows = np.repeat(np.arange(t1 - t0), K)
            np.subtract.at(G, (rows, ib_safe.ravel()), pb.ravel())
            G[~okb] = 0.0
            dH[t0:t1] = G @ Wd
            dW += G.T @ Hb
    out = {"loss": float(loss_rows.sum()), "loss_rows": loss_rows, "lse": lse}
    if want_grads:
        out["dH"] = dH
        out["dW"] = dW
    return out


def kd_oracle_rows(H, W, idx, p, rows, rows_per_block: int = 256):
    """lse, per-row loss and dH for the selected token rows only.

    Rows are independent in every one of these outputs, so this is
    ``kd_oracle`` on the sub-batch; it lets a test check sampled rows of a
    workload too large for the full fp64 computation."""
    rows = np.asarray(rows, dtype=np.int64)
    Hs = _f64(H[rows]) if not hasattr(H, "detach") else _f64(H[rows.tolist()])
    out = kd_oracle(Hs, W, np.asarray(idx)[rows], np.asarray(p)[rows],
                    want_grads=True, rows_per_block=rows_per_block)
    return {"rows": rows, "lse": out["lse"], "loss_rows": out["loss_rows"], "dH": out["dH"]}


def kd_oracle_dW_rows(H, W, idx, p, lse, vrows, rows_per_block: int = 1024):
    """Selected vocabulary rows of dW = G^T H, given lse_t for every token.

    dW_j = sum_t G_tj H_t with G_tj = M_t exp(z_tj - lse_t) - sum_{k: idx_tk = j}
    p_tk, the same G as ``kd_oracle`` (legiblepapers FAQ Q5 gradient), taken
    column by column: only z_tj = H_t . W_j for the selected j is formed, so a
    test can check chosen rows of dW for a sequence too long for the full fp64
    backward.  ``lse`` must be the oracle's own (``kd_oracle`` with
    ``want_grads=False``) for all T rows; rows with an id outside [0, V)
    contribute nothing.  ``vrows`` are distinct vocabulary ids; returns
    [len(vrows), d]."""
    Wd = _f64(W)
    idx = np.asarray(idx).astype(np.int64)
    pd = _f64(p)
    lse = np.asarray(lse, dtype=np.float64)
    vrows = np.asarray(vrows, dtype=np.int64)
    if np.unique(vrows).size != vrows.size:
        raise ValueError("vrows must be distinct")
    T, K = idx.shape
    V, d = Wd.shape
    ok = valid_rows(idx, V)
    col = np.full(V, -1, dtype=np.int64)                     # vocabulary id -> selected column
    col[vrows] = np.arange(vrows.size)
    Wj = Wd[vrows]                                           # [J, d]
    out = np.zeros((vrows.size, d))
    for t0 in range(0, T, rows_per_block):
        t1 = min(T, t0 + rows_per_block)
        Hb = _f64(H[t0:t1])
        zJ = Hb @ Wj.T                                       # [B, J]
        ib = idx[t0:t1]
        pb = pd[t0:t1]
        M = pb.sum(axis=1)
        G = M[:, None] * np.exp(zJ - lse[t0:t1, None])
        ib_safe = np.where(ok[t0:t1, None], ib, 0)
        c = col[ib_safe]                                     # [B, K], -1 where the id is not selected
        hit = c >= 0
        rows = np.repeat(np.arange(t1 - t0)[:, None], K, axis=1)
        np.subtract.at(G, (rows[hit], c[hit]), pb[hit])
        G[~ok[t0:t1]] = 0.0
        out += G.T @ Hb
    return out


def kd_oracle_naive(H, W, idx, p):
    """Pure-Python loops in fp64, for tiny inputs (brute-force cross-check).

    Written independently of ``kd_oracle``: explicit sums over d, V and K."""
    Hl = _f64(H).tolist()
    Wl = _f64(W).tolist()
    il = np.asarray(idx).astype(np.int64).tolist()
    pl = _f64(p).tolist()
    T, V, d = len(Hl), len(Wl), len(Wl[0])
    K = len(il[0]) if T else 0
    loss_rows, lses = [], []
    dH = [[0.0] * d for _ in range(T)]
    dW = [[0.0] * d for _ in range(V)]
    for t in range(T):
        z = [sum(Hl[t][c] * Wl[j][c] for c in range(d)) for j in range(V)]
        m = max(z)
        lse = m + math.log(sum(math.exp(zj - m) for zj in z))
        lses.append(lse)
        if not all(0 <= il[t][k] < V for k in range(K)):
            loss_rows.append(0.0)
            continue
        lt = 0.0
        for k in range(K):
            pk = pl[t][k]
            if pk > 0.0:
                lt += pk * (math.log(pk) - (z[il[t][k]] - lse))
        loss_rows.append(lt)
        mass = sum(pl[t])
        g = [mass * math.exp(z[j] - lse) for j in range(V)]
        for k in range(K):
            g[il[t][k]] -= pl[t][k]
        for c in range(d):
            dH[t][c] = sum(g[j] * Wl[j][c] for j in range(V))
        for j in range(V):
            for c in range(d):
                dW[j][c] += g[j] * Hl[t][c]
    return {"loss": math.fsum(loss_rows), "loss_rows": np.array(loss_rows),
            "lse": np.array(lses), "dH": np.array(dH).reshape(T, d),
            "dW": np.array(dW).reshape(V, d)}
