"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI
and compare with the fp64 oracle element by element.

Tolerances.  Loss: relative error <= 1e-3; dH, dW: max-abs error <=
2e-2 x max|ref| (the targets the method is built to).  lse and per-row loss
are not given a target, so they get one derived from the arithmetic: every
logit is an fp32 tensor-core sum of d bf16 products (relative error ~1e-6), the
normaliser is an fp32 sum of V terms 2^(x) from the special-function unit
(relative error ~2^-22 each, plus fp32 rounding over <= 256 terms per tile and
V/256 tiles combined in fp32), so lse carries an absolute error of order 1e-5;
1e-3 absolute leaves two orders of magnitude of margin while still catching a
dropped tile (which moves lse by >= log(1 + 1/(V/256)) ~ 2e-3 at V = 128256),
a missing top-K term or a wrong sign.  Per-row losses L_t = E_t - sum p z +
M_t lse_t inherit that bound (M_t <= 1): 2e-3 absolute.
"""
from __future__ import annotations

import numpy as np
import torch

from lm_head_top_tma_b300 import api
from oracle import kd_oracle, kd_oracle_rows

LOSS_RTOL = 1e-3
GRAD_FRAC = 2e-2
LSE_ATOL = 1e-3
LROW_ATOL = 2e-3


def to_dev(idx, p, dev):
    return (torch.as_tensor(np.ascontiguousarray(idx), dtype=torch.int32).to(dev),
            torch.as_tensor(np.ascontiguousarray(p), dtype=torch.float32).to(dev))


def grad_err(got: np.ndarray, ref: np.ndarray) -> float:
    scale = float(np.abs(ref).max())
    return float(np.abs(got - ref).max()) / max(scale, 1e-30)


def assert_close_full(got: dict, ref: dict, what=("loss", "lse", "loss_rows", "dH", "dW")):
    msgs = []
    if "loss" in what:
        rl = abs(float(got["loss"]) - ref["loss"]) / max(abs(ref["loss"]), 1e-30)
        if not rl <= LOSS_RTOL:
            msgs.append(f"loss rel err {rl:.3e} (gpu {float(got['loss'])!r}, ref {ref['loss']!r})")
    if "lse" in what:
        e = float(np.abs(got["lse"] - ref["lse"]).max())
        if not e <= LSE_ATOL:
            msgs.append(f"lse max abs err {e:.3e}")
    if "loss_rows" in what and "loss_rows" in got:
        e = float(np.abs(got["loss_rows"] - ref["loss_rows"]).max())
        if not e <= LROW_ATOL:
            msgs.append(f"loss_rows max abs err {e:.3e}")
    for k in ("dH", "dW"):
        if k in what and k in got:
            e = grad_err(got[k], ref[k])
            if not e <= GRAD_FRAC:
                msgs.append(f"{k} max abs err / max|ref| = {e:.3e}")
    assert not msgs, "; ".join(msgs)


def fused_to_host(res: dict) -> dict:
    torch.cuda.synchronize()
    out = {"loss": float(res["loss"].item()), "lse": res["lse"].double().cpu().numpy(),
           "dH": res["dH"].double().cpu().numpy(), "dW": res["dW"].double().cpu().numpy()}
    if "loss_rows" in res:
        out["loss_rows"] = res["loss_rows"].double().cpu().numpy()
    return out


def run_fused(H, W, idx_np, p_np, chunk, recompute=True, **kw):
    idx, p = to_dev(idx_np, p_np, H.device)
    fn = api.fused_step if recompute else api.fused_step_norecompute
    return fused_to_host(fn(H, W, idx, p, chunk, loss_rows=True, **kw))


__all__ = ["kd_oracle", "kd_oracle_rows", "to_dev", "grad_err", "assert_close_full", "fused_to_host",
           "run_fused", "LOSS_RTOL", "GRAD_FRAC", "LSE_ATOL", "LROW_ATOL"]


# ------------------------------------------------------------------ full-size cases
def sample_rows(T: int, chunk: int, n: int = 256, seed: int = 0) -> np.ndarray:
    """Token rows to check at a full sequence length: the first and last row
    of every chunk, topped up with seeded random rows to at least ``n``."""
    rng = np.random.default_rng(seed)
    edges = set()
    for c0 in range(0, T, chunk):
        edges.update({c0, min(T - 1, c0 + chunk - 1)})
    rows = set(edges)
    rest = np.setdiff1d(np.arange(T), np.fromiter(rows, dtype=np.int64))
    need = max(0, n - len(rows))
    rows.update(rng.choice(rest, size=min(need, rest.size), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def sample_vocab_rows(V: int, idx: np.ndarray, n: int = 256, seed: int = 0) -> np.ndarray:
    """Vocabulary rows of dW to check: both ends of the vocabulary, both sides
    of several 128- and 256-column tile boundaries (including the last,
    partial tile), the ids the teacher cache names most often (where the -p
    corrections pile up), and seeded random ids, at least ``n`` in all."""
    rng = np.random.default_rng(seed)
    rows = {0, 1, V - 2, V - 1}
    last_tile = (V - 1) // 256 * 256
    for b in [128, 256, 384, 512, last_tile, last_tile - 128, last_tile + 128] + \
             list(rng.choice(np.arange(256, V, 256), size=min(8, max(0, (V - 1) // 256)), replace=False)):
        for j in (int(b) - 1, int(b)):
            if 0 <= j < V:
                rows.add(j)
    ids, counts = np.unique(np.asarray(idx).ravel(), return_counts=True)
    ok = (ids >= 0) & (ids < V)
    rows.update(ids[ok][np.argsort(-counts[ok], kind="stable")][:32].tolist())
    rest = np.setdiff1d(np.arange(V), np.fromiter(rows, dtype=np.int64))
    need = max(0, n - len(rows))
    rows.update(rng.choice(rest, size=min(need, rest.size), replace=False).tolist())
    return np.array(sorted(rows), dtype=np.int64)


def projection_identities(H, W, dH, dW, r: int = 8, seed: int = 0):
    """<W A, dW> against <dH, H A^T> for r seeded rank-one matrices A = u v^T,
    in fp64 on the device.  Both equal trace(A^T W^T G^T H) for the same bf16
    G, so every one of them holds up to the fp32 accumulation of the two
    GEMMs; unlike the single identity with A = I they change when a group of
    dW rows is scaled, dropped, permuted or transposed.  Returns a list of
    (lhs, rhs, scale) with scale the quadrature norm of the summed terms,
    the size of a sum whose terms have independent signs."""
    import torch

    g = torch.Generator(device=H.device).manual_seed(1000 + seed)
    d = H.shape[1]
    U = torch.randn(d, r, generator=g, device=H.device, dtype=torch.float64)
    Vv = torch.randn(d, r, generator=g, device=H.device, dtype=torch.float64)
    out = []
    a = W.double() @ U
    b = dW.double() @ Vv
    c = dH.double() @ U
    e = H.double() @ Vv
    ab, ce = a * b, c * e
    lhs, rhs = ab.sum(0), ce.sum(0)
    ls, rs = ab.square().sum(0).sqrt(), ce.square().sum(0).sqrt()
    for i in range(r):
        out.append((lhs[i].item(), rhs[i].item(), max(ls[i].item(), rs[i].item())))
    return out


def assert_projection_identities(H, W, dH, dW, rtol: float = 1e-3, r: int = 8):
    """Every projection identity holds within rtol of its quadrature scale.
    The two sides differ only by fp32 accumulation order (relative ~1e-5
    per element), while losing one 256-row tile of dW at V = 128256 moves a
    sum by ~sqrt(256 / V) = 4.5% of its scale."""
    bad = [(l, rr, s) for l, rr, s in projection_identities(H, W, dH, dW, r=r) if abs(l - rr) > rtol * s]
    assert not bad, f"projection identities off: {bad}"


_CASE_CACHE: dict = {}


def full_case(name: str, T: int | None = None, oracle: str = "forward"):
    """Inputs of a workload at full size (H, W generated on the GPU) and the
    oracle's result, computed once and kept for the next test (one case at a
    time).  ``oracle``: "forward" (loss, per-row loss and lse of every row),
    "grads" (the same with dH and dW) or "rows" (lse, per-row loss and dH of
    the rows ``sample_rows`` picks, returned under ``rows``)."""
    import torch

    from lm_head_top_tma_b300.inputs import get_workload, make_inputs, sweep_workload

    key = (name, T, oracle)
    if key in _CASE_CACHE:
        return _CASE_CACHE[key]
    _CASE_CACHE.clear()
    wl = sweep_workload(int(name[5:])) if name.startswith("sweep") else get_workload(name)
    inp = make_inputs(wl, device=torch.device("cuda:0"), T=T)
    wl = inp["workload"]
    if oracle == "rows":
        rows = sample_rows(wl.T, wl.chunk)
        sel = torch.as_tensor(rows, device=inp["H"].device)
        ref = kd_oracle_rows(inp["H"][sel].cpu(), inp["W"].cpu(), inp["idx"][rows], inp["p"][rows],
                             np.arange(len(rows)))
        ref["rows"] = rows
    else:
        ref = kd_oracle(inp["H"].cpu(), inp["W"].cpu(), inp["idx"], inp["p"], want_grads=oracle == "grads",
                        rows_per_block=1024)
    _CASE_CACHE[key] = (inp, ref)
    return inp, ref


__all__ += ["sample_rows", "sample_vocab_rows", "projection_identities", "assert_projection_identities",
            "full_case"]
