"""Parity at the workloads' full sizes.

1. Every head shape (d, V, K) at full size with a few hundred tokens in
   ragged 128-row chunks: every output element against the fp64 oracle.
2. The benchmark's launch configuration (long-context head, chunk 2048) over
   two chunks, the second ragged: every element, dW included.
3. Full sequence lengths (8K, 32K, 128K, 256K tokens): lse, per-row loss and dH
   on sampled rows (first / last rows of chunks included) against the oracle,
   which computes each sampled row on its own; the loss equals the sum of the
   per-row losses; and dW is tied to dH by <W, dW> = <H, dH> (both are
   sum_tj G_tj z_tj for the same bf16 G), which fails if a chunk's dW is lost,
   offset or transposed.
"""
import numpy as np
import pytest
import torch

from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.inputs import get_workload, make_inputs, sweep_workload
from parity_util import (LROW_ATOL, LSE_ATOL, GRAD_FRAC, assert_close_full, kd_oracle, kd_oracle_rows,
                         run_fused, to_dev)

pytestmark = pytest.mark.gpu

HEADS = ["head3b", "bigvocab", "sweep4096"]


@pytest.mark.parametrize("name", HEADS)
def test_full_head_small_T(cuda_device, name):
    wl = get_workload(name)
    inp = make_inputs(wl, device=cuda_device, T=300)
    ref = kd_oracle(inp["H"].cpu(), inp["W"].cpu(), inp["idx"], inp["p"])
    got = run_fused(inp["H"], inp["W"], inp["idx"], inp["p"], 128)
    assert_close_full(got, ref)


def test_bench_launch_configuration_two_chunks(cuda_device):
    wl = get_workload("longctx")
    inp = make_inputs(wl, device=cuda_device, T=wl.chunk + 300)
    ref = kd_oracle(inp["H"].cpu(), inp["W"].cpu(), inp["idx"], inp["p"])
    got = run_fused(inp["H"], inp["W"], inp["idx"], inp["p"], wl.chunk)
    assert_close_full(got, ref)


def _sample_rows(T, chunk, n=40, seed=0):
    rng = np.random.default_rng(seed)
    edges = {0, T - 1}
    for c0 in range(0, T, chunk):
        edges.update({c0, min(T - 1, c0 + chunk - 1)})
    edges = sorted(edges)[:16]
    extra = rng.choice(T, size=n - len(edges), replace=False)
    return np.unique(np.concatenate([np.array(edges), extra]))


@pytest.mark.parametrize("name", ["head3b", "longctx", "bigvocab", "sweep262144"])
def test_full_T_sampled(cuda_device, name):
    wl = sweep_workload(262144) if name == "sweep262144" else get_workload(name)
    inp = make_inputs(wl, device=cuda_device)
    H, W = inp["H"], inp["W"]
    idx, p = to_dev(inp["idx"], inp["p"], cuda_device)
    res = api.fused_step(H, W, idx, p, wl.chunk, loss_rows=True)
    torch.cuda.synchronize()
    rows = _sample_rows(wl.T, wl.chunk)
    ref = kd_oracle_rows(H[torch.as_tensor(rows, device=cuda_device)].cpu(), W.cpu(),
                         inp["idx"][rows], inp["p"][rows], np.arange(len(rows)))
    lse = res["lse"].double().cpu().numpy()
    lrows = res["loss_rows"].double().cpu().numpy()
    dH_rows = res["dH"][torch.as_tensor(rows, device=cuda_device)].double().cpu().numpy()
    assert np.abs(lse[rows] - ref["lse"]).max() <= LSE_ATOL
    assert np.abs(lrows[rows] - ref["loss_rows"]).max() <= LROW_ATOL
    scale = np.abs(ref["dH"]).max()
    assert np.abs(dH_rows - ref["dH"]).max() <= GRAD_FRAC * scale
    # the loss is the fixed-order fp64 sum of the per-row losses (rounded to fp32 once)
    loss = res["loss"].item()
    assert abs(loss - lrows.sum()) <= 1e-5 * abs(lrows.sum()) + 1e-3
    # <W, dW> == <H, dH>
    lhs = torch.sum(W.double() * res["dW"].double()).item()
    rhs = torch.sum(H.double() * res["dH"].double()).item()
    assert abs(lhs - rhs) <= 1e-3 * max(abs(lhs), abs(rhs)), (lhs, rhs)
    assert torch.isfinite(res["dW"]).all()
