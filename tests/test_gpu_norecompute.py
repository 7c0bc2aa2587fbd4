"""The fused step without the backward recompute (kd_topk_kl_fused_step_norecompute)
against the fp64 oracle, element by element, on the same cases as the recomputing
fused step: every chunk size of the tiny workload, ragged and degenerate shapes,
duplicates / pads / zero-mass rows, bad ids, and dW accumulation with dloss (the
full-size cases, every head shape and full sequence lengths, are parametrised
over both fused steps in tests/test_gpu_fullsize.py).  Its G is rounded to bf16
twice (the kept exponentials, then G), so it is also compared with the
recomputing step, whose loss and lse it must reproduce exactly (the forward
arithmetic is the same up to the order of the exponent sums)."""
import numpy as np
import pytest
import torch

from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.inputs import make_cache, make_hw, make_inputs
from parity_util import GRAD_FRAC, assert_close_full, fused_to_host, grad_err, kd_oracle, run_fused, to_dev

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny(cuda_device):
    inp = make_inputs("tiny", device=cuda_device)
    ref = kd_oracle(inp["H"].cpu(), inp["W"].cpu(), inp["idx"], inp["p"])
    return inp, ref


@pytest.mark.parametrize("chunk", [64, 100, 128, 256, 1000])
def test_tiny_all_chunks(tiny, chunk):
    inp, ref = tiny
    got = run_fused(inp["H"], inp["W"], inp["idx"], inp["p"], chunk, recompute=False)
    assert_close_full(got, ref)


def test_matches_recomputing_step(tiny):
    inp, _ = tiny
    a = run_fused(inp["H"], inp["W"], inp["idx"], inp["p"], 128, recompute=True)
    b = run_fused(inp["H"], inp["W"], inp["idx"], inp["p"], 128, recompute=False)
    assert np.abs(a["lse"] - b["lse"]).max() <= 1e-5
    assert abs(a["loss"] - b["loss"]) <= 1e-5 * abs(a["loss"])
    # G differs by at most about two bf16 roundings per element
    assert grad_err(b["dH"], a["dH"]) <= 5e-3
    assert grad_err(b["dW"], a["dW"]) <= 5e-3


@pytest.mark.parametrize("T,d,V,K,chunk", [
    (250, 200, 4000, 16, 100),     # ragged T, V % 256 != 0, d % 64 != 0
    (1, 64, 300, 5, 64),           # one token, V below one vocabulary tile
    (129, 136, 520, 7, 128),       # one row past a tile, odd d
    (300, 256, 4096, 1, 128),      # K = 1 (cross-entropy)
    (64, 128, 512, 512, 64),       # K = V (full distribution)
    (200, 96, 2056, 100, 77),      # odd chunk
    (300, 64, 9000, 20, 256),      # V spans several 4096-column blocks of the G pass, ragged
])
def test_edge_shapes(cuda_device, T, d, V, K, chunk):
    H, W = make_hw(T, d, V, "uniform", seed=T + V, device=cuda_device)
    idx, p = make_cache(T, V, K, "uniform", seed=K)
    ref = kd_oracle(H.cpu(), W.cpu(), idx, p)
    got = run_fused(H, W, idx, p, chunk, recompute=False)
    assert_close_full(got, ref)


def test_duplicates_pads_zero_mass_and_bad_ids(cuda_device):
    T, d, V, K = 300, 128, 5000, 12
    H, W = make_hw(T, d, V, "uniform", seed=3, device=cuda_device)
    idx, p = make_cache(T, V, K, "uniform", seed=4)
    idx[0, 1] = idx[0, 0]
    idx[1, :] = idx[1, 0]               # one id repeated K times
    p[2, 3:] = 0.0                      # zero-probability pads
    p[3, :] = 0.0                       # no teacher mass
    idx[4, :] = np.arange(V - K, V)     # ids at the vocabulary tail
    idx[5, :] = np.arange(K)            # ids at the head
    idx[6, :] = 4090 + np.arange(K)     # ids straddling two G-pass column blocks
    idx[10, 2] = V + 5                  # bad ids: rows contribute nothing
    idx[150, 0] = -3
    ref = kd_oracle(H.cpu(), W.cpu(), idx, p)
    idx_d, p_d = to_dev(idx, p, cuda_device)
    res = api.fused_step_norecompute(H, W, idx_d, p_d, 128, loss_rows=True, check=False)
    got = fused_to_host(res)
    assert_close_full(got, ref)
    assert got["loss_rows"][3] == 0.0 and np.all(got["dH"][3] == 0.0)
    assert got["loss_rows"][10] == 0.0 and np.all(got["dH"][150] == 0.0)


def test_accumulate_and_dloss(tiny):
    inp, ref = tiny
    H, W = inp["H"], inp["W"]
    idx, p = to_dev(inp["idx"], inp["p"], H.device)
    g = torch.Generator(device=H.device).manual_seed(9)
    dW0 = torch.randn(W.shape, generator=g, device=H.device)
    dW = dW0.clone()
    res = api.fused_step_norecompute(H, W, idx, p, 128, dloss=-0.5, dW=dW, accumulate_dW=True)
    torch.cuda.synchronize()
    assert grad_err((dW - dW0).double().cpu().numpy(), -0.5 * ref["dW"]) <= GRAD_FRAC
    assert grad_err(res["dH"].double().cpu().numpy(), -0.5 * ref["dH"]) <= GRAD_FRAC
    assert abs(res["loss"].item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])

