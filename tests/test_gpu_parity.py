"""CUDA path (through the C ABI) against the fp64 oracle, element by element,
on the tiny workload and on edge cases: ragged T and V, d not a multiple of
the 64-wide k-block, chunks below / not a multiple of / above the 128-row
tile, duplicates, zero-probability pads, zero-mass rows, K = 1 and K = V,
bad ids, dW accumulation and the dloss scale; forward + backward as separate
calls must agree with the fused step."""
import numpy as np
import pytest
import torch

from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.inputs import make_cache, make_hw, make_inputs
from parity_util import (GRAD_FRAC, assert_close_full, fused_to_host, grad_err, kd_oracle, run_fused,
                         to_dev)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tiny(cuda_device):
    inp = make_inputs("tiny", device=cuda_device)
    ref = kd_oracle(inp["H"].cpu(), inp["W"].cpu(), inp["idx"], inp["p"])
    return inp, ref


@pytest.mark.parametrize("chunk", [64, 100, 128, 256, 1000])
def test_tiny_fused_all_chunks(tiny, chunk):
    inp, ref = tiny
    got = run_fused(inp["H"], inp["W"], inp["idx"], inp["p"], chunk)
    assert_close_full(got, ref)


def test_tiny_forward_then_backward(tiny):
    inp, ref = tiny
    H, W = inp["H"], inp["W"]
    idx, p = to_dev(inp["idx"], inp["p"], H.device)
    loss, lse, rows = api.forward(H, W, idx, p, 64, loss_rows=True)
    dH, dW = api.backward(H, W, idx, p, lse, 64)
    torch.cuda.synchronize()
    got = {"loss": loss.item(), "lse": lse.double().cpu().numpy(), "loss_rows": rows.double().cpu().numpy(),
           "dH": dH.double().cpu().numpy(), "dW": dW.double().cpu().numpy()}
    assert_close_full(got, ref)
    fused = run_fused(H, W, inp["idx"], inp["p"], 64)
    # same kernels, same order: the separate calls reproduce the fused step bit for bit
    assert got["loss"] == fused["loss"]
    assert np.array_equal(got["dH"], fused["dH"]) and np.array_equal(got["dW"], fused["dW"])


@pytest.mark.parametrize("T,d,V,K,chunk", [
    (250, 200, 4000, 16, 100),     # ragged T, V % 256 != 0, d % 64 != 0
    (1, 64, 300, 5, 64),           # one token, V below one vocabulary tile
    (129, 136, 520, 7, 128),       # one row past a tile, odd d
    (300, 256, 4096, 1, 128),      # K = 1 (cross-entropy)
    (64, 128, 512, 512, 64),       # K = V (full distribution)
    (200, 96, 2056, 100, 77),      # odd chunk
    # chunks of >= 256 rows run on two-CTA clusters (256-row tiles):
    (600, 200, 4000, 16, 256),     # ragged T, d tail in every GEMM, V % 256 != 0
    (513, 64, 300, 9, 513),        # 3 pair tiles, one ragged row; the peer's half of the
                                   # second vocabulary tile lies wholly past V
    (1100, 136, 1030, 32, 1024),   # two chunks of a pair-tiled size, dW grouped over both
    # degenerate and extreme sizes:
    (40, 64, 4096, 1024, 32),      # K at its maximum
    (700, 8, 2000, 10, 512),       # d at its minimum (one 16-byte row), pair tiles
    (50, 64, 1, 1, 16),            # a one-word vocabulary: softmax is 1, G = M - p
    (9, 32, 300, 3, 1),            # one row per chunk
])
def test_edge_shapes(cuda_device, T, d, V, K, chunk):
    H, W = make_hw(T, d, V, "uniform", seed=T + V, device=cuda_device)
    idx, p = make_cache(T, V, K, "uniform", seed=K)
    ref = kd_oracle(H.cpu(), W.cpu(), idx, p)
    got = run_fused(H, W, idx, p, chunk)
    assert_close_full(got, ref)


def test_duplicates_pads_and_zero_mass(cuda_device):
    T, d, V, K = 300, 128, 1000, 12
    H, W = make_hw(T, d, V, "uniform", seed=3, device=cuda_device)
    idx, p = make_cache(T, V, K, "uniform", seed=4)
    idx[0, 1] = idx[0, 0]
    idx[1, :] = idx[1, 0]               # one id repeated K times
    p[2, 3:] = 0.0                      # zero-probability pads
    p[3, :] = 0.0                       # no teacher mass
    idx[4, :] = np.arange(V - K, V)     # ids at the vocabulary tail
    idx[5, :] = np.arange(K)            # ids at the head
    ref = kd_oracle(H.cpu(), W.cpu(), idx, p)
    got = run_fused(H, W, idx, p, 128)
    assert_close_full(got, ref)
    assert got["loss_rows"][3] == 0.0
    assert np.all(got["dH"][3] == 0.0)


def test_bad_ids_zero_their_rows(cuda_device):
    T, d, V, K = 200, 64, 700, 6
    H, W = make_hw(T, d, V, "uniform", seed=5, device=cuda_device)
    idx, p = make_cache(T, V, K, "uniform", seed=6)
    idx[10, 2] = V + 5
    idx[150, 0] = -3
    ref = kd_oracle(H.cpu(), W.cpu(), idx, p)   # oracle reading: such rows contribute nothing
    idx_d, p_d = to_dev(idx, p, cuda_device)
    res = api.fused_step(H, W, idx_d, p_d, 64, loss_rows=True, check=False)
    got = fused_to_host(res)
    assert_close_full(got, ref)
    assert got["loss_rows"][10] == 0.0 and np.all(got["dH"][150] == 0.0)


def test_accumulate_and_dloss(tiny):
    inp, ref = tiny
    H, W = inp["H"], inp["W"]
    idx, p = to_dev(inp["idx"], inp["p"], H.device)
    g = torch.Generator(device=H.device).manual_seed(9)
    dW0 = torch.randn(W.shape, generator=g, device=H.device)
    dW = dW0.clone()
    res = api.fused_step(H, W, idx, p, 64, dloss=-0.5, dW=dW, accumulate_dW=True)
    torch.cuda.synchronize()
    got_dW = (dW - dW0).double().cpu().numpy()
    assert grad_err(got_dW, -0.5 * ref["dW"]) <= GRAD_FRAC
    assert grad_err(res["dH"].double().cpu().numpy(), -0.5 * ref["dH"]) <= GRAD_FRAC
    # the loss itself does not depend on dloss
    assert abs(res["loss"].item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])


@pytest.mark.parametrize("mode", ["separate", "fused", "fused_norecompute"])
def test_autograd_wrapper(tiny, mode):
    inp, ref = tiny
    H = inp["H"].clone().requires_grad_(True)
    W = inp["W"].clone().requires_grad_(True)
    idx, p = to_dev(inp["idx"], inp["p"], H.device)
    loss = api.TopKKLLoss.apply(H, W, idx, p, 64, mode)
    (2.0 * loss).backward()
    assert abs(loss.item() - ref["loss"]) <= 1e-3 * abs(ref["loss"])
    assert grad_err(H.grad.double().cpu().numpy(), 2.0 * ref["dH"]) <= GRAD_FRAC
    assert grad_err(W.grad.double().cpu().numpy(), 2.0 * ref["dW"]) <= GRAD_FRAC


def test_gradient_rows_sum_to_zero_on_gpu(tiny):
    """sum_j G_tj = 0, so the vocabulary sum of dW vanishes up to the bf16
    rounding of G (|sum| <= T * 2 * 2^-9 * max|H| per column)."""
    inp, _ = tiny
    got = run_fused(inp["H"], inp["W"], inp["idx"], inp["p"], 64)
    col = np.abs(got["dW"].sum(axis=0)).max()
    bound = inp["H"].shape[0] * 2 * 2.0 ** -9 * inp["H"].float().abs().max().item()
    assert col <= bound


@pytest.mark.parametrize("n", [1, 7, 4096, 1000003])
def test_grad_to_bf16_rounds_like_torch(cuda_device, n):
    """kd_grad_to_bf16: bf16(scale * x), round to nearest even, any length."""
    g = torch.Generator(device=cuda_device).manual_seed(n)
    x = torch.randn(n, generator=g, device=cuda_device) * 3.0
    got = api.grad_to_bf16(x, -0.37)
    ref = (x * -0.37).to(torch.bfloat16)   # fp32 product rounded once to bf16, the same two steps
    torch.cuda.synchronize()
    assert torch.equal(got.view(torch.int16), ref.view(torch.int16))
