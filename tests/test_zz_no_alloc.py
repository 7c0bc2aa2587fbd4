"""The forward entry point that allocates nothing.

Callers such as a plugin running inside another runtime's memory pool, a
process with a device-memory budget fixed at start-up, or a loop that cannot
take the synchronisation cudaMalloc may bring cannot hand the library a
workspace.  kd_topk_kl_forward_noalloc runs the same forward on a scratch
array the library owns (32 MiB per GPU).  These tests call it through the C
ABI and check it against kd_topk_kl_forward, with the tolerances of the other
parity tests, on two different problems called back to back (the scratch keeps
the previous call's contents) and once more on the first; sizes whose
workspace would not fit are rejected before anything runs.

This file is collected last on purpose: it exercises one optional entry point,
so a run that stops at the first failure has already run everything else.
"""
import pytest
import torch

from lm_head_top_tma_b300 import _native as N
from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.inputs import make_cache, make_hw, make_inputs
from parity_util import LOSS_RTOL, LROW_ATOL, LSE_ATOL, to_dev

pytestmark = pytest.mark.gpu


def _problem(dev, which):
    if which == 0:
        inp = make_inputs("tiny", device=dev)
        return inp["H"], inp["W"], *to_dev(inp["idx"], inp["p"], dev), 64
    H, W = make_hw(300, 128, 2056, "uniform", seed=11, device=dev)
    idx, p = make_cache(300, 2056, 20, "uniform", seed=12)
    return H, W, *to_dev(idx, p, dev), 128


def _check(H, W, idx, p, chunk):
    ref_loss, ref_lse, ref_rows = api.forward(H, W, idx, p, chunk, loss_rows=True)
    loss, lse, rows = api.forward_noalloc(H, W, idx, p, chunk, loss_rows=True)
    torch.cuda.synchronize()
    rl = abs(loss.item() - ref_loss.item()) / abs(ref_loss.item())
    assert rl <= LOSS_RTOL, rl
    assert (lse - ref_lse).abs().max().item() <= LSE_ATOL
    assert (rows - ref_rows).abs().max().item() <= LROW_ATOL


def test_noalloc_forward_matches_forward(cuda_device):
    for which in (0, 1, 0):        # two different problems back to back, then the first again
        _check(*_problem(cuda_device, which))


def test_noalloc_rejects_sizes_beyond_its_scratch(cuda_device):
    T, d, V, K, chunk = 4096, 64, 1_000_000, 1, 4096
    need = api.workspace_size(T, d, V, K, chunk, "forward")
    assert need > N.KD_NOALLOC_SCRATCH_BYTES
    H = torch.zeros(T, d, dtype=torch.bfloat16, device=cuda_device)
    W = torch.zeros(V, d, dtype=torch.bfloat16, device=cuda_device)
    idx = torch.zeros(T, K, dtype=torch.int32, device=cuda_device)
    p = torch.ones(T, K, dtype=torch.float32, device=cuda_device)
    with pytest.raises(N.KDError) as e:
        api.forward_noalloc(H, W, idx, p, chunk)
    assert e.value.code == N.KD_ERR_WORKSPACE
    # the same problem in smaller chunks fits
    loss, _ = api.forward_noalloc(H, W, idx, p, 128)
    torch.cuda.synchronize()
    assert torch.isfinite(loss).all()
