"""The token-parallel step on one GPU.

Two ranks each running the fused step on half of a sequence, followed by the
sum of their dW, are emulated by two calls on the two halves with the second
accumulating into the first one's dW.  With the split on a boundary of the
dW chunk groups, each row and each dW group sees exactly the arithmetic of
the one-call step, in the same order, so lse, dH and dW agree bit for bit and
the two losses add up to the one-call loss.  A split inside a chunk changes
the chunking (and the dW grouping) of the second half, so there the results
agree within fp32 accumulation error.  Without a process group the data-
parallel entry point is the plain fused step."""
import pytest
import torch

from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.dp import fused_step_data_parallel, shard_rows
from lm_head_top_tma_b300.inputs import make_inputs
from parity_util import to_dev

pytestmark = pytest.mark.gpu


def _halves(T, split, recompute):
    inp = make_inputs("longctx", device=torch.device("cuda:0"), T=T)
    H, W = inp["H"], inp["W"]
    idx, p = to_dev(inp["idx"], inp["p"], H.device)
    step = api.fused_step if recompute else api.fused_step_norecompute
    one = step(H, W, idx, p, 2048)
    a = step(H[:split], W, idx[:split], p[:split], 2048)
    b = step(H[split:], W, idx[split:], p[split:], 2048, dW=a["dW"], accumulate_dW=True)
    torch.cuda.synchronize()
    return one, a, b


@pytest.mark.parametrize("recompute", [True, False])
def test_two_halves_on_a_group_boundary_are_bit_identical(cuda_device, recompute):
    T = 16384
    t0, t1 = shard_rows(T, 2, 0)
    one, a, b = _halves(T, t1, recompute)
    assert torch.equal(torch.cat([a["lse"], b["lse"]]), one["lse"])
    assert torch.equal(torch.cat([a["dH"], b["dH"]]), one["dH"])
    assert torch.equal(b["dW"], one["dW"])
    total = a["loss"].double().item() + b["loss"].double().item()
    assert abs(total - one["loss"].double().item()) <= 2e-7 * abs(one["loss"].item())


def test_two_halves_split_inside_a_chunk(cuda_device):
    T = 5000
    one, a, b = _halves(T, 2501, True)
    assert (torch.cat([a["lse"], b["lse"]]) - one["lse"]).abs().max().item() <= 1e-5
    dH = torch.cat([a["dH"], b["dH"]])
    assert (dH - one["dH"]).abs().max().item() <= 1e-4 * one["dH"].abs().max().item()
    assert (b["dW"] - one["dW"]).abs().max().item() <= 1e-4 * one["dW"].abs().max().item()
    total = a["loss"].double().item() + b["loss"].double().item()
    assert abs(total - one["loss"].double().item()) <= 1e-6 * abs(one["loss"].item())


def test_data_parallel_entry_without_a_group_is_the_fused_step(cuda_device):
    inp = make_inputs("tiny", device=cuda_device)
    idx, p = to_dev(inp["idx"], inp["p"], cuda_device)
    ref = api.fused_step(inp["H"], inp["W"], idx, p, 64)
    got = fused_step_data_parallel(inp["H"], inp["W"], idx, p, 64)
    torch.cuda.synchronize()
    for k in ("loss", "lse", "dH", "dW"):
        assert torch.equal(got[k], ref[k]), k
    assert got["loss_f64"] == pytest.approx(ref["loss"].item(), rel=1e-7)
