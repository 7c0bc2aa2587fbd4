"""Calls on different streams with their own workspaces run concurrently and
give the same results as the calls made one at a time, bit for bit: apart
from the optional profiler the library keeps no mutable global state, and the
chunk loop's reductions have a fixed order."""
import pytest
import torch

from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.inputs import make_inputs
from parity_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("chunk", [128, 256])
def test_two_streams_match_one_at_a_time(cuda_device, chunk):
    cases = []
    for seed in (11, 12, 13):
        inp = make_inputs("tiny", device=cuda_device, seed=seed)
        idx, p = to_dev(inp["idx"], inp["p"], cuda_device)
        cases.append((inp["H"], inp["W"], idx, p))
    fns = (api.fused_step, api.fused_step_norecompute, api.fused_step)

    alone = []
    for (H, W, idx, p), fn in zip(cases, fns):
        r = fn(H, W, idx, p, chunk)
        alone.append({k: v.clone() for k, v in r.items()})
    torch.cuda.synchronize()

    streams = [torch.cuda.Stream(device=cuda_device) for _ in cases]
    spaces = [api.Workspace(cuda_device) for _ in cases]
    together = []
    for (H, W, idx, p), fn, st, ws in zip(cases, fns, streams, spaces):
        st.wait_stream(torch.cuda.current_stream(cuda_device))
        with torch.cuda.stream(st):
            together.append(fn(H, W, idx, p, chunk, workspace=ws, check=False))
    torch.cuda.synchronize()
    for ws in spaces:
        assert api.device_status(ws.buf, cuda_device) == 0
    for a, b in zip(alone, together):
        for k in ("loss", "lse", "dH", "dW"):
            assert torch.equal(a[k], b[k]), k
