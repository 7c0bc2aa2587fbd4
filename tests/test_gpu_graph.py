"""The fused steps can be captured in a CUDA graph and replayed: with the
workspace and outputs allocated up front, a captured step replayed on new
inputs (copied into the captured input buffers) gives, bit for bit, what the
eager call gives on those inputs."""
import pytest
import torch

from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.inputs import make_cache, make_hw
from parity_util import to_dev

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("fn_name,chunk", [("fused_step", 256), ("fused_step", 100),
                                           ("fused_step_norecompute", 256)])
def test_captured_step_replays_like_eager(cuda_device, fn_name, chunk):
    fn = getattr(api, fn_name)
    dev = cuda_device
    T, d, V, K = 700, 128, 3000, 12
    H1, W = make_hw(T, d, V, "uniform", seed=1, device=dev)
    H2, _ = make_hw(T, d, V, "uniform", seed=2, device=dev)
    idx1, p1 = to_dev(*make_cache(T, V, K, "uniform", seed=3), dev)
    idx2, p2 = to_dev(*make_cache(T, V, K, "uniform", seed=4), dev)
    work = api.Workspace(dev)
    work.get(api.workspace_size(T, d, V, K, chunk, "fused"))
    out = {"loss": torch.empty(1, device=dev), "lse": torch.empty(T, device=dev),
           "dH": torch.empty(T, d, device=dev), "dW": torch.empty(V, d, device=dev)}
    Hs, idxs, ps = H1.clone(), idx1.clone(), p1.clone()  # the captured input buffers

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):  # warm-up outside the graph (library load, attributes)
        fn(Hs, W, idxs, ps, chunk, workspace=work, out=out, check=False)
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize(dev)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn(Hs, W, idxs, ps, chunk, workspace=work, out=out, check=False)

    for H, idx, p in ((H1, idx1, p1), (H2, idx2, p2)):
        Hs.copy_(H)
        idxs.copy_(idx)
        ps.copy_(p)
        g.replay()
        torch.cuda.synchronize(dev)
        got = {k: v.clone() for k, v in out.items()}
        ref = fn(H, W, idx, p, chunk)
        torch.cuda.synchronize(dev)
        for k in ("loss", "lse", "dH", "dW"):
            assert torch.equal(got[k], ref[k]), k
