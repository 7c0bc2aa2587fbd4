"""Out-of-bounds writes: the workspace and every output get a guard band of
sentinel values right behind the bytes the call may write (the workspace is
passed with exactly kd_topk_kl_workspace_size bytes; outputs are the leading
rows of larger tensors).  After forward, backward, the fused step and the
no-recompute fused step on ragged shapes in both GEMM forms, every guard must
be untouched and the status must be KD_OK."""
import ctypes

import numpy as np
import pytest
import torch

from lm_head_top_tma_b300 import _native as N
from lm_head_top_tma_b300.inputs import make_cache, make_hw
from parity_util import to_dev

pytestmark = pytest.mark.gpu

GUARD = 65536      # bytes of workspace guard
PAD = 3            # guard rows behind each output


def ptr(t):
    return ctypes.c_void_p(t.data_ptr())


@pytest.mark.parametrize("T,d,V,K,chunk", [(600, 200, 4000, 16, 256), (333, 136, 1030, 7, 100),
                                           (2300, 64, 2056, 100, 1024)])
@pytest.mark.parametrize("call", ["forward", "backward", "fused", "fused_norecompute"])
def test_guards_untouched(cuda_device, T, d, V, K, chunk, call):
    lib = N.load()
    dev = cuda_device
    H, W = make_hw(T, d, V, "uniform", seed=T + d, device=dev)
    idx, p = to_dev(*make_cache(T, V, K, "uniform", seed=K), dev)
    what = {"forward": N.KD_WS_FORWARD, "backward": N.KD_WS_BACKWARD}.get(call, N.KD_WS_FUSED)
    ws_n = lib.kd_topk_kl_workspace_size(T, d, V, K, chunk, what)
    assert ws_n > 0
    ws_n_alloc = (ws_n + 255) // 256 * 256 + GUARD
    ws = torch.full((ws_n_alloc,), 0xA5, dtype=torch.uint8, device=dev)
    sentinel = float("nan")
    loss = torch.full((1 + PAD,), sentinel, device=dev)
    lse = torch.full((T + PAD,), sentinel, device=dev)
    lrows = torch.full((T + PAD,), sentinel, device=dev)
    dH = torch.full((T + PAD, d), sentinel, device=dev)
    dW = torch.full((V + PAD, d), sentinel, device=dev)
    stream = ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream)
    if call == "backward":  # a real lse for the backward to read
        lse_in = torch.empty(T, device=dev)
        ws_f = torch.empty(lib.kd_topk_kl_workspace_size(T, d, V, K, chunk, N.KD_WS_FORWARD), dtype=torch.uint8,
                           device=dev)
        N.check(lib.kd_topk_kl_forward(ptr(H), ptr(W), ptr(idx), ptr(p), T, d, V, K, chunk, ptr(loss), ptr(lse_in),
                                       ctypes.c_void_p(0), ptr(ws_f), ws_f.numel(), stream), "forward")
        rc = lib.kd_topk_kl_backward(ptr(H), ptr(W), ptr(idx), ptr(p), ptr(lse_in), T, d, V, K, chunk, 1.0, ptr(dH),
                                     ptr(dW), 0, ptr(ws), ws_n, stream)
    elif call == "forward":
        rc = lib.kd_topk_kl_forward(ptr(H), ptr(W), ptr(idx), ptr(p), T, d, V, K, chunk, ptr(loss), ptr(lse),
                                    ptr(lrows), ptr(ws), ws_n, stream)
    else:
        fn = lib.kd_topk_kl_fused_step if call == "fused" else lib.kd_topk_kl_fused_step_norecompute
        rc = fn(ptr(H), ptr(W), ptr(idx), ptr(p), T, d, V, K, chunk, 1.0, ptr(loss), ptr(lse), ptr(lrows), ptr(dH),
                ptr(dW), 0, ptr(ws), ws_n, stream)
    N.check(rc, call)
    N.check(lib.kd_topk_kl_device_status(ptr(ws), stream), call)
    torch.cuda.synchronize()
    tail = ws[ws_n:].cpu().numpy()
    assert np.all(tail == 0xA5), f"workspace guard overwritten at byte {ws_n + int(np.argmax(tail != 0xA5))}"
    writes_fwd = call in ("forward", "fused", "fused_norecompute")
    writes_bwd = call in ("backward", "fused", "fused_norecompute")
    if writes_fwd:
        assert torch.isnan(loss[1:]).all() and not torch.isnan(loss[0])
        assert torch.isnan(lse[T:]).all() and not torch.isnan(lse[:T]).any()
        assert torch.isnan(lrows[T:]).all() and not torch.isnan(lrows[:T]).any()
    if writes_bwd:
        assert torch.isnan(dH[T:]).all() and not torch.isnan(dH[:T]).any()
        assert torch.isnan(dW[V:]).all() and not torch.isnan(dW[:V]).any()
    else:
        assert torch.isnan(dH).all() and torch.isnan(dW).all()
