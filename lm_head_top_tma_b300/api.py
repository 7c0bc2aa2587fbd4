"""Torch-facing binding of the C ABI: argument checks and marshalling only.

Every step of the loss runs in the CUDA kernels of libkdtopk.so; torch only
provides device memory (inputs, outputs, workspace) and the current stream.
Names follow the C entry points: ``forward``, ``backward``, ``fused_step``.
"""
from __future__ import annotations

import ctypes

import torch

from . import _native as N

__all__ = ["workspace_size", "Workspace", "forward", "forward_noalloc", "backward", "fused_step",
           "fused_step_norecompute", "topk_cache_build", "grad_to_bf16",
           "device_status", "gemm_bf16", "debug_wait_timeout", "TopKKLLoss",
           "profile_enable", "profile_read"]


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(0)


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need(t, name, dtype, ndim, device=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if t.dim() != ndim:
        raise ValueError(f"{name} must have {ndim} dims, got {tuple(t.shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")


def _what(kind) -> int:
    return {"forward": N.KD_WS_FORWARD, "backward": N.KD_WS_BACKWARD,
            "fused": N.KD_WS_FUSED}[kind]


def workspace_size(T: int, d: int, V: int, K: int, chunk: int, what: str = "fused") -> int:
    n = N.load().kd_topk_kl_workspace_size(int(T), int(d), int(V), int(K), int(chunk), _what(what))
    if n == 0:
        raise ValueError(f"unsupported sizes T={T} d={d} V={V} K={K} chunk={chunk}")
    return int(n)


class Workspace:
    """Device scratch for the chunk loop, grown on demand and reused."""

    def __init__(self, device=None):
        self.device = torch.device(device or "cuda")
        self.buf = None

    def get(self, nbytes: int) -> torch.Tensor:
        if self.buf is None or self.buf.numel() < nbytes:
            self.buf = torch.empty(int(nbytes), dtype=torch.uint8, device=self.device)
        return self.buf

    @property
    def nbytes(self) -> int:
        return 0 if self.buf is None else self.buf.numel()


def _inputs(H, W, idx, p):
    _need(H, "H", torch.bfloat16, 2)
    dev = H.device
    _need(W, "W", torch.bfloat16, 2, dev)
    _need(idx, "idx", torch.int32, 2, dev)
    _need(p, "p", torch.float32, 2, dev)
    T, d = H.shape
    V, d2 = W.shape
    if d2 != d:
        raise ValueError("H and W disagree on d")
    if idx.shape != p.shape or idx.shape[0] != T:
        raise ValueError("idx and p must both be [T, K]")
    return dev, T, d, V, idx.shape[1]


def device_status(ws: torch.Tensor, device=None) -> int:
    return N.load().kd_topk_kl_device_status(_ptr(ws), _stream(device or ws.device))


def _finish(ws, dev, where, check):
    if check:
        N.check(device_status(ws, dev), where)


def forward(H, W, idx, p, chunk: int, *, loss_rows: bool = False, workspace: Workspace | None = None,
            check: bool = True):
    """Loss (1-element fp32 tensor), lse [T] and optionally per-row losses [T]."""
    dev, T, d, V, K = _inputs(H, W, idx, p)
    ws_n = workspace_size(T, d, V, K, chunk, "forward")
    ws = (workspace or Workspace(dev)).get(ws_n)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    lrows = torch.empty(T, dtype=torch.float32, device=dev) if loss_rows else None
    rc = N.load().kd_topk_kl_forward(_ptr(H), _ptr(W), _ptr(idx), _ptr(p), T, d, V, K, int(chunk),
                                     _ptr(loss), _ptr(lse), _ptr(lrows), _ptr(ws), ws.numel(), _stream(dev))
    N.check(rc, "kd_topk_kl_forward")
    _finish(ws, dev, "kd_topk_kl_forward", check)
    return (loss, lse, lrows) if loss_rows else (loss, lse)


def forward_noalloc(H, W, idx, p, chunk: int, *, loss_rows: bool = False):
    """``forward`` on the library's own 32 MiB per-GPU scratch array instead of
    a workspace, for callers that cannot allocate device memory.  Waits for
    the stream and raises on a device-side error (bad ids)."""
    dev, T, d, V, K = _inputs(H, W, idx, p)
    loss = torch.empty(1, dtype=torch.float32, device=dev)
    lse = torch.empty(T, dtype=torch.float32, device=dev)
    lrows = torch.empty(T, dtype=torch.float32, device=dev) if loss_rows else None
    rc = N.load().kd_topk_kl_forward_noalloc(_ptr(H), _ptr(W), _ptr(idx), _ptr(p), T, d, V, K, int(chunk),
                                             _ptr(loss), _ptr(lse), _ptr(lrows), _stream(dev))
    N.check(rc, "kd_topk_kl_forward_noalloc")
    return (loss, lse, lrows) if loss_rows else (loss, lse)


def backward(H, W, idx, p, lse, chunk: int, *, dloss: float = 1.0, dW: torch.Tensor | None = None,
             accumulate_dW: bool = False, workspace: Workspace | None = None, check: bool = True):
    """dH [T,d] fp32 and dW [V,d] fp32 (``dW`` is overwritten, or added to)."""
    dev, T, d, V, K = _inputs(H, W, idx, p)
    _need(lse, "lse", torch.float32, 1, dev)
    ws_n = workspace_size(T, d, V, K, chunk, "backward")
    ws = (workspace or Workspace(dev)).get(ws_n)
    dH = torch.empty(T, d, dtype=torch.float32, device=dev)
    if dW is None:
        if accumulate_dW:
            raise ValueError("accumulate_dW needs a dW tensor")
        dW = torch.empty(V, d, dtype=torch.float32, device=dev)
    _need(dW, "dW", torch.float32, 2, dev)
    rc = N.load().kd_topk_kl_backward(_ptr(H), _ptr(W), _ptr(idx), _ptr(p), _ptr(lse), T, d, V, K, int(chunk),
                                      float(dloss), _ptr(dH), _ptr(dW), int(bool(accumulate_dW)),
                                      _ptr(ws), ws.numel(), _stream(dev))
    N.check(rc, "kd_topk_kl_backward")
    _finish(ws, dev, "kd_topk_kl_backward", check)
    return dH, dW


def fused_step(H, W, idx, p, chunk: int, *, dloss: float = 1.0, dW: torch.Tensor | None = None,
               accumulate_dW: bool = False, loss_rows: bool = False, workspace: Workspace | None = None,
               check: bool = True, out: dict | None = None):
    """Forward + backward in one chunk loop.  Returns a dict with loss, lse,
    dH, dW (and loss_rows).  ``out`` may supply preallocated outputs."""
    return _fused(N.load().kd_topk_kl_fused_step, "kd_topk_kl_fused_step", H, W, idx, p, chunk, dloss, dW,
                  accumulate_dW, loss_rows, workspace, check, out)


def fused_step_norecompute(H, W, idx, p, chunk: int, *, dloss: float = 1.0, dW: torch.Tensor | None = None,
                           accumulate_dW: bool = False, loss_rows: bool = False,
                           workspace: Workspace | None = None, check: bool = True, out: dict | None = None):
    """``fused_step`` without the backward's second logits GEMM: G is formed
    elementwise from the exponentials the forward GEMM kept (same workspace)."""
    return _fused(N.load().kd_topk_kl_fused_step_norecompute, "kd_topk_kl_fused_step_norecompute", H, W, idx,
                  p, chunk, dloss, dW, accumulate_dW, loss_rows, workspace, check, out)


def _fused(fn, name, H, W, idx, p, chunk, dloss, dW, accumulate_dW, loss_rows, workspace, check, out):
    dev, T, d, V, K = _inputs(H, W, idx, p)
    ws_n = workspace_size(T, d, V, K, chunk, "fused")
    ws = (workspace or Workspace(dev)).get(ws_n)
    o = out if out is not None else {}
    loss = o.get("loss") if o.get("loss") is not None else torch.empty(1, dtype=torch.float32, device=dev)
    lse = o.get("lse") if o.get("lse") is not None else torch.empty(T, dtype=torch.float32, device=dev)
    dH = o.get("dH") if o.get("dH") is not None else torch.empty(T, d, dtype=torch.float32, device=dev)
    if dW is None:
        dW = o.get("dW") if o.get("dW") is not None else torch.empty(V, d, dtype=torch.float32, device=dev)
    lrows = None
    if loss_rows:
        lrows = o.get("loss_rows") if o.get("loss_rows") is not None else torch.empty(T, dtype=torch.float32, device=dev)
    rc = fn(_ptr(H), _ptr(W), _ptr(idx), _ptr(p), T, d, V, K, int(chunk), float(dloss), _ptr(loss), _ptr(lse),
            _ptr(lrows), _ptr(dH), _ptr(dW), int(bool(accumulate_dW)), _ptr(ws), ws.numel(), _stream(dev))
    N.check(rc, name)
    _finish(ws, dev, name, check)
    res = {"loss": loss, "lse": lse, "dH": dH, "dW": dW}
    if loss_rows:
        res["loss_rows"] = lrows
    return res


def topk_cache_build(Z, K: int, *, lse: bool = True, out=None):
    """Teacher cache from logits Z [T,V] (bf16 or fp32, CUDA): ids of the K
    largest logits (largest first, ties by ascending id), their softmax
    probabilities, and lse.  Returns (idx int32 [T,K], p fp32 [T,K], lse fp32 [T] or None).
    ``out`` = (idx, p, lse or None) reuses caller-owned output tensors."""
    if not isinstance(Z, torch.Tensor) or not Z.is_cuda or Z.dim() != 2 or not Z.is_contiguous():
        raise ValueError("Z must be a contiguous 2-D CUDA tensor")
    if Z.dtype not in (torch.bfloat16, torch.float32):
        raise TypeError("Z must be bf16 or fp32")
    T, V = Z.shape
    dev = Z.device
    if out is not None:
        idx, p, l = out
        _need(idx, "idx", torch.int32, 2, dev)
        _need(p, "p", torch.float32, 2, dev)
        if tuple(idx.shape) != (T, K) or tuple(p.shape) != (T, K):
            raise ValueError("out idx and p must be [T, K]")
        if l is not None:
            _need(l, "lse", torch.float32, 1, dev)
            if l.shape[0] != T:
                raise ValueError("out lse must be [T]")
    else:
        idx = torch.empty(T, K, dtype=torch.int32, device=dev)
        p = torch.empty(T, K, dtype=torch.float32, device=dev)
        l = torch.empty(T, dtype=torch.float32, device=dev) if lse else None
    rc = N.load().kd_topk_cache_build(_ptr(Z), int(Z.dtype == torch.bfloat16), T, V, int(K), _ptr(idx), _ptr(p),
                                      _ptr(l), _stream(dev))
    N.check(rc, "kd_topk_cache_build")
    return idx, p, l


def grad_to_bf16(g: torch.Tensor, scale: float = 1.0) -> torch.Tensor:
    """bf16(scale * g) for an fp32 CUDA gradient (kd_grad_to_bf16)."""
    _need(g, "g", torch.float32, g.dim())
    out = torch.empty(g.shape, dtype=torch.bfloat16, device=g.device)
    N.check(N.load().kd_grad_to_bf16(_ptr(g), _ptr(out), g.numel(), float(scale), _stream(g.device)),
            "kd_grad_to_bf16")
    return out


def gemm_bf16(A, B, M, N_, K, *, a_mn=False, b_mn=False, cta_pair=False, out=None, check=True):
    """D = A B^T on the library's tcgen05 GEMM (A [M,K] or [K,M]; B [N,K] or [K,N]);
    ``cta_pair`` selects the two-CTA-cluster form."""
    dev = A.device
    D = out if out is not None else torch.empty(M, N_, dtype=torch.float32, device=dev)
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    rc = N.load().kd_gemm_bf16(_ptr(A), _ptr(B), _ptr(D), M, N_, K, A.stride(0), B.stride(0), D.stride(0),
                               int(a_mn), int(b_mn), int(bool(cta_pair)), _ptr(ws), ws.numel(), _stream(dev))
    N.check(rc, "kd_gemm_bf16")
    _finish(ws, dev, "kd_gemm_bf16", check)
    return D


def debug_wait_timeout(limit_ms: int, device=None, cta_pair: bool = False) -> int:
    dev = torch.device(device or "cuda")
    ws = torch.zeros(256, dtype=torch.uint8, device=dev)
    return N.load().kd_debug_wait_timeout(int(limit_ms), int(bool(cta_pair)), _ptr(ws), ws.numel(), _stream(dev))


def profile_enable(on: bool = True):
    N.check(N.load().kd_profile_enable(int(bool(on))), "kd_profile_enable")


def profile_read(reset: bool = True) -> dict:
    lib = N.load()
    ms = (ctypes.c_double * N.KD_PROF_KINDS)()
    cnt = (ctypes.c_int64 * N.KD_PROF_KINDS)()
    lib.kd_profile_read(ms, cnt, N.KD_PROF_KINDS, int(bool(reset)))
    return {lib.kd_profile_kind_name(k).decode(): (float(ms[k]), int(cnt[k]))
            for k in range(N.KD_PROF_KINDS)}


class TopKKLLoss(torch.autograd.Function):
    """Autograd wrapper of the loss.

    ``mode="separate"`` (default): the forward calls kd_topk_kl_forward and the
    backward calls kd_topk_kl_backward (recomputing each chunk's logits) with
    the incoming gradient as dloss.
    ``mode="fused"`` / ``"fused_norecompute"``: the forward runs the whole fused
    step (kd_topk_kl_fused_step, or kd_topk_kl_fused_step_norecompute) and keeps
    dH, dW for dloss = 1; the loss is a scalar and the gradients are linear in
    dloss, so the backward only scales them.  The kept gradients occupy
    [T,d] + [V,d] fp32 from forward to backward."""

    @staticmethod
    def forward(ctx, H, W, idx, p, chunk, mode="separate"):
        if mode == "separate":
            loss, lse = forward(H, W, idx, p, chunk)
            ctx.save_for_backward(H, W, idx, p, lse)
            ctx.chunk = chunk
            ctx.grads = None
            return loss[0]
        fn = {"fused": fused_step, "fused_norecompute": fused_step_norecompute}.get(mode)
        if fn is None:
            raise ValueError(f"unknown mode {mode!r}")
        res = fn(H, W, idx, p, chunk)
        ctx.grads = (res["dH"], res["dW"])
        return res["loss"][0]

    @staticmethod
    def backward(ctx, g):
        if ctx.grads is not None:
            dH, dW = ctx.grads
            ctx.grads = None
            scale = float(g)
        else:
            H, W, idx, p, lse = ctx.saved_tensors
            dH, dW = backward(H, W, idx, p, lse, ctx.chunk, dloss=float(g))
            scale = 1.0
        # H and W are bf16 (the C ABI's input type): their gradients are too
        return grad_to_bf16(dH, scale), grad_to_bf16(dW, scale), None, None, None, None
