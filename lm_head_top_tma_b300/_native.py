"""ctypes view of libkdtopk.so (the C ABI in include/kdtopk.h).

Loading fails loudly: there is no fallback implementation of anything in
this package.
"""
from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkdtopk.so")

KD_OK = 0
KD_ERR_INVALID_ARG = 1
KD_ERR_UNSUPPORTED = 2
KD_ERR_WORKSPACE = 3
KD_ERR_BAD_INDEX = 4
KD_ERR_TIMEOUT = 5
KD_ERR_CUDA = 6

KD_WS_FORWARD = 1
KD_WS_BACKWARD = 2
KD_WS_FUSED = 3

KD_PROF_KINDS = 10
KD_NOALLOC_SCRATCH_BYTES = 32 << 20

_c_p = ctypes.c_void_p
_i32 = ctypes.c_int
_i64 = ctypes.c_int64
_f32 = ctypes.c_float
_sz = ctypes.c_size_t

# name -> (restype, argtypes); every symbol the header declares
SIGNATURES = {
    "kd_topk_kl_workspace_size": (_sz, [_i64, _i32, _i32, _i32, _i32, _i32]),
    "kd_topk_kl_forward": (_i32, [_c_p, _c_p, _c_p, _c_p, _i64, _i32, _i32, _i32, _i32,
                                  _c_p, _c_p, _c_p, _c_p, _sz, _c_p]),
    "kd_topk_kl_backward": (_i32, [_c_p, _c_p, _c_p, _c_p, _c_p, _i64, _i32, _i32, _i32, _i32,
                                   _f32, _c_p, _c_p, _i32, _c_p, _sz, _c_p]),
    "kd_topk_kl_fused_step": (_i32, [_c_p, _c_p, _c_p, _c_p, _i64, _i32, _i32, _i32, _i32,
                                     _f32, _c_p, _c_p, _c_p, _c_p, _c_p, _i32, _c_p, _sz, _c_p]),
    "kd_topk_kl_fused_step_norecompute": (_i32, [_c_p, _c_p, _c_p, _c_p, _i64, _i32, _i32, _i32, _i32,
                                                 _f32, _c_p, _c_p, _c_p, _c_p, _c_p, _i32, _c_p, _sz, _c_p]),
    "kd_topk_cache_build": (_i32, [_c_p, _i32, _i64, _i32, _i32, _c_p, _c_p, _c_p, _c_p]),
    "kd_grad_to_bf16": (_i32, [_c_p, _c_p, _i64, _f32, _c_p]),
    "kd_topk_kl_device_status": (_i32, [_c_p, _c_p]),
    "kd_topk_kl_forward_noalloc": (_i32, [_c_p, _c_p, _c_p, _c_p, _i64, _i32, _i32, _i32, _i32,
                                          _c_p, _c_p, _c_p, _c_p]),
    "kd_status_string": (ctypes.c_char_p, [_i32]),
    "kd_gemm_bf16": (_i32, [_c_p, _c_p, _c_p, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32, _i32,
                            _c_p, _sz, _c_p]),
    "kd_debug_wait_timeout": (_i32, [_i32, _i32, _c_p, _sz, _c_p]),
    "kd_profile_enable": (_i32, [_i32]),
    "kd_profile_read": (_i32, [ctypes.POINTER(ctypes.c_double), ctypes.POINTER(ctypes.c_int64), _i32, _i32]),
    "kd_profile_kind_name": (ctypes.c_char_p, [_i32]),
}

_lib = None


def load(path: str | None = None):
    """Load (once) and return the library handle with typed entry points."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    p = path or LIB_PATH
    if not os.path.exists(p):
        raise RuntimeError(
            f"libkdtopk.so not found at {p}; build it with "
            "`python -m lm_head_top_tma_b300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(p)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    if path is None:
        _lib = lib
    return lib


class KDError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = int(code)
        msg = load().kd_status_string(self.code).decode()
        super().__init__(f"{where}: {msg} (status {self.code})")


def check(code: int, where: str):
    if code != KD_OK:
        raise KDError(code, where)
