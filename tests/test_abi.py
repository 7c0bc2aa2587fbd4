"""The C-ABI library builds, loads and exports what include/kdtopk.h declares;
host-side argument checks and workspace sizing (no GPU needed)."""
import ctypes
import os
import re
import subprocess

import pytest

from lm_head_top_tma_b300 import _native as N
from lm_head_top_tma_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kdtopk.h")


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[A-Za-z_][\w\s\*]*?\b(kd_\w+)\s*\(", src, flags=re.M)))


@pytest.fixture(scope="module")
def lib():
    build()
    return N.load()


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("kd_topk_kl_forward", "kd_topk_kl_backward", "kd_topk_kl_fused_step",
                 "kd_topk_kl_workspace_size", "kd_status_string"):
        assert must in names


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", N.LIB_PATH], capture_output=True, text=True,
                         check=True).stdout
    exported = {ln.split()[-1] for ln in out.splitlines() if ln.strip()}
    for name in declared_functions():
        assert name in exported, name
        assert name in N.SIGNATURES, f"binding lacks {name}"
        getattr(lib, name)
    # nothing but the declared C ABI is exported
    ours = {n for n in exported if n.startswith("kd_")}
    assert ours == set(declared_functions())


def test_status_strings(lib):
    for code in range(7):
        assert lib.kd_status_string(code)
    assert lib.kd_status_string(N.KD_ERR_BAD_INDEX).decode().startswith("teacher id")


def test_host_argument_checks(lib):
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: checks fail first
    args = (fake, fake, fake, fake)
    # null pointers
    assert lib.kd_topk_kl_forward(null, fake, fake, fake, 64, 64, 128, 4, 64, fake, fake, null, fake,
                                  1 << 30, null) == N.KD_ERR_INVALID_ARG
    # d % 8 != 0 (TMA row stride must be a multiple of 16 bytes)
    assert lib.kd_topk_kl_forward(*args, 64, 60, 128, 4, 64, fake, fake, null, fake, 1 << 30,
                                  null) == N.KD_ERR_UNSUPPORTED
    # K > V, non-positive sizes
    assert lib.kd_topk_kl_forward(*args, 64, 64, 8, 16, 64, fake, fake, null, fake, 1 << 30,
                                  null) == N.KD_ERR_INVALID_ARG
    assert lib.kd_topk_kl_forward(*args, 0, 64, 128, 4, 64, fake, fake, null, fake, 1 << 30,
                                  null) == N.KD_ERR_INVALID_ARG
    assert lib.kd_topk_kl_backward(*args, null, 64, 64, 128, 4, 64, 1.0, fake, fake, 0, fake, 1 << 30,
                                   null) == N.KD_ERR_INVALID_ARG
    # K above the sort width
    assert lib.kd_topk_kl_forward(*args, 64, 64, 4096, 2000, 64, fake, fake, null, fake, 1 << 30,
                                  null) == N.KD_ERR_UNSUPPORTED
    # workspace too small
    need = lib.kd_topk_kl_workspace_size(64, 64, 128, 4, 64, N.KD_WS_FUSED)
    assert lib.kd_topk_kl_fused_step(*args, 64, 64, 128, 4, 64, 1.0, fake, fake, null, fake, fake, 0,
                                     fake, need - 1, null) == N.KD_ERR_WORKSPACE
    # misaligned H
    assert lib.kd_topk_kl_forward(ctypes.c_void_p((1 << 20) + 2), fake, fake, fake, 64, 64, 128, 4, 64,
                                  fake, fake, null, fake, 1 << 30, null) == N.KD_ERR_UNSUPPORTED


def test_cache_builder_argument_checks(lib):
    """kd_topk_cache_build rejects bad arguments before it touches the device:
    null pointers and sizes outside 1 <= K <= V (invalid), K above 1024 and
    logits or outputs not aligned to their element type (unsupported)."""
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)   # never dereferenced: checks fail first
    build_cache = lib.kd_topk_cache_build
    assert build_cache(null, 1, 8, 4096, 100, fake, fake, null, null) == N.KD_ERR_INVALID_ARG
    assert build_cache(fake, 1, 8, 4096, 100, null, fake, null, null) == N.KD_ERR_INVALID_ARG
    assert build_cache(fake, 1, 8, 4096, 100, fake, null, null, null) == N.KD_ERR_INVALID_ARG
    assert build_cache(fake, 1, 0, 4096, 100, fake, fake, null, null) == N.KD_ERR_INVALID_ARG
    assert build_cache(fake, 1, 8, 64, 65, fake, fake, null, null) == N.KD_ERR_INVALID_ARG
    assert build_cache(fake, 1, 8, 4096, 0, fake, fake, null, null) == N.KD_ERR_INVALID_ARG
    assert build_cache(fake, 1, 8, 4096, 1025, fake, fake, null, null) == N.KD_ERR_UNSUPPORTED
    odd = ctypes.c_void_p((1 << 20) + 1)
    two = ctypes.c_void_p((1 << 20) + 2)
    assert build_cache(odd, 1, 8, 4096, 100, fake, fake, null, null) == N.KD_ERR_UNSUPPORTED   # bf16
    assert build_cache(two, 0, 8, 4096, 100, fake, fake, null, null) == N.KD_ERR_UNSUPPORTED   # fp32
    assert build_cache(fake, 1, 8, 4096, 100, two, fake, null, null) == N.KD_ERR_UNSUPPORTED
    assert build_cache(fake, 1, 8, 4096, 100, fake, fake, two, null) == N.KD_ERR_UNSUPPORTED


def test_workspace_is_flat_in_T(lib):
    f = lambda T, what=N.KD_WS_FUSED: lib.kd_topk_kl_workspace_size(T, 3072, 128256, 100, 2048, what)
    # flat once T covers one dW group (two 2048-row chunks here); a single chunk needs less
    sizes = [f(T) for T in (4096, 32768, 262144)]
    assert len(set(sizes)) == 1 and sizes[0] > 0
    assert f(2048) <= f(4096)
    # chunk working set: [chunk, V] bf16 gradient operand dominates the backward
    assert f(32768) >= 2048 * 128256 * 2
    assert f(32768, N.KD_WS_FORWARD) < f(32768, N.KD_WS_BACKWARD)
    assert f(32768) < 2 * (1 << 30)
    # a chunk larger than T is clipped to T
    assert lib.kd_topk_kl_workspace_size(100, 256, 4096, 16, 4096, 3) == \
        lib.kd_topk_kl_workspace_size(100, 256, 4096, 16, 100, 3)
    assert lib.kd_topk_kl_workspace_size(0, 256, 4096, 16, 64, 3) == 0
    assert lib.kd_topk_kl_workspace_size(256, 250, 4096, 16, 64, 3) == 0


def test_missing_library_fails_loudly(tmp_path):
    """No fallback: a library that is not there is an error, not a slower path."""
    with pytest.raises(RuntimeError, match="not found"):
        N.load(str(tmp_path / "libkdtopk.so"))


def test_grad_to_bf16_argument_checks(lib):
    """kd_grad_to_bf16: null pointers and negative lengths are invalid, an empty
    range is a no-op, and a source off a 16-byte boundary or a destination off
    an 8-byte boundary is unsupported, all before any device work."""
    null = ctypes.c_void_p(0)
    fake = ctypes.c_void_p(1 << 20)
    assert lib.kd_grad_to_bf16(null, fake, 16, 1.0, null) == N.KD_ERR_INVALID_ARG
    assert lib.kd_grad_to_bf16(fake, null, 16, 1.0, null) == N.KD_ERR_INVALID_ARG
    assert lib.kd_grad_to_bf16(fake, fake, -1, 1.0, null) == N.KD_ERR_INVALID_ARG
    assert lib.kd_grad_to_bf16(fake, fake, 0, 1.0, null) == N.KD_OK
    assert lib.kd_grad_to_bf16(ctypes.c_void_p((1 << 20) + 4), fake, 16, 1.0, null) == N.KD_ERR_UNSUPPORTED
    assert lib.kd_grad_to_bf16(fake, ctypes.c_void_p((1 << 20) + 4), 16, 1.0, null) == N.KD_ERR_UNSUPPORTED
