"""The C ABI from plain C: tests/c_abi_client.c includes include/kdtopk.h,
allocates its own device buffers with cudaMalloc and calls
kd_topk_kl_fused_step on the legacy default stream, with no Python or torch in
the process.  On CPU the client must compile and link as C99 with every warning
an error (the header is usable from C); on a GPU its results for the tiny
workload must match the fp64 oracle."""
import os
import shutil
import subprocess

import numpy as np
import pytest

from lm_head_top_tma_b300 import _native as N
from lm_head_top_tma_b300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = "/usr/local/cuda"


def _compile(tmp_path):
    build()
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "c_abi_client")
    libdir = os.path.dirname(N.LIB_PATH)
    cmd = [cc, "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror", "-I", os.path.join(ROOT, "include"),
           "-I", os.path.join(CUDA, "include"), os.path.join(ROOT, "tests", "c_abi_client.c"), "-o", exe,
           "-L", libdir, "-lkdtopk", "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{libdir}:{os.path.join(CUDA, 'lib64')}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    return exe


def test_c_client_compiles_against_the_header(tmp_path):
    exe = _compile(tmp_path)
    assert os.path.exists(exe)


@pytest.mark.gpu
def test_c_client_matches_the_oracle(tmp_path, cuda_device):
    import torch

    from lm_head_top_tma_b300.inputs import make_inputs
    from parity_util import assert_close_full, kd_oracle

    exe = _compile(tmp_path)
    inp = make_inputs("tiny", device=cuda_device)
    H, W, idx, p = inp["H"].cpu(), inp["W"].cpu(), inp["idx"], inp["p"]
    T, d = H.shape
    V = W.shape[0]
    K = idx.shape[1]
    chunk = 64
    src = tmp_path / "in.bin"
    with open(src, "wb") as f:
        f.write(np.int64(T).tobytes())
        f.write(np.array([d, V, K, chunk], dtype=np.int32).tobytes())
        f.write(H.view(torch.int16).numpy().tobytes())
        f.write(W.view(torch.int16).numpy().tobytes())
        f.write(np.ascontiguousarray(idx, dtype=np.int32).tobytes())
        f.write(np.ascontiguousarray(p, dtype=np.float32).tobytes())
    dst = tmp_path / "out.bin"
    res = subprocess.run([exe, str(src), str(dst)], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stderr
    out = np.fromfile(dst, dtype=np.float32)
    assert out.size == 1 + T + T * d + V * d
    got = {"loss": float(out[0]), "lse": out[1:1 + T].astype(np.float64),
           "dH": out[1 + T:1 + T + T * d].reshape(T, d).astype(np.float64),
           "dW": out[1 + T + T * d:].reshape(V, d).astype(np.float64)}
    ref = kd_oracle(H, W, idx, p)
    assert_close_full(got, ref, what=("loss", "lse", "dH", "dW"))
