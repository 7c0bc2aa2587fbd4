"""Peak device memory of the fused step is linear in T, with a flat workspace.

The benchmark's peak-bytes-versus-T series (bench.peak_bytes_vs_T) is run on a
small head at three sequence lengths.  The library's workspace must be the same
at every T (its chunk working set is reused chunk after chunk; with 512-row
chunks and at least four chunks the dW grouping no longer changes either), and
the device peak during the step must grow by exactly the per-token bytes of the
caller's own inputs and outputs: H (2d) + dH (4d) + idx and p (8K) + lse (4).
This is the property the method is built for (aimodeling.com, "Second cut":
peak memory that grows only with the sequence, not with T x V logits)."""
import pytest
import torch

import bench
from lm_head_top_tma_b300.inputs import Workload, make_cache

pytestmark = pytest.mark.gpu


def test_workspace_flat_and_peak_linear_in_T(cuda_device):
    wl = Workload("peak_probe", 16384, 2048, 32768, 16, 512, 4, "zipf")
    Ts = (4096, 8192, 16384)
    idx, p = make_cache(4096, wl.V, wl.K, wl.kind, wl.seed)
    rows = bench.peak_bytes_vs_T(cuda_device, wl, idx, p, Ts)
    ws = {r["workspace_bytes"] for r in rows}
    assert len(ws) == 1, ws
    per_token = 6 * wl.d + 8 * wl.K + 4                      # 12,420 bytes
    peaks = [r["peak_bytes"] for r in rows]
    # The caching allocator may hand out a reused block up to ~1 MB larger than asked
    # for, so the slope over the whole range is held to 5% and the two halves to 10%;
    # a [T, V] term would add V * 2 = 64 KB per token here, five times the slope.
    whole = (peaks[2] - peaks[0]) / (Ts[2] - Ts[0])
    assert abs(whole - per_token) <= 0.05 * per_token, (peaks, whole, per_token)
    for i in (0, 1):
        half = (peaks[i + 1] - peaks[i]) / (Ts[i + 1] - Ts[i])
        assert abs(half - per_token) <= 0.10 * per_token, (peaks, half, per_token)
    # the constant part holds at least W and dW and the workspace
    const = peaks[0] - Ts[0] * per_token
    assert const >= wl.V * wl.d * 6 + next(iter(ws)) - (4 << 20)
    assert all(r["ms_per_step"] > 0 for r in rows)
