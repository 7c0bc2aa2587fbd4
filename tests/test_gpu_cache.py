"""Teacher-cache builder (kd_topk_cache_build) against the fp64 cache oracle.

The selection is integer work decided by exact comparisons of the same bf16 or
fp32 logits on both sides, so the ids must match bit for bit, ties included
(lower id first).  p = exp(z - lse) is computed in fp32 on the GPU: lse is an
fp32 sum of V terms 2^x from the special-function unit (relative error of
order 1e-6 for V ~ 1e5), so p carries a relative error of order 1e-6; the test
allows 1e-4 relative, which still catches a wrong lse (off by one term of the
sum moves p by ~1/V relative only for flat rows, but a missing max-shift,
a wrong base or a wrong id moves it by orders of magnitude).  Cases: teacher-
like bf16 and fp32 rows at the workloads' vocabulary sizes, V below the block
size, K = 1, K = V, K = 1024, heavily tied rows, rows that force the exact
fallback (thousands of equal maxima, all-equal rows), and masked -inf logits."""
import numpy as np
import pytest
import torch

from lm_head_top_tma_b300 import api
from lm_head_top_tma_b300.inputs import make_teacher_logits
from oracle import topk_cache_oracle

pytestmark = pytest.mark.gpu

P_RTOL = 1e-4
LSE_ATOL = 1e-4


def check(Z, K, rows=None):
    idx, p, lse = api.topk_cache_build(Z, K)
    torch.cuda.synchronize()
    sel = np.arange(Z.shape[0]) if rows is None else np.asarray(rows)
    Zs = Z[torch.as_tensor(sel, device=Z.device)].cpu()
    ref = topk_cache_oracle(Zs, K)
    gi = idx.cpu().numpy()[sel]
    assert np.array_equal(gi, ref["idx"]), np.argwhere(gi != ref["idx"])[:5]
    gp = p.double().cpu().numpy()[sel]
    np.testing.assert_allclose(gp, ref["p"], rtol=P_RTOL, atol=1e-30)
    gl = lse.double().cpu().numpy()[sel]
    fin = np.isfinite(ref["lse"])
    assert np.abs(gl[fin] - ref["lse"][fin]).max() <= LSE_ATOL
    return idx, p


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
@pytest.mark.parametrize("V,K", [(4096, 100), (128256, 100), (201088, 100)])
def test_teacher_like_rows(cuda_device, dtype, V, K):
    Z = make_teacher_logits(96, V, seed=V + K, device=cuda_device, dtype=dtype)
    check(Z, K)


@pytest.mark.parametrize("T,V,K", [(5, 300, 5), (3, 64, 64), (7, 1000, 1), (4, 5000, 1024), (2, 1024, 1024),
                                   (1, 1, 1), (9, 2047, 33),
                                   (3000, 520, 7),       # many short rows per block through the copy ring
                                   (700, 16392, 100)])   # rows of two chunks, the second nearly empty
def test_shapes(cuda_device, T, V, K):
    Z = make_teacher_logits(T, V, seed=T * V + K, device=cuda_device, dtype="bf16")
    check(Z, K)


def test_ties_and_fallback(cuda_device):
    T, V, K = 8, 20000, 100
    Z = make_teacher_logits(T, V, seed=11, device=cuda_device, dtype="bf16", noise=0.05)  # heavily tied
    Z[1] = 1.5                                    # all equal: every element reaches theta
    Z[2, 5000:11000] = Z[2].max() + 1.0           # 6000 equal maxima
    Z[3, ::3] = -float("inf")                     # masked logits
    Z[4] = -float("inf")
    Z[4, 123] = 0.0
    Z[4, 7] = 0.0                                 # 2 finite entries, K = 100: the rest are -inf, by id
    idx, p = check(Z, K)
    assert idx[1].tolist() == list(range(K))
    assert idx[2].tolist() == list(range(5000, 5000 + K))


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_signed_zeros_tie(cuda_device, dtype):
    """-0.0 and +0.0 are equal logits: they tie and go by ascending id."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    Z = torch.full((2, 4096), -3.0, device=cuda_device, dtype=tdt)
    Z[0, 10::400] = -0.0
    Z[0, 11::400] = 0.0
    Z[1, 4000:] = 0.0
    Z[1, :50] = -0.0
    idx, _ = check(Z, 40)
    assert idx[0, :4].tolist() == [10, 11, 410, 411]
    assert idx[1, :3].tolist() == [0, 1, 2]


def test_fp32_fallback_and_negative_values(cuda_device):
    Z = torch.full((3, 9000), -2.25, device=cuda_device)
    Z[1, 100:4200] = 3.0          # 4100 equal maxima
    Z[2, 8000:] = -1e-30          # tiny negatives above the rest
    check(Z, 64)


def test_full_size_sampled_rows(cuda_device):
    Z = make_teacher_logits(2048, 128256, seed=5, device=cuda_device, dtype="bf16")
    rng = np.random.default_rng(0)
    check(Z, 100, rows=np.sort(rng.choice(2048, 48, replace=False)))
