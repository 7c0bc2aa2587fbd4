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
fallback (thousands of equal maxima, all-equal rows), and masked -inf logits.
The builder keeps the maximum of every 32-byte group (16-byte group when the
row is not a multiple of 32 bytes) in shared memory and re-reads only the
groups that can hold a top-K element; the placement cases put the top K at the
row's end, its start, in one run, scattered, and the capacity cases take rows
at and just past the largest V each block shape and load width covers (longer
rows are scanned whole), and candidate lists at and one past each shape's
capacity."""
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
                                   (4, 5000, 512), (4, 5000, 513),  # the narrow shape's 512 slots bound K <= 512
                                   (1, 1, 1), (9, 2047, 33),
                                   (3000, 520, 7),       # many short rows per block
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


GMAX_GROUPS = 32768  # the wide shape's 16-byte group maxima (the narrow shape holds 16384 32-byte ones)


@pytest.mark.parametrize("dtype", ["bf16", "fp32"])
def test_topk_placement(cuda_device, dtype):
    """Top K at the row's end, at its start, in one run of 120 ids, K equal
    maxima scattered, and one half of the row uniformly above the other."""
    tdt = torch.bfloat16 if dtype == "bf16" else torch.float32
    V, K = 128256, 100
    mid = V // 4
    Z = make_teacher_logits(6, V, seed=21, device=cuda_device, dtype=dtype)
    g = torch.Generator(device="cpu").manual_seed(3)
    ramp = torch.linspace(-20.0, 20.0, V)
    Z[0] = ramp.to(tdt).to(cuda_device)                             # ascending: top K at the row's end
    Z[1] = ramp.flip(0).to(tdt).to(cuda_device)                     # descending: top K at its start
    Z[2, mid - 60:mid + 60] = (8.0 + torch.rand(120, generator=g)).to(tdt).to(cuda_device)
    Z[3, torch.randperm(V, generator=g)[:K].to(cuda_device)] = 9.0  # K equal maxima anywhere
    Z[4, mid:] = Z[4, mid:] + 3.0
    Z[5, :mid] = Z[5, :mid] + 3.0
    check(Z, K)


@pytest.mark.parametrize("dtype,V", [("bf16", GMAX_GROUPS * 8), ("bf16", GMAX_GROUPS * 8 + 8),
                                     ("bf16", GMAX_GROUPS * 8 - 3), ("fp32", GMAX_GROUPS * 4),
                                     ("fp32", GMAX_GROUPS * 4 + 4)])
def test_rows_around_group_maxima_capacity(cuda_device, dtype, V):
    """512 KB rows (32-byte loads, the narrow shape's group maxima exactly
    full), rows 16 bytes longer (16-byte loads, one group past the wide shape's
    32768 maxima: scanned whole), and a bf16 row just short of 512 KB whose
    length is not a multiple of 16 bytes (element-wise loads)."""
    Z = make_teacher_logits(6, V, seed=V, device=cuda_device, dtype=dtype)
    check(Z, 100)


# (dtype, V): the block shape and row access each row gets
SHAPE_ROWS = [
    ("bf16", 131072),   # 256 KB, 32-byte multiple: narrow shape, 32-byte loads
    ("bf16", 131064),   # a 16-byte but not 32-byte multiple: narrow shape, 16-byte loads, 16383 groups
    ("bf16", 131080),   # 16 bytes past 256 KB, not a 32-byte multiple: wide shape, 16-byte loads
    ("bf16", 262144),   # 512 KB: narrow shape, 32-byte loads, exactly its 16384 group maxima
    ("bf16", 262160),   # 32 bytes more: wide shape, 32-byte loads
    ("fp32", 131072),   # 512 KB of fp32: narrow shape, 32-byte loads, at capacity
    ("fp32", 131080),   # wide shape, 32-byte loads
    ("bf16", 524288),   # 1 MB: wide shape, 32-byte loads, exactly its 32768 group maxima
    ("bf16", 524304),   # one 32-byte group more: scanned whole
]


@pytest.mark.parametrize("dtype,V", SHAPE_ROWS)
def test_rows_around_the_block_shape_switches(cuda_device, dtype, V):
    """Rows on both sides of every switch between the block shapes (256
    threads, four blocks per SM, for rows of up to 512 KB; 512 threads, two per
    SM, above) and the load widths (32-byte loads when the row is a multiple of
    32 bytes, 16-byte loads otherwise), at and one group past each shape's
    group-maxima capacity."""
    Z = make_teacher_logits(4, V, seed=V + 1, device=cuda_device, dtype=dtype)
    check(Z, 100)


def test_rows_on_a_16_byte_boundary_only(cuda_device):
    """Rows whose start is 16- but not 32-byte aligned take the 16-byte loads:
    512 KB bf16 rows then fill the wide shape's 32768 group maxima exactly."""
    T, V = 4, 262144
    Z0 = make_teacher_logits(T, V, seed=9, device=cuda_device, dtype="bf16")
    buf = torch.empty(T * V + 8, device=cuda_device, dtype=torch.bfloat16)
    Z = buf[8:].view(T, V)                      # 16 bytes past a 32-byte boundary
    Z.copy_(Z0)
    assert Z.data_ptr() % 32 == 16
    check(Z, 100)


@pytest.mark.parametrize("V,n_eq", [(20000, 2048), (20000, 2049), (20008, 2049),
                                    (150000, 4096), (150000, 4097), (300000, 4097)])
def test_candidate_list_capacity(cuda_device, V, n_eq):
    """n_eq equal maxima in one run: every one of them reaches theta, so the
    candidate list holds exactly n_eq entries.  The narrow shape (40 KB rows,
    with 32- and with 16-byte loads) keeps 2048, the wide shape (a 300 KB row
    with 16-byte loads, a 600 KB row with 32-byte loads) 4096; one more takes
    the exact fallback."""
    Z = make_teacher_logits(3, V, seed=n_eq, device=cuda_device, dtype="bf16")
    top = float(Z.float().max()) + 2.0
    Z[0, 777:777 + n_eq] = top
    Z[1, V - n_eq:] = top
    Z[2, 0:n_eq] = top
    idx, _ = check(Z, 100)
    assert idx[0].tolist() == list(range(777, 877))
    assert idx[1].tolist() == list(range(V - n_eq, V - n_eq + 100))
    assert idx[2].tolist() == list(range(100))


@pytest.mark.parametrize("K", [1, 16, 17, 512, 1024])
def test_k_values_full_vocab(cuda_device, K):
    """K from 1 to the largest supported, on rows of the benchmark's vocabulary."""
    Z = make_teacher_logits(12, 128256, seed=K, device=cuda_device, dtype="bf16")
    check(Z, K)


def test_cache_feeds_the_loss(cuda_device):
    """The offline step and the loss together: the cache the GPU builds from
    teacher logits drives the fused step; the reference runs the oracle's cache
    through the loss oracle.  Chunks of 128 rows (pair GEMMs off) and 256
    (on), with a ragged last chunk."""
    from parity_util import assert_close_full, fused_to_host, kd_oracle
    from lm_head_top_tma_b300.inputs import make_hw

    T, d, V, K = 300, 256, 4096, 32
    Z = make_teacher_logits(T, V, seed=31, device=cuda_device, dtype="bf16")
    idx, p, _ = api.topk_cache_build(Z, K)
    ref_cache = topk_cache_oracle(Z.cpu(), K)
    assert np.array_equal(idx.cpu().numpy(), ref_cache["idx"])
    H, W = make_hw(T, d, V, "zipf", seed=5, device=cuda_device)
    ref = kd_oracle(H.cpu(), W.cpu(), ref_cache["idx"], ref_cache["p"])
    for chunk in (128, 256):
        got = fused_to_host(api.fused_step(H, W, idx, p, chunk, loss_rows=True))
        assert_close_full(got, ref)
