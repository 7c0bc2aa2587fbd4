"""Pins of the fp64 CPU oracle against things other than itself.

The pages print no worked values for the loss, so every pin comes from the
mathematics (see the oracle's module docstring for what is computed):

* hand-derived worked examples (tests/golden/handworked.json);
* central finite differences of L with respect to H and W;
* special cases that reduce to library routines: K = 1, p = 1 is
  torch's cross-entropy (sum reduction); distinct ids with any p is torch's
  KL divergence against a dense target that is zero off the top-K ids; both
  with gradients from torch autograd;
* closed forms (W = 0) and invariants (rows of G sum to zero, self-
  distillation gives zero, logit shift, scaling in p, permutations);
* brute force: the pure-Python loops against the blocked NumPy form.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

from oracle import kd_oracle, kd_oracle_dW_rows, kd_oracle_naive, kd_oracle_rows
from lm_head_top_tma_b300.inputs import make_cache, make_hw, make_inputs

pytestmark = pytest.mark.filterwarnings("ignore::RuntimeWarning")
GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "handworked.json")


def _rand_case(T, d, V, K, seed, distinct=True, scale_w=0.5):
    rng = np.random.default_rng(seed)
    H = rng.normal(size=(T, d))
    W = rng.normal(size=(V, d)) * scale_w
    if distinct:
        idx = np.stack([rng.permutation(V)[:K] for _ in range(T)])
    else:
        idx = rng.integers(0, V, size=(T, K))
    p = rng.random(size=(T, K))
    p = p / p.sum(axis=1, keepdims=True) * rng.uniform(0.5, 1.0, size=(T, 1))
    return H, W, idx.astype(np.int32), p


def _loss_only(H, W, idx, p):
    return kd_oracle(H, W, idx, p, want_grads=False)["loss"]


# ---------------------------------------------------------------- golden
def test_handworked_golden():
    cases = json.load(open(GOLDEN))["cases"]
    assert len(cases) >= 4
    for c in cases:
        H, W = np.array(c["H"]), np.array(c["W"])
        idx, p = np.array(c["idx"]), np.array(c["p"])
        for fn in (kd_oracle, kd_oracle_naive):
            out = fn(H, W, idx, p)
            assert out["loss"] == pytest.approx(c["loss"], abs=1e-14), (c["name"], fn.__name__)
            np.testing.assert_allclose(out["lse"], c["lse"], atol=1e-14)
            np.testing.assert_allclose(out["dH"], c["dH"], atol=1e-14)
            np.testing.assert_allclose(out["dW"], c["dW"], atol=1e-14)


# ---------------------------------------------------------------- P1
@pytest.mark.parametrize("distinct", [True, False])
def test_finite_differences(distinct):
    H, W, idx, p = _rand_case(3, 8, 12, 4, seed=11 if distinct else 12, distinct=distinct)
    out = kd_oracle(H, W, idx, p)
    h = 1e-6
    num_dH = np.zeros_like(H)
    for i in np.ndindex(H.shape):
        Hp, Hm = H.copy(), H.copy()
        Hp[i] += h
        Hm[i] -= h
        num_dH[i] = (_loss_only(Hp, W, idx, p) - _loss_only(Hm, W, idx, p)) / (2 * h)
    num_dW = np.zeros_like(W)
    for i in np.ndindex(W.shape):
        Wp, Wm = W.copy(), W.copy()
        Wp[i] += h
        Wm[i] -= h
        num_dW[i] = (_loss_only(H, Wp, idx, p) - _loss_only(H, Wm, idx, p)) / (2 * h)
    scale_h = np.abs(num_dH).max()
    scale_w = np.abs(num_dW).max()
    assert np.abs(out["dH"] - num_dH).max() <= 1e-7 * max(scale_h, 1.0)
    assert np.abs(out["dW"] - num_dW).max() <= 1e-7 * max(scale_w, 1.0)


# ---------------------------------------------------------------- P4
def test_cross_entropy_special_case():
    rng = np.random.default_rng(3)
    T, d, V = 7, 5, 9
    H, W = rng.normal(size=(T, d)), rng.normal(size=(V, d))
    tgt = rng.integers(0, V, size=T)
    out = kd_oracle(H, W, tgt[:, None], np.ones((T, 1)))
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    ce = torch.nn.functional.cross_entropy(Ht @ Wt.T, torch.tensor(tgt), reduction="sum")
    ce.backward()
    assert out["loss"] == pytest.approx(ce.item(), rel=1e-13)
    np.testing.assert_allclose(out["dH"], Ht.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(out["dW"], Wt.grad.numpy(), atol=1e-12)
    lse_ref = torch.logsumexp(torch.tensor(H @ W.T), dim=1).numpy()
    np.testing.assert_allclose(out["lse"], lse_ref, atol=1e-13)


def test_kl_div_special_case():
    """Distinct ids: L is torch's KL divergence of the softmax against a dense
    target equal to p at the ids and 0 elsewhere (sum reduction)."""
    T, d, V, K = 6, 7, 40, 9
    H, W, idx, p = _rand_case(T, d, V, K, seed=5)
    p[0, 3] = 0.0            # a zero-probability pad inside the support
    p[1, :] = 0.0            # a row with no teacher mass
    out = kd_oracle(H, W, idx, p)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    target = torch.zeros(T, V, dtype=torch.float64)
    target.scatter_(1, torch.tensor(idx, dtype=torch.int64), torch.tensor(p))
    logq = torch.log_softmax(Ht @ Wt.T, dim=1)
    kl = torch.nn.functional.kl_div(logq, target, reduction="sum")
    kl.backward()
    assert out["loss"] == pytest.approx(kl.item(), rel=1e-13)
    np.testing.assert_allclose(out["dH"], Ht.grad.numpy(), atol=1e-12)
    np.testing.assert_allclose(out["dW"], Wt.grad.numpy(), atol=1e-12)
    assert out["loss_rows"][1] == 0.0


# ---------------------------------------------------------------- P2
def test_gradient_rows_sum_to_zero():
    H, W, idx, p = _rand_case(5, 6, 30, 7, seed=2, distinct=False)
    out = kd_oracle(H, W, idx, p)
    # sum_j G_tj = 0 for every row  =>  sum over the vocabulary of dW is 0
    np.testing.assert_allclose(out["dW"].sum(axis=0), 0.0, atol=1e-12)
    # and <W, dW> = <H, dH> (both equal sum_tj G_tj z_tj)
    assert np.sum(W * out["dW"]) == pytest.approx(np.sum(H * out["dH"]), rel=1e-12)


# ---------------------------------------------------------------- P3
def test_self_distillation_is_zero():
    from scipy.special import softmax

    rng = np.random.default_rng(9)
    T, d, V = 4, 6, 10
    H, W = rng.normal(size=(T, d)), rng.normal(size=(V, d))
    q = softmax(H @ W.T, axis=1)
    idx = np.stack([rng.permutation(V) for _ in range(T)])
    p = np.take_along_axis(q, idx, axis=1)
    out = kd_oracle(H, W, idx, p)
    assert abs(out["loss"]) < 1e-13
    np.testing.assert_allclose(out["dH"], 0.0, atol=1e-13)
    np.testing.assert_allclose(out["dW"], 0.0, atol=1e-13)


# ---------------------------------------------------------------- P5
def test_zero_weights_closed_form():
    T, d, V, K = 5, 4, 16, 6
    H, _, idx, p = _rand_case(T, d, V, K, seed=4)
    W = np.zeros((V, d))
    out = kd_oracle(H, W, idx, p)
    M = p.sum(axis=1)
    E = (p * np.log(p)).sum(axis=1)
    assert out["loss"] == pytest.approx(float(np.sum(E + M * math.log(V))), rel=1e-13)
    np.testing.assert_allclose(out["lse"], math.log(V), atol=1e-14)
    G = np.repeat((M / V)[:, None], V, axis=1)
    for t in range(T):
        for k in range(K):
            G[t, idx[t, k]] -= p[t, k]
    np.testing.assert_allclose(out["dH"], 0.0, atol=1e-15)
    np.testing.assert_allclose(out["dW"], G.T @ H, atol=1e-13)


# ---------------------------------------------------------------- P6
def test_logit_shift_invariance():
    H, W, idx, p = _rand_case(4, 5, 20, 5, seed=6)
    b = np.random.default_rng(1).normal(size=5)
    a = kd_oracle(H, W, idx, p)
    s = kd_oracle(H, W + b[None, :], idx, p)
    assert s["loss"] == pytest.approx(a["loss"], rel=1e-12)
    np.testing.assert_allclose(s["lse"], a["lse"] + H @ b, atol=1e-12)
    np.testing.assert_allclose(s["dW"], a["dW"], atol=1e-12)


# ---------------------------------------------------------------- P7
def test_scaling_in_p():
    H, W, idx, p = _rand_case(4, 5, 20, 5, seed=7)
    alpha = 0.37
    a = kd_oracle(H, W, idx, p)
    s = kd_oracle(H, W, idx, alpha * p)
    M = p.sum(axis=1)
    expect = alpha * a["loss"] + alpha * math.log(alpha) * M.sum()
    assert s["loss"] == pytest.approx(expect, rel=1e-12)
    np.testing.assert_allclose(s["dH"], alpha * a["dH"], atol=1e-13)
    np.testing.assert_allclose(s["dW"], alpha * a["dW"], atol=1e-13)


# ---------------------------------------------------------------- P8
def test_permutation_invariance():
    T, d, V, K = 6, 5, 25, 7
    H, W, idx, p = _rand_case(T, d, V, K, seed=8)
    rng = np.random.default_rng(0)
    a = kd_oracle(H, W, idx, p)
    # within a row
    pk = np.stack([rng.permutation(K) for _ in range(T)])
    b = kd_oracle(H, W, np.take_along_axis(idx, pk, 1), np.take_along_axis(p, pk, 1))
    assert b["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(b["dW"], a["dW"], atol=1e-13)
    # over rows
    pt = rng.permutation(T)
    c = kd_oracle(H[pt], W, idx[pt], p[pt])
    assert c["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(c["dH"], a["dH"][pt], atol=1e-13)
    np.testing.assert_allclose(c["dW"], a["dW"], atol=1e-13)
    # over the vocabulary: W rows permuted, ids remapped, dW rows permute with them
    pv = rng.permutation(V)            # new row j holds old row pv[j]
    inv = np.argsort(pv)
    e = kd_oracle(H, W[pv], inv[idx], p)
    assert e["loss"] == pytest.approx(a["loss"], rel=1e-13)
    np.testing.assert_allclose(e["dW"], a["dW"][pv], atol=1e-13)
    np.testing.assert_allclose(e["dH"], a["dH"], atol=1e-13)


# ---------------------------------------------------------------- P9
def test_naive_matches_blocked():
    T, d, V, K = 7, 6, 23, 5
    H, W, idx, p = _rand_case(T, d, V, K, seed=10, distinct=False)
    idx[0, 1] = idx[0, 0]     # duplicate id
    p[2, 2] = 0.0             # zero-probability pad
    p[3, :] = 0.0             # row with M_t = 0
    idx[4, 3] = V + 2         # out-of-range id: the row contributes nothing
    a = kd_oracle_naive(H, W, idx, p)
    for rpb in (1, 3, 256):
        b = kd_oracle(H, W, idx, p, rows_per_block=rpb)
        assert b["loss"] == pytest.approx(a["loss"], rel=1e-13)
        np.testing.assert_allclose(b["loss_rows"], a["loss_rows"], atol=1e-13)
        np.testing.assert_allclose(b["lse"], a["lse"], atol=1e-13)
        np.testing.assert_allclose(b["dH"], a["dH"], atol=1e-13)
        np.testing.assert_allclose(b["dW"], a["dW"], atol=1e-13)
    assert a["loss_rows"][3] == 0.0 and a["loss_rows"][4] == 0.0
    assert np.all(a["dH"][4] == 0.0)


def test_rows_subset_matches_full():
    H, W, idx, p = _rand_case(9, 6, 30, 4, seed=13)
    full = kd_oracle(H, W, idx, p)
    rows = np.array([8, 0, 5])
    sub = kd_oracle_rows(H, W, idx, p, rows)
    np.testing.assert_allclose(sub["lse"], full["lse"][rows], atol=1e-13)
    np.testing.assert_allclose(sub["loss_rows"], full["loss_rows"][rows], atol=1e-13)
    np.testing.assert_allclose(sub["dH"], full["dH"][rows], atol=1e-13)


def test_dW_rows_finite_differences():
    """Selected rows of dW from the oracle's own lse equal central finite
    differences of L with respect to those rows of W (duplicates, pads and a
    zero-mass row included), independently of the full backward."""
    H, W, idx, p = _rand_case(4, 6, 14, 5, seed=31, distinct=False)
    idx[0, 1] = idx[0, 0]
    p[1, 2] = 0.0
    p[2, :] = 0.0
    lse = kd_oracle(H, W, idx, p, want_grads=False)["lse"]
    vrows = np.array([13, 0, int(idx[0, 0]) if idx[0, 0] not in (13, 0) else 5, 7])
    got = kd_oracle_dW_rows(H, W, idx, p, lse, vrows, rows_per_block=3)
    h = 1e-6
    num = np.zeros((len(vrows), W.shape[1]))
    for a, j in enumerate(vrows):
        for c in range(W.shape[1]):
            Wp, Wm = W.copy(), W.copy()
            Wp[j, c] += h
            Wm[j, c] -= h
            num[a, c] = (_loss_only(H, Wp, idx, p) - _loss_only(H, Wm, idx, p)) / (2 * h)
    assert np.abs(got - num).max() <= 1e-7 * max(np.abs(num).max(), 1.0)


def test_dW_rows_match_full_backward():
    T, d, V, K = 11, 5, 40, 6
    H, W, idx, p = _rand_case(T, d, V, K, seed=32, distinct=False)
    idx[0, 1] = idx[0, 0]          # duplicate id
    idx[1, :] = 39                 # one id K times, at the vocabulary end
    p[2, 3] = 0.0                  # zero-probability pad
    p[3, :] = 0.0                  # no teacher mass
    idx[4, 2] = V + 1              # bad id: the row contributes nothing
    idx[5, 0] = -2
    full = kd_oracle(H, W, idx, p)
    vrows = np.array([39, 0, int(idx[0, 0]), 17, 38]) if idx[0, 0] not in (39, 0, 17, 38) else np.array([39, 0, 17, 38])
    for rpb in (1, 4, 1024):
        got = kd_oracle_dW_rows(H, W, idx, p, full["lse"], vrows, rows_per_block=rpb)
        np.testing.assert_allclose(got, full["dW"][vrows], atol=1e-13)
    all_rows = kd_oracle_dW_rows(H, W, idx, p, full["lse"], np.arange(V))
    np.testing.assert_allclose(all_rows, full["dW"], atol=1e-13)
    with pytest.raises(ValueError):
        kd_oracle_dW_rows(H, W, idx, p, full["lse"], np.array([3, 3]))


def test_dW_rows_reject_a_wrong_lse():
    """The selected rows depend on every token's lse: an lse taken from the
    top-K ids only, or shifted by a constant, moves them visibly."""
    H, W, idx, p = _rand_case(6, 5, 30, 4, seed=33)
    full = kd_oracle(H, W, idx, p)
    vrows = np.arange(0, 30, 3)
    ref = full["dW"][vrows]
    z = H @ W.T
    zk = np.take_along_axis(z, idx.astype(np.int64), 1)
    lse_topk = zk.max(1) + np.log(np.exp(zk - zk.max(1, keepdims=True)).sum(1))
    for bad in (lse_topk, full["lse"] + 0.05, full["lse"][::-1].copy()):
        got = kd_oracle_dW_rows(H, W, idx, p, bad, vrows)
        assert np.abs(got - ref).max() > 1e-3 * np.abs(ref).max()


# ---------------------------------------------------------------- pin sensitivity
def test_pins_catch_planted_mistakes(monkeypatch):
    """A wrong oracle must fail the pins: plant three plausible mistakes in a
    copy of the gradient and check the library-autograd pin rejects each."""
    T, d, V, K = 4, 5, 15, 4
    H, W, idx, p = _rand_case(T, d, V, K, seed=21)
    Ht = torch.tensor(H, requires_grad=True)
    Wt = torch.tensor(W, requires_grad=True)
    target = torch.zeros(T, V, dtype=torch.float64)
    target.scatter_(1, torch.tensor(idx, dtype=torch.int64), torch.tensor(p))
    kl = torch.nn.functional.kl_div(torch.log_softmax(Ht @ Wt.T, 1), target, reduction="sum")
    kl.backward()
    z = H @ W.T
    q = np.exp(z - z.max(1, keepdims=True))
    q /= q.sum(1, keepdims=True)
    M = p.sum(1)
    P = target.numpy()
    good = M[:, None] * q - P
    wrong = {
        "dropped mass": q - P,                     # M_t taken as 1
        "sign": P - M[:, None] * q,
        "transposed": (M[:, None] * q - P)[:, ::-1],
    }
    np.testing.assert_allclose(good @ W, Ht.grad.numpy(), atol=1e-12)
    for name, G in wrong.items():
        assert np.abs(G @ W - Ht.grad.numpy()).max() > 1e-3, name


# ---------------------------------------------------------------- inputs
def test_inputs_follow_their_recipe():
    idx, p = make_cache(512, 128256, 100, "zipf", seed=1)
    assert idx.dtype == np.int32 and p.dtype == np.float32
    assert idx.shape == (512, 100) and p.shape == (512, 100)
    assert idx.min() >= 0 and idx.max() < 128256
    assert all(len(set(r)) == 100 for r in idx.tolist())
    M = p.sum(1)
    assert M.min() >= 0.85 - 1e-5 and M.max() <= 0.99 + 1e-5
    assert np.all(np.diff(p, axis=1) <= 1e-7)        # sorted-descending logits in draw order
    tidx, tp = make_cache(256, 4096, 16, "uniform", seed=0)
    assert all(len(set(r)) == 16 for r in tidx.tolist())
    assert tp.sum(1).min() >= 0.8 - 1e-5 and tp.sum(1).max() <= 1.0 + 1e-5
    H, W = make_hw(64, 32, 100, "uniform", 0)
    assert H.dtype == torch.bfloat16 and W.shape == (100, 32)
    assert 0.6 < H.float().std().item() < 1.4 and 0.01 < W.float().std().item() < 0.03
    a, b = make_cache(64, 1000, 8, "zipf", 3), make_cache(64, 1000, 8, "zipf", 3)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])
    inp = make_inputs("tiny", T=40)
    assert inp["H"].shape == (40, 256) and inp["idx"].shape == (40, 16)
