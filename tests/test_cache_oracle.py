"""Pins of the teacher-cache oracle (top-K selection and softmax, fp64) against
things other than itself: closed forms (strictly decreasing logits: a
geometric series; equal logits: the first K ids at 1/V each), invariants
(logit shift, K = V gives the whole distribution), brute force against the
pure-Python selection on tiny tied inputs, and torch.topk's values.  The last
test plants plausible mistakes in a copy of the oracle and checks that the
pins reject each one."""
import math

import numpy as np
import pytest
import torch

from oracle import topk_cache_naive, topk_cache_oracle
from lm_head_top_tma_b300.inputs import make_teacher_logits


def test_strictly_decreasing_logits_closed_form():
    V, K, a = 50, 7, 0.3
    Z = -a * np.arange(V, dtype=np.float64)[None, :]
    out = topk_cache_oracle(Z, K)
    assert out["idx"][0].tolist() == list(range(K))
    # p_k = e^{-ka} (1 - e^{-a}) / (1 - e^{-Va})
    ref = [math.exp(-k * a) * (1 - math.exp(-a)) / (1 - math.exp(-V * a)) for k in range(K)]
    np.testing.assert_allclose(out["p"][0], ref, rtol=1e-13)
    assert out["lse"][0] == pytest.approx(math.log((1 - math.exp(-V * a)) / (1 - math.exp(-a))), rel=1e-13)


def test_equal_logits_take_lowest_ids():
    V, K = 40, 9
    out = topk_cache_oracle(np.full((2, V), 1.75), K)
    assert out["idx"].tolist() == [list(range(K))] * 2
    np.testing.assert_allclose(out["p"], 1.0 / V, rtol=1e-14)


def test_reversed_ids_and_ties():
    # ids in reverse order of logit, with a tied pair: 3 and 5 share the top value
    z = np.array([[0.0, 1.0, 2.0, 5.0, 3.0, 5.0, -1.0]])
    out = topk_cache_oracle(z, 4)
    assert out["idx"][0].tolist() == [3, 5, 4, 2]


def test_shift_invariance_and_full_mass():
    rng = np.random.default_rng(0)
    Z = rng.normal(size=(5, 30))
    a = topk_cache_oracle(Z, 30)
    b = topk_cache_oracle(Z + 123.25, 30)
    assert np.array_equal(a["idx"], b["idx"])
    np.testing.assert_allclose(a["p"], b["p"], rtol=1e-12)
    np.testing.assert_allclose(a["p"].sum(axis=1), 1.0, rtol=1e-13)   # K = V: the whole distribution
    assert np.all(np.diff(a["p"], axis=1) <= 0)


def test_masked_logits_carry_no_mass():
    z = np.array([[0.5, -np.inf, 2.0, -np.inf, 1.0]])
    out = topk_cache_oracle(z, 3)
    assert out["idx"][0].tolist() == [2, 4, 0]
    np.testing.assert_allclose(out["p"].sum(), 1.0, rtol=1e-14)


@pytest.mark.parametrize("seed", range(5))
def test_brute_force_on_tied_bf16_rows(seed):
    Z = make_teacher_logits(6, 37, seed=seed, noise=0.5).float().numpy()
    Z[:, ::5] = Z[:, 1:2]                 # plant extra ties
    for K in (1, 5, 37):
        a = topk_cache_oracle(Z, K)
        b = topk_cache_naive(Z, K)
        assert np.array_equal(a["idx"], b["idx"])
        np.testing.assert_allclose(a["p"], b["p"], rtol=1e-13)
        np.testing.assert_allclose(a["lse"], b["lse"], rtol=1e-13)


def test_values_match_torch_topk():
    Z = make_teacher_logits(16, 3000, seed=3).float()
    out = topk_cache_oracle(Z, 100)
    vals = torch.topk(Z.double(), 100, dim=1).values.numpy()
    got = np.take_along_axis(Z.double().numpy(), out["idx"].astype(np.int64), axis=1)
    assert np.array_equal(got, vals)
    lse = torch.logsumexp(Z.double(), dim=1).numpy()
    np.testing.assert_allclose(out["lse"], lse, rtol=1e-13)


# ---------------------------------------------------------------- pin sensitivity
def _pins(fn):
    """The pins above as checks of a cache function fn(Z, K) -> {idx, p, lse};
    returns the names of the pins it fails."""
    failed = []
    V, K, a = 50, 7, 0.3
    out = fn(-a * np.arange(V, dtype=np.float64)[None, :], K)
    ref = [math.exp(-k * a) * (1 - math.exp(-a)) / (1 - math.exp(-V * a)) for k in range(K)]
    if out["idx"][0].tolist() != list(range(K)) or not np.allclose(out["p"][0], ref, rtol=1e-12):
        failed.append("geometric closed form")
    out = fn(np.full((1, 40), 1.75), 9)
    if out["idx"][0].tolist() != list(range(9)) or not np.allclose(out["p"], 1 / 40, rtol=1e-12):
        failed.append("equal logits")
    Z = make_teacher_logits(4, 300, seed=5).float()
    out = fn(Z, 20)
    vals = torch.topk(Z.double(), 20, dim=1).values.numpy()
    got = np.take_along_axis(Z.double().numpy(), out["idx"].astype(np.int64), axis=1)
    if not np.array_equal(got, vals) or not np.allclose(out["lse"], torch.logsumexp(Z.double(), 1).numpy(),
                                                          rtol=1e-12):
        failed.append("torch.topk values and logsumexp")
    Zt = make_teacher_logits(3, 23, seed=1, noise=0.5).float().numpy()
    Zt[:, ::4] = Zt[:, 2:3]
    a_, b_ = fn(Zt, 6), topk_cache_naive(Zt, 6)
    if not np.array_equal(a_["idx"], b_["idx"]) or not np.allclose(a_["p"], b_["p"], rtol=1e-12):
        failed.append("brute force")
    return failed


def _variant(mistake):
    """topk_cache_oracle with one plausible mistake planted (CPU, test-local)."""
    def fn(Z, K):
        Z = np.asarray(Z.double().numpy() if hasattr(Z, "double") else Z, dtype=np.float64)
        T, V = Z.shape
        ids = np.arange(V)
        idx = np.empty((T, K), dtype=np.int32)
        p = np.empty((T, K))
        lse = np.empty(T)
        for t in range(T):
            z = Z[t]
            order = np.lexsort((-ids if mistake == "ties by descending id" else ids, -z))
            if mistake == "ascending order":
                order = np.lexsort((ids, z))
            idx[t] = order[1:K + 1] if mistake == "off by one rank" and V > K else order[:K]
            m = z.max()
            terms = z[idx[t]] if mistake == "lse over the top K" else z
            lse[t] = m + math.log(np.exp(terms - m).sum())
            p[t] = np.exp(z[idx[t]] - lse[t])
            if mistake == "p renormalised over the top K":
                p[t] /= p[t].sum()
        return {"idx": idx, "p": p, "lse": lse}
    return fn


def test_pins_catch_planted_mistakes():
    assert _pins(topk_cache_oracle) == []
    for mistake in ("ties by descending id", "ascending order", "off by one rank", "lse over the top K",
                    "p renormalised over the top K"):
        assert _pins(_variant(mistake)), mistake
