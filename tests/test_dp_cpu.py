"""The token-parallel step's host logic on CPU: gloo ranks on 127.0.0.1.

Each rank takes its rows with ``shard_rows``, computes the fp64 oracle on
them (standing in for the GPU step, which needs a GPU), and exchanges loss and
dW with ``allreduce_loss_and_dW``.  The exchanged loss and dW, and the
concatenated per-rank lse and dH, must equal the oracle on the whole sequence:
the loss is a sum over tokens and dW = sum_t G_t^T H_t, so the token split is
exact.  Ragged splits (T not a multiple of the world size, a rank with no
rows) are covered."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from lm_head_top_tma_b300.dp import shard_rows


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _case(T, seed=0, d=6, V=29, K=5):
    rng = np.random.default_rng(seed)
    H = rng.normal(size=(T, d))
    W = rng.normal(size=(V, d)) * 0.5
    idx = rng.integers(0, V, size=(T, K)).astype(np.int32)
    p = rng.random(size=(T, K))
    p = p / p.sum(1, keepdims=True) * 0.9
    p[min(1, T - 1), :] = 0.0                       # a row with no teacher mass
    return H, W, idx, p


def _rank_main(rank, world, port, T, out):
    os.environ.update({"RANK": str(rank), "WORLD_SIZE": str(world), "MASTER_ADDR": "127.0.0.1",
                       "MASTER_PORT": str(port)})
    import torch.distributed as dist

    from lm_head_top_tma_b300.dp import allreduce_loss_and_dW
    from oracle import kd_oracle

    dist.init_process_group("gloo", rank=rank, world_size=world)
    H, W, idx, p = _case(T)
    t0, t1 = shard_rows(T, world, rank)
    V, d = W.shape
    if t1 > t0:
        ref = kd_oracle(H[t0:t1], W, idx[t0:t1], p[t0:t1])
        res = {"loss": torch.tensor([ref["loss"]], dtype=torch.float64), "dW": torch.from_numpy(ref["dW"]).clone()}
        lse, dH = ref["lse"], ref["dH"]
    else:                                            # a rank without rows still joins the exchange
        res = {"loss": torch.zeros(1, dtype=torch.float64), "dW": torch.zeros(V, d, dtype=torch.float64)}
        lse, dH = np.zeros(0), np.zeros((0, d))
    allreduce_loss_and_dW(res)
    out[rank] = (t0, t1, res["loss_f64"], res["dW"].numpy().copy(), lse, dH)
    dist.destroy_process_group()


@pytest.mark.parametrize("world,T", [(2, 17), (3, 2)])
def test_token_parallel_exchange_equals_whole_sequence(world, T):
    from oracle import kd_oracle

    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, T, out)) for r in range(world)]
    for pr in procs:
        pr.start()
    for pr in procs:
        pr.join(timeout=180)
        assert pr.exitcode == 0
    H, W, idx, p = _case(T)
    full = kd_oracle(H, W, idx, p)
    got = [out[r] for r in range(world)]
    assert [g[:2] for g in got] == [shard_rows(T, world, r) for r in range(world)]
    for g in got:                                    # every rank holds the sequence's loss and dW
        assert g[2] == pytest.approx(full["loss"], rel=1e-13)
        np.testing.assert_allclose(g[3], full["dW"], atol=1e-12)
    np.testing.assert_allclose(np.concatenate([g[4] for g in got]), full["lse"], atol=1e-13)
    np.testing.assert_allclose(np.concatenate([g[5] for g in got]), full["dH"], atol=1e-13)


def test_shard_rows_partition():
    for T in (0, 1, 5, 16, 17, 32768):
        for world in (1, 2, 3, 8):
            spans = [shard_rows(T, world, r) for r in range(world)]
            assert spans[0][0] == 0 and spans[-1][1] == T
            assert all(a[1] == b[0] for a, b in zip(spans, spans[1:]))
            sizes = [b - a for a, b in spans]
            assert max(sizes) - min(sizes) <= 1 and sum(sizes) == T
    with pytest.raises(ValueError):
        shard_rows(10, 2, 2)


def test_single_process_needs_no_group():
    """Without a process group the exchange is the identity (loss kept, fp64 copy made)."""
    from lm_head_top_tma_b300.dp import allreduce_loss_and_dW

    res = {"loss": torch.tensor([2.5]), "dW": torch.ones(3, 2)}
    allreduce_loss_and_dW(res)
    assert res["loss_f64"] == 2.5 and res["loss"].item() == 2.5 and torch.all(res["dW"] == 1)
