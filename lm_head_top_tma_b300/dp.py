"""Token-parallel (data-parallel) use of the fused step across processes.

Rows of the loss are independent: a token's loss, lse and dH need only its own
hidden state, the full W and its own teacher cache.  So a sequence of T tokens
splits into contiguous shards, one per rank, each with a full replica of W, and
each rank runs ``kd_topk_kl_fused_step`` on its own rows.  The one exchange
step is a sum over ranks of dW [V,d] (fp32) and of the scalar loss; dH and lse
stay with the rank that owns the rows.  The pages describe only the one-GPU
loss (aimodeling.com "Second cut": chunked over the sequence); the parallel
group their released code is written for appears only as entry names
(codewithpapers.app record, harvested samples: a tensor-parallel rank and
size), so the partition here is the plain token split the loss's row
independence allows.

All arithmetic of the step stays in the library's kernels; this module only
picks rows and calls ``torch.distributed.all_reduce`` (any backend: gloo for
host tensors, NCCL for device tensors).  Without an initialised process group
it runs the single-process step unchanged.
"""
from __future__ import annotations

import torch

from . import api

__all__ = ["shard_rows", "allreduce_loss_and_dW", "fused_step_data_parallel"]


def shard_rows(T: int, world_size: int, rank: int) -> tuple[int, int]:
    """Rows [t0, t1) of a T-token sequence that ``rank`` owns: contiguous,
    in rank order, sizes differing by at most one (the first T % world_size
    ranks take one extra row).  A rank may own no rows when T < world_size."""
    if world_size < 1 or not 0 <= rank < world_size or T < 0:
        raise ValueError(f"bad shard request T={T} world_size={world_size} rank={rank}")
    base, extra = divmod(int(T), int(world_size))
    t0 = rank * base + min(rank, extra)
    return t0, t0 + base + (1 if rank < extra else 0)


def _world(group):
    import torch.distributed as dist

    if not (dist.is_available() and dist.is_initialized()):
        return None, 1
    return dist, dist.get_world_size(group)


def allreduce_loss_and_dW(res: dict, group=None) -> dict:
    """Sum ``res["loss"]`` and ``res["dW"]`` over the ranks of ``group``, in
    place.  The loss is summed in fp64 (each rank's partial is itself an fp64
    sum rounded to fp32 once) and written back as fp32; ``res["loss_f64"]``
    keeps the fp64 total.  dW is summed in its own dtype.  With no process
    group (or one rank) nothing is exchanged."""
    dist, ws = _world(group)
    loss = res["loss"].reshape(-1)[:1].to(torch.float64)
    if ws > 1:
        dist.all_reduce(loss, op=dist.ReduceOp.SUM, group=group)
        dist.all_reduce(res["dW"], op=dist.ReduceOp.SUM, group=group)
    res["loss"].reshape(-1)[:1].copy_(loss.to(res["loss"].dtype))
    res["loss_f64"] = float(loss.item())
    return res


def fused_step_data_parallel(H, W, idx, p, chunk: int, *, group=None, dloss: float = 1.0,
                             recompute: bool = True, loss_rows: bool = False,
                             workspace: api.Workspace | None = None, out: dict | None = None,
                             check: bool = True) -> dict:
    """One fused forward + backward over this rank's rows, then the exchange.

    H [T_r,d], idx and p [T_r,K] are this rank's shard (``shard_rows`` gives
    the split of a sequence); W [V,d] is the full replica every rank holds.
    Returns the dict of ``api.fused_step``: ``loss`` and ``dW`` summed over
    the group (the loss and weight gradient of the whole sequence), ``lse``,
    ``dH`` (and ``loss_rows``) for this rank's rows only.  dW is always
    overwritten: accumulating into a caller's dW would add its previous
    contents once per rank, so a trainer accumulates after the exchange."""
    step = api.fused_step if recompute else api.fused_step_norecompute
    res = step(H, W, idx, p, chunk, dloss=dloss, loss_rows=loss_rows, workspace=workspace, out=out, check=check)
    return allreduce_loss_and_dW(res, group)
