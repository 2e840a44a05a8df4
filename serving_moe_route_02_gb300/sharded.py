"""Token-sharded routing and expert-parallel dispatch plans across ranks.

Plumbing around the library's kernels for multi-rank use.  Every arithmetic step is a
library call (``route``, ``route_index``, ``dispatch_counts``, ``alltoall_layout``);
this module only moves the small per-rank results between ranks with
``torch.distributed`` collectives (NCCL for CUDA tensors, gloo for CPU tensors).

Token-sharded routing (vLLM PR #59693, description: the residual stream is sharded over
tokens and the router's top-k results are gathered): rank r routes the contiguous rows
[T r / R, T (r + 1) / R) of the batch, the packed top-k values of all ranks are gathered,
and, routing being row-independent, the gathered values are the whole batch's; each rank
then builds the whole batch's counts, offsets and permutation from them.

Expert-parallel dispatch (vLLM PR #54606, description: a variable-size all-to-all driven
by a counts matrix, one layout helper for both transports): from a routing with global
ids, each rank's entries per destination rank are gathered into the counts matrix
[source][destination], from which every rank takes its send and receive displacements.
The transfer itself is out of scope here.

The collectives run on ``group`` (default: the world).  With no initialised process
group the calls run on one rank without collectives.  The ``*_fn`` arguments exist so
that the host-side logic can be exercised on CPU ranks with stand-in functions; their
defaults are the library's CUDA entry points.
"""
from __future__ import annotations

import torch
import torch.distributed as dist


def _world(group):
    if not (dist.is_available() and dist.is_initialized()):
        return 1, 0
    return dist.get_world_size(group), dist.get_rank(group)


def shard_bounds(T: int, world: int, rank: int) -> tuple[int, int]:
    """Rows [lo, hi) of a batch of T rows that rank `rank` of `world` routes."""
    return T * rank // world, T * (rank + 1) // world


def _gather_rows(x: torch.Tensor, group, world: int) -> torch.Tensor:
    """Concatenate every rank's x (same trailing shape, any number of rows) in rank order."""
    n = torch.tensor([x.shape[0]], dtype=torch.int64, device=x.device)
    sizes = [torch.empty_like(n) for _ in range(world)]
    dist.all_gather(sizes, n, group=group)
    sizes = [int(s.item()) for s in sizes]
    m = max(sizes)
    pad = torch.zeros((m,) + tuple(x.shape[1:]), dtype=x.dtype, device=x.device)
    pad[: x.shape[0]] = x
    parts = [torch.empty_like(pad) for _ in range(world)]
    dist.all_gather(parts, pad, group=group)
    return torch.cat([p[:s] for p, s in zip(parts, sizes)])


def token_sharded_route(logits_shard: torch.Tensor, bias: torch.Tensor, *, group=None,
                        route_fn=None, index_fn=None, **route_kw) -> dict:
    """Route this rank's rows, gather every rank's packed top-k values and index the
    whole batch.  Returns the whole batch's ``packed`` [T, k], ``counts``, ``offsets``,
    ``perm`` and this rank's ``shard`` = (first row, row count)."""
    if route_fn is None or index_fn is None:
        from . import route, route_index
        route_fn = route_fn or route
        index_fn = index_fn or route_index
    world, _ = _world(group)
    mine = route_fn(logits_shard, bias, **route_kw)
    NE = mine["counts"].numel()
    if world == 1:
        return dict(mine, shard=(0, logits_shard.shape[0]))
    rows = torch.tensor([logits_shard.shape[0]], dtype=torch.int64, device=mine["packed"].device)
    sizes = [torch.empty_like(rows) for _ in range(world)]
    dist.all_gather(sizes, rows, group=group)
    _, rank = _world(group)
    first = int(sum(int(s.item()) for s in sizes[:rank]))
    packed = _gather_rows(mine["packed"], group, world)
    full = index_fn(packed, NE)
    return dict(packed=packed, counts=full["counts"], offsets=full["offsets"], perm=full["perm"],
                shard=(first, logits_shard.shape[0]))


def dispatch_plan(offsets: torch.Tensor, num_ranks: int | None = None, *, group=None,
                  counts_fn=None, layout_fn=None) -> dict:
    """Expert-parallel dispatch layout of this rank's routing (global ids): entries per
    destination rank, the gathered counts matrix [source][destination], and this rank's
    send displacements, receive counts and receive displacements."""
    if counts_fn is None or layout_fn is None:
        from . import alltoall_layout, dispatch_counts
        counts_fn = counts_fn or dispatch_counts
        layout_fn = layout_fn or alltoall_layout
    world, rank = _world(group)
    R = world if num_ranks is None else num_ranks
    if R != world and world > 1:
        raise ValueError(f"num_ranks {R} differs from the group's {world} ranks")
    sc = counts_fn(offsets, R)
    if world > 1:
        rows = [torch.empty_like(sc["send_counts"]) for _ in range(world)]
        dist.all_gather(rows, sc["send_counts"].contiguous(), group=group)
        matrix = torch.stack(rows)
    else:
        matrix = sc["send_counts"].reshape(1, -1)
    lay = layout_fn(matrix, rank) if matrix.shape[0] == matrix.shape[1] else {}
    return dict(send_counts=sc["send_counts"], send_offsets=sc["send_offsets"], matrix=matrix, **lay)
