"""Multi-rank host logic on CPU ranks (gloo, world size 2 and 4).

Token-sharded routing and the expert-parallel dispatch plan exchange their per-rank
results with torch.distributed collectives.  Here the ranks are CPU processes and the
per-rank steps are stand-ins backed by the oracle (the library's CUDA kernels are
compared with the same oracle functions in the GPU tests), so what is under test is
the exchange: shard bounds, gathering of unequal shards in rank order, the counts
matrix and each rank's send/receive layout.
"""
import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _oracle_fns():
    import oracle

    def route_fn(logits, bias, **kw):
        cfg = kw["cfg"]
        sub = dict(cfg, logits=logits.numpy(), T=logits.shape[0])
        o = oracle.route_cfg(sub)
        return {k: torch.from_numpy(np.ascontiguousarray(o[k])) for k in ("packed", "counts", "offsets", "perm")}

    def index_fn(packed, NE):
        r = oracle.route_index(packed.numpy(), NE)
        return {k: torch.from_numpy(v) for k, v in r.items()}

    def layout_fn(matrix, rank):
        r = oracle.alltoall_layout(matrix.numpy(), rank)
        return {k: torch.from_numpy(v) for k, v in r.items()}

    return route_fn, index_fn, layout_fn


def _worker(rank, world, port, result_dir):
    for p in (ROOT, HERE):
        if p not in sys.path:
            sys.path.insert(0, p)
    import gen
    import oracle
    from serving_moe_route_02_gb300 import sharded

    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank, world_size=world)
    try:
        route_fn, index_fn, layout_fn = _oracle_fns()
        T = 997  # shards of unequal sizes
        cfg = gen.cfg3(T, off=784, cnt=112)
        lo, hi = sharded.shard_bounds(T, world, rank)
        shard = torch.from_numpy(np.ascontiguousarray(cfg["logits"][lo:hi]))
        out = sharded.token_sharded_route(shard, torch.from_numpy(cfg["bias"]), route_fn=route_fn,
                                          index_fn=index_fn, cfg=cfg)
        full = oracle.route_cfg(cfg)
        assert out["shard"] == (lo, hi - lo)
        for key in ("packed", "counts", "offsets", "perm"):
            got = out[key].numpy().reshape(full[key].shape)
            assert np.array_equal(got, full[key]), (rank, key)

        # dispatch: global ids of this rank's shard, one row of the counts matrix per rank
        g = dict(cfg, off=0, cnt=0, logits=cfg["logits"][lo:hi], T=hi - lo)
        mine = oracle.route_cfg(g)
        d = oracle.dispatch_counts(mine["ids"], 896, world)

        def counts_fn(offsets, R):
            return {k: torch.from_numpy(v) for k, v in d.items()}

        plan = sharded.dispatch_plan(torch.from_numpy(mine["offsets"]), counts_fn=counts_fn,
                                     layout_fn=layout_fn)
        m = plan["matrix"].numpy()
        assert m.shape == (world, world) and np.array_equal(m[rank], d["send_counts"])
        np.save(os.path.join(result_dir, f"plan{rank}.npy"),
                np.concatenate([m.ravel(), plan["send_displs"].numpy(), plan["recv_counts"].numpy(),
                                plan["recv_displs"].numpy()]))
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("world", [2, 4])
def test_token_sharded_and_dispatch_on_cpu_ranks(tmp_path, world):
    mp.spawn(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world, join=True)
    # every rank saw the same matrix; what rank s sends to rank d is what d receives from s
    plans = [np.load(tmp_path / f"plan{r}.npy") for r in range(world)]
    W = world
    mats = [p[: W * W].reshape(W, W) for p in plans]
    for m in mats[1:]:
        assert np.array_equal(m, mats[0])
    m = mats[0]
    for r, p in enumerate(plans):
        sd = p[W * W: W * W + W + 1]
        rc = p[W * W + W + 1: W * W + 2 * W + 1]
        rd = p[W * W + 2 * W + 1:]
        assert np.array_equal(sd, np.concatenate([[0], np.cumsum(m[r])]))
        assert np.array_equal(rc, m[:, r])
        assert np.array_equal(rd, np.concatenate([[0], np.cumsum(m[:, r])]))
    assert m.sum() == 997 * 16


def test_single_rank_runs_without_collectives():
    import gen
    import oracle
    from serving_moe_route_02_gb300 import sharded
    route_fn, index_fn, layout_fn = _oracle_fns()
    cfg = gen.cfg1(8)
    out = sharded.token_sharded_route(torch.from_numpy(cfg["logits"]), torch.from_numpy(cfg["bias"]),
                                      route_fn=route_fn, index_fn=index_fn, cfg=cfg)
    full = oracle.route_cfg(cfg)
    assert out["shard"] == (0, 8)
    assert np.array_equal(out["packed"].numpy(), full["packed"])
    assert sharded.shard_bounds(10, 3, 0) == (0, 3) and sharded.shard_bounds(10, 3, 2) == (6, 10)
