"""Index from packed ids, dispatch counts and all-to-all layout on the GPU, against the
oracle, bit for bit; token-sharded routing on one rank through the library."""
import numpy as np
import pytest
import torch

import gen
import oracle

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    import serving_moe_route_02_gb300 as mr
    mr.load()
    mr.reserve()
    return mr


def routed(mr, cfg):
    dev = torch.device("cuda")
    lg = torch.from_numpy(np.ascontiguousarray(cfg["logits"]).view(np.int16)).to(dev).view(torch.bfloat16)
    return mr.route(lg, torch.from_numpy(cfg["bias"]).to(dev), local_offset=cfg["off"],
                    local_count=cfg["cnt"], want_ids=True)


@pytest.mark.parametrize("T,off,cnt", [(1, 0, 0), (8, 336, 112), (17, 0, 0), (50, 336, 112), (64, 0, 0), (65, 784, 112),
                                       (1001, 0, 0), (16384, 784, 112), (65536, 0, 0)])
def test_index_of_routed_packed(mr, T, off, cnt):
    """Indexing the routing's own packed ids gives the routing's counts, offsets, perm
    (decode kernel for T <= 64, persistent kernel above), equal to the oracle's index."""
    cfg = gen.cfg3(T, off=off, cnt=cnt) if T > 64 else gen.cfg1(T, off=off, cnt=cnt)
    out = routed(mr, cfg)
    NE = out["counts"].numel()
    idx = mr.route_index(out["packed"], NE)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    for key in ("counts", "offsets", "perm"):
        assert torch.equal(idx[key], out[key]), key
    ref = oracle.route_index(out["packed"].cpu().numpy(), NE)
    for key in ("counts", "offsets", "perm"):
        assert np.array_equal(idx[key].cpu().numpy(), ref[key]), key


def test_index_of_unaligned_packed(mr):
    """Packed values 4 bytes off a 16-byte boundary (the approximate-score kernel copies
    aligned rows, so the exact-score kernel takes them): the same outputs as the oracle."""
    T = 5000
    cfg = gen.cfg3(T)
    out = routed(mr, cfg)
    NE = out["counts"].numel()
    buf = torch.empty(T * 16 + 1, dtype=torch.int32, device="cuda")
    view = buf[1:].view(T, 16)
    view.copy_(out["packed"])
    assert view.data_ptr() % 16 == 4
    idx = mr.route_index(view, NE)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    ref = oracle.route_index(out["packed"].cpu().numpy(), NE)
    for key in ("counts", "offsets", "perm"):
        assert np.array_equal(idx[key].cpu().numpy(), ref[key]), key


def distinct_rows(T, k, NE, seed):
    """T rows of k distinct ids below NE: the k smallest of NE seeded draws per row."""
    r = gen.raw64(seed, T * NE).reshape(T, NE)
    return np.argsort(r, axis=1, kind="stable")[:, :k].astype(np.int64)


@pytest.mark.parametrize("T,k,NE", [(5, 3, 7), (64, 32, 1056), (3000, 8, 128), (40000, 1, 1)])
def test_index_of_arbitrary_packed(mr, T, k, NE):
    """Arbitrary ids (distinct within a row, any order), k other than 16."""
    ids = distinct_rows(T, k, NE, 4000 + T)
    packed = ((ids << 16) | 0x3E20).astype(np.int32).reshape(T, k)
    idx = mr.route_index(torch.from_numpy(packed).cuda(), NE)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    ref = oracle.route_index(packed, NE)
    for key in ("counts", "offsets", "perm"):
        assert np.array_equal(idx[key].cpu().numpy(), ref[key]), key


@pytest.mark.parametrize("T", [16, 500])
@pytest.mark.parametrize("fault", ["too_large", "repeated"])
def test_index_reports_bad_id(mr, T, fault):
    """An id at or above NE, or repeated within a row, is reported by the status word on
    both kernels; the other entries stay within the outputs."""
    ids = distinct_rows(T, 4, 9, 4100 + T)
    if fault == "too_large":
        ids[T // 2, 1] = 9
    else:
        ids[T // 2, 1] = ids[T // 2, 3]
    packed = ((ids << 16) | 0x3E20).astype(np.int32)
    idx = mr.route_index(torch.from_numpy(packed).cuda(), 9)
    assert mr.device_status() == mr.E_BAD_ID
    assert mr.device_status() == 0  # cleared by the read
    assert int(idx["counts"].sum()) <= T * 4


@pytest.mark.parametrize("T", [16, 5000])
@pytest.mark.parametrize("k,NE", [(8, 40), (16, 896), (16, 128)])
def test_index_leaves_out_every_bad_entry(mr, T, k, NE):
    """Rows with an id repeated three times, a repeated pair and an id >= NE: every kernel
    (decode-size, and for T > 64 the exact-score one or, at k = 16, the approximate-score
    one) leaves out exactly those entries (every occurrence of a repeated id), so the
    counts are the histogram of the remaining ones and the permutation holds exactly them."""
    ids = distinct_rows(T, k, NE, 4200 + T + k)
    bad_rows = sorted({1, T // 3, T // 2, T - 1})
    ids[bad_rows[0], 2] = ids[bad_rows[0], 5] = ids[bad_rows[0], 0]   # three times
    ids[bad_rows[1], 7] = ids[bad_rows[1], 3]                         # a pair
    ids[bad_rows[2], 4] = NE + 3                                      # out of range
    ids[bad_rows[3], 1] = ids[bad_rows[3], 6]
    ids[bad_rows[3], 0] = NE
    packed = ((ids << 16) | 0x3E20).astype(np.int32)
    idx = mr.route_index(torch.from_numpy(packed).cuda(), NE)
    assert mr.device_status() == mr.E_BAD_ID
    valid = ids < NE
    for t in range(T):
        u, c = np.unique(ids[t], return_counts=True)
        valid[t] &= ~np.isin(ids[t], u[c > 1])
    flat = np.flatnonzero(valid.ravel())
    assert np.array_equal(idx["counts"].cpu().numpy(), np.bincount(ids.ravel()[flat], minlength=NE))
    n = len(flat)
    assert int(idx["offsets"][-1]) == n
    got = np.sort(idx["perm"].cpu().numpy()[:n])
    assert np.array_equal(got, flat)


@pytest.mark.parametrize("R", [1, 2, 4, 7, 8, 16, 56])
def test_dispatch_counts(mr, R):
    cfg = gen.cfg3(3000)
    out = routed(mr, cfg)
    d = mr.dispatch_counts(out["offsets"], R)
    torch.cuda.synchronize()
    ref = oracle.dispatch_counts(out["ids"].cpu().numpy(), 896, R)
    assert np.array_equal(d["send_counts"].cpu().numpy(), ref["send_counts"])
    assert np.array_equal(d["send_offsets"].cpu().numpy(), ref["send_offsets"])


@pytest.mark.parametrize("R", [1, 3, 8, 64, 1024])
def test_alltoall_layout(mr, R):
    m = (gen.raw64(5000 + R, R * R) % np.uint64(1 << 14)).astype(np.int32).reshape(R, R)
    md = torch.from_numpy(m).cuda()
    for rank in sorted({0, R // 2, R - 1}):
        L = mr.alltoall_layout(md, rank)
        ref = oracle.alltoall_layout(m, rank)
        for key in ("send_displs", "recv_counts", "recv_displs"):
            assert np.array_equal(L[key].cpu().numpy(), ref[key]), (rank, key)


def test_rejects(mr):
    lib = mr.load()
    s = torch.cuda.current_stream().cuda_stream
    x = torch.zeros(1024, dtype=torch.int32, device="cuda")
    assert lib.moe_route_index(x.data_ptr(), 4, 33, 8, x.data_ptr(), x.data_ptr(), x.data_ptr(), s) == mr.E_UNSUPPORTED
    assert lib.moe_route_index(x.data_ptr(), 4, 4, 2000, x.data_ptr(), x.data_ptr(), x.data_ptr(), s) == mr.E_UNSUPPORTED
    assert lib.moe_route_dispatch_counts(x.data_ptr(), 896, 3, x.data_ptr(), None, s) == mr.E_INVALID_ARG
    assert lib.moe_route_alltoall_layout(x.data_ptr(), 4, 4, None, None, None, s) == mr.E_INVALID_ARG
    assert lib.moe_route_alltoall_layout(x.data_ptr(), 2000, 0, None, None, None, s) == mr.E_UNSUPPORTED


def test_token_sharded_single_rank(mr):
    """Without a process group the sharded call is one rank routing the whole batch."""
    from serving_moe_route_02_gb300 import sharded
    cfg = gen.cfg3(500, off=784, cnt=112)
    dev = torch.device("cuda")
    lg = torch.from_numpy(cfg["logits"].view(np.int16)).to(dev).view(torch.bfloat16)
    out = sharded.token_sharded_route(lg, torch.from_numpy(cfg["bias"]).to(dev),
                                      local_offset=784, local_count=112)
    o = oracle.route_cfg(cfg)
    for key in ("packed", "counts", "offsets", "perm"):
        assert np.array_equal(out[key].cpu().numpy().reshape(o[key].shape), o[key]), key
    g = routed(mr, dict(cfg, off=0, cnt=0))
    plan = sharded.dispatch_plan(g["offsets"], 8)
    ref = oracle.dispatch_counts(g["ids"].cpu().numpy(), 896, 8)
    assert np.array_equal(plan["send_counts"].cpu().numpy(), ref["send_counts"])
