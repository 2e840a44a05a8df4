"""moe_route_noalloc against moe_route.

Some callers cannot call cudaMalloc: a serving engine that reserves all free HBM at
start-up, code under a memory pool that forbids raw allocations, a plugin that may only
use the buffers it is handed.  moe_route_noalloc serves them with scratch held in a
static array inside the library.  This file checks, through the C ABI, that two calls in
a row of the no-allocation entry point give exactly the outputs of moe_route (bit-exact,
the bar the other parity tests apply to the same kernels) and meet the oracle under the
same bar as moe_route (bit-exact for bf16 logits; the near-tie rule for float32 logits),
also for T = 0 and for a decode-size batch.  Its name makes pytest collect it last; it
passes alone in a fresh process and after the other tests.
"""
import ctypes

import numpy as np
import pytest
import torch

import gen
import oracle
import parity

pytestmark = pytest.mark.gpu


def _dev(cfg):
    dev = torch.device("cuda")
    if cfg["dtype"] == "bf16":
        lg = torch.from_numpy(np.ascontiguousarray(cfg["logits"]).view(np.int16)).to(dev).view(
            torch.bfloat16)
    else:
        lg = torch.from_numpy(np.ascontiguousarray(cfg["logits"], dtype=np.float32)).to(dev)
    return lg, torch.from_numpy(cfg["bias"]).to(dev)


@pytest.mark.parametrize("cfg", [gen.cfg3(16384), gen.cfg3(3001, off=784, cnt=112),
                                 gen.cfg4(T=2048, off=336, cnt=112), gen.cfg1(24),
                                 gen.cfg1(1, off=0, cnt=0)],
                         ids=["prefill16k", "prefill_local_ragged", "ties_f32_local", "decode24",
                              "decode1_global"])
def test_noalloc_matches_moe_route_twice(cfg):
    import serving_moe_route_02_gb300 as mr
    lib = mr.load()
    lg, bias = _dev(cfg)
    T, off, cnt = cfg["T"], cfg["off"], cfg["cnt"]
    ref = mr.route(lg, bias, local_offset=off, local_count=cnt, want_ids=True)
    torch.cuda.synchronize()
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    dt = mr.BF16 if cfg["dtype"] == "bf16" else mr.F32
    for _ in range(2):
        out = mr.alloc_outputs(T, 896, 16, cnt, lg.device, want_ids=True)
        for v in out.values():
            v.fill_(-1)
        rc = lib.moe_route_noalloc(P(lg), dt, P(bias), T, 896, 16, 8, 4, 2.5, off, cnt,
                                   P(out["packed"]), P(out["counts"]), P(out["offsets"]),
                                   P(out["perm"]), P(out["ids"]), P(status), stream)
        assert rc == mr.OK, mr.strerror(rc)
        torch.cuda.synchronize()
        assert int(status.item()) == 0
        for key in ("packed", "counts", "offsets", "perm", "ids"):
            assert torch.equal(out[key], ref[key]), key
    got = {k: v.cpu().numpy() for k, v in out.items()}
    parity.compare(got, oracle.route_cfg(cfg), cfg, exact=cfg["dtype"] == "bf16")


def test_noalloc_empty_batch_against_oracle():
    import serving_moe_route_02_gb300 as mr
    lib = mr.load()
    cfg = gen.cfg1(8)
    lg, bias = _dev(cfg)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    status = torch.full((1,), 12345, dtype=torch.int32, device="cuda")
    out = mr.alloc_outputs(0, 896, 16, 112, lg.device)
    out["counts"].fill_(-7)
    out["offsets"].fill_(-7)
    rc = lib.moe_route_noalloc(P(lg), mr.BF16, P(bias), 0, 896, 16, 8, 4, 2.5, 336, 112,
                               P(out["packed"]), P(out["counts"]), P(out["offsets"]),
                               P(out["perm"]), None, P(status), stream)
    assert rc == mr.OK, mr.strerror(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = oracle.route_cfg(dict(cfg, logits=cfg["logits"][:0], T=0))
    assert np.array_equal(out["counts"].cpu().numpy(), ref["counts"])
    assert np.array_equal(out["offsets"].cpu().numpy(), ref["offsets"])


def test_noalloc_rejects_what_moe_route_rejects():
    import serving_moe_route_02_gb300 as mr
    lib = mr.load()
    cfg = gen.cfg1(8)
    lg, bias = _dev(cfg)
    out = mr.alloc_outputs(8, 896, 16, 0, lg.device)
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    args = lambda **kw: [P(lg), 1, P(bias), kw.get("T", 8), kw.get("E", 896), 16, kw.get("G", 8),  # noqa: E731
                         4, 2.5, 0, kw.get("cnt", 0), P(out["packed"]), P(out["counts"]),
                         P(out["offsets"]), P(out["perm"]), None, None, stream]
    assert lib.moe_route_noalloc(*args(G=5)) == mr.E_INVALID_ARG
    assert lib.moe_route_noalloc(*args(cnt=-1)) == mr.E_INVALID_ARG
    assert lib.moe_route_noalloc(*args(E=256)) == mr.E_UNSUPPORTED
