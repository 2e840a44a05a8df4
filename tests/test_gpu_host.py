"""moe_route_host (logits and results in host memory) against the oracle and against
moe_route on the same inputs, bit for bit; back-to-back calls that share the two
staging slots; pageable host memory; argument errors and capture."""
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


def host_logits(cfg, pin=True):
    lg = np.ascontiguousarray(cfg["logits"])
    if cfg["dtype"] == "bf16":
        t = torch.from_numpy(lg.view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(lg.astype(np.float32))
    return t.pin_memory() if pin else t.clone()


def dev_bias(cfg):
    return torch.from_numpy(np.ascontiguousarray(cfg["bias"], dtype=np.float32)).cuda()


def kw(cfg):
    return dict(k=cfg["k"], n_group=cfg["G"], topk_group=cfg["Kg"], scale=cfg["scale"],
                local_offset=cfg.get("off", 0), local_count=cfg.get("cnt", 0))


def check_against_oracle(out, cfg):
    ref = oracle.route_cfg(cfg)
    T = cfg["T"]
    for key in ("packed", "counts", "offsets", "perm"):
        got = out[key].numpy().reshape(ref[key].shape)
        assert np.array_equal(got, ref[key]), key
    if out.get("ids") is not None and T > 0:
        assert np.array_equal(out["ids"].numpy().reshape(T, -1), ref["ids"])


@pytest.mark.parametrize("case", ["cfg0_8", "cfg1_64", "cfg3_65", "cfg3_5000", "cfg3_0"])
def test_host_matches_oracle(mr, case):
    name, T = case.split("_")
    T = int(T)
    cfg = {"cfg0": lambda: gen.cfg0(T), "cfg1": lambda: gen.cfg1(T),
           "cfg3": lambda: gen.cfg3(T, off=784, cnt=112)}[name]()
    x = host_logits(cfg)
    out = mr.route_host(x, dev_bias(cfg), want_ids=True, **kw(cfg))
    assert mr.device_status() == 0
    ref = mr.route(x.cuda(), dev_bias(cfg), want_ids=True, **kw(cfg))
    torch.cuda.synchronize()
    for key in ("packed", "counts", "offsets", "perm", "ids"):
        assert torch.equal(out[key], ref[key].cpu()), key
    if cfg["dtype"] == "bf16":  # float32 scores are compared under the near-tie rule elsewhere
        check_against_oracle(out, cfg)


def test_back_to_back_calls_share_slots(mr):
    """Four calls of different sizes and dtypes without a synchronisation in between:
    every result equals moe_route's on the same input (the two slots alternate, the
    second pair reuses them and the larger inputs grow them)."""
    cfgs = [gen.cfg3(3000), gen.cfg0(8), gen.cfg3(20000, off=336, cnt=112), gen.cfg1(40)]
    ins = [host_logits(c) for c in cfgs]
    outs = [mr.route_host(x, dev_bias(c), synchronize=False, **kw(c)) for x, c in zip(ins, cfgs)]
    torch.cuda.synchronize()
    for c, x, o in zip(cfgs, ins, outs):
        ref = mr.route(x.cuda(), dev_bias(c), **kw(c))
        torch.cuda.synchronize()
        for key in ("packed", "counts", "offsets", "perm"):
            assert torch.equal(o[key], ref[key].cpu()), key


def test_pageable_host_memory(mr):
    cfg = gen.cfg3(1000)
    x = host_logits(cfg, pin=False)
    out = {k: (torch.empty(v.shape, dtype=v.dtype) if v is not None else None)  # pageable
           for k, v in mr.alloc_host_outputs(1000, 896).items()}
    assert not x.is_pinned() and not out["perm"].is_pinned()
    mr.route_host(x, dev_bias(cfg), out=out, **kw(cfg))
    check_against_oracle(out, cfg)


def test_full_size_sampled(mr):
    """65,536 rows (the prefill workload): counts and offsets against the oracle's
    histogram of the host results' ids, sampled rows against the oracle."""
    T = 65536
    cfg = gen.cfg3(T)
    out = mr.route_host(host_logits(cfg), dev_bias(cfg), want_ids=True, **kw(cfg))
    ids = out["ids"].numpy()
    assert np.array_equal(out["counts"].numpy(), np.bincount(ids.ravel(), minlength=896))
    assert int(out["offsets"][-1]) == T * 16
    rows = np.unique(gen.raw64(77, 64) % np.uint64(T)).astype(np.int64)
    sub = dict(cfg, logits=cfg["logits"][rows], T=len(rows))
    ref = oracle.route_cfg(sub)
    assert np.array_equal(out["packed"].numpy()[rows], ref["packed"])
    perm = out["perm"].numpy()
    assert np.array_equal(np.sort(perm), np.arange(T * 16))


@pytest.mark.filterwarnings("ignore:The CUDA Graph is empty")
def test_rejects(mr):
    lib = mr.load()
    cfg = gen.cfg1(8)
    x = host_logits(cfg)
    b = dev_bias(cfg)
    out = mr.alloc_host_outputs(8, 896)
    s = torch.cuda.current_stream().cuda_stream
    P = lambda t: t.data_ptr()
    args = lambda E, ng: (P(x), 1, P(b), 8, E, 16, ng, 4, 2.5, 0, 0, P(out["packed"]),
                          P(out["counts"]), P(out["offsets"]), P(out["perm"]), None, s)
    assert lib.moe_route_host(*args(896, 5)) == mr.E_INVALID_ARG
    assert lib.moe_route_host(*args(900, 9)) == mr.E_UNSUPPORTED
    with pytest.raises(ValueError):
        mr.route_host(x.cuda(), b)
    # capture: refused, nothing enqueued
    g = torch.cuda.CUDAGraph()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        st.wait_stream(torch.cuda.current_stream())
        with torch.cuda.graph(g, stream=st):
            rc = lib.moe_route_host(*args(896, 8)[:-1], st.cuda_stream)
    assert rc == mr.E_UNSUPPORTED
    assert lib.moe_route_host_release() == 0
    out2 = mr.route_host(x, b, **kw(cfg))  # slots allocated again
    check_against_oracle(out2, cfg)
