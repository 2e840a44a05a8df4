"""The persistent kernel on approximate scores (bf16 logits, k = 16, keep 4 groups: the
kernel moe_route runs for prefill batches of the Kimi-K3 instance) against the oracle and
against the persistent kernel that computes every score exactly (path 3), on inputs that
drive each decision onto its hardest path: equal and nearly equal group scores (exact
group scores from the table), 33 to 64 experts within the approximation's error band
of the cutoff (the 64-key sort), more than 64 experts sharing the k-th score (the slow
extraction), negative biased scores (no 32-bit keys), large biases (a wider error
bound), and rows where every score ties."""
import numpy as np
import pytest
import torch

import gen
import oracle
import parity

pytestmark = pytest.mark.gpu

KINDS = ("flat", "group_copy", "group_near", "negative", "large_bias", "plateau", "band")
KEYS = ("packed", "counts", "offsets", "perm", "ids")


@pytest.fixture(scope="module")
def mr():
    import serving_moe_route_02_gb300 as mr
    mr.load()
    mr.reserve()
    return mr


def run(mr, cfg, path):
    dev = torch.device("cuda")
    lg = torch.from_numpy(np.ascontiguousarray(cfg["logits"]).view(np.int16)).to(dev).view(torch.bfloat16)
    bias = torch.from_numpy(np.ascontiguousarray(cfg["bias"], dtype=np.float32)).to(dev)
    prev = mr.set_path(path)
    try:
        out = mr.route(lg, bias, local_offset=cfg["off"], local_count=cfg["cnt"], want_ids=True)
    finally:
        mr.set_path(prev)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    return {k: v.cpu().numpy() for k, v in out.items()}


def check_both(mr, cfg):
    fast = run(mr, cfg, path=2)
    exact = run(mr, cfg, path=3)
    for key in KEYS:
        assert np.array_equal(fast[key], exact[key]), key
    rep = parity.compare(fast, oracle.route_cfg(cfg), cfg, exact=True)
    print(rep)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("off,cnt", [(0, 0), (784, 112)])
def test_decision_edges(mr, kind, off, cnt):
    check_both(mr, gen.cfg_decision_edges(kind, 3000, off=off, cnt=cnt))


@pytest.mark.parametrize("T", [65, 2432, 2433, 9999, 40000])
def test_prefill_sizes(mr, T):
    """Ragged splits over the CTAs and warps (2,432 = 152 CTAs x 16 warps)."""
    check_both(mr, gen.cfg3(T, off=336, cnt=112))


@pytest.mark.parametrize("off,cnt", [(0, 0), (448, 112)])
def test_every_bf16_magnitude(mr, off, cnt):
    check_both(mr, gen.cfg_bf16_patterns(3000, off=off, cnt=cnt))


def test_ties_every_rank(mr):
    for off in (0, 336, 784):
        check_both(mr, gen.cfg4(dtype="bf16", off=off, cnt=112))


def test_graph_replay_twice(mr):
    """Captured once, replayed twice: the grid barrier words return to their start state."""
    cfg = gen.cfg3(5000)
    dev = torch.device("cuda")
    lg = torch.from_numpy(cfg["logits"].view(np.int16)).to(dev).view(torch.bfloat16)
    bias = torch.from_numpy(cfg["bias"]).to(dev)
    out = mr.alloc_outputs(5000, 896, 16, 0, dev, want_ids=True)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        mr.route(lg, bias, out=out, stream=st)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            mr.route(lg, bias, out=out, stream=st)
    ref = oracle.route_cfg(cfg)
    for _ in range(2):
        for v in out.values():
            v.fill_(-1)
        g.replay()
        torch.cuda.synchronize()
        assert mr.device_status() == 0
        parity.compare({k: v.cpu().numpy() for k, v in out.items()}, ref, cfg, exact=True)
