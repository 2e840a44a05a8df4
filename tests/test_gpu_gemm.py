"""Fused router contraction + routing (moe_router_gemm_route) against the oracle.

Logits: |gpu - ref| <= 1e-3 * max(|ref|, 1e-2 * max_row |ref|), ref accumulated in
double.  Routing: the oracle router applied to the GPU's own float32 logits must give
the GPU's packed ids, counts, offsets and permutation bit for bit.
"""
import numpy as np
import pytest
import torch

import gen
import oracle
import parity

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def mr():
    import serving_moe_route_02_gb300 as mr
    mr.load()
    mr.reserve()
    return mr


@pytest.fixture(scope="module")
def weight():
    cfg = gen.cfg2(1)
    return cfg["w"], torch.from_numpy(cfg["w"].view(np.int16)).cuda()


def logits_close(got, ref):
    scale = np.maximum(np.abs(ref), 1e-2 * np.abs(ref).max(axis=1, keepdims=True))
    err = np.abs(got.astype(np.float64) - ref) / scale
    return float(err.max())


@pytest.mark.parametrize("T", [1, 4, 8, 16, 32, 64])
@pytest.mark.parametrize("off,cnt", [(0, 0), (0, 112)])
def test_router_gemm_route(mr, weight, T, off, cnt):
    w_np, w_dev = weight
    cfg = gen.cfg2(T, off=off, cnt=cnt)
    hid = torch.from_numpy(cfg["hidden"].view(np.int16)).cuda()
    bias = torch.from_numpy(cfg["bias"]).cuda()
    out = mr.router_gemm_route(hid, w_dev, bias, local_offset=off, local_count=cnt, want_ids=True)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    logits = out["logits"].cpu().numpy()
    ref = oracle.router_gemm(cfg["hidden"], w_np)
    rel = logits_close(logits, ref)
    print(f"T={T} max relative logit error {rel:.2e}")
    assert rel <= 1e-3
    rcfg = dict(logits=logits, dtype="f32", bias=cfg["bias"], T=T, E=896, k=16, G=8, Kg=4,
                scale=2.5, off=off, cnt=cnt)
    o = oracle.route_cfg(rcfg)
    g = {k: v.cpu().numpy() for k, v in out.items() if v is not None and k != "logits"}
    parity.compare(g, o, rcfg, exact=True)


@pytest.mark.parametrize("H", [1024, 2048, 14336, 21504])
def test_router_gemm_hidden_sizes(mr, H):
    """Hidden sizes other than 7168: one 64-column block per CTA (1024), a ring of two
    stages (2048), and K slices longer than the ring, refilled once (14336) and twice
    (21504) as the MMAs free its stages; row counts that are not multiples of 4 or 16."""
    cfg0 = gen.cfg2(1, H=H)
    w_dev = torch.from_numpy(cfg0["w"].view(np.int16)).cuda()
    for T in (1, 17, 64):
        cfg = gen.cfg2(T, H=H)
        hid = torch.from_numpy(cfg["hidden"].view(np.int16)).cuda()
        bias = torch.from_numpy(cfg["bias"]).cuda()
        out = mr.router_gemm_route(hid, w_dev, bias, want_ids=True)
        torch.cuda.synchronize()
        assert mr.device_status() == 0
        logits = out["logits"].cpu().numpy()
        ref = oracle.router_gemm(cfg["hidden"], cfg0["w"])
        rel = logits_close(logits, ref)
        print(f"H={H} T={T} max relative logit error {rel:.2e}")
        assert rel <= 1e-3
        rcfg = dict(logits=logits, dtype="f32", bias=cfg["bias"], T=T, E=896, k=16, G=8, Kg=4,
                    scale=2.5, off=0, cnt=0)
        o = oracle.route_cfg(rcfg)
        g = {k: v.cpu().numpy() for k, v in out.items() if v is not None and k != "logits"}
        parity.compare(g, o, rcfg, exact=True)


def test_router_gemm_without_logits_out(mr, weight):
    w_np, w_dev = weight
    cfg = gen.cfg2(16)
    hid = torch.from_numpy(cfg["hidden"].view(np.int16)).cuda()
    bias = torch.from_numpy(cfg["bias"]).cuda()
    a = mr.router_gemm_route(hid, w_dev, bias, want_logits=True)
    b = mr.router_gemm_route(hid, w_dev, bias, want_logits=False)
    torch.cuda.synchronize()
    for key in ("packed", "counts", "offsets", "perm"):
        assert torch.equal(a[key], b[key]), key


def test_router_gemm_rejects(mr, weight):
    _, w_dev = weight
    hid = torch.zeros((65, 7168), dtype=torch.int16, device="cuda")
    bias = torch.zeros(896, dtype=torch.float32, device="cuda")
    with pytest.raises(mr.MoeRouteError) as e:
        mr.router_gemm_route(hid, w_dev, bias)
    assert e.value.status == mr.E_UNSUPPORTED
    # H / 64 = 15 blocks: not a multiple of the K-split count (16, or 8)
    hid = torch.zeros((8, 960), dtype=torch.int16, device="cuda")
    w = torch.zeros((896, 960), dtype=torch.int16, device="cuda")
    with pytest.raises(mr.MoeRouteError) as e:
        mr.router_gemm_route(hid, w, bias)
    assert e.value.status == mr.E_UNSUPPORTED
    torch.cuda.synchronize()
    assert mr.device_status() == 0


def test_router_gemm_repeated_and_replayed(mr, weight):
    """Back-to-back calls chain the contraction and the routing as programmatic
    dependents: outputs cleared before each call come back whole, over calls of two batch
    shapes in turn on one stream and over replays of a captured graph of them."""
    _, w_dev = weight
    cases = []
    for T, off, cnt in ((8, 0, 0), (24, 0, 112)):
        cfg = gen.cfg2(T, off=off, cnt=cnt)
        hid = torch.from_numpy(cfg["hidden"].view(np.int16)).cuda()
        bias = torch.from_numpy(cfg["bias"]).cuda()
        ref = mr.router_gemm_route(hid, w_dev, bias, local_offset=off, local_count=cnt, want_ids=True)
        torch.cuda.synchronize()
        ref = {k: v.clone() for k, v in ref.items() if v is not None}
        out = mr.alloc_outputs(T, 896, 16, cnt, hid.device, True)
        out["logits"] = torch.empty((T, 896), dtype=torch.float32, device=hid.device)
        cases.append((hid, bias, off, cnt, ref, out))

    def run(stream=None):
        for i in range(6):
            hid, bias, off, cnt, _, out = cases[i % 2]
            for v in out.values():
                if v is not None:
                    v.fill_(-1)
            mr.router_gemm_route(hid, w_dev, bias, local_offset=off, local_count=cnt, out=out,
                                 want_ids=True, stream=stream)

    def check():
        torch.cuda.synchronize()
        assert mr.device_status() == 0
        for *_, ref, out in cases:
            for key, v in ref.items():
                assert torch.equal(out[key], v), key

    run()
    check()
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        st.wait_stream(torch.cuda.current_stream())
        run(st)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            run(st)
    for _ in range(3):
        for *_, out in cases:
            for v in out.values():
                if v is not None:
                    v.fill_(-7)
        torch.cuda.synchronize()
        g.replay()
        check()
