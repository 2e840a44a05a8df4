"""The expert-GEMM layout (moe_route_layout) against the oracle, bit for bit.

The layout is built on the GPU from the GPU routing's own counts, offsets and perm,
and compared with the oracle's layout of those same arrays (the routing itself is
compared with the oracle's routing in test_gpu_route.py).
"""
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
    lg = torch.from_numpy(np.ascontiguousarray(cfg["logits"]).view(
        np.int16 if cfg["dtype"] == "bf16" else np.float32)).to(dev)
    if cfg["dtype"] == "bf16":
        lg = lg.view(torch.bfloat16)
    bias = torch.from_numpy(cfg["bias"]).to(dev)
    return mr.route(lg, bias, k=cfg["k"], n_group=cfg["G"], topk_group=cfg["Kg"], scale=cfg["scale"],
                    local_offset=cfg["off"], local_count=cfg["cnt"])


def check_layout(mr, out, tile):
    L = mr.route_layout(out, tile)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    counts, offsets, perm = (out[k].cpu().numpy() for k in ("counts", "offsets", "perm"))
    ref = oracle.route_layout(counts, offsets, perm, tile, capacity=L["padded_rows"].numel())
    for key in ("inv_perm", "padded_offsets", "padded_rows", "m_indices"):
        got = L[key].cpu().numpy()
        assert np.array_equal(got, ref[key]), (key, np.nonzero(got != ref[key])[0][:8])
    return L, ref


CASES = {
    "decode8_local": lambda: gen.cfg1(8),
    "decode64_global": lambda: gen.cfg1(64, off=0, cnt=0),
    "prefill1001_global": lambda: gen.cfg3(1001),
    "prefill1001_local": lambda: gen.cfg3(1001, off=784, cnt=112),
    "ties4096_local": lambda: gen.cfg4(dtype="bf16", off=336, cnt=112),
}


@pytest.mark.parametrize("tile", [1, 8, 128])
@pytest.mark.parametrize("case", sorted(CASES))
def test_layout_matches_oracle(mr, case, tile):
    check_layout(mr, routed(mr, CASES[case]()), tile)


def test_layout_full_size(mr):
    """65,536 rows, global ids, tile 128: the size the benchmark times."""
    L, ref = check_layout(mr, routed(mr, gen.cfg3(65536)), 128)
    assert ref["total"] <= L["padded_rows"].numel()


def test_layout_empty(mr):
    """T = 0: every padded offset is 0 and every row is padding."""
    cfg = gen.cfg1(8)
    dev = torch.device("cuda")
    out = mr.alloc_outputs(0, 896, 16, 112, dev)
    lg = torch.zeros((0, 896), dtype=torch.bfloat16, device=dev)
    mr.route(lg, torch.from_numpy(cfg["bias"]).to(dev), local_offset=336, local_count=112, out=out)
    L = mr.route_layout(out, 8)
    torch.cuda.synchronize()
    assert torch.all(L["padded_offsets"] == 0)
    assert torch.all(L["padded_rows"] == -1) and torch.all(L["m_indices"] == -1)
    assert L["inv_perm"].numel() == 0


def test_layout_partial_outputs(mr):
    """Any subset of the outputs may be asked for; the others are left alone."""
    out = routed(mr, gen.cfg1(16))
    full = mr.route_layout(out, 16)
    only_inv = mr.route_layout(out, 16, padded=False)
    only_pad = mr.route_layout(out, 16, inv=False)
    torch.cuda.synchronize()
    assert torch.equal(full["inv_perm"], only_inv["inv_perm"])
    for key in ("padded_offsets", "padded_rows", "m_indices"):
        assert torch.equal(full[key], only_pad[key])


def test_layout_rejects(mr):
    out = routed(mr, gen.cfg1(8))
    lib = mr.load()
    P = lambda t: t.data_ptr()  # noqa: E731
    s = torch.cuda.current_stream().cuda_stream
    rows = torch.empty(100, dtype=torch.int32, device="cuda")
    NE = out["counts"].numel()
    call = lambda tile, cap: lib.moe_route_layout(  # noqa: E731
        P(out["counts"]), P(out["offsets"]), P(out["perm"]), 8, 16, NE, tile, None, None,
        P(rows), None, cap, s)
    assert call(0, 100) == mr.E_INVALID_ARG
    assert call(8, 100) == mr.E_INVALID_ARG          # below 128 + 128 * 7
    assert lib.moe_route_padded_capacity(8, 16, 128, 8) == 8 * 16 + 128 * 7
    assert lib.moe_route_padded_capacity(-1, 16, 128, 8) == mr.E_INVALID_ARG


def test_layout_in_graph(mr):
    """Routing and layout captured in one CUDA graph and replayed."""
    cfg = gen.cfg1(32)
    dev = torch.device("cuda")
    lg = torch.from_numpy(cfg["logits"].view(np.int16)).to(dev).view(torch.bfloat16)
    bias = torch.from_numpy(cfg["bias"]).to(dev)
    out = mr.alloc_outputs(32, 896, 16, 112, dev)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        mr.route(lg, bias, local_offset=336, local_count=112, out=out)
        L = mr.route_layout(out, 64)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            mr.route(lg, bias, local_offset=336, local_count=112, out=out)
            mr.route_layout(out, 64, layout=L)
    for v in list(out.values()) + list(L.values()):
        if v is not None:
            v.fill_(-7)
    g.replay()
    torch.cuda.synchronize()
    o = oracle.route_cfg(cfg)
    ref = oracle.route_layout(o["counts"], o["offsets"], o["perm"], 64, capacity=L["padded_rows"].numel())
    for key in ("inv_perm", "padded_offsets", "padded_rows", "m_indices"):
        assert np.array_equal(L[key].cpu().numpy(), ref[key]), key


@pytest.mark.parametrize("cfg,path", [
    (gen.cfg1(8), 0), (gen.cfg1(64, off=0, cnt=0), 0),           # decode kernel
    (gen.cfg3(3000), 0), (gen.cfg3(3001, off=784, cnt=112), 0),  # approximate-score kernel
    (gen.cfg3(3000, off=336, cnt=112), 3),                        # exact-score kernel
    (gen.cfg4(T=2048, off=112, cnt=112), 0),                      # float32 logits (exact kernel)
    (gen.cfg_decision_edges("plateau", 1500), 0),                 # slow extraction path
], ids=["decode8_local", "decode64", "fast3000", "fast3001_local", "exact3000_local", "f32_2048",
        "plateau"])
def test_routing_writes_the_inverse(mr, cfg, path):
    """moe_route_ex's inv_perm is the inverse of its perm and equals the oracle layout's
    inverse of that perm; the other outputs equal moe_route's."""
    dev = torch.device("cuda")
    lg = torch.from_numpy(np.ascontiguousarray(cfg["logits"]).view(
        np.int16 if cfg["dtype"] == "bf16" else np.float32)).to(dev)
    if cfg["dtype"] == "bf16":
        lg = lg.view(torch.bfloat16)
    bias = torch.from_numpy(cfg["bias"]).to(dev)
    prev = mr.set_path(path)
    try:
        ex = mr.route(lg, bias, local_offset=cfg["off"], local_count=cfg["cnt"], want_inv=True,
                      want_ids=True)
        plain = mr.route(lg, bias, local_offset=cfg["off"], local_count=cfg["cnt"], want_ids=True)
    finally:
        mr.set_path(prev)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    for key in ("packed", "counts", "offsets", "perm", "ids"):
        assert torch.equal(ex[key], plain[key]), key
    perm = ex["perm"].cpu().numpy()
    inv = ex["inv_perm"].cpu().numpy()
    assert np.array_equal(perm[inv], np.arange(perm.size, dtype=np.int32))
    ref = oracle.route_layout(ex["counts"].cpu().numpy(), ex["offsets"].cpu().numpy(), perm, tile=1)
    assert np.array_equal(inv, ref["inv_perm"])


WITH_LAYOUT_CASES = {
    "decode8_local": (lambda: gen.cfg1(8), 0),
    "prefill1001_global": (lambda: gen.cfg3(1001), 0),
    "prefill1001_local": (lambda: gen.cfg3(1001, off=784, cnt=112), 0),
    "prefill1001_local_exact": (lambda: gen.cfg3(1001, off=784, cnt=112), 3),
    "prefill40000_global": (lambda: gen.cfg3(40000), 0),
    "prefill65536_local": (lambda: gen.cfg3(65536, off=336, cnt=112), 0),
    "ties4096_f32_local": (lambda: gen.cfg4(dtype="f32", off=336, cnt=112), 0),
}


@pytest.mark.parametrize("tile", [1, 64, 128])
@pytest.mark.parametrize("case", sorted(WITH_LAYOUT_CASES))
def test_route_with_layout(mr, case, tile):
    """moe_route_with_layout: the same routing, and the layout that moe_route_layout builds
    from it (the bf16 prefill kernel writes the layout itself; the other paths run the
    layout kernel after routing), equal to the oracle's layout of the routing's arrays."""
    make, path = WITH_LAYOUT_CASES[case]
    cfg = make()
    prev = mr.set_path(path)
    try:
        ref = routed(mr, cfg)
        dev = torch.device("cuda")
        lg = torch.from_numpy(np.ascontiguousarray(cfg["logits"]).view(
            np.int16 if cfg["dtype"] == "bf16" else np.float32)).to(dev)
        if cfg["dtype"] == "bf16":
            lg = lg.view(torch.bfloat16)
        bias = torch.from_numpy(cfg["bias"]).to(dev)
        got = mr.route(lg, bias, k=cfg["k"], n_group=cfg["G"], topk_group=cfg["Kg"], scale=cfg["scale"],
                       local_offset=cfg["off"], local_count=cfg["cnt"], layout_tile=tile)
        torch.cuda.synchronize()
    finally:
        mr.set_path(prev)
    assert mr.device_status() == 0
    for key in ("packed", "counts", "offsets", "perm"):
        assert torch.equal(got[key], ref[key]), key
    counts, offsets, perm = (ref[k].cpu().numpy() for k in ("counts", "offsets", "perm"))
    want = oracle.route_layout(counts, offsets, perm, tile, capacity=got["padded_rows"].numel())
    for key in ("padded_offsets", "padded_rows", "m_indices"):
        g = got[key].cpu().numpy()
        assert np.array_equal(g, want[key]), (key, np.nonzero(g != want[key])[0][:8])
