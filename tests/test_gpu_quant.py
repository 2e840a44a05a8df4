"""The fused route+quant decode launch (moe_route_quant) against the oracle: routing
outputs as moe_route's (bit-exact), MXFP4 codes and E8M0 scales of the activations
bit-exact against the oracle's quantiser (the OCP Microscaling v1.0 MXFP4 reading), at
T = 1..64, on normal activations, every bf16 bit pattern, exact rounding ties and
saturating values."""
import ctypes

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


def dev_bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def logits_dev(cfg):
    if cfg["dtype"] == "bf16":
        return dev_bf16(cfg["logits"])
    return torch.from_numpy(np.ascontiguousarray(cfg["logits"], dtype=np.float32)).cuda()


def check(mr, cfg, x_bits):
    lg = logits_dev(cfg)
    bias = torch.from_numpy(cfg["bias"]).cuda()
    out = mr.route_quant(lg, bias, dev_bf16(x_bits), local_offset=cfg["off"],
                         local_count=cfg["cnt"], want_ids=True)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    q = oracle.mxfp4_quant(x_bits)
    got_q, got_s = out["x_q"].cpu().numpy(), out["x_scales"].cpu().numpy()
    bad = np.nonzero(got_q != q["q"])
    assert bad[0].size == 0, (bad[0][:4], bad[1][:4], got_q[bad][:4], q["q"][bad][:4])
    assert np.array_equal(got_s, q["scales"])
    g = {k: v.cpu().numpy() for k, v in out.items() if k not in ("x_q", "x_scales")}
    parity.compare(g, oracle.route_cfg(cfg), cfg, exact=cfg["dtype"] == "bf16")
    ref = mr.route(lg, bias, local_offset=cfg["off"], local_count=cfg["cnt"], want_ids=True)
    torch.cuda.synchronize()
    for key in ("packed", "counts", "offsets", "perm", "ids"):
        assert torch.equal(out[key], ref[key]), key


@pytest.mark.parametrize("T", [1, 2, 7, 8, 16, 24, 33, 64])
def test_route_quant_normal(mr, T):
    check(mr, gen.cfg1(T), gen.mx_activations(T))


@pytest.mark.parametrize("kind", ["patterns", "ties"])
@pytest.mark.parametrize("T", [5, 64])
def test_route_quant_edge_values(mr, kind, T):
    check(mr, gen.cfg1(T, off=0, cnt=0), gen.mx_activations(T, kind=kind))


def test_route_quant_f32_logits_other_width(mr):
    cfg = gen.cfg0()
    check(mr, cfg, gen.mx_activations(8, H=4096, kind="ties"))


@pytest.mark.parametrize("T,H", [(64, 32), (64, 21504), (3, 28672)])
def test_route_quant_quantising_clusters(mr, T, H):
    """The quantisation runs on the clusters after the routing cluster, as many as give
    every quantising warp at most one pass: one quantising cluster with a single short
    step in all (64 rows of 32), three quantising clusters of 16 CTAs (64 rows of
    21,504), three one-CTA quantising clusters beside a one-CTA routing cluster (3 rows
    of 28,672)."""
    check(mr, gen.cfg1(T), gen.mx_activations(T, H=H))


def test_route_quant_empty_and_errors(mr):
    lib = mr.load()
    cfg = gen.cfg1(8)
    lg = logits_dev(cfg)
    bias = torch.from_numpy(cfg["bias"]).cuda()
    x = dev_bf16(gen.mx_activations(65, H=256))
    out = mr.alloc_outputs(65, 896, 16, 0, lg.device)
    xq = torch.empty((65, 128), dtype=torch.uint8, device="cuda")
    xs = torch.empty((65, 8), dtype=torch.uint8, device="cuda")
    P = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())  # noqa: E731
    st = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call(T=8, H=256, xp=None, qp=None):
        return lib.moe_route_quant(P(lg), 1, P(bias), T, 896, 16, 8, 4, 2.5, 0, 0,
                                   xp if xp is not None else P(x), H,
                                   qp if qp is not None else P(xq), P(xs), P(out["packed"]),
                                   P(out["counts"]), P(out["offsets"]), P(out["perm"]), None, st)

    assert call(T=65) == mr.E_UNSUPPORTED
    assert call(H=100) == mr.E_INVALID_ARG
    assert call(H=0) == mr.E_INVALID_ARG
    assert call(xp=ctypes.c_void_p(x.data_ptr() + 2)) == mr.E_INVALID_ARG
    assert call(qp=ctypes.c_void_p(xq.data_ptr() + 1)) == mr.E_INVALID_ARG
    assert call(qp=ctypes.c_void_p(xq.data_ptr() + 2)) == mr.E_INVALID_ARG
    out["counts"].fill_(-1)
    assert call(T=0) == mr.OK
    torch.cuda.synchronize()
    assert torch.all(out["counts"] == 0)
    assert mr.device_status() == 0


def test_route_quant_graph_replay(mr):
    cfg = gen.cfg1(24)
    xb = gen.mx_activations(24)
    lg = logits_dev(cfg)
    bias = torch.from_numpy(cfg["bias"]).cuda()
    x = dev_bf16(xb)
    out = mr.route_quant(lg, bias, x, local_offset=336, local_count=112)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        st.wait_stream(torch.cuda.current_stream())
        mr.route_quant(lg, bias, x, local_offset=336, local_count=112, out=out, stream=st)
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            mr.route_quant(lg, bias, x, local_offset=336, local_count=112, out=out, stream=st)
    out["x_q"].fill_(0)
    out["x_scales"].fill_(0)
    g.replay()
    torch.cuda.synchronize()
    q = oracle.mxfp4_quant(xb)
    assert np.array_equal(out["x_q"].cpu().numpy(), q["q"])
    assert np.array_equal(out["x_scales"].cpu().numpy(), q["scales"])
