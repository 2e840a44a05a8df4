"""Parity of the CUDA routing path (through the C ABI) with the CPU oracle."""
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


def to_dev(cfg):
    dev = torch.device("cuda")
    lg = cfg["logits"]
    if cfg["dtype"] == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(lg).view(np.int16)).to(dev).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(lg, dtype=np.float32)).to(dev)
    return t, torch.from_numpy(np.ascontiguousarray(cfg["bias"], dtype=np.float32)).to(dev)


def run_gpu(mr, cfg, path=0, want_ids=True):
    lg, bias = to_dev(cfg)
    prev = mr.set_path(path)
    try:
        out = mr.route(lg, bias, k=cfg["k"], n_group=cfg["G"], topk_group=cfg["Kg"],
                       scale=cfg["scale"], local_offset=cfg.get("off", 0),
                       local_count=cfg.get("cnt", 0), want_ids=want_ids)
    finally:
        mr.set_path(prev)
    torch.cuda.synchronize()
    assert mr.device_status() == 0
    return {k: (None if v is None else v.cpu().numpy()) for k, v in out.items()}


def check(mr, cfg, exact, path=0):
    g = run_gpu(mr, cfg, path=path)
    o = oracle.route_cfg(cfg)
    rep = parity.compare(g, o, cfg, exact=exact)
    print(rep)
    return g, o, rep


# ----------------------------------------------------------------- step a1
def test_sigmoid_bf16_every_value(mr):
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    xs = gen.bf16_bits_to_f32(bits)
    bits = bits[np.isfinite(xs)]
    x = torch.from_numpy(bits.view(np.int16)).cuda().view(torch.bfloat16)
    got = mr.sigmoid(x).cpu().numpy()
    want = oracle.sigmoid(bits, "bf16")
    bad = np.nonzero(got.view(np.uint32) != want.view(np.uint32))[0]
    assert bad.size == 0, (bad[:5], xs[np.isfinite(xs)][bad[:5]])


def test_sigmoid_f32_within_1ulp(mr):
    """float32 logits: within one ulp of the oracle everywhere, equal almost everywhere."""
    x = np.concatenate([gen.uniform_f32(11, 1 << 20, -40.0, 40.0), gen.normal_f32(12, 1 << 20),
                        gen.normal_f32(13, 1 << 18) * np.float32(1e-4),
                        gen.uniform_f32(14, 1 << 16, -104.0, -80.0),
                        gen.uniform_f32(18, 1 << 16, 60.0, 200.0),
                        gen.cfg_f32_edges("bits", 64)["logits"].ravel()]).astype(np.float32)
    got = mr.sigmoid(torch.from_numpy(x).cuda()).cpu().numpy()
    want = oracle.sigmoid(x, "f32")
    d = np.abs(got.view(np.int32).astype(np.int64) - want.view(np.int32).astype(np.int64))
    frac_exact = float((d == 0).mean())
    print("f32 sigmoid: max ulp", int(d.max()), "fraction exact", frac_exact)
    bad = np.nonzero(d)[0]
    if bad.size:
        import oracle_pins
        for i in bad[:: max(1, bad.size // 12)][:12]:
            exact, near = oracle_pins.exact_sigmoid_f32(float(x[i]))
            print(f"x={x[i]!r} gpu={got[i]!r} oracle={want[i]!r} exact={exact!r} near_mid={near}")
        ranges = np.histogram(x[bad], bins=[-200, -87.4, -20, -1, -1e-3, 0, 1e-3, 1, 20, 200])[0]
        print("mismatches by x range", ranges.tolist())
    assert d.max() <= 1
    assert frac_exact >= 0.9999


# ------------------------------------------------------------- full routing
def test_cfg0_smallest(mr):
    check(mr, gen.cfg0(), exact=False)


@pytest.mark.parametrize("T", [5, 6, 7, 8, 9, 16, 17, 24, 32, 41, 57, 63, 64])  # 1..16 CTAs, ragged splits
@pytest.mark.parametrize("local", [True, False])
def test_cfg1_decode_sweep(mr, T, local):
    cfg = gen.cfg1(T) if local else gen.cfg1(T, off=0, cnt=0)
    check(mr, cfg, exact=True)


@pytest.mark.parametrize("T", [1, 2, 7, 33, 64])
def test_decode_and_persistent_paths_agree(mr, T):
    cfg = gen.cfg1(T)
    a = run_gpu(mr, cfg, path=1)
    b = run_gpu(mr, cfg, path=2)
    for key in ("packed", "counts", "offsets", "perm", "ids"):
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("T", [65, 1001, 16384])
@pytest.mark.parametrize("off,cnt", [(0, 0), (784, 112)])
def test_cfg3_prefill(mr, T, off, cnt):
    check(mr, gen.cfg3(T, off=off, cnt=cnt), exact=True)


@pytest.mark.parametrize("off,cnt", [(0, 0), (784, 112)])
def test_cfg3_full_size(mr, off, cnt):
    """65,536 rows, the launch the benchmark times; every row against the oracle."""
    check(mr, gen.cfg3(65536, off=off, cnt=cnt), exact=True)


@pytest.mark.parametrize("off", [0, 112, 224, 336, 448, 560, 672, 784])
def test_cfg4_ties_every_rank_bf16(mr, off):
    cfg = gen.cfg4(dtype="bf16", off=off, cnt=112)
    check(mr, cfg, exact=True)


@pytest.mark.parametrize("off,cnt", [(0, 0), (336, 112)])
def test_cfg4_ties_f32(mr, off, cnt):
    cfg = gen.cfg4(off=off, cnt=cnt)
    g, o, rep = check(mr, cfg, exact=False)
    # hot rows: 16 equal hot experts with zero bias -> weights 2.5/16 exactly where all 16 win
    assert rep["mismatched_rows"] <= rep.get("near_tie_rows", 0)


@pytest.mark.parametrize("T,path", [(64, 1), (3000, 2)])
@pytest.mark.parametrize("off,cnt", [(0, 0), (448, 112)])
def test_every_bf16_magnitude(mr, T, path, off, cnt):
    """bf16 logits over all finite bit patterns (zeros, subnormals, magnitudes below
    2^-26 and above 112, both signs) reach the clamped score-table lookups of the row
    routine on both paths; many exact ties in b."""
    check(mr, gen.cfg_bf16_patterns(T, off=off, cnt=cnt), exact=True, path=path)


@pytest.mark.parametrize("T,paths", [(8, (1, 4)), (64, (1, 4)), (3000, (2, 3))])
@pytest.mark.parametrize("kind", ["cfg0", "cfg4", "bits", "ulps"])
def test_f32_approximate_scores_agree(mr, T, paths, kind):
    """float32 logits: routing that starts from approximate scores (paths 1 and 2) equals
    routing that computes every score exactly (paths 4 and 3), on the decode and the
    persistent kernel, including logits where the score saturates and experts whose
    scores differ by less than the approximation's error bound."""
    if kind == "cfg0":
        cfg = dict(gen.cfg0(max(T, 8)))
    elif kind == "cfg4":
        cfg = gen.cfg4(T=T, off=336, cnt=112)
    else:
        cfg = gen.cfg_f32_edges(kind, T)
    a = run_gpu(mr, cfg, path=paths[0])
    b = run_gpu(mr, cfg, path=paths[1])
    for key in ("packed", "counts", "offsets", "perm", "ids"):
        assert np.array_equal(a[key], b[key]), key


@pytest.mark.parametrize("kind", ["bits", "ulps"])
def test_f32_edges_oracle(mr, kind):
    check(mr, gen.cfg_f32_edges(kind, 3000, off=784, cnt=112), exact=False)


def test_t_zero(mr):
    cfg = gen.cfg1(8)
    lg, bias = to_dev(cfg)
    for path in (1, 2):
        prev = mr.set_path(path)
        out = mr.alloc_outputs(0, 896, 16, 112, lg.device)
        out["counts"].fill_(-7)
        out["offsets"].fill_(-7)
        mr.route(lg[:0], bias, local_offset=336, local_count=112, out=out)
        mr.set_path(prev)
        assert torch.all(out["counts"] == 0) and torch.all(out["offsets"] == 0)


def test_rows_are_independent(mr):
    """Routing rows in pieces gives the rows of routing them together."""
    cfg = gen.cfg3(3000)
    whole = run_gpu(mr, cfg)
    pieces = []
    for lo, hi in ((0, 64), (64, 1000), (1000, 1001), (1001, 3000)):
        sub = dict(cfg, logits=cfg["logits"][lo:hi], T=hi - lo)
        pieces.append(run_gpu(mr, sub)["packed"])
    assert np.array_equal(np.concatenate(pieces), whole["packed"])


@pytest.mark.parametrize("Kg,k", [(1, 16), (2, 16), (8, 16), (4, 1), (4, 8), (4, 32), (3, 24)])
def test_group_and_k_variants(mr, Kg, k):
    """Other topk_group / k: exercises the pool sizes and the exact slow path."""
    for cfg in (gen.cfg1(64, off=336, cnt=112), gen.cfg3(700), gen.cfg4(T=512, dtype="bf16")):
        cfg = dict(cfg, Kg=Kg, k=k)
        check(mr, cfg, exact=True)


def test_invalid_and_unsupported(mr):
    cfg = gen.cfg1(8)
    lg, bias = to_dev(cfg)
    lib = mr.load()
    out = mr.alloc_outputs(8, 896, 16, 0, lg.device)
    P = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    s = torch.cuda.current_stream().cuda_stream

    def call(E=896, k=16, G=8, Kg=4, off=0, cnt=0, T=8, logits=lg):
        return lib.moe_route(P(logits), 1, P(bias), T, E, k, G, Kg, 2.5, off, cnt, P(out["packed"]),
                             P(out["counts"]), P(out["offsets"]), P(out["perm"]), None, s)

    assert call(G=5) == mr.E_INVALID_ARG
    assert call(Kg=0) == mr.E_INVALID_ARG
    assert call(Kg=9) == mr.E_INVALID_ARG
    assert call(k=0) == mr.E_INVALID_ARG
    assert call(off=800, cnt=112) == mr.E_INVALID_ARG
    assert call(cnt=-1) == mr.E_INVALID_ARG
    assert call(T=-1) == mr.E_INVALID_ARG
    assert call(k=33, Kg=8) == mr.E_UNSUPPORTED
    assert call(E=256, G=8) == mr.E_UNSUPPORTED
    assert lib.moe_route(P(lg) + 2, 1, P(bias), 8, 896, 16, 8, 4, 2.5, 0, 0, P(out["packed"]),
                         P(out["counts"]), P(out["offsets"]), P(out["perm"]), None, s) == \
        mr.E_INVALID_ARG
    assert call() == mr.OK
    torch.cuda.synchronize()
    assert mr.device_status() == 0


def test_graph_capture_and_replay(mr):
    cfg = gen.cfg1(16)
    lg, bias = to_dev(cfg)
    out = mr.alloc_outputs(16, 896, 16, 112, lg.device, want_ids=True)
    st = torch.cuda.Stream()
    with torch.cuda.stream(st):
        mr.route(lg, bias, local_offset=336, local_count=112, out=out)  # warm
        st.synchronize()
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=st):
            mr.route(lg, bias, local_offset=336, local_count=112, out=out)
    for v in out.values():
        v.fill_(-1)
    g.replay()
    torch.cuda.synchronize()
    o = oracle.route_cfg(cfg)
    parity.compare({k: v.cpu().numpy() for k, v in out.items()}, o, cfg, exact=True)
