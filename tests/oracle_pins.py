"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes a loaded oracle library (ctypes) and raises
AssertionError when the oracle disagrees with:
  * the exact sigmoid (mpmath at 100 bits, rounded correctly to float32),
  * torch's float32 -> bfloat16 conversion (library routine),
  * a brute-force full sort of every row (group scores, group choice, top-k),
  * numpy's stable argsort / bincount / cumsum for histogram, scan, permutation,
  * closed forms (equal scores give weights 2.5/16 = 0x3E20 in bf16),
  * exact rational renormalisation (fractions),
  * invariants stated for the method (unique ids, ids inside kept groups,
    counts summing to T*k, perm a permutation, weights summing to the scale,
    rank-local ids unique, < count+k, round-tripping to the global ids),
  * facts printed on the pages (num_experts 128 at EP8, router size),
  * for the expert-GEMM layout: numpy's argsort (inverse permutation), numpy.repeat
    (unpadded row index), a padded layout built by appending entries and padding,
    and its invariants.
The same functions are run against deliberately broken copies of the oracle in
test_oracle_mutations.py to show that each plausible mistake is caught.
"""
from __future__ import annotations

import math
import os
from fractions import Fraction

import numpy as np

import gen
import oracle

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# --------------------------------------------------------------------- helpers

def exact_sigmoid_f32(x: float):
    """(correctly rounded float32 of sigma(x), True if sigma(x) lies within 2^-44
    relative of a float32 rounding midpoint), via mpmath at 120 bits."""
    import mpmath
    with mpmath.workprec(120):
        v = 1 / (1 + mpmath.exp(-mpmath.mpf(float(x))))
        f = np.float32(float(v))
        best, bd = None, None
        cands = (np.nextafter(f, np.float32(-np.inf)), f, np.nextafter(f, np.float32(np.inf)))
        for c in cands:
            d = abs(mpmath.mpf(float(c)) - v)
            if bd is None or d < bd:
                best, bd = c, d
        # distance to the nearest midpoint between best and a neighbour
        lo = mpmath.mpf(float(np.nextafter(best, np.float32(-np.inf))))
        hi = mpmath.mpf(float(np.nextafter(best, np.float32(np.inf))))
        b = mpmath.mpf(float(best))
        dm = min(abs(v - (b + lo) / 2), abs(v - (b + hi) / 2))
        near_mid = bool(dm <= abs(v) * mpmath.mpf(2) ** -44)
        return np.float32(best), near_mid


def lib_sigmoid(lib, x: np.ndarray) -> np.ndarray:
    return np.array([lib.oracle_sigmoid(float(v)) for v in np.asarray(x, np.float32).ravel()],
                    dtype=np.float32).reshape(np.shape(x))


def logits_f32(cfg) -> np.ndarray:
    if cfg["dtype"] == "f32":
        return np.asarray(cfg["logits"], np.float32)
    return gen.bf16_bits_to_f32(cfg["logits"])


def brute_force_rows(x: np.ndarray, s: np.ndarray, bias: np.ndarray, G: int, Kg: int, k: int):
    """Full-sort reference of the selection: returns (ids [T,k], kept groups [T,Kg])."""
    T, E = x.shape
    gsz = E // G
    b = (s.astype(np.float32) + bias.astype(np.float32)[None, :]).astype(np.float32)
    ids = np.zeros((T, k), dtype=np.int64)
    kept_all = np.zeros((T, Kg), dtype=np.int64)
    for t in range(T):
        row = b[t]
        gs = []
        for g in range(G):
            top2 = sorted((float(v) for v in row[g * gsz:(g + 1) * gsz]), reverse=True)[:2]
            gs.append(np.float32(np.float32(top2[0]) + np.float32(top2[1])))
        order = sorted(range(G), key=lambda g: (-float(gs[g]), g))
        kept = sorted(order[:Kg])
        cand = [e for e in range(E) if e // gsz in kept]
        cand.sort(key=lambda e: (-float(row[e]), e))
        ids[t] = cand[:k]
        kept_all[t] = kept
    return ids, kept_all


def unpack(packed: np.ndarray):
    p = packed.astype(np.int64) & 0xFFFFFFFF
    return (p >> 16).astype(np.int64), (p & 0xFFFF).astype(np.uint16)


def run(lib, cfg, off=None, cnt=None):
    return oracle.route(cfg["logits"], cfg["dtype"], cfg["bias"], cfg["T"], cfg["E"], cfg["k"],
                        cfg["G"], cfg["Kg"], cfg["scale"],
                        cfg.get("off", 0) if off is None else off,
                        cfg.get("cnt", 0) if cnt is None else cnt, lib=lib)


def small_cfg(T, E, G, Kg, k, seed, levels=5, bias_levels=(0.0, 0.25, -0.25), dtype="f32",
              scale=2.5):
    """Tiny instance with many exact ties: logits on a small integer grid."""
    r = gen.raw64(1000 + seed, T * E)
    x = ((r % np.uint64(levels)).astype(np.int64) - levels // 2).astype(np.float32) * 0.5
    rb = gen.raw64(2000 + seed, E)
    bias = np.array(bias_levels, dtype=np.float32)[(rb % np.uint64(len(bias_levels))).astype(np.int64)]
    logits = x.reshape(T, E)
    if dtype == "bf16":
        logits = gen.f32_to_bf16_bits(logits)
    return dict(logits=logits, dtype=dtype, bias=bias, T=T, E=E, k=k, G=G, Kg=Kg, scale=scale,
                off=0, cnt=0)


# ------------------------------------------------------------------------ pins

def pin_sigmoid_exact(lib, n_random: int = 4000):
    """The oracle's sigmoid (double evaluation, one rounding to float) equals the
    correctly rounded value on every finite bf16 input below 20 in magnitude, a
    sparse sample beyond, and random float32 inputs -- except where sigma(x) lies
    within 2^-44 of a float32 midpoint, where double rounding may pick either
    neighbour; there it must be within one ulp.  sigma(0) = 0.5."""
    assert lib.oracle_sigmoid(0.0) == 0.5
    bits = np.arange(0, 1 << 16, dtype=np.uint32).astype(np.uint16)
    xs = gen.bf16_bits_to_f32(bits)
    xs = xs[np.isfinite(xs)]
    core = xs[(np.abs(xs) < 20.0)]
    rest = xs[(np.abs(xs) >= 20.0)][::97]
    rnd = gen.uniform_f32(77, n_random, -30.0, 30.0)
    n_mid = 0
    for x in np.concatenate([core, rest, rnd]):
        got = np.float32(lib.oracle_sigmoid(float(x)))
        want, near_mid = exact_sigmoid_f32(float(x))
        if near_mid:
            n_mid += 1
            assert abs(float(got) - float(want)) <= float(np.spacing(want)), float(x)
        else:
            assert got == want, (float(x), float(got), float(want))
    # the midpoint zone is a small set (tiny |x|, where sigma(x) ~ 1/2 + x/4)
    assert n_mid < 400, n_mid


def pin_sigmoid_symmetry(lib):
    """sigma(-x) = 1 - sigma(x): checked in exact arithmetic within one ulp of each."""
    xs = gen.uniform_f32(78, 2000, -12.0, 12.0)
    for x in xs:
        a = Fraction(float(lib.oracle_sigmoid(float(x))))
        b = Fraction(float(lib.oracle_sigmoid(float(-x))))
        ulp = Fraction(float(np.spacing(np.float32(max(a, b)))))
        assert abs(a + b - 1) <= ulp, float(x)


def pin_bf16_rounding(lib):
    import torch
    vals = np.concatenate([
        gen.uniform_f32(79, 5000, -3.0, 3.0),
        gen.normal_f32(80, 5000) * np.float32(1e-3),
        # exact halfway cases between two bf16 values (ties to even)
        gen.bf16_bits_to_f32(np.arange(0x3F00, 0x3F40, dtype=np.uint16)) *
        np.float32(1.0 + 2.0 ** -8),
        np.array([0.15625, 2.5, 1.0, 0.0, -0.0, 1e-30, 3.0e38], dtype=np.float32),
    ]).astype(np.float32)
    want = torch.from_numpy(vals).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([lib.oracle_f32_to_bf16(float(v)) for v in vals], dtype=np.uint16)
    assert np.array_equal(got, want)


def pin_selection_brute_force(lib):
    """Tiny shapes with many ties: ids and slot order equal a full sort per row."""
    cases = [
        (8, 2, 1, 2), (8, 2, 2, 3), (8, 4, 2, 2), (16, 4, 2, 4), (16, 8, 3, 4), (16, 1, 1, 4),
        (32, 4, 2, 4), (32, 8, 4, 16), (32, 2, 1, 16), (64, 8, 4, 16), (64, 16, 5, 8),
    ]
    for i, (E, G, Kg, k) in enumerate(cases):
        cfg = small_cfg(T=40, E=E, G=G, Kg=Kg, k=k, seed=i)
        out = run(lib, cfg)
        x = logits_f32(cfg)
        ids_bf, _ = brute_force_rows(x, lib_sigmoid(lib, x), cfg["bias"], G, Kg, k)
        assert np.array_equal(out["ids"], ids_bf), (E, G, Kg, k)
        lid, _ = unpack(out["packed"])
        assert np.array_equal(lid, ids_bf)


def pin_selection_exhaustive(lib):
    """E=8, 2 groups of 4, keep 1 group, top 2: every logit vector in {-1,0,1}^8."""
    E, G, Kg, k = 8, 2, 1, 2
    grid = np.array(np.meshgrid(*([np.array([-1.0, 0.0, 1.0], np.float32)] * E), indexing="ij"))
    x = grid.reshape(E, -1).T.copy().astype(np.float32)
    bias = np.array([0.0, 0.0, 0.25, -0.25, 0.0, 0.25, 0.0, -0.25], dtype=np.float32)
    cfg = dict(logits=x, dtype="f32", bias=bias, T=x.shape[0], E=E, k=k, G=G, Kg=Kg, scale=2.5)
    out = run(lib, cfg)
    ids_bf, _ = brute_force_rows(x, lib_sigmoid(lib, x), bias, G, Kg, k)
    assert np.array_equal(out["ids"], ids_bf)


def pin_selection_kimi_shape(lib):
    """Kimi shape (896, 8 groups, keep 4, top 16) on tie-heavy rows: full-sort reference."""
    cfg = gen.cfg4(T=48, n_hot=12)
    out = run(lib, cfg)
    x = logits_f32(cfg)
    ids_bf, kept = brute_force_rows(x, lib_sigmoid(lib, x), cfg["bias"], cfg["G"], cfg["Kg"],
                                    cfg["k"])
    assert np.array_equal(out["ids"], ids_bf)
    cfg0 = gen.cfg0()
    out0 = run(lib, cfg0)
    x0 = logits_f32(cfg0)
    ids0, _ = brute_force_rows(x0, lib_sigmoid(lib, x0), cfg0["bias"], 8, 4, 16)
    assert np.array_equal(out0["ids"], ids0)


def pin_plain_topk(lib):
    """One group, keep it: the method reduces to plain top-k (numpy lexsort)."""
    cfg = small_cfg(T=64, E=32, G=1, Kg=1, k=8, seed=91)
    out = run(lib, cfg)
    x = logits_f32(cfg)
    b = (lib_sigmoid(lib, x) + cfg["bias"][None, :]).astype(np.float32)
    for t in range(cfg["T"]):
        order = np.lexsort((np.arange(32), -b[t].astype(np.float64)))
        assert np.array_equal(out["ids"][t], order[:8])


def pin_keep_all_groups_is_noop(lib):
    """Keeping every group gives the same ids as a single group of all experts."""
    base = small_cfg(T=64, E=64, G=8, Kg=8, k=16, seed=92)
    a = run(lib, base)
    one = dict(base, G=1, Kg=1)
    b = run(lib, one)
    assert np.array_equal(a["ids"], b["ids"])


def pin_weights(lib):
    """Weights: within one bf16 ulp of the exact rational s_j / sum(s) * scale; they sum
    to the scale within 1e-2; equal scores give 2.5/16 = 0.15625 = bf16 0x3E20."""
    for cfg in (gen.cfg0(), small_cfg(T=32, E=64, G=8, Kg=4, k=16, seed=93)):
        out = run(lib, cfg)
        x = logits_f32(cfg)
        s = lib_sigmoid(lib, x)
        _, wb = unpack(out["packed"])
        w = gen.bf16_bits_to_f32(wb).astype(np.float64)
        assert np.all(np.abs(w.sum(axis=1) - cfg["scale"]) <= 1e-2)
        for t in range(cfg["T"]):
            sel = [Fraction(float(s[t, e])) for e in out["ids"][t]]
            den = sum(sel)
            for j, sj in enumerate(sel):
                exact = sj / den * Fraction(cfg["scale"])
                ulp = Fraction(2) ** (math.frexp(float(exact))[1] - 8)
                assert abs(Fraction(float(w[t, j])) - exact) <= ulp, (t, j)
    # closed form: 16 equal chosen scores (identical logits, zero bias, one group) -> 5/32
    E = 896
    x = np.full((2, E), -4.0, np.float32)
    x[:, 112:128] = 3.0
    cfg = dict(logits=x, dtype="f32", bias=np.zeros(E, np.float32), T=2, E=E, k=16, G=8, Kg=4,
               scale=2.5)
    out = run(lib, cfg)
    _, wb = unpack(out["packed"])
    assert np.all(wb == 0x3E20)
    assert np.array_equal(out["ids"][0], np.arange(112, 128))


def pin_histogram_scan_perm(lib):
    """counts = bincount, offsets = [0, cumsum], perm = stable argsort of the ids."""
    for cfg in (gen.cfg0(), gen.cfg1(24), gen.cfg4(T=200, n_hot=50, off=336, cnt=112),
                small_cfg(T=50, E=32, G=4, Kg=2, k=4, seed=94)):
        out = run(lib, cfg)
        lid, _ = unpack(out["packed"])
        flat = lid.ravel()
        NE = out["NE"]
        assert np.array_equal(out["counts"], np.bincount(flat, minlength=NE))
        assert np.array_equal(out["offsets"], np.concatenate([[0], np.cumsum(out["counts"])]))
        assert np.array_equal(out["perm"], np.argsort(flat, kind="stable"))


def check_invariants(out, cfg, kept_groups=None):
    T, k, E, G = cfg["T"], cfg["k"], cfg["E"], cfg["G"]
    off, cnt = cfg.get("off", 0), cfg.get("cnt", 0)
    gsz = E // G
    ids = out["ids"]
    lid, wb = unpack(out["packed"])
    for t in range(T):
        assert len(set(ids[t].tolist())) == k
        if kept_groups is not None:
            assert set((ids[t] // gsz).tolist()) <= set(kept_groups[t].tolist())
        assert len(set(lid[t].tolist())) == k
    assert out["counts"].sum() == T * k
    assert out["offsets"][-1] == T * k and np.all(np.diff(out["offsets"]) >= 0)
    assert np.array_equal(np.sort(out["perm"]), np.arange(T * k))
    w = gen.bf16_bits_to_f32(wb).astype(np.float64)
    assert np.all(np.abs(w.sum(axis=1) - cfg["scale"]) <= 1e-2)
    NE = out["NE"]
    assert np.all(lid < NE)
    if cnt > 0:
        # num_experts: a multiple of 4 covering count + top_k, and nothing more
        assert NE % 4 == 0 and cnt + k <= NE < cnt + k + 4
        assert np.all(lid < cnt + k) and np.all(out["counts"][cnt + k:] == 0)
        # round trip: local id -> global id
        back = np.where(lid < cnt, lid + off,
                        np.take_along_axis(ids, np.clip(lid - cnt, 0, k - 1), axis=1))
        assert np.array_equal(back, ids)
        # rank-local ids of other ranks' experts sit in the slot they occupy
        other = lid >= cnt
        assert np.array_equal((lid - cnt)[other], np.nonzero(other)[1])
    else:
        assert np.array_equal(lid, ids)


def pin_invariants(lib):
    for cfg in (gen.cfg0(), gen.cfg1(64), gen.cfg4(T=256, n_hot=64, cnt=112, off=448),
                gen.cfg3(96, off=784, cnt=112), gen.cfg1(16, off=101, cnt=30),
                gen.cfg1(9, off=0, cnt=113), small_cfg(T=40, E=32, G=4, Kg=2, k=4, seed=95)):
        out = run(lib, cfg)
        x = logits_f32(cfg)
        _, kept = brute_force_rows(x, lib_sigmoid(lib, x), cfg["bias"], cfg["G"], cfg["Kg"],
                                   cfg["k"])
        check_invariants(out, cfg, kept)


def pin_rank_local_matrix(lib):
    """The page's test matrix: EP 2/8/16, first/middle/last rank, 1..64 tokens.  Local
    ids are valid and round-trip, and the global outputs do not change."""
    E, k = 896, 16
    full = gen.cfg1(64, off=0, cnt=0)
    g_out = run(lib, full)
    for ep in (2, 8, 16):
        cnt = E // ep
        for rank in (0, ep // 2, ep - 1):
            off = rank * cnt
            for T in (1, 2, 7, 16, 33, 64):
                cfg = gen.cfg1(T, off=off, cnt=cnt)
                out = run(lib, cfg)
                check_invariants(out, cfg)
                assert np.array_equal(out["ids"], g_out["ids"][:T])
                # entries of this rank's experts: same (token, slot, weight) in the same order
                glid, gw = unpack(g_out["packed"][:T])
                llid, lw = unpack(out["packed"])
                assert np.array_equal(gw, lw)
                gflat = glid.ravel()
                gperm = np.argsort(gflat, kind="stable")
                lperm = out["perm"]
                for e in range(cnt):
                    ge = gperm[gflat[gperm] == off + e]
                    le = lperm[out["offsets"][e]:out["offsets"][e + 1]]
                    assert np.array_equal(ge, le)


def pin_page_facts(lib):
    with open(os.path.join(GOLDEN, "page1_rank_local.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for E, k, ep, cnt, ne in ((int(v) for v in r) for r in rows):
        assert E // ep == cnt
        assert lib.oracle_num_experts(E, k, 3 * cnt, cnt) == ne
    assert lib.oracle_num_experts(896, 16, 0, 0) == 896
    with open(os.path.join(GOLDEN, "router_params.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for E, H, L, billions in rows:
        assert round(int(E) * int(H) * int(L) / 1e9, 2) == float(billions)


def pin_router_gemm(lib):
    """Double accumulation agrees with exact integer arithmetic on sampled outputs
    (bf16 values are dyadic rationals) and with numpy's float64 matmul."""
    T, H, E = 3, 256, 40
    hid = gen.f32_to_bf16_bits(gen.normal_f32(501, T * H).reshape(T, H))
    w = gen.f32_to_bf16_bits(gen.normal_f32(502, E * H, std=0.02).reshape(E, H))
    out = oracle.router_gemm(hid, w, lib=lib)
    hf = gen.bf16_bits_to_f32(hid).astype(np.float64)
    wf = gen.bf16_bits_to_f32(w).astype(np.float64)
    ref = hf @ wf.T
    assert np.allclose(out, ref, rtol=1e-12, atol=1e-12)
    for t, e in ((0, 0), (1, 17), (2, 39)):
        exact = sum(Fraction(float(hf[t, h])) * Fraction(float(wf[e, h])) for h in range(H))
        assert abs(Fraction(float(out[t, e])) - exact) <= abs(exact) * Fraction(1, 1 << 40) + \
            Fraction(1, 1 << 60)


def pin_rejects_invalid(lib):
    cfg = gen.cfg0()
    bad = [dict(G=5), dict(G=448, Kg=4, k=16), dict(Kg=0), dict(Kg=9), dict(k=113, Kg=1), dict(cnt=-1),
           dict(off=800, cnt=112)]
    for b in bad:
        c = dict(cfg, **b)
        try:
            run(lib, c)
        except ValueError:
            continue
        raise AssertionError(f"oracle accepted {b}")


def _layout_cases(lib):
    """Routing results the layout pins start from: decode, rank-local, ties, tiny."""
    for cfg in (gen.cfg1(8), gen.cfg1(64, off=0, cnt=0), gen.cfg4(T=300, n_hot=80, off=224, cnt=112),
                small_cfg(T=40, E=32, G=4, Kg=2, k=4, seed=95), small_cfg(T=1, E=8, G=2, Kg=1, k=2, seed=96)):
        out = run(lib, cfg)
        yield cfg, out


def layout(lib, out, tile, capacity=None):
    return oracle.route_layout(out["counts"], out["offsets"], out["perm"], tile, capacity, lib=lib)


def pin_layout_inverse(lib):
    """inv_perm is the inverse permutation: numpy's argsort of perm, and perm[inv] = id."""
    for _, out in _layout_cases(lib):
        L = layout(lib, out, 8)
        n = out["perm"].size
        assert np.array_equal(L["inv_perm"], np.argsort(out["perm"], kind="stable"))
        assert np.array_equal(out["perm"][L["inv_perm"]], np.arange(n))


def pin_layout_tile_one(lib):
    """tile = 1 is the unpadded layout: padded offsets = offsets, padded rows = perm,
    m_indices = numpy.repeat of the bins by their counts, nothing else written."""
    for _, out in _layout_cases(lib):
        n, NE = out["perm"].size, out["counts"].size
        L = layout(lib, out, 1, capacity=n + 5)
        assert L["total"] == n
        assert np.array_equal(L["padded_offsets"], out["offsets"])
        assert np.array_equal(L["padded_rows"][:n], out["perm"])
        assert np.array_equal(L["m_indices"][:n], np.repeat(np.arange(NE), out["counts"]))
        assert np.all(L["padded_rows"][n:] == -1) and np.all(L["m_indices"][n:] == -1)


def pin_layout_append(lib):
    """Padded layout built by a different method: append each bin's entries, then -1
    until the length is a multiple of the tile; pad to the capacity with -1."""
    for _, out in _layout_cases(lib):
        lid, _ = unpack(out["packed"])
        flat = lid.ravel()
        NE = out["counts"].size
        for tile in (2, 3, 8, 128):
            rows, mind, starts = [], [], []
            for e in range(NE):
                starts.append(len(rows))
                for x in range(flat.size):      # entries of bin e in (token, slot) order
                    if flat[x] == e:
                        rows.append(x)
                        mind.append(e)
                while len(rows) % tile:
                    rows.append(-1)
                    mind.append(-1)
            starts.append(len(rows))
            cap = len(rows) + 7
            L = layout(lib, out, tile, capacity=cap)
            assert L["total"] == len(rows)
            assert np.array_equal(L["padded_offsets"], np.array(starts))
            assert np.array_equal(L["padded_rows"], np.array(rows + [-1] * 7))
            assert np.array_equal(L["m_indices"], np.array(mind + [-1] * 7))


def pin_layout_invariants(lib):
    """Every block is the smallest multiple of the tile that holds its bin; a real padded
    row's entry carries the bin's id in its packed value; the padded total is within the
    bound n + NE (tile - 1) that callers size their buffers by."""
    for _, out in _layout_cases(lib):
        lid, _ = unpack(out["packed"])
        flat = lid.ravel()
        n, NE = flat.size, out["counts"].size
        for tile in (4, 16, 128):
            L = layout(lib, out, tile)
            size = np.diff(L["padded_offsets"])
            assert np.all(size % tile == 0)
            assert np.all(size >= out["counts"]) and np.all(size < out["counts"] + tile)
            assert L["total"] <= n + NE * (tile - 1)
            real = L["padded_rows"] >= 0
            assert real.sum() == n
            assert np.array_equal(flat[L["padded_rows"][real]], L["m_indices"][real])
            assert np.all(L["m_indices"][~real] == -1)


def pin_layout_rejects(lib):
    out = run(lib, gen.cfg1(8))
    for tile, cap in ((0, 1000), (8, 10)):
        try:
            layout(lib, out, tile, capacity=cap)
        except ValueError:
            continue
        raise AssertionError(f"layout accepted tile={tile} capacity={cap}")


def pin_route_index(lib):
    """Histogram, scan and stable permutation from packed values alone: numpy bincount,
    cumsum and stable argsort of the ids, for routing outputs and for arbitrary packed
    arrays (repeated ids in a row included); ids >= NE are rejected."""
    for cfg in (gen.cfg1(24), gen.cfg1(64, off=0, cnt=0), gen.cfg4(T=200, n_hot=50, off=336, cnt=112)):
        out = run(lib, cfg)
        r = oracle.route_index(out["packed"], out["NE"], lib=lib)
        for key in ("counts", "offsets", "perm"):
            assert np.array_equal(r[key], out[key]), key
    for seed, (T, k, NE) in enumerate(((1, 1, 1), (7, 3, 5), (50, 16, 128), (33, 8, 1056))):
        ids = (gen.raw64(3000 + seed, T * k) % np.uint64(NE)).astype(np.int64)
        packed = ((ids << 16) | 0x3E20).astype(np.int32).reshape(T, k)
        r = oracle.route_index(packed, NE, lib=lib)
        assert np.array_equal(r["counts"], np.bincount(ids, minlength=NE))
        assert np.array_equal(r["offsets"], np.concatenate([[0], np.cumsum(np.bincount(ids, minlength=NE))]))
        assert np.array_equal(r["perm"], np.argsort(ids, kind="stable"))
    bad = np.array([[5 << 16]], dtype=np.int32)
    try:
        oracle.route_index(bad, 5, lib=lib)
    except ValueError:
        return
    raise AssertionError("route_index accepted an id >= NE")


def pin_token_sharded(lib):
    """Rows are independent: routing contiguous token shards and gathering their packed
    values gives the full batch's packed values, and the index built from the gathered
    values is the full batch's counts, offsets and perm."""
    cfg = gen.cfg3(1000, off=784, cnt=112)
    full = run(lib, cfg)
    for R in (2, 3, 8):
        parts = []
        for r in range(R):
            lo, hi = 1000 * r // R, 1000 * (r + 1) // R
            sub = dict(cfg, logits=cfg["logits"][lo:hi], T=hi - lo)
            parts.append(run(lib, sub)["packed"])
        gathered = np.concatenate(parts)
        assert np.array_equal(gathered, full["packed"])
        r = oracle.route_index(gathered, full["NE"], lib=lib)
        for key in ("counts", "offsets", "perm"):
            assert np.array_equal(r[key], full[key]), (R, key)


def pin_dispatch_counts(lib):
    """Entries per destination rank = numpy bincount of id // (E / R); offsets = cumsum;
    with global-id routing they are the expert offsets sampled at the rank boundaries."""
    out = run(lib, gen.cfg3(500))
    ids = out["ids"].ravel()
    for R in (1, 2, 4, 7, 8, 16):
        d = oracle.dispatch_counts(ids, 896, R, lib=lib)
        ref = np.bincount(ids // (896 // R), minlength=R)
        assert np.array_equal(d["send_counts"], ref)
        assert np.array_equal(d["send_offsets"], np.concatenate([[0], np.cumsum(ref)]))
        assert np.array_equal(d["send_offsets"], out["offsets"][np.arange(R + 1) * (896 // R)])
    for bad in ((ids, 896, 5), (np.array([896]), 896, 8)):
        try:
            oracle.dispatch_counts(*bad, lib=lib)
        except ValueError:
            continue
        raise AssertionError(f"dispatch_counts accepted {bad[1:]}")


def pin_alltoall_layout(lib):
    """A hand-worked 3-rank case; numpy cumsum of the matrix row and column; what rank s
    sends to rank d is what rank d expects from rank s, for every pair."""
    m = np.arange(9, dtype=np.int32).reshape(3, 3)
    L = oracle.alltoall_layout(m, 1, lib=lib)
    assert L["send_displs"].tolist() == [0, 3, 7, 12]
    assert L["recv_counts"].tolist() == [1, 4, 7]
    assert L["recv_displs"].tolist() == [0, 1, 5, 12]
    R = 8
    m = (gen.raw64(3100, R * R) % np.uint64(1000)).astype(np.int32).reshape(R, R)
    lay = [oracle.alltoall_layout(m, me, lib=lib) for me in range(R)]
    for me in range(R):
        assert np.array_equal(lay[me]["send_displs"], np.concatenate([[0], np.cumsum(m[me])]))
        assert np.array_equal(lay[me]["recv_displs"], np.concatenate([[0], np.cumsum(m[:, me])]))
        for d in range(R):
            sent = lay[me]["send_displs"][d + 1] - lay[me]["send_displs"][d]
            assert sent == lay[d]["recv_counts"][me]
    assert sum(int(l["recv_displs"][-1]) for l in lay) == int(m.sum())


# ------------------------------------------------------------------ MXFP4 quantiser
# Pins of oracle_mxfp4_quant, the reading of the route+quant activation format taken
# from the OCP Microscaling (MX) v1.0 MXFP4 format: E2M1 elements (1 sign, 2 exponent
# bits with bias 1, 1 mantissa bit; exponent 0 is the subnormal range), 32-element
# blocks, an E8M0 shared scale 2^(floor(log2 amax) - 2), round to nearest with ties to
# the even code, saturation at the largest magnitude.

def e2m1_value(code: int) -> float:
    """Value of a 4-bit E2M1 code from its bit fields."""
    sign = -1.0 if code & 8 else 1.0
    ex, m = (code >> 1) & 3, code & 1
    mag = 0.5 * m if ex == 0 else 2.0 ** (ex - 1) * (1.0 + 0.5 * m)
    return sign * mag


def e2m1_by_thresholds(v: float) -> int:
    """Code by comparisons against the midpoints of consecutive magnitudes; at a midpoint
    the neighbour whose code ends in 0 wins, so the test is > below an odd code and >=
    below an even one."""
    a = abs(v)
    mag = (int(a > 0.25) + int(a >= 0.75) + int(a > 1.25) + int(a >= 1.75) + int(a > 2.5)
           + int(a >= 3.5) + int(a > 5.0))
    return (8 if np.signbit(v) else 0) | mag


def pin_e2m1_codes(lib):
    vals = [e2m1_value(c) for c in range(8)]
    assert vals == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    grid = np.concatenate([np.arange(0, 8.0, 1.0 / 64), [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0,
                                                        6.0, 7.999, 100.0, 1e30]])
    for v in grid:
        for sv in (float(v), -float(v)):
            got = oracle.e2m1_encode(sv, lib)
            assert got == e2m1_by_thresholds(sv), (sv, got)
            # nearest representable magnitude (saturating), brute force over the 8 codes
            a = min(abs(sv), 6.0)
            dist = [abs(a - abs(e2m1_value(c))) for c in range(8)]
            assert dist[got & 7] == min(dist), (sv, got)
    assert oracle.e2m1_encode(-0.0, lib) == 8 and oracle.e2m1_encode(0.0, lib) == 0
    assert oracle.e2m1_encode(-0.1, lib) == 8 and oracle.e2m1_encode(-7.0, lib) == 15


def _bf16(x):
    return gen.f32_to_bf16_bits(np.asarray(x, dtype=np.float32))


def pin_mx_scale(lib):
    rng = np.random.default_rng(21)
    for j in range(-130, 128, 3):
        # a block whose largest magnitude lies in [2^j, 2^(j+1)): scale exponent j - 2
        amax = np.float32(2.0 ** j * (1.0 + rng.random() * 0.99))
        if not np.isfinite(amax) or amax == 0:
            continue
        blk = (rng.random(32).astype(np.float32) * amax).astype(np.float32)
        blk[rng.integers(32)] = -amax
        xb = _bf16(blk).reshape(1, 32)
        real = float(np.abs(gen.bf16_bits_to_f32(xb)).max())
        if real == 0.0:
            continue
        want = min(max(int(np.floor(np.log2(real))) - 2, -127), 127)
        got = int(oracle.mxfp4_quant(xb, lib)["scales"][0, 0])
        assert got == want + 127, (j, real, got, want)
    zero = np.zeros((1, 32), np.uint16)
    zero[0, 5] = 0x8000  # -0
    r = oracle.mxfp4_quant(zero, lib)
    assert int(r["scales"][0, 0]) == 0 and int(r["q"][0, 2]) == 0x80
    big = np.full((1, 32), 0x7F7F, np.uint16)  # the largest bf16, 2^127 * (2 - 2^-7)
    assert int(oracle.mxfp4_quant(big, lib)["scales"][0, 0]) == 125 + 127


def pin_mx_roundtrip(lib):
    """Blocks of exact E2M1 multiples of 2^s with one element at +-4 or +-6 quantise to
    exactly those codes and that scale."""
    rng = np.random.default_rng(22)
    for trial in range(300):
        s = int(rng.integers(-120, 120))
        codes = rng.integers(0, 16, 32)
        codes[rng.integers(32)] = int(rng.choice([6, 7, 14, 15]))
        vals = np.array([e2m1_value(int(c)) * 2.0 ** s for c in codes], dtype=np.float32)
        xb = _bf16(vals).reshape(1, 32)
        assert np.array_equal(gen.bf16_bits_to_f32(xb).ravel(), vals)  # exact in bf16
        r = oracle.mxfp4_quant(xb, lib)
        assert int(r["scales"][0, 0]) == s + 127
        q = r["q"][0]
        got = np.empty(32, np.int64)
        got[0::2] = q & 0xF
        got[1::2] = q >> 4
        # +0 and -0 are the same value: compare values, and codes where nonzero
        deq = np.array([e2m1_value(int(c)) for c in got])
        want = np.array([e2m1_value(int(c)) for c in codes])
        assert np.array_equal(deq, want), trial
        nz = want != 0
        assert np.array_equal(got[nz], codes[nz]), trial


def pin_mx_nearest(lib):
    """Every element of random blocks is the nearest (saturating) multiple of the scale."""
    x = gen.f32_to_bf16_bits(gen.normal_f32(23, 8 * 256, std=3.0).reshape(8, 256))
    r = oracle.mxfp4_quant(x, lib)
    xf = gen.bf16_bits_to_f32(x).astype(np.float64)
    for t in range(8):
        for b in range(8):
            e = int(r["scales"][t, b]) - 127
            for i in range(32):
                byte = int(r["q"][t, b * 16 + i // 2])
                c = (byte >> 4) if i & 1 else (byte & 0xF)
                v = xf[t, b * 32 + i] / 2.0 ** e
                assert c == e2m1_by_thresholds(v), (t, b, i, v, c)


def pin_mx_layout(lib):
    """Element 2i in the low nibble of byte i of its block, block b at bytes 16b.., the
    scale of block b of row t at t * H / 32 + b."""
    H = 128
    x = np.zeros((2, H), np.float32)
    x[:, 0::32] = 6.0            # fixes every scale at 2^0
    x[1, 33] = 1.0               # row 1, block 1, element 1: high nibble of byte 16
    x[1, 66] = -0.5              # row 1, block 2, element 2: low nibble of byte 33
    x[0, 127] = 5.5              # row 0, block 3, element 31: high nibble of byte 63 (-> 6)
    r = oracle.mxfp4_quant(_bf16(x), lib)
    assert np.all(r["scales"] == 127)
    assert int(r["q"][1, 16]) == (0x2 << 4) | 0x7
    assert int(r["q"][1, 33]) == 0x9
    assert int(r["q"][0, 63]) == 0x7 << 4
    assert int(r["q"][0, 0]) == 0x7 and int(r["q"][0, 1]) == 0
    assert r["q"].shape == (2, H // 2) and r["scales"].shape == (2, H // 32)


ALL_PINS = [
    pin_sigmoid_exact, pin_sigmoid_symmetry, pin_bf16_rounding, pin_selection_brute_force,
    pin_selection_exhaustive, pin_selection_kimi_shape, pin_plain_topk, pin_keep_all_groups_is_noop,
    pin_weights, pin_histogram_scan_perm, pin_invariants, pin_rank_local_matrix, pin_page_facts,
    pin_router_gemm, pin_rejects_invalid, pin_layout_inverse, pin_layout_tile_one, pin_layout_append,
    pin_layout_invariants, pin_layout_rejects, pin_route_index, pin_token_sharded,
    pin_dispatch_counts, pin_alltoall_layout, pin_e2m1_codes, pin_mx_scale, pin_mx_roundtrip,
    pin_mx_nearest, pin_mx_layout,
]
