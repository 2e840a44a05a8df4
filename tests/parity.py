"""Helpers that compare the CUDA routing path with the CPU oracle.

Acceptance (the stated bar for this path):
  * packed ids, counts, offsets and perm bit-exact wherever the oracle's decision
    margins exceed 4 float32 ulp; rows with a smaller margin ("near-tie" rows) are
    counted and reported;
  * bf16 weights within 1 bf16 ulp;
  * counts / offsets / perm always bit-exact against the oracle's histogram, scan and
    stable permutation applied to the GPU's own packed ids (numpy bincount, cumsum and
    stable argsort, which the oracle's pins tie to the oracle).

Near-tie reading: a row is near-tie if any of these gaps is at most 4 ulp, where ulp is
taken at the larger magnitude of the two compared values and of their unbiased scores:
(i) the k-th vs (k+1)-th biased score among kept experts, (ii) two adjacent biased
scores inside the top-k (they fix slot order), (iii) the topk_group-th vs the next
group score.  Equal values that come from identical (logit, bias) inputs are not
near-ties: both sides compute the same number and the tie-break decides.
"""
from __future__ import annotations

import numpy as np

import gen
import oracle

ULPS = 4


def logits_np(cfg) -> np.ndarray:
    return np.ascontiguousarray(cfg["logits"])


def oracle_scores(cfg):
    s = oracle.sigmoid(cfg["logits"], cfg["dtype"])
    b = (s + cfg["bias"].astype(np.float32)[None, :]).astype(np.float32)
    return s, b


def _ulp(x):
    return np.spacing(np.abs(np.asarray(x, np.float32))).astype(np.float64)


def near_tie_rows(cfg) -> np.ndarray:
    """Boolean [T]: rows whose decisions have a margin of at most 4 ulp."""
    T, E, G, Kg, k = cfg["T"], cfg["E"], cfg["G"], cfg["Kg"], cfg["k"]
    gsz = E // G
    s, b = oracle_scores(cfg)
    x = np.asarray(cfg["logits"]).reshape(T, E)
    bias = cfg["bias"].astype(np.float32)
    near = np.zeros(T, dtype=bool)
    eidx = np.arange(E)
    for t in range(T):
        row = b[t]
        # group scores and the kept-set margin (iii)
        gb = row.reshape(G, gsz)
        top = np.argsort(-gb.astype(np.float64), axis=1, kind="stable")[:, :3]
        g1 = gb[np.arange(G), top[:, 0]]
        g2 = gb[np.arange(G), top[:, 1]]
        gs = (g1 + g2).astype(np.float32)
        gorder = np.lexsort((np.arange(G), -gs.astype(np.float64)))
        if Kg < G:
            a, c = gorder[Kg - 1], gorder[Kg]
            gap = abs(float(gs[a]) - float(gs[c]))
            u = max(_ulp(gs[a]), _ulp(gs[c]))
            same = (np.array_equal(np.sort(x[t, a * gsz + top[a, :2]]), np.sort(x[t, c * gsz + top[c, :2]]))
                    and np.array_equal(np.sort(bias[a * gsz + top[a, :2]]), np.sort(bias[c * gsz + top[c, :2]])))
            if gap <= ULPS * u and not same:
                near[t] = True
                continue
            # a 2nd/3rd swap inside a group changes its score
            for g in (a, c):
                d = abs(float(gb[g, top[g, 1]]) - float(gb[g, top[g, 2]]))
                if d <= ULPS * max(_ulp(gb[g, top[g, 1]]), _ulp(gb[g, top[g, 2]])):
                    i1, i2 = g * gsz + top[g, 1], g * gsz + top[g, 2]
                    if not (x[t, i1] == x[t, i2] and bias[i1] == bias[i2]):
                        near[t] = True
        if near[t]:
            continue
        kept = np.sort(gorder[:Kg])
        cand = eidx[np.isin(eidx // gsz, kept)]
        order = cand[np.lexsort((cand, -row[cand].astype(np.float64)))]
        pairs = [(order[j], order[j + 1]) for j in range(min(k, len(order) - 1))]
        for i1, i2 in pairs:
            gap = abs(float(row[i1]) - float(row[i2]))
            u = max(_ulp(row[i1]), _ulp(row[i2]), _ulp(s[t, i1]), _ulp(s[t, i2]))
            if gap <= ULPS * u and not (x[t, i1] == x[t, i2] and bias[i1] == bias[i2]):
                near[t] = True
                break
    return near


def unpack(packed: np.ndarray):
    p = np.asarray(packed).astype(np.int64) & 0xFFFFFFFF
    return (p >> 16).astype(np.int64), (p & 0xFFFF).astype(np.int64)


def derived_from_packed(packed: np.ndarray, NE: int):
    lid, _ = unpack(packed)
    flat = lid.ravel()
    counts = np.bincount(flat, minlength=NE).astype(np.int32)
    offsets = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    perm = np.argsort(flat, kind="stable").astype(np.int32)
    return counts, offsets, perm


def compare(gpu: dict, orc: dict, cfg: dict, exact: bool) -> dict:
    """Asserts the acceptance bar; returns a report.  exact=True demands every row
    bit-exact (bf16 logits: the GPU scores are the oracle's scores)."""
    T, k = cfg["T"], cfg["k"]
    NE = orc["NE"]
    gp = np.asarray(gpu["packed"]).reshape(T, k)
    op = orc["packed"]
    glid, gw = unpack(gp)
    olid, ow = unpack(op)
    row_bad = np.any(gp != op, axis=1)
    rep = dict(T=T, mismatched_rows=int(row_bad.sum()))
    # counts / offsets / perm: always exact vs the GPU's own packed ids
    c2, o2, p2 = derived_from_packed(gp, NE)
    assert np.array_equal(np.asarray(gpu["counts"]), c2), "counts != histogram of GPU packed ids"
    assert np.array_equal(np.asarray(gpu["offsets"]), o2), "offsets != scan of GPU counts"
    assert np.array_equal(np.asarray(gpu["perm"]), p2), "perm != stable order of GPU packed ids"
    if exact:
        assert not row_bad.any(), f"{int(row_bad.sum())} rows differ: first {np.nonzero(row_bad)[0][:8]}"
        assert np.array_equal(np.asarray(gpu["counts"]), orc["counts"])
        assert np.array_equal(np.asarray(gpu["offsets"]), orc["offsets"])
        assert np.array_equal(np.asarray(gpu["perm"]), orc["perm"])
        if gpu.get("ids") is not None:
            assert np.array_equal(np.asarray(gpu["ids"]).reshape(T, k), orc["ids"])
        rep["near_tie_rows"] = None
        return rep
    near = near_tie_rows(cfg) if row_bad.any() else np.zeros(T, bool)
    rep["near_tie_rows"] = int(near.sum()) if row_bad.any() else 0
    # ids bit-exact on all non-near-tie rows
    bad_ids = np.any(glid != olid, axis=1)
    if gpu.get("ids") is not None:
        bad_ids |= np.any(np.asarray(gpu["ids"]).reshape(T, k) != orc["ids"], axis=1)
    assert not np.any(bad_ids & ~near), f"id mismatch outside near-tie rows: {np.nonzero(bad_ids & ~near)[0][:8]}"
    # weights within 1 bf16 ulp where ids agree
    same = ~bad_ids
    dw = np.abs(gw[same] - ow[same])  # same sign (positive): bit distance = ulp distance
    assert dw.size == 0 or dw.max() <= 1, f"weight differs by {dw.max()} bf16 ulp"
    rep["max_weight_ulp"] = int(dw.max()) if dw.size else 0
    if not row_bad.any():
        assert np.array_equal(np.asarray(gpu["counts"]), orc["counts"])
        assert np.array_equal(np.asarray(gpu["offsets"]), orc["offsets"])
        assert np.array_equal(np.asarray(gpu["perm"]), orc["perm"])
    return rep
