"""Seeded synthetic inputs for the MoE routing step.

This module only draws random numbers and lays them out; it holds none of the
routing arithmetic (no sigmoid, no selection, no renormalisation).  Both the
CPU oracle and the CUDA path consume exactly the arrays produced here.

Generator: SplitMix64 (Steele, Lea and Flood, "Fast splittable pseudorandom
number generators", OOPSLA 2014) used as a counter-based generator: draw i of
stream (seed, sub) is mix64(key(seed, sub) + (i + 1) * golden_gamma).
Uniforms keep the top 24 bits; normals use the Box-Muller transform in float64
and are rounded once to float32.  float64 log/cos come from numpy, so the last
bit of a normal draw may differ between CPU architectures; nothing stores a
generated input, every comparison regenerates both sides from the seed.

Workload shapes follow the Kimi-K3 routing described on the pages: 896 routed
experts, top_k 16, 8 groups of 112 (sglang PR #37, description: FlashInfer's
Tier<896, 16> specialisation, 112 experts per rank at EP8); hidden 7168 for the router
contraction.
"""
from __future__ import annotations

import numpy as np

E_KIMI = 896
K_KIMI = 16
G_KIMI = 8
KG_KIMI = 4
SCALE_KIMI = 2.5
H_KIMI = 7168

_GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)


def _mix64(z: np.ndarray) -> np.ndarray:
    z = z.copy()
    z ^= z >> np.uint64(30)
    z *= _M1
    z ^= z >> np.uint64(27)
    z *= _M2
    z ^= z >> np.uint64(31)
    return z


def raw64(seed: int, n: int, sub: int = 0) -> np.ndarray:
    """n raw 64-bit draws of stream (seed, sub)."""
    with np.errstate(over="ignore"):
        key = _mix64(np.array([(seed * 0x100000001B3 + sub * 0x632BE59BD9B4E019) & 0xFFFFFFFFFFFFFFFF],
                              dtype=np.uint64))[0]
        ctr = np.arange(1, n + 1, dtype=np.uint64) * _GAMMA + key
        return _mix64(ctr)


def uniform24(seed: int, n: int, sub: int = 0) -> np.ndarray:
    """n uniforms in [0, 1) with 24 random bits each (float64)."""
    return (raw64(seed, n, sub) >> np.uint64(40)).astype(np.float64) * (1.0 / (1 << 24))


def normal_f32(seed: int, n: int, mean: float = 0.0, std: float = 1.0, sub: int = 0) -> np.ndarray:
    """n normal draws (Box-Muller, float64) rounded once to float32."""
    r = raw64(seed, 2 * n, sub)
    u1 = ((r[0::2] >> np.uint64(40)).astype(np.float64) + 1.0) * (1.0 / (1 << 24))  # (0, 1]
    u2 = (r[1::2] >> np.uint64(40)).astype(np.float64) * (1.0 / (1 << 24))          # [0, 1)
    z = np.sqrt(-2.0 * np.log(u1)) * np.cos(2.0 * np.pi * u2)
    return (mean + std * z).astype(np.float32)


def uniform_f32(seed: int, n: int, lo: float, hi: float, sub: int = 0) -> np.ndarray:
    return (lo + (hi - lo) * uniform24(seed, n, sub)).astype(np.float32)


def permutation(seed: int, n: int, sub: int = 0) -> np.ndarray:
    """A seeded permutation of 0..n-1 (argsort of distinct 64-bit draws)."""
    return np.argsort(raw64(seed, n, sub), kind="stable").astype(np.int64)


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 to bfloat16 (nearest, ties to even); returns uint16 bit patterns.
    Inputs are finite by construction."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return (u >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(h: np.ndarray) -> np.ndarray:
    return (np.asarray(h, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


# --------------------------------------------------------------------------
# The five workloads (sizes and distributions as stated for the Kimi-K3 shape)
# --------------------------------------------------------------------------

def bias_standard(E: int = E_KIMI) -> np.ndarray:
    """Correction bias ~ U(-0.1, 0.1), seed 1."""
    return uniform_f32(1, E, -0.1, 0.1)


def cfg0(T: int = 8, E: int = E_KIMI) -> dict:
    """Smallest instance: fp32 logits ~N(0,1) seed 0, global ids."""
    return dict(logits=normal_f32(0, T * E).reshape(T, E), dtype="f32", bias=bias_standard(E),
                T=T, E=E, k=K_KIMI, G=G_KIMI, Kg=KG_KIMI, scale=SCALE_KIMI, off=0, cnt=0)


def cfg1(T: int, E: int = E_KIMI, off: int = 336, cnt: int = 112) -> dict:
    """Decode sweep: bf16 logits ~N(0,1) (first T rows of a 64-row draw, seed 0),
    rank-local ids for rank 3 of 8 (offset 336, count 112)."""
    assert 1 <= T <= 64
    full = normal_f32(0, 64 * E).reshape(64, E)
    return dict(logits=f32_to_bf16_bits(full[:T]), dtype="bf16", bias=bias_standard(E),
                T=T, E=E, k=K_KIMI, G=G_KIMI, Kg=KG_KIMI, scale=SCALE_KIMI, off=off, cnt=cnt)


def cfg2(T: int, H: int = H_KIMI, E: int = E_KIMI, off: int = 0, cnt: int = 0) -> dict:
    """Router contraction at decode: hidden bf16 ~N(0,1) seed 2, router weight
    bf16 ~N(0, 0.02) seed 3 (row e of the weight is expert e)."""
    hidden = f32_to_bf16_bits(normal_f32(2, T * H).reshape(T, H))
    w = f32_to_bf16_bits(normal_f32(3, E * H, std=0.02).reshape(E, H))
    return dict(hidden=hidden, w=w, bias=bias_standard(E), T=T, H=H, E=E, k=K_KIMI, G=G_KIMI,
                Kg=KG_KIMI, scale=SCALE_KIMI, off=off, cnt=cnt)


def zipf_offsets(E: int = E_KIMI) -> np.ndarray:
    """Per-expert popularity offset 0.5*ln(r^-1.1) = -0.55*ln(r), r = 1 + position of
    the expert in a seeded permutation (seed 5)."""
    perm = permutation(5, E)
    rank = np.empty(E, dtype=np.float64)
    rank[perm] = np.arange(1, E + 1, dtype=np.float64)
    return -0.55 * np.log(rank)


def cfg3(T: int, E: int = E_KIMI, off: int = 0, cnt: int = 0) -> dict:
    """Prefill scale: bf16 logits = RNE(N(0,1) seed 4 + Zipf popularity offset)."""
    z = normal_f32(4, T * E).reshape(T, E).astype(np.float64) + zipf_offsets(E)[None, :]
    return dict(logits=f32_to_bf16_bits(z.astype(np.float32)), dtype="bf16", bias=bias_standard(E),
                T=T, E=E, k=K_KIMI, G=G_KIMI, Kg=KG_KIMI, scale=SCALE_KIMI, off=off, cnt=cnt)


def cfg4(T: int = 4096, E: int = E_KIMI, off: int = 0, cnt: int = 0, dtype: str = "f32",
         n_hot: int | None = None) -> dict:
    """Adversarial ties: logits j/64 for integer j uniform in [-128, 128] (seed 6);
    a seeded quarter of the rows (seed 7) put logit 3.0 on a fixed 16-expert hot set
    inside one seeded group (seed 7); the bias of a seeded half of the experts
    (seed 8) is zero."""
    G = G_KIMI
    gsz = E // G
    j = (raw64(6, T * E) % np.uint64(257)).astype(np.int64) - 128
    logits = (j.astype(np.float64) / 64.0).astype(np.float32).reshape(T, E)
    n_hot = T // 4 if n_hot is None else n_hot
    hot_rows = permutation(7, T, sub=1)[:n_hot]
    hot_group = int(raw64(7, 1, sub=2)[0] % np.uint64(G))
    hot_experts = hot_group * gsz + permutation(7, gsz, sub=3)[:K_KIMI]
    logits[np.ix_(hot_rows, hot_experts)] = 3.0
    bias = bias_standard(E)
    bias[permutation(8, E)[: E // 2]] = 0.0
    out = dict(logits=logits, dtype="f32", bias=bias, T=T, E=E, k=K_KIMI, G=G, Kg=KG_KIMI,
               scale=SCALE_KIMI, off=off, cnt=cnt, hot_rows=np.sort(hot_rows),
               hot_experts=np.sort(hot_experts), hot_group=hot_group)
    if dtype == "bf16":
        out["logits"] = f32_to_bf16_bits(logits)
        out["dtype"] = "bf16"
    return out


def cfg_bf16_patterns(T: int, E: int = E_KIMI, off: int = 0, cnt: int = 0, seed: int = 9) -> dict:
    """bf16 logits drawn uniformly over bit patterns (seed 9), non-finite patterns made
    finite by clearing the top exponent bit: zeros, subnormals, magnitudes far below and
    far above the range where the score varies, both signs."""
    h = (raw64(seed, T * E) >> np.uint64(48)).astype(np.uint16)
    inf_nan = (h & np.uint16(0x7F80)) == np.uint16(0x7F80)
    h[inf_nan] ^= np.uint16(0x4000)
    return dict(logits=h.reshape(T, E), dtype="bf16", bias=bias_standard(E), T=T, E=E, k=K_KIMI,
                G=G_KIMI, Kg=KG_KIMI, scale=SCALE_KIMI, off=off, cnt=cnt)


def cfg_f32_edges(kind: str, T: int, E: int = E_KIMI, off: int = 0, cnt: int = 0) -> dict:
    """float32 inputs at the edges of the approximate float32 scores:
      bits   logits drawn uniformly over finite float32 bit patterns (seed 15): zeros,
             subnormals, magnitudes where the score is 0 or 1 (many exact ties), both signs;
      ulps   N(0,1) logits (seed 16) with 64 seeded experts per row (seed 17) at 2.5 plus
             0..63 float steps and a zero bias, so that their biased scores differ by less
             than the approximation's error bound.
    """
    bias = bias_standard(E)
    if kind == "bits":
        u = (raw64(15, T * E) >> np.uint64(32)).astype(np.uint32)
        nonfinite = (u & np.uint32(0x7F800000)) == np.uint32(0x7F800000)
        u[nonfinite] ^= np.uint32(0x40000000)
        logits = u.view(np.float32).reshape(T, E)
    elif kind == "ulps":
        logits = normal_f32(16, T * E).reshape(T, E)
        cols = (raw64(17, T * 64) % np.uint64(E)).astype(np.int64).reshape(T, 64)
        steps = np.arange(64, dtype=np.uint32)
        near = (np.float32(2.5).view(np.uint32) + steps).view(np.float32)
        logits[np.arange(T)[:, None], cols] = near[None, :]
        bias[np.unique(cols)] = 0.0
    else:
        raise ValueError(kind)
    return dict(logits=np.ascontiguousarray(logits, dtype=np.float32), dtype="f32", bias=bias, T=T, E=E,
                k=K_KIMI, G=G_KIMI, Kg=KG_KIMI, scale=SCALE_KIMI, off=off, cnt=cnt)


def cfg_decision_edges(kind: str, T: int = 3000, E: int = E_KIMI, off: int = 0, cnt: int = 0) -> dict:
    """bf16 inputs that put every decision of the routing on its hardest path:
      flat        all logits 0 and bias 0: every score, group score and top-k value ties;
      group_copy  prefill logits with group 5 a copy of group 2 (logits and bias), so two
                  group scores are equal in every row;
      group_near  as group_copy, but group 5's biases are one float step above group 2's,
                  so the two group scores differ by a few float steps;
      negative    prefill logits, bias ~U(-2.1, -1.9): every biased score is negative;
      large_bias  prefill logits, bias ~U(-50, 50);
      plateau     N(0,1) logits (seed 10) with 200 seeded experts per row (seed 11) at 4.0 and
                  bias 0, so the k-th largest score is shared by far more than k experts;
      band        N(0,1) logits (seed 10) with 48 seeded experts per row (seed 13), 12 in each
                  of groups 0-3, at 3.0; the biases of groups 0-3 are distinct multiples of
                  2^-21 (a seeded permutation, seed 14), the others' -0.5, so that about 48
                  biased scores of a row lie within 2.2e-4 of each other: distinct, but
                  closer than the approximate scores can tell apart.
    """
    G = G_KIMI
    gsz = E // G
    base = cfg3(T, E, off, cnt)
    logits = base["logits"].copy()
    bias = base["bias"].copy()
    if kind == "flat":
        logits[:] = 0
        bias[:] = 0.0
    elif kind in ("group_copy", "group_near"):
        logits[:, 5 * gsz:6 * gsz] = logits[:, 2 * gsz:3 * gsz]
        bias[5 * gsz:6 * gsz] = bias[2 * gsz:3 * gsz]
        if kind == "group_near":
            bias[5 * gsz:6 * gsz] = np.nextafter(bias[5 * gsz:6 * gsz], np.float32(np.inf))
    elif kind == "negative":
        bias = uniform_f32(1, E, -2.1, -1.9)
    elif kind == "large_bias":
        bias = uniform_f32(1, E, -50.0, 50.0)
    elif kind == "plateau":
        x = normal_f32(10, T * E).reshape(T, E)
        cols = (raw64(11, T * 200) % np.uint64(E)).astype(np.int64).reshape(T, 200)
        x[np.arange(T)[:, None], cols] = 4.0
        logits = f32_to_bf16_bits(x)
        bias[:] = 0.0
    elif kind == "band":
        x = normal_f32(10, T * E).reshape(T, E)
        pick = (raw64(13, T * 48) % np.uint64(gsz)).astype(np.int64).reshape(T, 4, 12)
        cols = (pick + (np.arange(4) * gsz)[None, :, None]).reshape(T, 48)
        x[np.arange(T)[:, None], cols] = 3.0
        logits = f32_to_bf16_bits(x)
        bias = np.full(E, -0.5, dtype=np.float32)
        bias[:4 * gsz] = (permutation(14, 4 * gsz).astype(np.float64) * 2.0 ** -21).astype(np.float32)
    else:
        raise ValueError(kind)
    return dict(base, logits=logits, bias=bias)


def mx_activations(T: int, H: int = H_KIMI, kind: str = "normal", seed: int = 12) -> np.ndarray:
    """bf16 activations [T, H] for the fused route+quant launch:
      normal    N(0,1) (seed 12), the decode batch's hidden states;
      patterns  bf16 bit patterns drawn uniformly (seed 13), non-finite ones made finite by
                clearing the top exponent bit: zeros, subnormals, huge and tiny values;
      ties      blocks of 32 whose elements sit on the midpoints between E2M1 magnitudes
                (0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5) or in (6, 8), times 2^s, with 7 * 2^s
                in each block (so that the block scale is 2^s), random signs and s
                (seed 14); every fourth block all zeros.
    """
    if kind == "normal":
        return f32_to_bf16_bits(normal_f32(seed, T * H).reshape(T, H))
    if kind == "patterns":
        h = (raw64(13, T * H) >> np.uint64(48)).astype(np.uint16)
        bad = (h & np.uint16(0x7F80)) == np.uint16(0x7F80)
        h[bad] ^= np.uint16(0x4000)
        return h.reshape(T, H)
    if kind == "ties":
        nb = T * H // 32
        mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 6.5, 7.5, 6.0, 0.0])
        pick = (raw64(14, nb * 32, sub=1) % np.uint64(mids.size)).astype(np.int64).reshape(nb, 32)
        vals = mids[pick]
        vals[:, 0] = 7.0
        sign = np.where((raw64(14, nb * 32, sub=2) & np.uint64(1)).reshape(nb, 32) == 1, -1.0, 1.0)
        s = (raw64(14, nb, sub=3) % np.uint64(200)).astype(np.int64) - 100
        v = (vals * sign * np.exp2(s.astype(np.float64))[:, None]).astype(np.float32)
        v[::4] = 0.0
        return f32_to_bf16_bits(v.reshape(T, H))
    raise ValueError(kind)


def num_local_experts(E: int, ep: int) -> int:
    return E // ep
