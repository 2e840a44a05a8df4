// route_fast.cuh -- row routine for bfloat16 logits with k = 16 and topk_group = 4 (the
// Kimi-K3 instance), built on a cheap approximate score and exact scores only where a
// decision needs them.  The result is identical to route_row's.
//
// The exact score of a bf16 logit is a table lookup (common.cuh); its index depends on
// the data, so a warp's 32 lookups fall on shared-memory banks unevenly (about 3.5-way
// conflicts), and for all 896 experts of a row that is the costliest part of routing.
// Here every expert first gets an approximate biased score
//     b' = fma(0.5, tanh(x / 2), 0.5 + bias)      one MUFU tanh and two FMA-pipe ops
// whose distance from the exact b = s + bias is at most eps:
//     eps = E_half + (2 + B) 2^-22 + 2^-24,
// where E_half bounds |0.5 tanh.approx(x / 2) - (sigmoid(x) - 0.5)| over every bf16
// input (measured exhaustively on the device when the library state is created; about
// 3.5e-6 on sm_103a) and the other terms cover the roundings of the two additions for
// biases up to B = max |bias| in magnitude.  Each decision is then either certain from
// b' or taken on exact scores:
//   group choice: a group score is fl(m1 + m2) of the group's two largest b, so its
//     approximate value is within delta = 2 eps + (2 + 2B) 2^-22 of the exact one.  When
//     the topk_group-th and the next approximate group scores differ by more than
//     2 delta the kept set is certain; otherwise (about one row in 10^4 on the prefill
//     workload) the exact group scores are computed from the table.
//   top-k: p16 = the 16th largest of a pool of 32 approximate values, the two largest of
//     each kept lane (32 distinct kept experts).  At least 16 kept experts have
//     b' >= p16, so the exact 16th largest tau satisfies tau >= p16 - eps, and every
//     kept expert with exact b >= tau has b' >= p16 - 2 eps; every other expert has
//     exact b < tau.  The experts with b' >= p16 - 2 eps ("survivors", 17-22 on the
//     prefill workload, always at least 16) are looked up in the table, one per lane,
//     and ranked exactly by (b descending, id ascending).
//   weights: from the exact scores of the 16 winners, summed in slot order.
#pragma once
#include "route_row.cuh"

namespace moe {

// Per-warp shared scratch of route_row_fast.
struct FastScratch {
  float pool[32];          // threshold pool (approximate scores)
  uint32_t skey[32];       // survivor keys
  int32_t sid[32];         // survivor expert ids, ascending
  int32_t slot_id[16];     // expert id of each slot
  float slot_s[16];        // exact score of each slot
};

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// a - b rounded toward -infinity
__device__ __forceinline__ float fsub_down(float a, float b) {
  float y;
  asm("sub.rm.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

// Error bounds of the approximate scores for biases of magnitude at most bmax:
// eps bounds |b' - b| per expert, delta bounds the error of a group score.
struct ApproxBounds {
  float eps, delta;
};

__device__ __forceinline__ ApproxBounds approx_bounds(float e_half, float bmax) {
  ApproxBounds r;
  r.eps = e_half + (2.0f + bmax) * 0x1p-22f + 0x1p-24f;
  r.delta = 2.0f * r.eps + (2.0f + 2.0f * bmax) * 0x1p-22f;
  return r;
}

// Exact biased score of expert `id` of a bf16 row in shared memory.
__device__ __forceinline__ float exact_b(const uint16_t* row, const float* bias_s, const float* stab,
                                         int id, float* s_out) {
  const float s = stab[sig_index(row[id])];
  *s_out = s;
  return __fadd_rn(s, bias_s[id]);
}

// Routes one bf16 row with k = 16, topk_group = 4.  `row`: the row's 896 bf16 logits in
// shared memory (16-byte aligned); `bias_s`: the biases in shared memory; `c`: this
// lane's 28 values 0.5 + bias (registers); `stab`: the exact score table (shared memory).
// All 32 lanes must call it.  Lanes 0..15 return slots 0..15.
__device__ __forceinline__ SlotOut route_row_fast(const void* row_v, const float* bias_s,
                                                  const float* stab, const float (&c)[kEPL],
                                                  ApproxBounds bnd, const RouteArgs& a,
                                                  FastScratch& ws) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int K = 16, KG = 4;
  const int lane = threadIdx.x & 31;
  const int e0 = lane * kEPL;
  const uint16_t* row = static_cast<const uint16_t*>(row_v);
  const uint2* p = reinterpret_cast<const uint2*>(row + e0);

  // ---- approximate biased scores and the lane's two largest (two independent chains)
  float b[kEPL];
  float xa1 = -INFINITY, xa2 = -INFINITY, xb1 = -INFINITY, xb2 = -INFINITY;
#pragma unroll
  for (int q = 0; q < kEPL / 4; ++q) {
    const uint2 v = p[q];
    const float x0 = __uint_as_float(v.x << 16), x1 = __uint_as_float(v.x & 0xFFFF0000u);
    const float x2 = __uint_as_float(v.y << 16), x3 = __uint_as_float(v.y & 0xFFFF0000u);
    b[4 * q + 0] = __fmaf_rn(0.5f, tanh_approx(__fmul_rn(x0, 0.5f)), c[4 * q + 0]);
    b[4 * q + 1] = __fmaf_rn(0.5f, tanh_approx(__fmul_rn(x1, 0.5f)), c[4 * q + 1]);
    b[4 * q + 2] = __fmaf_rn(0.5f, tanh_approx(__fmul_rn(x2, 0.5f)), c[4 * q + 2]);
    b[4 * q + 3] = __fmaf_rn(0.5f, tanh_approx(__fmul_rn(x3, 0.5f)), c[4 * q + 3]);
    top2_pair(xa1, xa2, b[4 * q + 0], b[4 * q + 1]);
    top2_pair(xb1, xb2, b[4 * q + 2], b[4 * q + 3]);
  }
  const float lm1 = fmaxf(xa1, xb1);
  const float lm2 = fmax3(fminf(xa1, xb1), xa2, xb2);

  // ---- approximate group scores: 4-lane merge of the lanes' top-2 lists
  float gm1 = lm1, gm2 = lm2;
#pragma unroll
  for (int o = 1; o < kLanesPerGroup; o <<= 1) {
    const float p1 = __shfl_xor_sync(FULL, gm1, o);
    const float p2 = __shfl_xor_sync(FULL, gm2, o);
    gm2 = fmax3(fminf(gm1, p1), gm2, p2);
    gm1 = fmaxf(gm1, p1);
  }
  const float gs = __fadd_rn(gm1, gm2);

  // ---- kept groups: the 4th and 5th largest distinct approximate scores (the 4 lanes
  //      of a group hold the same key), certain when exactly 4 groups reach the 4th and
  //      its margin over the 5th exceeds 2 delta
  const uint32_t key = fkey(gs);
  uint32_t kx = __reduce_max_sync(FULL, key);
#pragma unroll
  for (int r = 1; r < KG; ++r) kx = __reduce_max_sync(FULL, key < kx ? key : 0u);
  const uint32_t k4 = kx;
  const uint32_t k5 = __reduce_max_sync(FULL, key < k4 ? key : 0u);
  bool kept = key >= k4;
  uint32_t kept_lanes = __ballot_sync(FULL, kept);
  const bool certain = __popc(kept_lanes) == KG * kLanesPerGroup && k5 != 0u &&
                       __fsub_rn(fkey_inv(k4), fkey_inv(k5)) > 2.0f * bnd.delta;
  if (!certain) {
    // exact group scores from the table, ranked with ties to the lower group
    const float* tab_lo = stab - kSigLo;
    const float4* bq = reinterpret_cast<const float4*>(bias_s + e0);
    float ya1 = -INFINITY, ya2 = -INFINITY, yb1 = -INFINITY, yb2 = -INFINITY;
#pragma unroll
    for (int q = 0; q < kEPL / 4; ++q) {
      const uint2 v = p[q];
      const float4 bb = bq[q];
      float s0, s1, s2, s3;
      sig_bf16_pair(tab_lo, v.x, s0, s1);
      sig_bf16_pair(tab_lo, v.y, s2, s3);
      top2_pair(ya1, ya2, __fadd_rn(s0, bb.x), __fadd_rn(s1, bb.y));
      top2_pair(yb1, yb2, __fadd_rn(s2, bb.z), __fadd_rn(s3, bb.w));
    }
    float h1 = fmaxf(ya1, yb1), h2 = fmax3(fminf(ya1, yb1), ya2, yb2);
#pragma unroll
    for (int o = 1; o < kLanesPerGroup; o <<= 1) {
      const float p1 = __shfl_xor_sync(FULL, h1, o);
      const float p2 = __shfl_xor_sync(FULL, h2, o);
      h2 = fmax3(fminf(h1, p1), h2, p2);
      h1 = fmaxf(h1, p1);
    }
    const float egs = __fadd_rn(h1, h2);
    const int my_g = lane / kLanesPerGroup;
    int grank = 0;
#pragma unroll
    for (int g = 0; g < kG; ++g) {
      const float o = __shfl_sync(FULL, egs, g * kLanesPerGroup);
      grank += (o > egs || (o == egs && g < my_g)) ? 1 : 0;
    }
    kept = grank < KG;
    kept_lanes = __ballot_sync(FULL, kept);
  }
  const int ki = __popc(kept_lanes & ((1u << lane) - 1u));

  // ---- p16: 16th largest (with multiplicity) of the kept lanes' two largest values,
  //      by rank counting; survivors are the kept experts with b' >= p16 - 2 eps
  if (kept) {
    ws.pool[2 * ki] = lm1;
    ws.pool[2 * ki + 1] = lm2;
  }
  __syncwarp();
  float cut;
  {
    const float v = ws.pool[lane];
    const float4* p4 = reinterpret_cast<const float4*>(ws.pool);
    int g0 = 0, g1 = 0, g2 = 0, g3 = 0;
#pragma unroll
    for (int q = 0; q < 8; ++q) {
      const float4 u = p4[q];
      g0 += u.x > v;
      g1 += u.y > v;
      g2 += u.z > v;
      g3 += u.w > v;
    }
    const uint32_t cand = (g0 + g1 + g2 + g3 <= K - 1) ? fkey(v) : 0xFFFFFFFFu;
    const float p16 = fkey_inv(__reduce_min_sync(FULL, cand));
    cut = fsub_down(p16, 2.0f * bnd.eps);
  }
  uint32_t smask = 0;
  if (kept) {
#pragma unroll
    for (int i = 0; i < kEPL; ++i) smask |= (b[i] >= cut) ? (1u << i) : 0u;
  }
  const int cnt = __popc(smask);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int n = __shfl_up_sync(FULL, incl, o);
    if (lane >= o) incl += n;
  }
  const int total = __shfl_sync(FULL, incl, 31);

  if (total <= 32) {
    // survivors one per lane, in ascending id order
    int pos = incl - cnt;
    for (uint32_t m = smask; m; m &= m - 1u) ws.sid[pos++] = e0 + __ffs(m) - 1;
    __syncwarp();
    int id = 0;
    float s = 0.0f, bx = 0.0f;
    if (lane < total) {
      id = ws.sid[lane];
      bx = exact_b(row, bias_s, stab, id, &s);
    }
    // every survivor's exact b is at least cut - eps
    const float base = fsub_down(cut, bnd.eps);
    bool keys32 = false;
    if (base > 0.0f) {
      const uint32_t bmax = __reduce_max_sync(FULL, lane < total ? __float_as_uint(bx) : 0u);
      keys32 = (bmax - __float_as_uint(base)) < (1u << 26);
    }
    if (keys32) {
      // unique 32-bit keys (b relative to base, then id: lower id larger); a
      // survivor's slot is the number of survivors with a larger key
      const uint32_t kk =
          lane < total ? (((__float_as_uint(bx) - __float_as_uint(base) + 1u) << 5) | uint32_t(31 - lane))
                       : 0u;
      ws.skey[lane] = kk;
      __syncwarp();
      const uint4* k4p = reinterpret_cast<const uint4*>(ws.skey);
      int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
#pragma unroll
      for (int q = 0; q < 6; ++q) {
        const uint4 u = k4p[q];
        r0 += u.x > kk;
        r1 += u.y > kk;
        r2 += u.z > kk;
        r3 += u.w > kk;
      }
      if (total > 24) {
#pragma unroll
        for (int q = 6; q < 8; ++q) {
          const uint4 u = k4p[q];
          r0 += u.x > kk;
          r1 += u.y > kk;
          r2 += u.z > kk;
          r3 += u.w > kk;
        }
      }
      const int rank = r0 + r1 + r2 + r3;
      if (lane < total && rank < K) {
        ws.slot_id[rank] = id;
        ws.slot_s[rank] = s;
      }
    } else {
      // K rounds of a warp maximum; equal scores go to the lower lane (lower id)
      uint32_t kk = lane < total ? fkey(bx) : 0u;
      for (int j = 0; j < K; ++j) {
        const uint32_t top = __reduce_max_sync(FULL, kk);
        const int win = __ffs(__ballot_sync(FULL, kk == top)) - 1;
        if (lane == win) {
          ws.slot_id[j] = id;
          ws.slot_s[j] = s;
          kk = 0u;
        }
      }
    }
  } else {
    // more than 32 survivors: K rounds, each lane offering its best remaining survivor
    // (exact scores recomputed from the table; ties to the lower id)
    uint32_t rem = smask;
    for (int j = 0; j < K; ++j) {
      uint32_t best = 0u;
      int bi = -1;
      float bs = 0.0f;
      for (uint32_t m = rem; m; m &= m - 1u) {
        const int i = __ffs(m) - 1;
        float si;
        const uint32_t kq = fkey(exact_b(row, bias_s, stab, e0 + i, &si));
        if (kq > best) {
          best = kq;
          bi = i;
          bs = si;
        }
      }
      const uint32_t top = __reduce_max_sync(FULL, best);
      const int win = __ffs(__ballot_sync(FULL, best == top && bi >= 0)) - 1;
      if (lane == win) {
        ws.slot_id[j] = e0 + bi;
        ws.slot_s[j] = bs;
        rem &= ~(1u << bi);
      }
    }
  }
  __syncwarp();

  // ---- weights from the exact scores, summed in slot order; relabel; pack
  SlotOut out;
  out.id = 0;
  out.lid = 0;
  out.packed = 0;
  float den = 0.0f;
  {
    const float4* s4 = reinterpret_cast<const float4*>(ws.slot_s);
#pragma unroll
    for (int q = 0; q < K / 4; ++q) {
      const float4 u = s4[q];
      den = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(den, u.x), u.y), u.z), u.w);
    }
  }
  if (lane < K) {
    out.id = ws.slot_id[lane];
    const float s = ws.slot_s[lane];
    const float w = __fmul_rn(__fdiv_rn(s, den), a.scale);
    const uint32_t wb = f32_to_bf16_bits(w);
    int lid = out.id;
    if (a.cnt > 0) lid = (out.id >= a.off && out.id < a.off + a.cnt) ? out.id - a.off : a.cnt + lane;
    out.lid = lid;
    out.packed = static_cast<int32_t>((static_cast<uint32_t>(lid) << 16) | wb);
  }
  __syncwarp();
  return out;
}

}  // namespace moe
