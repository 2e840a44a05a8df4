// route_row.cuh -- one warp routes one token row of 896 router logits.
//
// Steps per row (the method, as defined in moe_route.h):
//   s = sigmoid(x), b = s + bias                    lane l owns experts [28 l, 28 l + 28)
//   group score = top-2 sum of b over 112 experts   lane top-2, then a 4-lane merge
//   keep topk_group groups                          rank of each group among the 8 scores
//   top-k of b over kept experts, ties to lower id  threshold + compaction + ranks
//   weights, relabel, pack                          lanes 0..k-1 hold slots 0..k-1
//
// Selection.  tau0 = the k-th largest value of a pool made of the two largest b of
// every kept lane (a subset of the candidates, so at least k candidates reach tau0),
// found by rank counting: each lane counts the pool values above its own.
// Candidates with b >= tau0 ("survivors", typically 17-22 for k = 16) are compacted
// one per lane in expert-id order with 32-bit keys (b relative to tau0, then position,
// so exact ties go to the lower id); a survivor's slot is the number of larger keys.
// When the key range does not allow such keys, k rounds of a warp maximum pick the
// slots.  33 to 64 survivors are ranked the same way, two per lane; beyond that a
// slower exact path extracts the k winners from per-lane maxima.  Rank counting reads the pool and the keys from shared memory, so
// its latency is a few loads instead of a chain of shuffles.
#pragma once
#include "common.cuh"

namespace moe {

struct RouteArgs {
  const void* logits;     // [T, E] f32 or bf16 bits
  const float* bias;      // [E]
  const float* stab;      // sigmoid table (bf16 logits), global
  const float2* etab;     // 2^(j/64) float-float table (float32 logits), global
  int32_t* packed;        // [T, k]
  int32_t* counts;        // [NE]
  int32_t* offsets;       // [NE + 1]
  int32_t* perm;          // [T * k]
  int32_t* ids;           // [T, k] or nullptr
  int32_t* inv = nullptr; // [T * k] or nullptr: position of entry t * k + j in perm
  // the expert-GEMM layout written by the routing itself (moe_route_with_layout), where
  // the kernel supports it: tile-padded offsets [NE + 1], padded rows and their bins
  // [capacity] (-1 for padding); all nullptr when not asked
  int32_t* poffs = nullptr;
  int32_t* prows = nullptr;
  int32_t* midx = nullptr;
  int tile = 1, capacity = 0;
  int* err;               // device status word
  int T, k, Kg, off, cnt, NE;
  float scale;
  float eps_half;         // bound on |0.5 tanh.approx(x / 2) - (sigmoid(x) - 0.5)| over
                          // bf16 x, measured on the device (route_pair.cuh)
  uint64_t barrier_wait_ns = kWaitLimitNs;  // limit of each grid-barrier wait of the
                                            // persistent kernels
  int barrier_skip_cta = -1;  // CTA that leaves before the first grid barrier (-1: none;
                              // a test of the timeout path)
  // MXFP4 quantisation of the decode batch's activations in the same launch
  // (moe_route_quant); unused when qx is null
  const uint16_t* qx = nullptr;  // [T, qH] bf16 bits
  uint8_t* qcodes = nullptr;     // [T, qH / 2] two E2M1 codes per byte, even element low
  uint8_t* qscales = nullptr;    // [T, qH / 32] E8M0
  int qH = 0;
  // bound on |0.5 tanh.approx(x / 2) + 0.5 - sig_f32(x)| over every float32 x, measured on
  // the device (k_approx_err_f32); negative: float32 scores are all computed exactly
  float eps_f32 = -1.0f;
};

// Per-warp shared scratch of the row routine.  NB = biased scores parked by the kept
// lanes: 28 per kept lane (448 when 4 of the 8 groups are kept, 896 at most).
template <int NB>
struct WarpScratchT {
  float b[NB];            // biased scores of the kept lanes (kept lane i at [28 i, 28 i + 28))
  float pool[32];         // threshold pool
  uint32_t skey[64];      // survivor keys
  int32_t sid[64];        // survivor expert ids
  int32_t slot_id[kMaxK]; // expert id of each slot
};
using WarpScratch = WarpScratchT<kEPL * 32>;

// Row input kinds: float32 logits, bfloat16 logits, float32 scores already equal to
// sigmoid(logit) (the fused contraction computes them in its epilogue), or packed
// values (id << 16 | weight) that are only indexed (histogram, scan, permutation).
enum { DT_F32 = 0, DT_BF16 = 1, DT_SCORE = 2, DT_PACKED = 3 };

template <int DT>
__device__ __forceinline__ float row_sigmoid(const void* row, int e, const float* stab,
                                             const float2* etab) {
  if constexpr (DT == DT_BF16) {
    return sig_bf16(stab, static_cast<const uint16_t*>(row)[e]);
  } else if constexpr (DT == DT_SCORE) {
    return static_cast<const float*>(row)[e];
  } else {
    return sig_f32(static_cast<const float*>(row)[e], etab);
  }
}


// Result of one routed row, valid in lanes j < k.
struct SlotOut {
  int32_t id;      // global expert id of slot j
  int32_t lid;     // relabelled id (== id when cnt == 0)
  int32_t packed;  // (lid << 16) | bf16 weight bits
};

__device__ __forceinline__ float fmax3(float a, float b, float c) {
  float r;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
  return r;
}

// Inverse of fkey.
__device__ __forceinline__ float fkey_inv(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Adds the pair (u, v) to the top-2 list (m1 >= m2); counts equal values with
// multiplicity.
__device__ __forceinline__ void top2_pair(float& m1, float& m2, float u, float v) {
  const float hi = fmaxf(u, v), lo = fminf(u, v);
  m2 = fmax3(m2, lo, fminf(m1, hi));
  m1 = fmaxf(m1, hi);
}

// bfloat16 logits: the scores of the two bf16 values packed in v (low half first).
// Both table indices are formed at once in 16-bit lanes: magnitude clamped to the
// table's range, plus the entries of one sign (N) for negative values.  `tab_lo` is the
// table shifted down by the first magnitude it covers, so it is indexed by magnitude.
__device__ __forceinline__ void sig_bf16_pair(const float* tab_lo, uint32_t v, float& s0, float& s1) {
  uint32_t m = v & 0x7FFF7FFFu;
  m = __vmaxu2(m, kSigLo * 0x10001u);
  m = __vminu2(m, kSigHi * 0x10001u);
  uint32_t neg;  // 0xFFFF in each half whose sign bit is set
  asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(neg) : "r"(v));
  const uint32_t i2 = m + (neg & (uint32_t(kSigN) * 0x10001u));
  s0 = tab_lo[i2 & 0xFFFFu];
  s1 = tab_lo[i2 >> 16];
}

// a - b rounded toward -infinity
__device__ __forceinline__ float sub_rm(float a, float b) {
  float y;
  asm("sub.rm.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

// Approximate biased score of a float32 logit: fma(0.5, tanh.approx(x / 2), bias + 0.5),
// within eps_f32 + (4 + 4 max|bias|) 2^-24 of fl(sig_f32(x) + bias) (route_row).
__device__ __forceinline__ float approx_b_f32(float x, float bias) {
  float t;
  asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(__fmul_rn(x, 0.5f)));
  return __fmaf_rn(0.5f, t, __fadd_rn(bias, 0.5f));
}

// Routes one row.  `row` points to the row's E logits (or scores) in shared memory
// (16-byte aligned); `bias_s` to the E biases in shared memory (16-byte aligned).  All
// 32 lanes must call it.  KC and KGC fix k and topk_group at compile time (the Kimi-K3
// instance: 16 and 4); 0 reads them from `a`.
template <int DT, int KC = 0, int KGC = 0, class WS>
__device__ __forceinline__ SlotOut route_row(const void* row, const float* bias_s,
                                             const float* stab, const RouteArgs& a, WS& ws) {
  const unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int e0 = lane * kEPL;
  const int k = KC ? KC : a.k;
  const int Kg = KGC ? KGC : a.Kg;

  // ---- a1, a2: scores, biased scores, lane top-2 (two independent lists)
  const float4* bq = reinterpret_cast<const float4*>(bias_s + e0);
  float b[kEPL];
  float xa1 = -INFINITY, xa2 = -INFINITY, xb1 = -INFINITY, xb2 = -INFINITY;
  // float32 logits with a measured approximation bound take approximate scores first
  const bool apx = DT == DT_F32 && a.eps_f32 >= 0.0f;
  float bmag = 0.0f;  // max |bias| over this lane's experts (approximate path)
  if constexpr (DT == DT_BF16) {
    const float* tab_lo = stab - kSigLo;
    const uint2* p = reinterpret_cast<const uint2*>(static_cast<const uint16_t*>(row) + e0);
#pragma unroll
    for (int q = 0; q < kEPL / 4; ++q) {
      const uint2 v = p[q];
      const float4 bb = bq[q];
      float s0, s1, s2, s3;
      sig_bf16_pair(tab_lo, v.x, s0, s1);
      sig_bf16_pair(tab_lo, v.y, s2, s3);
      b[4 * q + 0] = __fadd_rn(s0, bb.x);
      b[4 * q + 1] = __fadd_rn(s1, bb.y);
      b[4 * q + 2] = __fadd_rn(s2, bb.z);
      b[4 * q + 3] = __fadd_rn(s3, bb.w);
      top2_pair(xa1, xa2, b[4 * q + 0], b[4 * q + 1]);
      top2_pair(xb1, xb2, b[4 * q + 2], b[4 * q + 3]);
    }
  } else if (apx) {
    // float32 logits: approximate biased scores (one tanh.approx each), exact ones below
    // only for the experts a decision can depend on
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(row) + e0);
#pragma unroll
    for (int q = 0; q < kEPL / 4; ++q) {
      const float4 v = p[q];
      const float4 bb = bq[q];
      b[4 * q + 0] = approx_b_f32(v.x, bb.x);
      b[4 * q + 1] = approx_b_f32(v.y, bb.y);
      b[4 * q + 2] = approx_b_f32(v.z, bb.z);
      b[4 * q + 3] = approx_b_f32(v.w, bb.w);
      bmag = fmaxf(fmaxf(bmag, fmaxf(fabsf(bb.x), fabsf(bb.y))), fmaxf(fabsf(bb.z), fabsf(bb.w)));
      top2_pair(xa1, xa2, b[4 * q + 0], b[4 * q + 1]);
      top2_pair(xb1, xb2, b[4 * q + 2], b[4 * q + 3]);
    }
  } else {
    const float4* p = reinterpret_cast<const float4*>(static_cast<const float*>(row) + e0);
#pragma unroll
    for (int q = 0; q < kEPL / 4; ++q) {
      const float4 v = p[q];
      const float4 bb = bq[q];
      const float x[4] = {v.x, v.y, v.z, v.w};
      const float bi[4] = {bb.x, bb.y, bb.z, bb.w};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const float sc = (DT == DT_SCORE) ? x[r] : sig_f32(x[r], a.etab);
        b[4 * q + r] = __fadd_rn(sc, bi[r]);
      }
      top2_pair(xa1, xa2, b[4 * q + 0], b[4 * q + 1]);
      top2_pair(xb1, xb2, b[4 * q + 2], b[4 * q + 3]);
    }
  }
  float lm1 = fmaxf(xa1, xb1);
  float lm2 = fmax3(fminf(xa1, xb1), xa2, xb2);
  // exact biased scores of this lane's experts whose bits are set in m, two at a time;
  // f(i, b) is called for each
  auto exact_f32 = [&](uint32_t m, auto&& f) {
    const float* xr = static_cast<const float*>(row) + e0;
    while (m) {
      const int i0 = __ffs(m) - 1;
      m &= m - 1u;
      const int i1 = m ? __ffs(m) - 1 : i0;
      m &= m - 1u;
      const float v0 = __fadd_rn(sig_f32(xr[i0], a.etab), bias_s[e0 + i0]);
      const float v1 = __fadd_rn(sig_f32(xr[i1], a.etab), bias_s[e0 + i1]);
      f(i0, v0);
      if (i1 != i0) f(i1, v1);
    }
  };
  float eps = 0.0f;
  if (apx) {
    // |approximate - exact| <= eps for every expert of the row: the measured bound plus the
    // roundings of bias + 0.5, of the fma and of the exact sum (each within 2^-24 of its
    // magnitude, at most 1 + max|bias|), with slack for the float arithmetic here
    const float B = __uint_as_float(__reduce_max_sync(FULL, __float_as_uint(bmag)));
    eps = (a.eps_f32 + (4.0f + 4.0f * B) * 0x1p-24f) * (1.0f + 0x1p-20f);
    // the lane's exact top two: two experts have approximate scores >= lm2, so the exact
    // second largest is >= lm2 - eps, and either of the two has an approximate score of
    // at least lm2 - 2 eps
    const float thr = sub_rm(lm2, 2.0f * eps);
    uint32_t cm = 0;
#pragma unroll
    for (int i = 0; i < kEPL; ++i) cm |= (b[i] >= thr) ? (1u << i) : 0u;
    float e1 = -INFINITY, e2 = -INFINITY;
    exact_f32(cm, [&](int, float e) {
      e2 = fmaxf(e2, fminf(e1, e));
      e1 = fmaxf(e1, e);
    });
    lm1 = e1;
    lm2 = e2;
  }

  // ---- a3: group score = sum of the group's two largest b (4-lane merge of top-2 lists)
  float gm1 = lm1, gm2 = lm2;
#pragma unroll
  for (int o = 1; o < kLanesPerGroup; o <<= 1) {
    const float p1 = __shfl_xor_sync(FULL, gm1, o);
    const float p2 = __shfl_xor_sync(FULL, gm2, o);
    gm2 = fmax3(fminf(gm1, p1), gm2, p2);
    gm1 = fmaxf(gm1, p1);
  }
  const float gs = __fadd_rn(gm1, gm2);

  // ---- a4: keep the topk_group best groups, ties to the lower group index
  const int my_g = lane / kLanesPerGroup;
  int grank = 0;
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    const float o = __shfl_sync(FULL, gs, g * kLanesPerGroup);
    grank += (o > gs || (o == gs && g < my_g)) ? 1 : 0;
  }
  const bool kept = grank < Kg;
  const uint32_t kept_lanes = __ballot_sync(FULL, kept);
  const int nk = KGC ? KGC * kLanesPerGroup : __popc(kept_lanes);
  const int ki = __popc(kept_lanes & ((1u << lane) - 1u));

  // kept lanes park their biased scores for the survivor extraction below
  if (kept) {
    float4* d = reinterpret_cast<float4*>(ws.b + ki * kEPL);
#pragma unroll
    for (int q = 0; q < kEPL / 4; ++q)
      d[q] = make_float4(b[4 * q], b[4 * q + 1], b[4 * q + 2], b[4 * q + 3]);
  }

  // ---- a5: threshold tau0 = k-th largest (with multiplicity) of a pool of candidates
  //      made of the kept lanes' two largest values; at least k candidates reach it.
  //      Rank counting: lane l holds pool[l]; tau0 is the smallest pool value with at
  //      most k - 1 pool values strictly above it.
  int pool_n;
  if (2 * nk <= 32) {
    if (!KGC || 2 * nk < 32) ws.pool[lane] = -INFINITY;
    __syncwarp();
    if (kept) {
      ws.pool[2 * ki] = lm1;
      ws.pool[2 * ki + 1] = lm2;
    }
    pool_n = 2 * nk;
  } else {
    ws.pool[lane] = -INFINITY;
    __syncwarp();
    if (kept) {
      ws.pool[ki] = lm1;
      if (ki < 32 - nk) ws.pool[nk + ki] = lm2;
    }
    pool_n = 32;
  }
  __syncwarp();
  float tau0 = -INFINITY;
  if (pool_n >= k) {
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
    const uint32_t cand = (g0 + g1 + g2 + g3 <= k - 1) ? fkey(v) : 0xFFFFFFFFu;
    tau0 = fkey_inv(__reduce_min_sync(FULL, cand));
  }

  uint32_t smask = 0;
  if (kept) {
    if (apx) {
      // survivors have exact b >= tau0, so approximate b >= tau0 - eps: those get their
      // exact score, parked over the approximate one (the others stay below tau0)
      const float thr = sub_rm(tau0, eps);
      uint32_t dm = 0;
#pragma unroll
      for (int i = 0; i < kEPL; ++i) dm |= (b[i] >= thr) ? (1u << i) : 0u;
      exact_f32(dm, [&](int i, float e) {
        ws.b[ki * kEPL + i] = e;
        smask |= (e >= tau0) ? (1u << i) : 0u;
      });
    } else {
#pragma unroll
      for (int i = 0; i < kEPL; ++i) smask |= (b[i] >= tau0) ? (1u << i) : 0u;
    }
  }
  // inclusive prefix of the per-lane counts c (0..28, five bits) by bit slices: five
  // independent ballots instead of a five-step shuffle chain
  const int c = __popc(smask);
  const uint32_t le = 0xffffffffu >> (31 - lane);  // lanes 0..lane
  int incl = 0, total = 0;
#pragma unroll
  for (int bit = 0; bit < 5; ++bit) {
    const uint32_t bal = __ballot_sync(FULL, (c >> bit) & 1);
    incl += __popc(bal & le) << bit;
    total += __popc(bal) << bit;
  }
  __syncwarp();  // ws.b visible to the warp

  // composite 32-bit keys (b, position) need tau0 > 0 and survivors within 2^26 float
  // steps of it (b >= 0 there, so float bits order like the values)
  bool keys32 = false, keys64 = false;
  if (total <= 64 && tau0 > 0.0f) {
    const uint32_t bmax = __reduce_max_sync(FULL, kept ? __float_as_uint(lm1) : 0u);
    keys32 = total <= 32 && (bmax - __float_as_uint(tau0)) < (1u << 26);
    // float32 rows only: compiled into the bf16 and score instances, the 64-key ranking
    // cost their common rows 0.05-0.3 us per call (decode and contraction + routing)
    if constexpr (DT == DT_F32)
      keys64 = total > 32 && (bmax - __float_as_uint(tau0)) < (1u << 26) - 1u;  // 6 position bits
  }

  if (total <= 32) {
    if (keys32 && lane >= total) ws.skey[lane] = 0u;  // below every survivor's key
    int pos = incl - c;
    while (smask) {
      const int i = __ffs(smask) - 1;
      smask &= smask - 1u;
      const float bv = ws.b[ki * kEPL + i];
      ws.skey[pos] = keys32 ? (((__float_as_uint(bv) - __float_as_uint(tau0) + 1u) << 5) |
                               uint32_t(31 - pos))
                            : fkey(bv);
      ws.sid[pos] = e0 + i;
      ++pos;
    }
    __syncwarp();
    if (keys32) {
      // unique keys: a survivor's slot is the number of survivors with a larger key
      // (slots past `total` hold 0, below every key; almost always total <= 24)
      const uint32_t key = ws.skey[lane];
      const uint4* k4 = reinterpret_cast<const uint4*>(ws.skey);
      int r0 = 0, r1 = 0, r2 = 0, r3 = 0;
#pragma unroll
      for (int q = 0; q < 6; ++q) {
        const uint4 u = k4[q];
        r0 += u.x > key;
        r1 += u.y > key;
        r2 += u.z > key;
        r3 += u.w > key;
      }
      if (total > 24) {
#pragma unroll
        for (int q = 6; q < 8; ++q) {
          const uint4 u = k4[q];
          r0 += u.x > key;
          r1 += u.y > key;
          r2 += u.z > key;
          r3 += u.w > key;
        }
      }
      const int rank = r0 + r1 + r2 + r3;
      if (lane < total && rank < k) ws.slot_id[rank] = ws.sid[lane];
    } else {
      uint32_t key = (lane < total) ? ws.skey[lane] : 0u;
      const int my_id = (lane < total) ? ws.sid[lane] : 0;
      for (int j = 0; j < k; ++j) {
        const uint32_t top = __reduce_max_sync(FULL, key);
        const int win = __ffs(__ballot_sync(FULL, key == top)) - 1;
        if (lane == win) {
          ws.slot_id[j] = my_id;
          key = 0u;
        }
      }
    }
  } else if (DT == DT_F32 && keys64) {
    // 33 to 64 survivors (ties or near ties around tau0): two per lane, the same keys with
    // 6 position bits, each ranked against all 64 (positions past `total` hold 0)
    if (lane + 32 >= total) ws.skey[lane + 32] = 0u;
    int pos = incl - c;
    while (smask) {
      const int i = __ffs(smask) - 1;
      smask &= smask - 1u;
      const float bv = ws.b[ki * kEPL + i];
      ws.skey[pos] = ((__float_as_uint(bv) - __float_as_uint(tau0) + 1u) << 6) | uint32_t(63 - pos);
      ws.sid[pos] = e0 + i;
      ++pos;
    }
    __syncwarp();
    const uint32_t key0 = ws.skey[lane], key1 = ws.skey[lane + 32];
    const uint4* k4 = reinterpret_cast<const uint4*>(ws.skey);
    int r0 = 0, r1 = 0, q0 = 0, q1 = 0;
#pragma unroll
    for (int q = 0; q < 16; ++q) {
      const uint4 u = k4[q];
      r0 += int(u.x > key0) + int(u.y > key0);
      r1 += int(u.z > key0) + int(u.w > key0);
      q0 += int(u.x > key1) + int(u.y > key1);
      q1 += int(u.z > key1) + int(u.w > key1);
    }
    if (r0 + r1 < k) ws.slot_id[r0 + r1] = ws.sid[lane];  // lane < 32 < total
    if (lane + 32 < total && q0 + q1 < k) ws.slot_id[q0 + q1] = ws.sid[lane + 32];
  } else {
    // exact slow path: k rounds of (warp max over lane maxima), winner lane rescans
    uint32_t taken = 0;
    auto lane_best = [&](uint32_t& bk, int& bi) {
      bk = 0u;
      bi = -1;
      if (!kept) return;
      // the lane's 28 parked scores in seven 16-byte loads, all in flight at once
      const float4* p = reinterpret_cast<const float4*>(ws.b + ki * kEPL);
#pragma unroll
      for (int q = 0; q < kEPL / 4; ++q) {
        const float4 u = p[q];
        const float v[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int r = 0; r < 4; ++r) {
          const int i = 4 * q + r;
          const uint32_t kk = ((taken >> i) & 1u) ? 0u : fkey(v[r]);
          if (kk > bk) {
            bk = kk;
            bi = i;
          }
        }
      }
    };
    uint32_t bk;
    int bi;
    lane_best(bk, bi);
    for (int j = 0; j < k; ++j) {
      const uint32_t top = __reduce_max_sync(FULL, bk);
      const int win = __ffs(__ballot_sync(FULL, bk == top)) - 1;
      if (lane == win) {
        ws.slot_id[j] = e0 + bi;
        taken |= 1u << bi;
        lane_best(bk, bi);
      }
    }
  }
  __syncwarp();

  // ---- a6..a8: renormalise the unbiased scores, relabel, pack
  SlotOut out;
  out.id = 0;
  out.lid = 0;
  out.packed = 0;
  float s = 0.0f;
  if (lane < k) {
    out.id = ws.slot_id[lane];
    s = row_sigmoid<DT>(row, out.id, stab, a.etab);
  }
  // sequential sum in slot order, read back from shared memory; lanes >= k hold s = 0,
  // and adding +0 to den > 0 is exact
  ws.pool[lane] = s;
  __syncwarp();
  float den = 0.0f;
  {
    const float4* s4 = reinterpret_cast<const float4*>(ws.pool);
#pragma unroll
    for (int q = 0; q < (KC ? (KC + 3) / 4 : kMaxK / 4); ++q) {
      const float4 u = s4[q];
      den = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(den, u.x), u.y), u.z), u.w);
    }
  }
  if (lane < k) {
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

// ---------------------------------------------------------------- block scan
// Exclusive scan of in[0..n) into out[0..n], out[n] = total.  All threads of the
// block call it; `tmp` holds at least 32 ints.  in and out may alias.
__device__ __forceinline__ void block_exclusive_scan(const int* in, int* out, int n, int* tmp) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, wid = tid >> 5, nw = (nt + 31) >> 5;
  const int per = (n + nt - 1) / nt;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int sum = 0;
  for (int i = lo; i < hi; ++i) sum += in[i];
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) tmp[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    int v = (lane < nw) ? tmp[lane] : 0;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int u = __shfl_up_sync(0xffffffffu, inc, o);
      if (lane >= o) inc += u;
    }
    if (lane < nw) tmp[lane] = inc - v;
  }
  __syncthreads();
  int run = tmp[wid] + incl - sum;
  __syncthreads();  // everyone has read tmp; in may alias out
  for (int i = lo; i < hi; ++i) {
    const int v = in[i];
    out[i] = run;
    run += v;
  }
  if (hi == n && lo < hi) out[n] = run;
  if (n == 0 && tid == 0) out[0] = 0;
  __syncthreads();
}

}  // namespace moe
