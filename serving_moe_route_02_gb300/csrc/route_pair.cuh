// route_pair.cuh -- one warp routes two bf16 rows at once (k = 16, topk_group = 4, the
// Kimi-K3 instance): lanes 0-15 route the first row, lanes 16-31 the second.  The result
// is identical to route_row's.
//
// Why approximate scores.  The exact score of a bf16 logit is a table lookup (common.cuh)
// whose index depends on the data, so a warp's 32 lookups fall on shared-memory banks
// unevenly (about 3.5-way conflicts); for all 896 experts of a row that is the costliest
// part of routing.  Here every expert first gets a cheap approximate score, and the exact
// table is read only for the experts a decision depends on: the survivors of the top-k
// step (about 18 of 896 per row) and, when the group choice is uncertain, the few
// candidates for each group's top two.
//
// Layout.  Lane h of a half (h = lane & 15) owns the 56 experts [56 h, 56 h + 56) as two
// "chains" of 28: chain a = [56 h, 56 h + 28) and chain b = [56 h + 28, 56 h + 56), each a
// quarter of a group of 112; a group is lanes 2g and 2g + 1.  Approximate scores are kept
// as packed f16 pairs: word j holds element j of chain a (low half) and of chain b (high
// half), so one packed max/min step tracks the two largest values of both chains at once.
//
// Approximate scores (the halving and the fma on f32 pairs, which round like the scalar
// forms):
//   b'' = f16(fma(0.5, tanh.approx(x / 2), c'')),  c'' = bias + (0.5 - o),
// where o centres the values (|b''| <= R = (bias_max - bias_min + 1) / 2), so the f16
// rounding error is at most half an f16 ulp at R.  With the offset added back, b'' + o is
// within eps of the exact b = s + bias:
//   eps = E_half + ulp_f16(R) / 2 + (2 + B) 2^-22 + 2^-24,   B = max |bias|,
// where E_half bounds |0.5 tanh.approx(x / 2) - (sigmoid(x) - 0.5)| over every bf16 input
// (measured exhaustively on the device when the library state is created; about 3.5e-6
// on sm_103a) and the other terms cover the roundings of the additions.  A group score is
// fl(m1 + m2) of the group's two largest b, so its approximate value is within
// delta = 2 eps + (2 + 2B) 2^-22 of the exact one.
// Steps per row (everything in the row's half-warp):
//   group choice: the 4th and 5th approximate group scores differ by more than 2 delta,
//     so the kept set is certain; otherwise (about one row in 80) the group scores are
//     computed exactly, from the table values of the experts that can be among each
//     group's top two (b'' at least the group's approximate second largest less 2 eps);
//   top-k: p16 = the 16th largest of the 32 kept chains' top-2 values (a bitonic sort of
//     packed f16 pairs across the half).  At least 16 kept experts have b'' >= p16, so the
//     exact 16th largest tau satisfies tau >= p16 + o - eps, and every kept expert whose
//     exact b reaches tau has b'' >= p16 - 2 eps; every other expert has exact b < tau.
//     The experts with b'' >= p16 - 2 eps ("survivors", 17-22 on the prefill workload,
//     always at least 16) get packed compares (a bit per expert), are compacted in
//     ascending id order, looked up in the exact table (two per lane) and ranked by a
//     bitonic sort of 32-bit keys (exact b, then id), which gives slots 0..15;
//   weights from the exact scores in slot order, relabel, pack.
// Rare cases: 33 to 64 survivors in a row are ranked the same way, four per lane in a
// 64-key sort; more than 64, or keys that do not fit 32 bits, take an exact extraction
// (16 rounds of a half-warp maximum over the survivors).
#pragma once
#include "route_row.cuh"

namespace moe {

__device__ __forceinline__ float tanh_approx(float x) {
  float y;
  asm("tanh.approx.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// a - b and a + b rounded toward -infinity
__device__ __forceinline__ float fsub_down(float a, float b) {
  float y;
  asm("sub.rm.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

constexpr int kPairEPL = 56;   // experts per lane
constexpr int kChain = 28;     // experts per chain

// c'' in shared memory: per lane, the pairs (chain a, chain b) of its 28 words, 60 floats
// apart (56 used), so that 8 lanes' 16-byte loads fall on distinct banks
constexpr int kCppStride = 60;
constexpr int kCppFloats = 16 * kCppStride;

// One packed approximate score word: b'' for x = (xa, xb) and c'' = (ca, cb), f16 pair
// (xa's low).  The halving and the fma run on f32 pairs (mul.rn.f32x2, fma.rn.f32x2),
// which round like their scalar forms, so each half equals
// f16(fma(0.5, tanh.approx(x * 0.5), c)).
__device__ __forceinline__ uint32_t approx_word(float xa, float xb, uint64_t c2) {
  uint32_t v;
  asm("{\n\t.reg .b64 x, q, t, r;\n\t.reg .b32 t0, t1, r0, r1;\n\t"
      "mov.b64 x, {%1, %2};\n\tmul.rn.f32x2 q, x, %4;\n\tmov.b64 {t0, t1}, q;\n\t"
      "tanh.approx.f32 t0, t0;\n\ttanh.approx.f32 t1, t1;\n\tmov.b64 t, {t0, t1};\n\t"
      "fma.rn.f32x2 r, t, %4, %3;\n\tmov.b64 {r0, r1}, r;\n\tcvt.rn.f16x2.f32 %0, r1, r0;\n\t}"
      : "=r"(v)
      : "f"(xa), "f"(xb), "l"(c2), "l"(0x3F0000003F000000ull));
  return v;
}

// Per-warp shared scratch of route_pair.
struct PairScratch {
  uint32_t pool[2][16];   // per row: the 32 kept chains' top-2 values, f16 pairs
  int32_t sid[2][32];     // survivors' expert ids, ascending
  float ss[2][32];        // survivors' exact scores
  int32_t slot_id[2][16]; // expert id of each slot
  float slot_s[2][16];    // exact score of each slot
};

__device__ __forceinline__ uint32_t h2max(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("max.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ uint32_t h2min(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("min.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
// f16 pair (lo, hi), round to nearest
__device__ __forceinline__ uint32_t h2pack(float lo, float hi) {
  uint32_t r;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
  return r;
}
// 0xFFFF in each half where a >= b
__device__ __forceinline__ uint32_t h2ge(uint32_t a, uint32_t b) {
  uint32_t r;
  asm("set.ge.u32.f16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
  return r;
}
__device__ __forceinline__ float h_lo(uint32_t v) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, l;\n\t}" : "=f"(f) : "r"(v));
  return f;
}
__device__ __forceinline__ float h_hi(uint32_t v) {
  float f;
  asm("{\n\t.reg .b16 l, h;\n\tmov.b32 {l, h}, %1;\n\tcvt.f32.f16 %0, h;\n\t}" : "=f"(f) : "r"(v));
  return f;
}
// f16 rounded toward -infinity, in both halves
__device__ __forceinline__ uint32_t h2dup_down(float x) {
  uint16_t h;
  asm("cvt.rm.f16.f32 %0, %1;" : "=h"(h) : "f"(x));
  return uint32_t(h) * 0x10001u;
}
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
  uint32_t r;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
  return r;
}
__device__ __forceinline__ float fadd_down(float a, float b) {
  float y;
  asm("add.rm.f32 %0, %1, %2;" : "=f"(y) : "f"(a), "f"(b));
  return y;
}

// Per-CTA constants of the approximation: offset o, d0 = 0.5 - o (both exact), eps, delta,
// and whether the f16 range holds every value (otherwise every row takes the exact paths).
struct PairBounds {
  float o, d0, eps, delta;
  bool ok;
};

__device__ __forceinline__ PairBounds pair_bounds(float e_half, float bmin, float bmax) {
  PairBounds r;
  // o = (bmin + bmax + 1) / 2 rounded to a multiple of 2^-8, so that 0.5 - o is exact
  r.o = rintf((bmin + bmax + 1.0f) * 128.0f) * 0x1p-8f;
  r.d0 = 0.5f - r.o;
  const float babs = fmaxf(fabsf(bmin), fabsf(bmax));
  // |b''| <= R: the values' half range, plus the offset's rounding (2^-9) and slack
  const float R = fmaxf(fmaxf(bmax + 1.0f - r.o, r.o - bmin), 0.5f) + 0x1p-8f;
  r.ok = R < 8192.0f;
  // half an f16 ulp at R: 2^(e - 11) for R in [2^e, 2^(e+1))
  const int e = int((__float_as_uint(R) >> 23) & 0xFFu) - 127;
  const float hhalf = __int_as_float((e - 11 + 127) << 23);
  r.eps = e_half + hhalf + (2.0f + babs) * 0x1p-22f + 0x1p-24f;
  r.delta = 2.0f * r.eps + (2.0f + 2.0f * babs) * 0x1p-22f;
  return r;
}

// Descending bitonic sort of 32 f16 values held as one pair per lane of a half-warp
// (positions 2h and 2h + 1 in the low and high halves of lane h's word).
__device__ __forceinline__ uint32_t bitonic32_h2(uint32_t v, int h) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j >= 1; j >>= 1) {
      const bool desc = ((2 * h) & k) == 0;
      if (j == 1) {
        const uint32_t sw = prmt(v, v, 0x1032u);
        const uint32_t mx = h2max(v, sw), mn = h2min(v, sw);
        v = desc ? prmt(mx, mn, 0x7610u) : prmt(mn, mx, 0x7610u);
      } else {
        const uint32_t p = __shfl_xor_sync(0xffffffffu, v, j >> 1);
        const bool lower = ((2 * h) & j) == 0;
        v = (lower == desc) ? h2max(v, p) : h2min(v, p);
      }
    }
  }
  return v;
}

// Descending bitonic sort of 32 uint32 keys held two per lane of a half-warp.
__device__ __forceinline__ void bitonic32_u32(uint32_t& k0, uint32_t& k1, int h) {
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int j = k >> 1; j >= 1; j >>= 1) {
      const bool desc = ((2 * h) & k) == 0;
      if (j == 1) {
        const uint32_t mx = max(k0, k1), mn = min(k0, k1);
        k0 = desc ? mx : mn;
        k1 = desc ? mn : mx;
      } else {
        const uint32_t p0 = __shfl_xor_sync(0xffffffffu, k0, j >> 1);
        const uint32_t p1 = __shfl_xor_sync(0xffffffffu, k1, j >> 1);
        const bool lower = ((2 * h) & j) == 0;
        const bool keep_max = lower == desc;
        k0 = keep_max ? max(k0, p0) : min(k0, p0);
        k1 = keep_max ? max(k1, p1) : min(k1, p1);
      }
    }
  }
}

// Descending bitonic sort of 64 uint32 keys held four per lane of a half-warp (lane h
// holds positions 4 h .. 4 h + 3).
__device__ __forceinline__ void bitonic64_u32(uint32_t (&k)[4], int h) {
#pragma unroll
  for (int kk = 2; kk <= 64; kk <<= 1) {
#pragma unroll
    for (int j = kk >> 1; j >= 1; j >>= 1) {
      if (j >= 4) {
        // partner in lane h ^ (j / 4), same element; direction and side depend on h only
        const bool desc = ((4 * h) & kk) == 0;
        const bool keep_max = (((4 * h) & j) == 0) == desc;
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const uint32_t p = __shfl_xor_sync(0xffffffffu, k[e], j >> 2);
          k[e] = keep_max ? max(k[e], p) : min(k[e], p);
        }
      } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          if (e & j) continue;
          const bool desc = ((4 * h + e) & kk) == 0;
          const uint32_t mx = max(k[e], k[e | j]), mn = min(k[e], k[e | j]);
          k[e] = desc ? mx : mn;
          k[e | j] = desc ? mn : mx;
        }
      }
    }
  }
}

// Maximum over the lanes of a half-warp.
__device__ __forceinline__ uint32_t half_max(uint32_t v) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float half_maxf(float v) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}
__device__ __forceinline__ float half_minf(float v) {
#pragma unroll
  for (int o = 8; o >= 1; o >>= 1) v = fminf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

// Bits of the words of a lane whose values reach `thr2` (an f16 pair holding the same
// threshold twice): bit q of *ma for element q of chain a, of *mb for chain b.
__device__ __forceinline__ void chain_masks(const uint32_t (&bp)[kChain], uint32_t thr2, uint32_t& ma,
                                            uint32_t& mb) {
  uint32_t acc0 = 0, acc1 = 0;
#pragma unroll
  for (int q = 0; q < kChain; ++q) {
    const uint32_t pat = (1u << (q % 14)) * 0x10001u;
    const uint32_t t = h2ge(bp[q], thr2) & pat;
    if (q < 14) acc0 |= t;
    else acc1 |= t;
  }
  ma = (acc0 & 0x3FFFu) | ((acc1 & 0x3FFFu) << 14);
  mb = (acc0 >> 16) | ((acc1 >> 16) << 14);
}

// Routes two bf16 rows: `row0` for lanes 0-15, `row1` for lanes 16-31 (shared memory,
// 16-byte aligned; both may be the same row).  `bias_s`: biases; `cpp_s`: c'' = bias + d0
// (shared memory); `stab`: the exact score table (global memory, read-only).  All 32 lanes call it;
// lane h of each half returns slot h of its row.
__device__ __forceinline__ SlotOut route_pair(const void* row0, const void* row1, const float* bias_s,
                                              const float* cpp_s, const float* stab, const PairBounds& pb,
                                              const RouteArgs& a, PairScratch& ws) {
  constexpr unsigned FULL = 0xffffffffu;
  constexpr int K = 16, KG = 4;
  const int lane = threadIdx.x & 31;
  const int half = lane >> 4, h = lane & 15;
  const int hbase = lane & 16;  // first lane of this half
  const int e0 = h * kPairEPL;
  const uint16_t* row = static_cast<const uint16_t*>(half ? row1 : row0);

  // ---- approximate scores, packed (chain a low, chain b high); two independent top-2
  //      trackers (even and odd words) shorten the dependent chain
  uint32_t bp[kChain];
  uint32_t m1e = 0xFC00FC00u, m2e = 0xFC00FC00u, m1o = 0xFC00FC00u, m2o = 0xFC00FC00u;  // -inf
  {
    const uint2* pa = reinterpret_cast<const uint2*>(row + e0);
    const uint2* pb = reinterpret_cast<const uint2*>(row + e0 + kChain);
    const ulonglong2* cq = reinterpret_cast<const ulonglong2*>(cpp_s + h * kCppStride);
#pragma unroll
    for (int q = 0; q < kChain / 4; ++q) {
      const uint2 va = pa[q], vb = pb[q];
      const ulonglong2 c01 = cq[2 * q], c23 = cq[2 * q + 1];
      const float xa[4] = {__uint_as_float(va.x << 16), __uint_as_float(va.x & 0xFFFF0000u),
                           __uint_as_float(va.y << 16), __uint_as_float(va.y & 0xFFFF0000u)};
      const float xb[4] = {__uint_as_float(vb.x << 16), __uint_as_float(vb.x & 0xFFFF0000u),
                           __uint_as_float(vb.y << 16), __uint_as_float(vb.y & 0xFFFF0000u)};
      const uint64_t cc[4] = {c01.x, c01.y, c23.x, c23.y};
#pragma unroll
      for (int r = 0; r < 4; ++r) {
        const uint32_t v = approx_word(xa[r], xb[r], cc[r]);
        bp[4 * q + r] = v;
        if (r & 1) {
          const uint32_t t = h2min(m1o, v);
          m1o = h2max(m1o, v);
          m2o = h2max(m2o, t);
        } else {
          const uint32_t t = h2min(m1e, v);
          m1e = h2max(m1e, v);
          m2e = h2max(m2e, t);
        }
      }
    }
  }
  // merge the two trackers: chains' top-2 (packed)
  const uint32_t m1 = h2max(m1e, m1o);
  const uint32_t m2 = h2max(h2min(m1e, m1o), h2max(m2e, m2o));

  // ---- approximate group scores (f32): lane top-2 over both chains, then the partner lane
  float gs, g2;
  {
    const float a1 = h_lo(m1), a2 = h_lo(m2), b1 = h_hi(m1), b2 = h_hi(m2);
    float l1 = fmaxf(a1, b1), l2 = fmax3(fminf(a1, b1), a2, b2);
    const float p1 = __shfl_xor_sync(FULL, l1, 1), p2 = __shfl_xor_sync(FULL, l2, 1);
    g2 = fmax3(fminf(l1, p1), l2, p2);
    gs = __fadd_rn(fmaxf(l1, p1), g2);
  }
  // exact biased score of an expert of this half's row
  auto exact_b = [&](int id) -> float { return __fadd_rn(__ldg(stab + sig_index(row[id])), bias_s[id]); };

  // ---- kept groups per half: rank among the 8 (ties to the lower group); certain when
  //      min(kept) - max(dropped) > 2 delta
  const int my_g = h >> 1;
  int grank = 0;
#pragma unroll
  for (int g = 0; g < kG; ++g) {
    const float o = __shfl_sync(FULL, gs, hbase + 2 * g);
    grank += (o > gs || (o == gs && g < my_g)) ? 1 : 0;
  }
  bool kept = grank < KG;
  {
    const float kmin = half_minf(kept ? gs : INFINITY);
    const float nmax = half_maxf(kept ? -INFINITY : gs);
    const bool certain = pb.ok && __fsub_rn(kmin, nmax) > 2.0f * pb.delta;
    if (!__all_sync(FULL, certain)) {
      // exact group scores for both rows.  Two experts of the group have b'' >= g2 (its
      // approximate second largest), so its exact second largest is at least g2 + o - eps,
      // and an expert among its exact top-2 has b'' >= g2 - 2 eps: only those
      // ("candidates", one or two per lane as a rule) are looked up, four at a time.
      uint32_t ra, rb;
      chain_masks(bp, pb.ok ? h2dup_down(fsub_down(g2, 2.0f * pb.eps)) : 0xFC00FC00u, ra, rb);
      float y1 = -INFINITY, y2 = -INFINITY;
      do {
        int id[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          id[i] = -1;
          if (ra) {
            id[i] = e0 + __ffs(ra) - 1;
            ra &= ra - 1u;
          } else if (rb) {
            id[i] = e0 + kChain + __ffs(rb) - 1;
            rb &= rb - 1u;
          }
        }
        float v[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) v[i] = id[i] >= 0 ? exact_b(id[i]) : -INFINITY;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          y2 = fmaxf(y2, fminf(y1, v[i]));
          y1 = fmaxf(y1, v[i]);
        }
      } while (ra | rb);
      const float p1 = __shfl_xor_sync(FULL, y1, 1), p2 = __shfl_xor_sync(FULL, y2, 1);
      const float egs = __fadd_rn(fmaxf(y1, p1), fmax3(fminf(y1, p1), y2, p2));
      int er = 0;
#pragma unroll
      for (int g = 0; g < kG; ++g) {
        const float o = __shfl_sync(FULL, egs, hbase + 2 * g);
        er += (o > egs || (o == egs && g < my_g)) ? 1 : 0;
      }
      kept = er < KG;
    }
  }
  const uint32_t kept_lanes = __ballot_sync(FULL, kept);
  const uint32_t half_lanes = kept_lanes & (0xFFFFu << hbase);
  const int ki = __popc(half_lanes & ((1u << lane) - 1u));  // 0..7 among the half's kept lanes

  // ---- p16: 16th largest of the kept chains' top-2 values (packed f16), bitonic sort
  if (kept) {
    ws.pool[half][2 * ki] = prmt(m1, m2, 0x5410u);      // chain a: (m1, m2)
    ws.pool[half][2 * ki + 1] = prmt(m1, m2, 0x7632u);  // chain b: (m1, m2)
  }
  __syncwarp();
  const uint32_t srt = bitonic32_h2(ws.pool[half][h], h);
  const float p16 = h_hi(__shfl_sync(FULL, srt, hbase + 7));  // position 15
  // cutoff in b'' units, rounded down to f16; every exact top-k expert reaches it
  const float cutf = pb.ok ? fsub_down(p16, 2.0f * pb.eps) : -INFINITY;
  const uint32_t cut2 = pb.ok ? h2dup_down(cutf) : 0xFC00FC00u;

  // ---- survivors: a bit per kept expert with b'' >= cut (chain a: bits of ma, b: mb)
  uint32_t ma, mb;
  chain_masks(bp, cut2, ma, mb);
  if (!kept) ma = mb = 0u;
  const int cnt = __popc(ma) + __popc(mb);
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 16; o <<= 1) {
    const int n = __shfl_up_sync(FULL, incl, o, 16);
    if (h >= o) incl += n;
  }
  const int total = __shfl_sync(FULL, incl, hbase + 15);

  // exact biased score of a survivor, and its 32-bit key relative to `base`
  const float* bias_l = bias_s;
  auto exact = [&](int id, float* s_out) -> float {
    const float s = __ldg(stab + sig_index(row[id]));
    *s_out = s;
    return __fadd_rn(s, bias_l[id]);
  };
  // every survivor has b'' >= the f16 cutoff applied above, so its exact b is at least
  // (that cutoff + o) - eps
  const float base = fsub_down(fadd_down(h_lo(cut2), pb.o), pb.eps);

  bool slow = __any_sync(FULL, total > 32) || !pb.ok;
  if (!slow) {
    int pos = incl - cnt;
    for (uint32_t m = ma; m; m &= m - 1u) ws.sid[half][pos++] = e0 + __ffs(m) - 1;
    for (uint32_t m = mb; m; m &= m - 1u) ws.sid[half][pos++] = e0 + kChain + __ffs(m) - 1;
    __syncwarp();
    // survivors 2h and 2h + 1 of this half (total >= 16, so both indices below exist;
    // the lookups of lanes past the total are discarded)
    const bool v0 = 2 * h < total, v1 = 2 * h + 1 < total;
    uint32_t k0 = 0, k1 = 0;
    float s0, s1;
    const float bx0 = exact(ws.sid[half][min(2 * h, total - 1)], &s0);
    const float bx1 = exact(ws.sid[half][min(2 * h + 1, total - 1)], &s1);
    if (v0) ws.ss[half][2 * h] = s0;
    if (v1) ws.ss[half][2 * h + 1] = s1;
    __syncwarp();  // the survivors' exact scores are read by the slot owners below
    // keys of 32 bits: every survivor's exact b is at least base, so they fit when base is
    // positive and each lies less than 2^26 float steps above it
    const uint32_t bb = __float_as_uint(base);
    const bool keys32 = base > 0.0f && (!v0 || __float_as_uint(bx0) - bb < (1u << 26)) &&
                        (!v1 || __float_as_uint(bx1) - bb < (1u << 26));
    if (__all_sync(FULL, keys32)) {
      if (v0) k0 = ((__float_as_uint(bx0) - bb + 1u) << 5) | uint32_t(31 - 2 * h);
      if (v1) k1 = ((__float_as_uint(bx1) - bb + 1u) << 5) | uint32_t(30 - 2 * h);
      bitonic32_u32(k0, k1, h);
      // positions 0..15 (lanes 0..7 of the half) are slots 0..15
      if (h < 8) {
        const int p0 = 31 - int(k0 & 31u), p1 = 31 - int(k1 & 31u);
        ws.slot_id[half][2 * h] = ws.sid[half][p0];
        ws.slot_s[half][2 * h] = ws.ss[half][p0];
        ws.slot_id[half][2 * h + 1] = ws.sid[half][p1];
        ws.slot_s[half][2 * h + 1] = ws.ss[half][p1];
      }
    } else {
      slow = true;
    }
  }
  if (slow) {
    if (pb.ok && !__any_sync(FULL, total > 64)) {
      // 33 to 64 survivors (many experts within the error band of the cutoff): four per
      // lane, their ids as 16-bit values in the id scratch, 32-bit keys (exact b relative
      // to the cutoff, then position) in a 64-key sort; the 16 winners' scores are looked
      // up again by the slot lanes
      uint16_t* sid16 = reinterpret_cast<uint16_t*>(ws.sid[half]);
      int pos = incl - cnt;
      for (uint32_t m = ma; m; m &= m - 1u) sid16[pos++] = static_cast<uint16_t>(e0 + __ffs(m) - 1);
      for (uint32_t m = mb; m; m &= m - 1u) sid16[pos++] = static_cast<uint16_t>(e0 + kChain + __ffs(m) - 1);
      __syncwarp();
      const uint32_t bb = __float_as_uint(base);
      uint32_t kq[4];
      bool fit = base > 0.0f;
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int q = 4 * h + e;
        float se;
        const float bx = exact(sid16[min(q, total - 1)], &se);
        kq[e] = 0u;
        if (q < total) {
          fit = fit && __float_as_uint(bx) - bb < (1u << 26) - 1u;  // (range + 1) << 6 fits
          kq[e] = ((__float_as_uint(bx) - bb + 1u) << 6) | uint32_t(63 - q);
        }
      }
      if (__all_sync(FULL, fit)) {
        bitonic64_u32(kq, h);
        // positions 0..15 (lanes 0..3 of the half) are slots 0..15
        if (h < 4) {
#pragma unroll
          for (int e = 0; e < 4; ++e) ws.slot_id[half][4 * h + e] = sid16[63 - int(kq[e] & 63u)];
        }
        __syncwarp();
        ws.slot_s[half][h] = __ldg(stab + sig_index(row[ws.slot_id[half][h]]));
        slow = false;
      }
      __syncwarp();  // the id scratch is rewritten below when the keys did not fit
    }
    if (slow) {
      // exact extraction: 16 rounds, each lane offering its best remaining survivor; equal
      // scores go to the lower lane (lower ids)
      uint32_t ra = ma, rb = mb;
      const uint32_t hmask = 0xFFFFu << hbase;
      for (int j = 0; j < K; ++j) {
        uint32_t best = 0u;
        int bid = -1;
        float bs = 0.0f;
        for (uint32_t m = ra; m; m &= m - 1u) {
          const int id = e0 + __ffs(m) - 1;
          float si;
          const uint32_t kq = fkey(exact(id, &si));
          if (kq > best) {
            best = kq;
            bid = id;
            bs = si;
          }
        }
        for (uint32_t m = rb; m; m &= m - 1u) {
          const int id = e0 + kChain + __ffs(m) - 1;
          float si;
          const uint32_t kq = fkey(exact(id, &si));
          if (kq > best) {
            best = kq;
            bid = id;
            bs = si;
          }
        }
        const uint32_t top = half_max(best);
        const uint32_t cand = __ballot_sync(FULL, best == top && bid >= 0) & hmask;
        const int win = __ffs(cand) - 1;
        if (lane == win) {
          ws.slot_id[half][j] = bid;
          ws.slot_s[half][j] = bs;
          if (bid < e0 + kChain) ra &= ~(1u << (bid - e0));
          else rb &= ~(1u << (bid - e0 - kChain));
        }
      }
    }
  }
  __syncwarp();

  // ---- weights from the exact scores in slot order; relabel; pack (lane h = slot h)
  SlotOut out;
  float den = 0.0f;
  {
    const float4* s4 = reinterpret_cast<const float4*>(ws.slot_s[half]);
#pragma unroll
    for (int q = 0; q < K / 4; ++q) {
      const float4 u = s4[q];
      den = __fadd_rn(__fadd_rn(__fadd_rn(__fadd_rn(den, u.x), u.y), u.z), u.w);
    }
  }
  out.id = ws.slot_id[half][h];
  const float s = ws.slot_s[half][h];
  const float w = __fmul_rn(__fdiv_rn(s, den), a.scale);
  const uint32_t wb = f32_to_bf16_bits(w);
  int lid = out.id;
  if (a.cnt > 0) lid = (out.id >= a.off && out.id < a.off + a.cnt) ? out.id - a.off : a.cnt + h;
  out.lid = lid;
  out.packed = static_cast<int32_t>((static_cast<uint32_t>(lid) << 16) | wb);
  __syncwarp();
  return out;
}

}  // namespace moe
