// router_gemm.cu -- step a0: logits[t][e] = sum_h hidden[t][h] * W[e][h] for decode
// batches (T <= 64), bf16 operands, fp32 accumulation, on the 5th-generation tensor
// cores.  The epilogue also applies the score function s = sigmoid(logit), so the
// routing kernel that follows starts from float32 scores.
//
// The router weight (896 x 7168 bf16, 12.85 MB) dominates the traffic: at T <= 64 the
// contraction does at most ~64 flop per weight byte, so it is bound by reading W once.
// Layout of the work (swap-AB, so the experts fill the MMA's M = 128 and the few
// tokens its N = T rounded up to 16):
//   grid = 7 expert tiles x C K-splits, one thread-block cluster of C CTAs per tile
//   (C = 16 when the GPU schedules such clusters, else 8);
//   each CTA streams its 128 x (H / C) slice of W with 2-D TMA loads (128-byte swizzle)
//   into a ring of shared-memory stages, issued at entry (the weight is a constant);
//   after the dependency wait, one 3-D TMA load brings the matching hidden columns of
//   the first ring's worth of stages (one 64-column tile per stage);
//   one elected lane of a converged warp issues tcgen05.mma (kind::f16, bf16 x bf16 ->
//   fp32) into a 128 x N accumulator in tensor memory, back to back over the ring;
//   the 4 warps read the accumulator (tcgen05.ld) into local staging rows (the T valid
//   token columns of each expert row), and C lanes each send one bulk copy to one
//   cluster CTA with the rows of the experts it owns (distributed shared memory,
//   completion counted on the owner's mbarrier); each CTA sums its 128 / C experts' C
//   partial rows in a fixed order (deterministic) and writes their logits and scores.
// Only the thread that loads the hidden rows waits for the preceding kernel early; the
// rest wait just before the global writes.
// All mbarrier waits are bounded; tensor memory is released on every path; every CTA
// sends its copies whatever its own waits gave, and none leaves while a peer's copy may
// still land in it.
#include <cuda.h>
#include <cooperative_groups.h>

#include "launch.h"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kGemmThreads = 128;
constexpr int kBM = 128;               // experts per tile (MMA M)
constexpr int kBK = 64;                // K per stage: one 128-byte swizzle row of bf16
constexpr int kStageW = kBM * kBK * 2; // 16 KB of W per stage
constexpr int kStageH = 64 * kBK * 2;  // room for N <= 64 token rows: 8 KB per stage
constexpr int kMaxStages = 7;
constexpr int kTmemCols = 64;
constexpr int kRowPad = 64 + 4;       // longest partial row: 64 token sums + padding
constexpr int kRecvBytes = kBM * kRowPad * 4;  // receive rows: C sources x (128/C) rows

struct GemmArgs {
  float* logits;  // [T, E] fp32 logits out, or nullptr
  float* scores;  // [T, E] fp32 sigmoid(logits) out (read by the routing kernel)
  const float2* etab;  // 2^(j/64) table of the float32 score function
  int T, Tpad, E;
  int kb_per_cta; // 64-wide K blocks per CTA
  int stages;     // ring depth (the first `stages` hidden tiles come in one 3-D load)
  int* err;
};

__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  // tcgen05 shared-memory matrix descriptor: K-major operand, 128-byte swizzle, 8-row
  // groups 1024 bytes apart (stride byte offset), descriptor version 1.
  uint64_t d = uint64_t((saddr & 0x3FFFFu) >> 4);
  d |= uint64_t(16 >> 4) << 16;    // leading byte offset (unused for swizzled K-major)
  d |= uint64_t(1024 >> 4) << 32;  // stride byte offset
  d |= uint64_t(1) << 46;          // version
  d |= uint64_t(2) << 61;          // SWIZZLE_128B
  return d;
}

__device__ __forceinline__ uint32_t mma_idesc(int n) {
  // kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major, M = 128, N = n
  return (1u << 4) | (1u << 7) | (1u << 10) | (uint32_t(n >> 3) << 17) | (uint32_t(kBM >> 4) << 24);
}

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* tm, int x, int y,
                                            int z, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes "
      "[%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
      "l"(tm), "r"(x), "r"(y), "r"(z), "r"(bar)
      : "memory");
}

// One MMA (or commit) issued by a single lane that elect.sync picks; the whole warp
// executes the instruction stream, so the operands are warp-uniform.
__device__ __forceinline__ void mma_bf16_elect(uint32_t tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                               int accumulate) {
  asm volatile(
      "{\n\t.reg .pred e, p;\n\telect.sync _|e, 0xffffffff;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "@e tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void mma_commit_elect(uint32_t bar) {
  asm volatile(
      "{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\t"
      "@e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(bar)
      : "memory");
}

__device__ __forceinline__ uint32_t mapa_cluster(uint32_t local_saddr, int rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(local_saddr), "r"(rank));
  return r;
}


// This warp's 32 accumulator lanes (one expert row each), columns 0 .. n-1 for the
// narrowest load shape that covers n = Tpad (16, 32 or 64 columns) into v[0 ..].
__device__ __forceinline__ void tmem_ld_row(uint32_t ta, uint32_t (&v)[64], int n) {
  if (n <= 16) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15])
                 : "r"(ta)
                 : "memory");
  } else if (n <= 32) {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31])
                 : "r"(ta)
                 : "memory");
  } else {
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
                 : "=r"(v[0]), "=r"(v[1]), "=r"(v[2]), "=r"(v[3]), "=r"(v[4]), "=r"(v[5]), "=r"(v[6]), "=r"(v[7]), "=r"(v[8]), "=r"(v[9]), "=r"(v[10]), "=r"(v[11]), "=r"(v[12]), "=r"(v[13]), "=r"(v[14]), "=r"(v[15]), "=r"(v[16]), "=r"(v[17]), "=r"(v[18]), "=r"(v[19]), "=r"(v[20]), "=r"(v[21]), "=r"(v[22]), "=r"(v[23]), "=r"(v[24]), "=r"(v[25]), "=r"(v[26]), "=r"(v[27]), "=r"(v[28]), "=r"(v[29]), "=r"(v[30]), "=r"(v[31]), "=r"(v[32]), "=r"(v[33]), "=r"(v[34]), "=r"(v[35]), "=r"(v[36]), "=r"(v[37]), "=r"(v[38]), "=r"(v[39]), "=r"(v[40]), "=r"(v[41]), "=r"(v[42]), "=r"(v[43]), "=r"(v[44]), "=r"(v[45]), "=r"(v[46]), "=r"(v[47]), "=r"(v[48]), "=r"(v[49]), "=r"(v[50]), "=r"(v[51]), "=r"(v[52]), "=r"(v[53]), "=r"(v[54]), "=r"(v[55]), "=r"(v[56]), "=r"(v[57]), "=r"(v[58]), "=r"(v[59]), "=r"(v[60]), "=r"(v[61]), "=r"(v[62]), "=r"(v[63])
                 : "r"(ta)
                 : "memory");
  }
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__global__ void __launch_bounds__(kGemmThreads, 1)
    k_router_gemm(const __grid_constant__ CUtensorMap tmW, const __grid_constant__ CUtensorMap tmH,
                  const __grid_constant__ CUtensorMap tmH3, GemmArgs g) {
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  // 1024-byte alignment for the swizzled stages
  // (offset from the shared array itself, so the compiler keeps shared-memory accesses)
  uint8_t* smem = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  cg::cluster_group cluster = cg::this_cluster();
  const int C = static_cast<int>(cluster.num_blocks());
  const int r = static_cast<int>(cluster.block_rank());
  const int R = kBM / C;  // experts whose logits this CTA finishes
  const int mtile = blockIdx.x / C;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int NS = g.stages;
  // the routing kernel that reads this kernel's scores may launch now; it waits for
  // this grid's completion (griddepcontrol.wait) before it reads them
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");

  // [W ring: NS x 16 KB][hidden ring: NS x Tpad x 128 B][receive rows][barriers][table]
  uint8_t* wring = smem;
  uint8_t* hring = smem + kMaxStages * kStageW;
  const uint32_t htile = uint32_t(g.Tpad * kBK * 2);  // bytes of one stage's hidden tile
  float* recv = reinterpret_cast<float*>(smem + kMaxStages * (kStageW + kStageH));  // [C][R][rs]
  uint64_t* fullW = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(recv) + kRecvBytes);
  uint64_t* fullH = fullW + kMaxStages;  // refills of the hidden ring (stage kb >= NS)
  uint64_t* empty = fullH + kMaxStages;
  uint64_t* hfirst = empty + kMaxStages;  // the first NS hidden tiles (one 3-D load)
  uint64_t* done = hfirst + 1;
  uint64_t* recv_bar = done + 1;  // the 128 partial rows this CTA receives
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(recv_bar + 1);
  // the 2^(j/64) table of the epilogue's score function, staged once (512 bytes)
  float2* etab_s = reinterpret_cast<float2*>(recv_bar + 2);
  if (threadIdx.x < kExpTable) etab_s[threadIdx.x] = g.etab[threadIdx.x];
  const int kb0 = r * g.kb_per_cta;
  const int n0 = NS < g.kb_per_cta ? NS : g.kb_per_cta;  // stages of the first fill
  // partial and receive rows hold the T token sums, rounded up to whole float4s, + 4
  // floats of padding
  const int rs = ((g.T + 3) & ~3) + 4;

  if (threadIdx.x == 0) {
    // barriers, then the first fill of the W ring (the ring holds the whole K slice when
    // it fits; otherwise the producer loop below refills freed stages)
    for (int s = 0; s < NS; ++s) {
      mbar_init(fullW + s, 1);
      mbar_init(fullH + s, 1);
      mbar_init(empty + s, 1);
    }
    mbar_init(hfirst, 1);
    mbar_init(done, 1);
    mbar_init(recv_bar, 1);
    fence_mbar_init();
    // the weight is read as a constant: its loads start before the preceding kernel on
    // the stream has completed (this grid is a programmatic dependent)
    for (int kb = 0; kb < n0; ++kb) {
      mbar_expect_tx(fullW + kb, kStageW);
      tma_load_2d(smem_addr(wring + kb * kStageW), &tmW, (kb0 + kb) * kBK, mtile * kBM,
                  smem_addr(fullW + kb));
    }
  }
  if (warp == 1) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_addr(tmem_slot)),
                 "r"(kTmemCols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  // every CTA of the cluster runs, with its barriers initialised, before any peer stores
  // into its shared memory; the arrive is relaxed so that it does not wait for this
  // CTA's TMA loads in flight
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = *tmem_slot;

  if (threadIdx.x == 0) {
    // the hidden rows depend on the preceding kernel.  Only this thread waits for it
    // here: the others wait just before the global writes at the end, and the MMA warp
    // and the epilogue touch only shared and tensor memory.  (While every thread of the
    // CTA sat in this wait, most of the weight tiles issued above did not land until
    // it returned.)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    // hidden tiles of the first fill: box (64 columns, Tpad rows, n0 K blocks), rows past
    // T read as zeros; lands as n0 consecutive Tpad x 64 tiles
    mbar_expect_tx(hfirst, htile * uint32_t(n0));
    tma_load_3d(smem_addr(hring), &tmH3, 0, 0, kb0, smem_addr(hfirst));
    mbar_expect_tx(recv_bar, uint32_t(C * R * rs * 4));  // C partial blocks will arrive
    // producer: refill stages freed by the MMAs (only when the K slice exceeds the ring)
    for (int kb = NS; kb < g.kb_per_cta; ++kb) {
      const int s = kb % NS;
      if (!mbar_wait_bounded(empty + s, uint32_t((kb / NS - 1) & 1), g.err)) break;
      const int k = (kb0 + kb) * kBK;
      mbar_expect_tx(fullW + s, kStageW);
      tma_load_2d(smem_addr(wring + s * kStageW), &tmW, k, mtile * kBM, smem_addr(fullW + s));
      mbar_expect_tx(fullH + s, htile);
      tma_load_2d(smem_addr(hring + s * htile), &tmH, k, 0, smem_addr(fullH + s));
    }
  } else if (warp == 1) {
    // MMA issuer: 4 MMAs of K = 16 per 64-wide stage, from one elected lane (every lane
    // waits, so the lane that elect.sync picks has observed the data).  The first fill is
    // unrolled over the ring with compile-time descriptor offsets and no waits between
    // its MMAs: issued from a runtime loop with a wait per stage, these small MMAs went
    // out at about a third of the rate.
    const uint32_t idesc = mma_idesc(g.Tpad);
    const uint64_t ad0 = sw128_desc(smem_addr(wring));
    const uint64_t bd0 = sw128_desc(smem_addr(hring));
    const uint32_t hstep = htile >> 4;  // descriptor units (16 bytes) per hidden tile
    // the weight tiles land first (they were issued at entry), then the hidden tiles
    bool ok = true;
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s)
      if (s < n0 && ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(fullW + s, 0, g.err));
    if (ok) ok = __all_sync(0xffffffffu, mbar_wait_bounded(hfirst, 0, g.err));
#pragma unroll
    for (int s = 0; s < kMaxStages; ++s) {
      if (s < n0 && ok) {
        const uint64_t ad = ad0 + uint64_t(s * (kStageW >> 4));
        const uint64_t bd = bd0 + uint64_t(s) * hstep;
#pragma unroll
        for (int k = 0; k < kBK / 16; ++k)
          mma_bf16_elect(tmem, ad + uint64_t(2 * k), bd + uint64_t(2 * k), idesc, (s | k) != 0);
        // the producer refills this stage only when the K slice exceeds the ring
        if (s + NS < g.kb_per_cta) mma_commit_elect(smem_addr(empty + s));
      }
    }
    for (int kb = NS; ok && kb < g.kb_per_cta; ++kb) {
      const int s = kb % NS, f = kb / NS;
      bool mine = mbar_wait_bounded(fullW + s, uint32_t(f & 1), g.err);
      if (mine) mine = mbar_wait_bounded(fullH + s, uint32_t((f - 1) & 1), g.err);
      ok = __all_sync(0xffffffffu, mine);
      if (!ok) break;
      const uint64_t ad = ad0 + uint64_t(s * (kStageW >> 4));
      const uint64_t bd = bd0 + uint64_t(s) * hstep;
#pragma unroll
      for (int k = 0; k < kBK / 16; ++k)
        mma_bf16_elect(tmem, ad + uint64_t(2 * k), bd + uint64_t(2 * k), idesc, 1);
      if (kb + NS < g.kb_per_cta) mma_commit_elect(smem_addr(empty + s));
      __syncwarp();
    }
    // arrives once every MMA issued above has completed (at once if none was issued)
    mma_commit_elect(smem_addr(done));
    __syncwarp();
  }
  __syncwarp();

  // ---- epilogue: accumulator -> this thread's expert row of partial sums (its T valid
  // columns) -> the cluster CTA that owns the expert
  const bool acc_ok = mbar_wait_bounded(done, 0, g.err);
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const int e_row = warp * 32 + lane;  // this thread's expert row of the tile
  const int Tq = (g.T + 3) & ~3;       // columns sent, rounded up to whole float4s
  float* stage_rows = reinterpret_cast<float*>(wring);  // [128][rs]: the ring is free now
  if (acc_ok) {
    uint32_t v[64];
    tmem_ld_row(tmem + (uint32_t(warp * 32) << 16), v, g.Tpad);
    float4* d4 = reinterpret_cast<float4*>(stage_rows + e_row * rs);
#pragma unroll
    for (int c = 0; c < 16; ++c)
      if (4 * c < Tq)
        d4[c] = make_float4(__uint_as_float(v[4 * c]), __uint_as_float(v[4 * c + 1]),
                            __uint_as_float(v[4 * c + 2]), __uint_as_float(v[4 * c + 3]));
  }
  fence_proxy_async_smem();  // staging rows visible to the bulk-copy engine
  // the accumulator reads are complete: warp 1 frees tensor memory
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  if (warp == 1)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols)
                 : "memory");
  if (warp == 0 && lane < C) {
    // lane o sends rows [o R, o R + R) to CTA o, into its receive slot for source r
    const uint32_t src = smem_addr(stage_rows + lane * R * rs);
    const uint32_t dst = mapa_cluster(smem_addr(recv + r * R * rs), lane);
    const uint32_t bar = mapa_cluster(smem_addr(recv_bar), lane);
    asm volatile(
        "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
        "[%3];" ::"r"(dst),
        "r"(src), "r"(uint32_t(R * rs * 4)), "r"(bar)
        : "memory");
    asm volatile("cp.async.bulk.commit_group;" ::: "memory");
  }
  const bool recv_ok = mbar_wait_bounded(recv_bar, 0, g.err);

  // ---- this CTA's R experts: sum the C partial rows in source order, then the scores
  // (written only once the preceding kernel, which may still read the last ones, is done)
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (!recv_ok) {
    // a peer's rows may still be on their way: every peer sends them once its own
    // bounded waits (at most kb_per_cta + 2 of them, each ending at the first one that
    // runs out) are over; wait that long again before leaving
    const uint64_t t0 = globaltimer_ns();
    const uint64_t limit = uint64_t(g.kb_per_cta + 3) * kWaitLimitNs;
    while (!mbar_try_wait(recv_bar, 0) && globaltimer_ns() - t0 < limit) {
    }
  } else if (R * g.T <= kGemmThreads) {
    // few tokens: one (expert, token) pair per thread, shortest chain
    const int idx = threadIdx.x;
    if (idx < R * g.T) {
      const int t = idx % g.T, i = idx / g.T;
      float acc = 0.0f;
#pragma unroll 8
      for (int c = 0; c < C; ++c) acc = __fadd_rn(acc, recv[(c * R + i) * rs + t]);
      const int e = mtile * kBM + r * R + i;
      if (g.logits) g.logits[size_t(t) * g.E + e] = acc;
      g.scores[size_t(t) * g.E + e] = sig_f32(acc, etab_s);
    }
  } else {
    const int ngrp = R / 4;
    for (int idx = threadIdx.x; idx < ngrp * g.T; idx += kGemmThreads) {
      const int t = idx % g.T, i0 = (idx / g.T) * 4;
      float acc[4] = {0.0f, 0.0f, 0.0f, 0.0f};
#pragma unroll 4
      for (int c = 0; c < C; ++c) {
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[q] = __fadd_rn(acc[q], recv[(c * R + i0 + q) * rs + t]);
      }
      const int e = mtile * kBM + r * R + i0;
      if (g.logits)
        *reinterpret_cast<float4*>(g.logits + size_t(t) * g.E + e) =
            make_float4(acc[0], acc[1], acc[2], acc[3]);
      *reinterpret_cast<float4*>(g.scores + size_t(t) * g.E + e) =
          make_float4(sig_f32(acc[0], etab_s), sig_f32(acc[1], etab_s), sig_f32(acc[2], etab_s),
                      sig_f32(acc[3], etab_s));
    }
  }
  if (warp == 0 && lane < C) asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// ------------------------------------------------------------------- host side
namespace {

using EncodeTiled = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                 const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                 const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                 CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiled g_encode = nullptr;
int g_cluster = 0;

bool make_map(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_inner,
              uint32_t box_outer) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {inner * 2};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t estr[2] = {1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// hidden [T][H] as a 3-D tensor (64 columns, T rows, H / 64 column blocks): a box of
// (64, Tpad, n) lands as n consecutive Tpad x 64 tiles, one per K block
bool make_map_blocks(CUtensorMap* m, const void* base, uint64_t H, uint64_t T, uint32_t Tpad,
                     uint32_t n) {
  const cuuint64_t dims[3] = {uint64_t(kBK), T, H / kBK};
  const cuuint64_t strides[2] = {H * 2, uint64_t(kBK) * 2};
  const cuuint32_t box[3] = {uint32_t(kBK), Tpad, n};
  const cuuint32_t estr[3] = {1, 1, 1};
  return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// 24 mbarriers + the tensor-memory slot fit the 256 bytes after the receive rows
constexpr int kGemmSmem = kMaxStages * (kStageW + kStageH) + kRecvBytes + 1024 /*align*/ +
                          256 /*barriers*/ + kExpTable * 8 /*score table*/;
static_assert((3 * kMaxStages + 3) * 8 + 8 <= 256, "barriers exceed their room");
static_assert(kGemmSmem <= 227 * 1024, "router contraction smem exceeds 227 KB");

}  // namespace

cudaError_t setup_router_gemm() {
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                     cudaEnableDefault, &q);
    if (e != cudaSuccess || fn == nullptr || q != cudaDriverEntryPointSuccess)
      return e != cudaSuccess ? e : cudaErrorNotSupported;
    g_encode = reinterpret_cast<EncodeTiled>(fn);
  }
  cudaError_t e =
      cudaFuncSetAttribute(k_router_gemm, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem);
  if (e != cudaSuccess) return e;
  // prefer clusters of 16 K-splits when the GPU can schedule 7 of them at once
  g_cluster = 8;
  if (cudaFuncSetAttribute(k_router_gemm, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) ==
      cudaSuccess) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(7 * 16, 1, 1);
    cfg.blockDim = dim3(kGemmThreads, 1, 1);
    cfg.dynamicSmemBytes = kGemmSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int nclusters = 0;
    if (cudaOccupancyMaxActiveClusters(&nclusters, k_router_gemm, &cfg) == cudaSuccess &&
        nclusters >= 7)
      g_cluster = 16;
  }
  cudaGetLastError();  // clear a refused query
  return cudaSuccess;
}

int router_gemm_cluster() { return g_cluster; }

cudaError_t launch_router_gemm(const uint16_t* hidden, const uint16_t* w, float* logits,
                               float* scores, const float2* etab, int T, int H, int E, int* err,
                               cudaStream_t st) {
  const int Tpad = (T + 15) / 16 * 16;
  const int C = g_cluster;
  const int nkb = H / kBK;
  if (Tpad > 64 || nkb % C != 0 || E % kBM != 0) return cudaErrorInvalidValue;
  const int kb_per_cta = nkb / C;
  const int stages = kb_per_cta < kMaxStages ? kb_per_cta : kMaxStages;
  // tensor maps depend only on (pointer, shape): reuse the last ones when unchanged
  static thread_local CUtensorMap tmW, tmH, tmH3;
  static thread_local const void* w_key = nullptr;
  static thread_local int w_h = 0, w_e = 0;
  static thread_local const void* h_key = nullptr;
  static thread_local int h_t = 0, h_h = 0, h_n = 0;
  if (w != w_key || H != w_h || E != w_e) {
    w_key = nullptr;
    if (!make_map(&tmW, w, uint64_t(H), uint64_t(E), kBK, kBM)) return cudaErrorInvalidValue;
    w_key = w;
    w_h = H;
    w_e = E;
  }
  if (hidden != h_key || T != h_t || H != h_h || stages != h_n) {
    h_key = nullptr;
    if (!make_map(&tmH, hidden, uint64_t(H), uint64_t(T), kBK, uint32_t(Tpad)) ||
        !make_map_blocks(&tmH3, hidden, uint64_t(H), uint64_t(T), uint32_t(Tpad), uint32_t(stages)))
      return cudaErrorInvalidValue;
    h_key = hidden;
    h_t = T;
    h_h = H;
    h_n = stages;
  }
  GemmArgs g = {};
  g.logits = logits;
  g.scores = scores;
  g.etab = etab;
  g.T = T;
  g.Tpad = Tpad;
  g.E = E;
  g.kb_per_cta = kb_per_cta;
  g.stages = stages;
  g.err = err;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((E / kBM) * C, 1, 1);
  cfg.blockDim = dim3(kGemmThreads, 1, 1);
  cfg.dynamicSmemBytes = kGemmSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_router_gemm, tmW, tmH, tmH3, g);
}

}  // namespace moe
