// route_prefill_fast.cu -- prefill-size routing of bf16 logits for the Kimi-K3 instance
// (E = 896 in 8 groups, k = 16, keep 4 groups) in one persistent, cooperative launch:
// one CTA of 20 warps per SM, a contiguous row range per CTA and per warp.  The exact
// score table stays in global memory (read through the L1 cache): only the survivors of
// each row, about 18 of 896, and the rare exact group scores look it up.
//
// Phase 1 (streaming): every warp keeps D pairs of rows in flight with one-dimensional
//   bulk copies into a private ring in shared memory and routes each pair with route_pair
//   (lanes 0-15 the first row, 16-31 the second; approximate scores, exact table lookups
//   only where a decision needs them).  Lane h of each half stores slot h, then counts
//   its relabelled id into the warp's own 16-bit counters (two per 32-bit word), first
//   row first; the counter's old value is the entry's rank among this warp's entries of
//   the same id, in (token, slot) order, since a warp routes its rows in order and ids
//   are unique in a row.  (id, rank) is kept in shared memory.
// CTA tail of phase 1: a column pass over the warps' counters gives each warp's prefix
//   per id and the CTA's histogram, which goes to the expert-major matrix hist[bin][cta].
//   The CTA then arrives at grid barrier 1 and, before it waits, a block scan gives the
//   CTA-local bin offsets and every entry is placed at its CTA-local position (bin
//   offset + warp prefix + rank) in a buffer that replaces the ring: the CTA's entries
//   sorted by (id, token, slot).
// Grid barrier 1 (wait), column scan over CTAs (prefixes and totals), grid barrier 2 (the
//   CTAs that own bins of the scan place their entries after it, before they wait).
// Phase 3: offsets from the totals (CTA 0 writes counts and offsets); the sorted buffer
//   goes to perm in runs of consecutive addresses, one run per bin.
// Index mode (moe_route_index, k = 16): phase 1 takes each warp's rows of given packed
//   ids in one bulk copy and only ranks them; everything after it is the same.
// Every wait is bounded in time; a wait that runs out sets the status word and the CTA
// leaves (through grid_exit, which restores the barrier words once all CTAs have left).
#include <cooperative_groups.h>

#include "persist.cuh"
#include "route_pair.cuh"

namespace moe {

namespace {

__host__ __device__ constexpr int f_align(int x, int a) { return (x + a - 1) / a * a; }

struct FastSmem {
  static constexpr int NW = 20;                    // warps per CTA
  static constexpr int D = 2;                      // pairs of rows in flight per warp
  static constexpr int ROWB = kE * 2;              // one bf16 row: 1,792 bytes
  static constexpr int SLOTB = 2 * ROWB;           // a pair of rows
  static constexpr int WORDS = kFastBins / 2;      // 16-bit counters, two per word
  static constexpr int o_bias = 0;
  static constexpr int o_cpp = f_align(o_bias + kE * 4, 128);   // c'' = bias + 0.5 - o, in pairs
  static constexpr int o_ring = f_align(o_cpp + kCppFloats * 4, 128);
  static constexpr int o_wcnt = o_ring + NW * D * SLOTB;
  static constexpr int o_ws = f_align(o_wcnt + NW * WORDS * 4, 128);
  static constexpr int o_hist = f_align(o_ws + NW * int(sizeof(PairScratch)), 128);
  static constexpr int o_lbase = f_align(o_hist + (kFastBins + 1) * 4, 128);
  static constexpr int o_gbase = f_align(o_lbase + (kFastBins + 1) * 4, 128);
  static constexpr int o_tmp = f_align(o_gbase + (kFastBins + 1) * 4, 128);
  static constexpr int o_mbar = f_align(o_tmp + 64 * 4, 128);
  static constexpr int o_ent = f_align(o_mbar + (NW * D + 1) * 8, 128);
  // (id, rank) of each entry, 16 bits (id | rank << 10), per warp, in the room left
  static constexpr int ENT_PER_WARP = (227 * 1024 - o_ent) / (NW * 2) / 32 * 32;
  static constexpr int ROWS_PER_WARP = ENT_PER_WARP / 16;
  static constexpr int total = o_ent + NW * ENT_PER_WARP * 2;
  // the CTA's sorted entries, in the ring once phase 1 is over: values, then bins
  static constexpr int SORT_CAP = (NW * D * SLOTB) / 6 / 8 * 8;
  static constexpr int o_sval = o_ring;
  static constexpr int o_sbin = o_ring + SORT_CAP * 4;
};

static_assert(FastSmem::total <= 227 * 1024, "fast prefill smem exceeds 227 KB");
static_assert(FastSmem::SORT_CAP >= FastSmem::NW * FastSmem::ENT_PER_WARP, "sorted entries fit the ring");
static_assert(FastSmem::ROWS_PER_WARP >= 22, "room for 65,536 rows on 152 SMs");
static_assert(FastSmem::ROWS_PER_WARP <= 64, "a rank within a warp fits 6 bits");
static_assert(kFastBins <= 1024, "an id fits 10 bits");
static_assert(2 * FastSmem::NW + 2 <= 64, "the bias range reduction and the barrier flag fit tmp");
static_assert(2 * (kFastBins + 1) * 4 <= FastSmem::NW * int(sizeof(PairScratch)),
              "phase 3's offsets and padded offsets fit the routing scratch");
static_assert(FastSmem::ROWB % 128 == 0, "row slots keep 128-byte alignment");
static_assert(160 * FastSmem::NW * 4 <= FastSmem::NW * FastSmem::D * FastSmem::SLOTB,
              "the column scan's tile for up to 160 CTAs fits the ring");

// Column scan over CTAs for the bins this CTA owns (warp w: bin blockIdx.x * NW + w, and
// further chunks grid * NW bins apart; called by every thread of every CTA): totals go to
// counts[e], and each CTA's exclusive prefix to the CTA-major matrix
// prefix[c * kMaxBins + e] through a [grid][NW] tile in shared memory (`tile`), so that a
// chunk's prefixes leave as one contiguous piece per CTA and phase 3 reads its own row of
// the matrix contiguously.
__device__ __forceinline__ void column_scan_cta_major(const PrefillWS& pw, int NE, int grid, int* tile) {
  constexpr int NW = FastSmem::NW, NT = NW * 32;
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e0 = int(blockIdx.x) * NW; e0 < NE; e0 += grid * NW) {  // uniform over the CTA
    const int e = e0 + w;
    if (e < NE) {
      const int* hrow = pw.hist + size_t(e) * pw.grid_max;
      int carry = 0;
      for (int c0 = 0; c0 < grid; c0 += 256) {
        const int span = min(256, grid - c0);
        const int per = (span + 31) / 32;
        const int cl = c0 + lane * per;
        int v[8];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          v[i] = (i < per && cl + i < c0 + span) ? __ldcg(hrow + cl + i) : 0;
          sum += v[i];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const int n = __shfl_up_sync(0xffffffffu, incl, o);
          if (lane >= o) incl += n;
        }
        int run = carry + incl - sum;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          if (i < per && cl + i < c0 + span) tile[(cl + i) * NW + w] = run;
          run += v[i];
        }
        carry += __shfl_sync(0xffffffffu, incl, 31);
      }
      if (lane == 0) pw.counts[e] = carry;
    }
    __syncthreads();
    const int nb = min(NW, NE - e0);
    for (int x = threadIdx.x; x < grid * nb; x += NT) {
      const int c = x / nb, j = x - c * nb;
      pw.prefix[size_t(c) * kMaxBins + e0 + j] = tile[c * NW + j];
    }
    __syncthreads();
  }
}

}  // namespace

int fast_prefill_rows_per_warp() { return FastSmem::ROWS_PER_WARP; }
int fast_prefill_warps() { return FastSmem::NW; }

// INDEX: index mode (moe_route_index for k = 16): phase 1 reads the given packed ids of
// each row (a.logits, 16-byte aligned: each warp's rows come in one bulk copy) instead of
// routing; an id >= NE, and every occurrence of an id that appears twice in its row, is
// reported (kErrBadId) and left out of every output.
// LAYOUT: phase 3 also writes the expert-GEMM layout (a.poffs, a.prows, a.midx).
template <bool INDEX, bool LAYOUT>
__global__ void __launch_bounds__(FastSmem::NW * 32, 1)
    k_route_prefill_fast(RouteArgs a, PrefillWS pw) {
  using L = FastSmem;
  constexpr int NW = L::NW;
  constexpr int NT = NW * 32;
  constexpr int K = 16;
  extern __shared__ __align__(128) uint8_t smem[];
  float* bias_s = reinterpret_cast<float*>(smem + L::o_bias);
  float* cpp_s = reinterpret_cast<float*>(smem + L::o_cpp);
  uint8_t* ring_all = smem + L::o_ring;
  uint32_t* wcnt_all = reinterpret_cast<uint32_t*>(smem + L::o_wcnt);
  PairScratch* wsp = reinterpret_cast<PairScratch*>(smem + L::o_ws);
  int* hist_s = reinterpret_cast<int*>(smem + L::o_hist);
  int* lbase_s = reinterpret_cast<int*>(smem + L::o_lbase);
  int* gbase_s = reinterpret_cast<int*>(smem + L::o_gbase);
  int* tmp = reinterpret_cast<int*>(smem + L::o_tmp);
  uint64_t* mbar_all = reinterpret_cast<uint64_t*>(smem + L::o_mbar);
  int* sval = reinterpret_cast<int*>(smem + L::o_sval);
  uint16_t* sbin = reinterpret_cast<uint16_t*>(smem + L::o_sbin);

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int grid = gridDim.x, cta = blockIdx.x;
  const int r0 = int((long long)a.T * cta / grid);
  const int r1 = int((long long)a.T * (cta + 1) / grid);
  const int per_warp = (r1 - r0 + NW - 1) / NW;
  const int wr0 = min(r1, r0 + w * per_warp);
  const int wr1 = min(r1, wr0 + per_warp);
  const int nw = wr1 - wr0;  // <= ROWS_PER_WARP (checked by the launcher)
  const int npairs = (nw + 1) / 2;
  uint8_t* ring = ring_all + w * L::D * L::SLOTB;
  uint64_t* mb = mbar_all + w * L::D;
  uint32_t* wcnt = wcnt_all + w * L::WORDS;
  uint16_t* ent = reinterpret_cast<uint16_t*>(smem + L::o_ent) + w * L::ENT_PER_WARP;
  const uint8_t* logits = static_cast<const uint8_t*>(a.logits);
  const int nwords = a.NE / 2;  // NE is a multiple of 4

  // the next launch on the stream (a programmatic dependent) may start now: before its
  // griddepcontrol.wait it touches only its own shared memory
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  // ---- setup: mbarriers, counters, score table and bias, first rows in flight
  uint64_t* tab_bar = mbar_all + NW * L::D;
  if (lane == 0) {
    for (int d = 0; d < L::D; ++d) mbar_init(mb + d, 1);
    if (w == 0) mbar_init(tab_bar, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < NW * L::WORDS; i += NT) wcnt_all[i] = 0u;
  __syncthreads();
  // inputs, outputs, the workspace and the grid barrier's words belong to the preceding
  // launch until it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0 && !INDEX) {
    mbar_expect_tx(tab_bar, uint32_t(kE * 4));
    bulk_g2s(bias_s, a.bias, kE * 4, tab_bar);
  }
  // rows 2p and 2p + 1 of this warp (the second may not exist) into slot p % D
  auto issue_pair = [&](int p) {
    const int slot = p % L::D;
    const uint32_t bytes = uint32_t(min(2, nw - 2 * p)) * L::ROWB;
    mbar_expect_tx(mb + slot, bytes);
    bulk_g2s(ring + slot * L::SLOTB, logits + size_t(wr0 + 2 * p) * L::ROWB, bytes, mb + slot);
  };
  if (lane == 0 && !INDEX) {
    for (int d = 0; d < L::D && d < npairs; ++d) issue_pair(d);
  }
  if (INDEX && lane == 0 && nw > 0) {
    // index mode: the warp's rows of packed ids (64 bytes each) in one bulk copy
    const uint32_t bytes = uint32_t(nw) * K * 4;
    mbar_expect_tx(mb, bytes);
    bulk_g2s(ring, static_cast<const uint8_t*>(a.logits) + size_t(wr0) * K * 4, bytes, mb);
  }
  // first row whose wait ran out (-1: none); 0 also when the table never arrived
  int fail_at = -1;
  if constexpr (!INDEX) fail_at = mbar_wait_bounded(tab_bar, 0, a.err) ? -1 : 0;

  const int half = lane >> 4, h = lane & 15;
  if constexpr (INDEX) {
    // ---- phase 1 (index mode): the warp's rows two at a time (lanes 0-15 and 16-31)
    //      from its bulk copy; ranks as in routing
    __syncthreads();
    if (nw > 0 && !mbar_wait_bounded(mb, 0, a.err)) fail_at = 0;
    const uint32_t* ids = reinterpret_cast<const uint32_t*>(ring);
    {
      for (int p = 0; p < npairs && fail_at < 0; ++p) {
        const int i = 2 * p + half;
        const bool valid = i < nw;
        const int lid = int((valid ? ids[i * K + h] : 0u) >> 16);
        const bool inr = valid && lid < a.NE;
        const uint32_t sh = uint32_t(lid & 1) * 16u;
        // ranks: the first row's entries before the second row's.  Ids must be distinct
        // within a row (the ranks count rows per id): after a row's increments, a lane whose
        // counter rose by more than one shares its id with another lane of the row (in
        // every repeat the lane that counted first sees it); only then is every occurrence
        // found (a match over the half) and its increments taken back.
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          const bool mine = half == hh && inr;
          uint32_t old = 0u;
          if (mine) old = atomicAdd(wcnt + (lid >> 1), 1u << sh);
          __syncwarp();
          const uint32_t rank = (old >> sh) & 0xFFFFu;
          const bool suspect = mine && ((wcnt[lid >> 1] >> sh) & 0xFFFFu) - rank != 1u;
          bool dup = false;
          if (__any_sync(0xffffffffu, suspect)) {
            const uint32_t same = __match_any_sync(0xffffffffu, uint32_t(lid) | (uint32_t(half) << 16));
            dup = mine && __popc(same) > 1;
            __syncwarp();
            if (dup) atomicSub(wcnt + (lid >> 1), 1u << sh);
          }
          if (half == hh && valid) {
            if (!inr || dup) atomicExch(a.err, kErrBadId);
            ent[i * K + h] = (inr && !dup) ? static_cast<uint16_t>(uint32_t(lid) | (rank << 10)) : uint16_t(0xFFFFu);
          }
          __syncwarp();
        }
      }
    }
  } else {
    // error bounds of the approximate scores: the biases' range
    PairBounds pbnd;
    {
      float mx = -INFINITY, mn = INFINITY;
      for (int e = tid; e < kE; e += NT) {
        mx = fmaxf(mx, bias_s[e]);
        mn = fminf(mn, bias_s[e]);
      }
      // order-preserving keys, so that integer reductions give the float max and min
      const uint32_t kmx = __reduce_max_sync(0xffffffffu, fkey(mx));
      const uint32_t kmn = __reduce_min_sync(0xffffffffu, fkey(mn));
      if (lane == 0) {
        tmp[w] = int(kmx);
        tmp[NW + w] = int(kmn);
      }
      __syncthreads();
      uint32_t bmx = 0u, bmn = 0xFFFFFFFFu;
  #pragma unroll
      for (int i = 0; i < NW; ++i) {
        bmx = max(bmx, uint32_t(tmp[i]));
        bmn = min(bmn, uint32_t(tmp[NW + i]));
      }
      pbnd = pair_bounds(a.eps_half, fkey_inv(bmn), fkey_inv(bmx));
    }
    // c'' in the pair order route_pair reads: lane h's word j pairs expert 56 h + j with
    // expert 56 h + 28 + j
    for (int e = tid; e < kE; e += NT) {
      const int hh = e / kPairEPL, r = e - hh * kPairEPL;
      const int c = r >= kChain ? 1 : 0, j = r - c * kChain;
      cpp_s[hh * kCppStride + 2 * j + c] = __fadd_rn(bias_s[e], pbnd.d0);
    }
    __syncthreads();

    // ---- phase 1: route this warp's rows two at a time, rank their entries within the warp
    for (int p = 0; p < npairs && fail_at < 0; ++p) {
      const int slot = p % L::D;
      const uint32_t par = uint32_t(p / L::D) & 1u;
      if (!mbar_wait_bounded(mb + slot, par, a.err)) {
        fail_at = p;
        break;
      }
      const uint8_t* r0p = ring + slot * L::SLOTB;
      const bool has1 = 2 * p + 1 < nw;
      const SlotOut o = route_pair(r0p, has1 ? r0p + L::ROWB : r0p, bias_s, cpp_s, a.stab, pbnd, a, wsp[w]);
      const int i = 2 * p + half;  // this half's row within the warp
      const bool valid = i < nw;
      const int t = wr0 + i;
      if (valid) {
        a.packed[size_t(t) * K + h] = o.packed;
        if (a.ids) a.ids[size_t(t) * K + h] = o.id;
      }
      // ranks: the first row's entries before the second row's
      const uint32_t sh = uint32_t(o.lid & 1) * 16u;
      if (half == 0) {
        const uint32_t old = atomicAdd(wcnt + (o.lid >> 1), 1u << sh);
        ent[i * K + h] = static_cast<uint16_t>(uint32_t(o.lid) | (((old >> sh) & 0xFFFFu) << 10));
      }
      __syncwarp();
      if (half == 1 && valid) {
        const uint32_t old = atomicAdd(wcnt + (o.lid >> 1), 1u << sh);
        ent[i * K + h] = static_cast<uint16_t>(uint32_t(o.lid) | (((old >> sh) & 0xFFFFu) << 10));
      }
      __syncwarp();
      if (lane == 0 && p + L::D < npairs) {
        fence_proxy_async_smem();
        issue_pair(p + L::D);
      }
    }
  }
  // after a wait that ran out, the copies issued for pairs fail_at .. fail_at + D - 1 may
  // still be owed to the ring: wait for them (bounded) before the ring is reused
  if (fail_at >= 0 && lane == 0) {
    if (INDEX) {
      if (nw > 0) mbar_wait_bounded(mb, 0, nullptr);  // the one bulk copy of index mode
    } else {
      if (w == 0) mbar_wait_bounded(tab_bar, 0, nullptr);
      for (int q = fail_at; q < npairs && q < fail_at + L::D; ++q)
        mbar_wait_bounded(mb + q % L::D, uint32_t(q / L::D) & 1u, nullptr);
    }
  }
  __syncthreads();

  // ---- CTA tail of phase 1: warp prefixes per id (in place) and the CTA histogram
  for (int q = tid; q < nwords; q += NT) {
    uint32_t run = 0u;
#pragma unroll 4
    for (int w2 = 0; w2 < NW; ++w2) {
      const uint32_t v = wcnt_all[w2 * L::WORDS + q];
      wcnt_all[w2 * L::WORDS + q] = run;
      run += v;  // each half stays below 2^16: at most one entry per row and id
    }
    hist_s[2 * q] = int(run & 0xFFFFu);
    hist_s[2 * q + 1] = int(run >> 16);
  }
  __syncthreads();
  for (int e = tid; e < a.NE; e += NT) pw.hist[size_t(e) * pw.grid_max + cta] = hist_s[e];
  // grid barrier 1, split: arrive once the histogram is out; the CTA-local work below
  // overlaps the wait for the other CTAs
  const unsigned arrival = grid_arrive(pw.bar, grid, a.barrier_skip_cta);
  block_scan_fast(hist_s, lbase_s, a.NE, tmp);
  // every routed entry to its CTA-local sorted position (the ring is free now); after a
  // wait that ran out only the rows before it were routed and counted
  const int nrouted = fail_at < 0 ? nw : 2 * fail_at;
  auto place = [&]() {
#pragma unroll 4
    for (int x = lane; x < nrouted * K; x += 32) {
      const uint32_t v = ent[x];
      const int l = int(v & 0x3FFu);
      if (INDEX && l >= a.NE) continue;  // an id left out (index mode)
      const uint32_t wp = (wcnt[l >> 1] >> (uint32_t(l & 1) * 16u)) & 0xFFFFu;
      const int lp = lbase_s[l] + int(wp) + int(v >> 10);
      sval[lp] = (wr0 + x / K) * K + (x % K);
      sbin[lp] = static_cast<uint16_t>(l);
    }
  };
  // the CTAs that own bins of the column scan place their entries after it, while they
  // wait at grid barrier 2, so that the scan starts as soon as barrier 1 opens
  const bool scanner = cta * NW < a.NE;
  if (!scanner) place();

  int* flag_s = tmp + 32;
  if (!grid_wait(pw.bar, arrival, a.err, flag_s, a.barrier_wait_ns, a.barrier_skip_cta)) {
    grid_exit(pw.bar, grid);
    return;
  }
  // the ring is free in the CTAs that scan: they place their entries afterwards
  column_scan_cta_major(pw, a.NE, grid, reinterpret_cast<int*>(ring_all));
  const unsigned arrival2 = grid_arrive(pw.bar, grid);
  if (scanner) place();
  if (!grid_wait(pw.bar, arrival2, a.err, flag_s, a.barrier_wait_ns)) {
    grid_exit(pw.bar, grid);
    return;
  }

  // ---- phase 3: offsets, then the sorted entries to perm, one run per bin
  {
    // at most two bins per thread (NE <= 912 < 2 NT): all four loads in flight at once
    static_assert(kFastBins <= 2 * NT, "two bins per thread cover the bins");
    const int e0 = tid, e1 = tid + NT;
    const int c0 = e0 < a.NE ? __ldcg(pw.counts + e0) : 0;
    const int c1 = e1 < a.NE ? __ldcg(pw.counts + e1) : 0;
    const int g0 = e0 < a.NE ? __ldcg(pw.prefix + size_t(cta) * kMaxBins + e0) : 0;
    const int g1 = e1 < a.NE ? __ldcg(pw.prefix + size_t(cta) * kMaxBins + e1) : 0;
    if (e0 < a.NE) {
      hist_s[e0] = c0;
      gbase_s[e0] = g0;
    }
    if (e1 < a.NE) {
      hist_s[e1] = c1;
      gbase_s[e1] = g1;
    }
  }
  __syncthreads();
  int* off_s = reinterpret_cast<int*>(smem + L::o_ws);  // the routing scratch is free
  block_scan_fast(hist_s, off_s, a.NE, tmp);
  if (cta == 0) {
    for (int e = tid; e < a.NE; e += NT) {
      a.counts[e] = hist_s[e];
      a.offsets[e] = off_s[e];
    }
    if (tid == 0) a.offsets[a.NE] = off_s[a.NE];
  }
  // the expert-GEMM layout, when asked: tile-padded offsets (an exclusive scan of the
  // padded bin sizes, in the routing scratch after the offsets)
  int* poff_s = off_s + kFastBins + 1;
  if constexpr (LAYOUT) {
    for (int e = tid; e < a.NE; e += NT) poff_s[e] = (hist_s[e] + a.tile - 1) / a.tile * a.tile;
    __syncthreads();
    block_scan_fast(poff_s, poff_s, a.NE, tmp);
    if (cta == 0 && a.poffs)
      for (int e = tid; e <= a.NE; e += NT) a.poffs[e] = poff_s[e];
  }
  // global place of CTA-local position 0 of bin e
  for (int e = tid; e < a.NE; e += NT) gbase_s[e] += off_s[e] - lbase_s[e];
  __syncthreads();
  const int nvalid = lbase_s[a.NE];
  if constexpr (!LAYOUT) {
#pragma unroll 4
    for (int i = tid; i < nvalid; i += NT) a.perm[gbase_s[sbin[i]] + i] = sval[i];
  } else {
    // entry at perm position p of bin l goes to padded row p - offsets[l] + padded_offsets[l]
#pragma unroll 4
    for (int i = tid; i < nvalid; i += NT) {
      const int l = sbin[i];
      const int p = gbase_s[l] + i, v = sval[i];
      a.perm[p] = v;
      const int r = p - off_s[l] + poff_s[l];
      if (a.prows) a.prows[r] = v;
      if (a.midx) a.midx[r] = l;
    }
    // the padding rows of bins cta, cta + grid, ... and a share of the rows past the
    // padded total
    for (int e = cta; e < a.NE; e += grid) {
      for (int r = poff_s[e] + hist_s[e] + tid; r < poff_s[e + 1]; r += NT) {
        if (a.prows) a.prows[r] = -1;
        if (a.midx) a.midx[r] = -1;
      }
    }
    for (int r = poff_s[a.NE] + cta * NT + tid; r < a.capacity; r += grid * NT) {
      if (a.prows) a.prows[r] = -1;
      if (a.midx) a.midx[r] = -1;
    }
  }
  if (a.inv) {
    // each entry's place in perm, in token order (coalesced): warp prefix + rank within
    // the warp give its CTA-local position, gbase the rest
    for (int x = lane; x < nrouted * K; x += 32) {
      const uint32_t v = ent[x];
      const int l = int(v & 0x3FFu);
      if (INDEX && l >= a.NE) continue;
      const uint32_t wp = (wcnt[l >> 1] >> (uint32_t(l & 1) * 16u)) & 0xFFFFu;
      a.inv[size_t(wr0) * K + x] = gbase_s[l] + lbase_s[l] + int(wp) + int(v >> 10);
    }
  }
  grid_exit(pw.bar, grid);
}

cudaError_t setup_prefill_fast(int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(k_route_prefill_fast<true, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, FastSmem::total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_route_prefill_fast<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FastSmem::total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_route_prefill_fast<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           FastSmem::total);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_route_prefill_fast<false, false>,
                                                       FastSmem::NW * 32, FastSmem::total);
}

bool prefill_fast_fits(int T, int grid) {
  if (T <= 0 || grid < 1) return false;
  const long long per_cta = (static_cast<long long>(T) + grid - 1) / grid;
  const long long per_warp = (per_cta + FastSmem::NW - 1) / FastSmem::NW;
  return per_warp <= FastSmem::ROWS_PER_WARP;
}

cudaError_t launch_route_prefill_fast(const RouteArgs& a, const PrefillWS& ws, int grid,
                                      cudaStream_t st) {
  if (!prefill_fast_fits(a.T, grid) || a.k != 16 || a.NE > kFastBins) return cudaErrorInvalidValue;
  const bool index = a.Kg == 0;  // moe_route_index sets topk_group 0
  if (!index && a.Kg != 4) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(FastSmem::NW * 32, 1, 1);
  cfg.dynamicSmemBytes = FastSmem::total;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  if (index) return cudaLaunchKernelEx(&cfg, k_route_prefill_fast<true, false>, a, ws);
  if (a.poffs || a.prows || a.midx) return cudaLaunchKernelEx(&cfg, k_route_prefill_fast<false, true>, a, ws);
  return cudaLaunchKernelEx(&cfg, k_route_prefill_fast<false, false>, a, ws);
}

// ------------------------------------------------------------ approximation error
// E_half = max over every finite bf16 x of |0.5 tanh.approx(x * 0.5) - (sigmoid(x) - 0.5)|,
// the reference sigmoid evaluated in double (its error, about 1e-16, is covered by the
// 2^-40 added), rounded up to float.  Written to *out as the bits of a non-negative
// float (atomicMax on the bits orders like the values); *out must start at 0.
__global__ void k_approx_err(unsigned* out) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  unsigned m = 0u;
  if (h < 65536 && (h & 0x7F80) != 0x7F80) {
    const float x = __uint_as_float(uint32_t(h) << 16);
    const float t = tanh_approx(__fmul_rn(x, 0.5f));
    const double sd = 1.0 / (1.0 + exp(-static_cast<double>(x)));
    const double err = fabs(0.5 * static_cast<double>(t) - (sd - 0.5)) + 0x1p-40;
    m = __float_as_uint(__double2float_ru(err));
  }
  const unsigned wm = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && wm != 0u) atomicMax(out, wm);
}

cudaError_t launch_approx_err(unsigned* out, cudaStream_t st) {
  k_approx_err<<<256, 256, 0, st>>>(out);
  return cudaGetLastError();
}

}  // namespace moe
