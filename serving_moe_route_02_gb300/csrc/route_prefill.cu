// route_prefill.cu -- prefill-size routing (thousands of rows) in one persistent,
// cooperative launch: one CTA per SM, a contiguous row range per CTA and a contiguous
// sub-range per warp.  The bf16 Kimi-K3 instance (k = 16, keep 4 groups) runs 24 warps
// per SM (scratch sized for 448 kept candidates, 2 rows in flight per warp); other
// instances run 16 warps.
//
// Phase 1 (the streaming part): every warp is its own row engine.  Its lane 0 keeps D
//   rows in flight with one-dimensional bulk copies (cp.async.bulk, completion on a
//   per-slot mbarrier) into a private ring in shared memory; the warp routes each row
//   (route_row), writes packed ids coalesced, and counts the relabelled ids into the
//   CTA's histogram, which goes to the expert-major matrix hist[bin][cta].
// Grid barrier 1, then a column scan: for each bin one warp turns hist[bin][0..grid)
//   into exclusive prefixes over CTAs and the bin's total.
// Grid barrier 2, then phase 3: every CTA scans the totals into offsets (CTA 0 writes
//   counts and offsets) and adds its own CTA prefix; each warp stages its packed ids in
//   shared memory (the ring and scratch are free by then), counts its bins, a column
//   pass over the warps turns the counts into warp prefixes, and each warp walks its
//   rows in order: the entry (t, j) with relabelled id l goes to
//   perm[offsets[l] + cta prefix + warp prefix + running count of l in this warp],
//   which is its stable (id, token, slot) position, since ids are unique in a row.
// Every wait (mbarrier, grid barrier) is bounded in time; a wait that runs out sets
// the device status word and the kernel returns.
#include <cooperative_groups.h>

#include "persist.cuh"

namespace moe {

__host__ __device__ constexpr int p_align(int x, int a) { return (x + a - 1) / a * a; }

template <int DT, bool SPEC>
struct PrefillSmem {
  static constexpr bool WIDE = (DT == DT_BF16) && SPEC;
  static constexpr bool INDEX = DT == DT_PACKED;              // histogram/scan/perm of packed ids
  static constexpr int NW = WIDE ? 24 : 16;                  // warps per CTA
  // (index mode streams no rows: its "ring" is only phase-3 room)
  static constexpr int ROWB = INDEX ? 4096 : (DT == DT_BF16) ? kE * 2 : kE * 4;
  static constexpr int D = INDEX ? 1 : WIDE ? 2 : ((DT == DT_BF16) ? 3 : 2);  // rows in flight
  static constexpr int NB = SPEC ? 4 * kLanesPerGroup * kEPL : kEPL * 32;
  using WS = WarpScratchT<NB>;
  static constexpr int STAB = (DT == DT_BF16) ? kSigTablePad * 4 : 0;
  static constexpr int o_stab = 0;
  static constexpr int o_bias = p_align(o_stab + STAB, 128);
  static constexpr int o_ring = p_align(o_bias + kE * 4, 128);
  static constexpr int o_ws = o_ring + NW * D * ROWB;         // 128-aligned: ROWB is
  static constexpr int o_hist = p_align(o_ws + NW * int(sizeof(WS)), 128);
  static constexpr int o_base = p_align(o_hist + (kMaxBins + 1) * 4, 128);
  static constexpr int o_tmp = p_align(o_base + (kMaxBins + 1) * 4, 128);
  static constexpr int o_mbar = p_align(o_tmp + 33 * 4, 128);
  // each warp keeps its rows' relabelled ids (16-bit) for phase 3 in the room left
  static constexpr int o_lid = p_align(o_mbar + NW * D * 8 + 64, 128);
  static constexpr int LID_ENTRIES = (227 * 1024 - o_lid) / (NW * 2) / 64 * 64;
  static constexpr int total = o_lid + NW * LID_ENTRIES * 2;
  // phase 3 reuses [0, o_hist) (score table, bias, ring, scratch): warp prefixes, a
  // staging buffer per warp, the CTA-local bin offsets, then the CTA's entries sorted by
  // bin (values, then bins) when they fit
  static constexpr int STAGE_INTS = 256;
  static constexpr int o3_wpre = 0;
  static constexpr int o3_stage = o3_wpre + NW * kMaxBins * 4;
  static constexpr int o3_lbase = o3_stage + NW * STAGE_INTS * 4;
  static constexpr int o3_cpre = o3_lbase + (kMaxBins + 1) * 4;
  static constexpr int o3_sval = p_align(o3_cpre + kMaxBins * 4, 16);
  static constexpr int SORT_CAP = (o_hist - o3_sval) / 6 / 8 * 8;
  static constexpr int o3_sbin = o3_sval + SORT_CAP * 4;
};

static_assert(PrefillSmem<DT_F32, false>::total <= 227 * 1024, "prefill smem (f32) exceeds 227 KB");
static_assert(PrefillSmem<DT_F32, true>::total <= 227 * 1024, "prefill smem (f32) exceeds 227 KB");
static_assert(PrefillSmem<DT_BF16, false>::total <= 227 * 1024, "prefill smem (bf16) exceeds 227 KB");
static_assert(PrefillSmem<DT_BF16, true>::total <= 227 * 1024, "prefill smem (bf16) exceeds 227 KB");
static_assert(PrefillSmem<DT_PACKED, false>::total <= 227 * 1024, "prefill smem (index) exceeds 227 KB");
static_assert(PrefillSmem<DT_PACKED, false>::SORT_CAP >= 4096 && PrefillSmem<DT_BF16, true>::SORT_CAP >= 4096 &&
                  PrefillSmem<DT_BF16, false>::SORT_CAP >= 4096 &&
                  PrefillSmem<DT_F32, true>::SORT_CAP >= 4096 &&
                  PrefillSmem<DT_F32, false>::SORT_CAP >= 4096,
              "phase 3 keeps room for the CTA-local sort");
static_assert(PrefillSmem<DT_BF16, true>::LID_ENTRIES >= 512 && PrefillSmem<DT_BF16, false>::LID_ENTRIES >= 512 &&
                  PrefillSmem<DT_F32, true>::LID_ENTRIES >= 512 && PrefillSmem<DT_F32, false>::LID_ENTRIES >= 512 &&
                  PrefillSmem<DT_PACKED, false>::LID_ENTRIES >= 512,
              "room for the kept ids");
static_assert(PrefillSmem<DT_BF16, true>::ROWB % 128 == 0 && PrefillSmem<DT_F32, true>::ROWB % 128 == 0,
              "row slots keep 128-byte alignment");

// Index mode: true in the lanes of kmask whose id appears more than once among the
// row's k ids held by lanes 0..k-1 (all lanes of kmask must call it).
__device__ __forceinline__ bool repeated_in_row(int l, unsigned kmask, int k) {
  int n = 0;
  for (int j = 0; j < k; ++j) n += __shfl_sync(kmask, l, j) == l;
  return n > 1;
}

// SPEC: k = 16 and topk_group = 4 compiled in (the Kimi-K3 instance).
template <int DT, bool SPEC>
__global__ void __launch_bounds__(PrefillSmem<DT, SPEC>::NW * 32, 1)
    k_route_prefill(RouteArgs a, PrefillWS pw) {
  using L = PrefillSmem<DT, SPEC>;
  using WS = typename L::WS;
  constexpr int NW = L::NW;
  constexpr int NT = NW * 32;
  extern __shared__ __align__(128) uint8_t smem[];
  float* stab = reinterpret_cast<float*>(smem + L::o_stab);
  float* bias_s = reinterpret_cast<float*>(smem + L::o_bias);
  uint8_t* ring_all = smem + L::o_ring;
  WS* wsp = reinterpret_cast<WS*>(smem + L::o_ws);
  int* hist_s = reinterpret_cast<int*>(smem + L::o_hist);
  int* base_s = reinterpret_cast<int*>(smem + L::o_base);
  int* tmp = reinterpret_cast<int*>(smem + L::o_tmp);
  uint64_t* mbar_all = reinterpret_cast<uint64_t*>(smem + L::o_mbar);
  uint16_t* lid16 = reinterpret_cast<uint16_t*>(smem + L::o_lid) + (threadIdx.x >> 5) * L::LID_ENTRIES;

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int grid = gridDim.x, cta = blockIdx.x;
  const int r0 = int((long long)a.T * cta / grid);
  const int r1 = int((long long)a.T * (cta + 1) / grid);
  // this warp's rows: [wr0, wr1)
  const int per_warp = (r1 - r0 + NW - 1) / NW;
  const int wr0 = min(r1, r0 + w * per_warp);
  const int wr1 = min(r1, wr0 + per_warp);
  const int nw = wr1 - wr0;
  uint8_t* ring = ring_all + w * L::D * L::ROWB;
  uint64_t* mb = mbar_all + w * L::D;
  const uint8_t* logits = static_cast<const uint8_t*>(a.logits);

  // packed ids phase 3 reads: written by phase 1, or given (index mode)
  const int32_t* pk = L::INDEX ? static_cast<const int32_t*>(a.logits) : a.packed;

  // ---- setup: mbarriers, histogram, score table and bias, first rows in flight
  if (lane == 0) {
    for (int d = 0; d < L::D; ++d) mbar_init(mb + d, 1);
    fence_mbar_init();
  }
  uint64_t* tab_bar = mbar_all + NW * L::D;
  if (tid == 0) {
    mbar_init(tab_bar, 1);
    fence_mbar_init();
  }
  for (int e = tid; e < a.NE; e += NT) hist_s[e] = 0;
  __syncthreads();
  const unsigned kmask = (a.k == 32) ? 0xffffffffu : ((1u << a.k) - 1u);
  if constexpr (L::INDEX) {
    // ---- phase 1 (index mode): count this warp's given packed ids, 8 rows of loads in
    //      flight.  Ids must be distinct within a row: an id >= NE, and every occurrence
    //      of an id that appears twice in its row, is reported and left out here and in
    //      phase 3 alike (kept as 0xFFFF, never a bin).  Repeats are found with two
    //      bitmaps of the row's ids in the warp's (otherwise unused) ring slot: ids seen,
    //      and ids seen twice; both are cleared after each row.
    constexpr int kWords = kMaxBins / 32;
    uint32_t* seen = reinterpret_cast<uint32_t*>(ring);
    uint32_t* twice = seen + kWords;
    for (int i = lane; i < 2 * kWords; i += 32) seen[i] = 0u;
    __syncwarp();
    for (int i0 = 0; i0 < nw; i0 += 8) {
      int32_t v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q)
        v[q] = (i0 + q < nw && lane < a.k) ? pk[size_t(wr0 + i0 + q) * a.k + lane] : 0;
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const bool act = i0 + q < nw && lane < a.k;
        const int l = act ? int(uint32_t(v[q]) >> 16) : 0;
        const bool inb = act && l < a.NE;
        const int wd = inb ? (l >> 5) : 0;  // bitmap word, in range on every lane
        const uint32_t bit = 1u << (l & 31);
        if (inb && (atomicOr(&seen[wd], bit) & bit) != 0u) atomicOr(&twice[wd], bit);
        __syncwarp();
        const bool bad = act && (!inb || (twice[wd] & bit) != 0u);
        if (act) {
          if ((i0 + q) * a.k + lane < L::LID_ENTRIES)
            lid16[(i0 + q) * a.k + lane] = static_cast<uint16_t>(bad ? 0xFFFF : l);
          if (!bad) atomicAdd(&hist_s[l], 1);
          else atomicExch(a.err, kErrBadId);
        }
        __syncwarp();  // every lane has read `twice` before the clear
        if (inb) {
          seen[wd] = 0u;
          twice[wd] = 0u;
        }
        __syncwarp();
      }
    }
  } else {
  if (tid == 0) {
    mbar_expect_tx(tab_bar, uint32_t(L::STAB + kE * 4));
    if (L::STAB) bulk_g2s(stab, a.stab, L::STAB, tab_bar);
    bulk_g2s(bias_s, a.bias, kE * 4, tab_bar);
  }
  if (lane == 0) {
    for (int d = 0; d < L::D && d < nw; ++d) {
      mbar_expect_tx(mb + d, L::ROWB);
      bulk_g2s(ring + d * L::ROWB, logits + size_t(wr0 + d) * L::ROWB, L::ROWB, mb + d);
    }
  }
  mbar_wait_bounded(tab_bar, 0, a.err);

  // ---- phase 1: route this warp's rows
  for (int i = 0; i < nw; ++i) {
    const int slot = i % L::D;
    const uint32_t par = uint32_t(i / L::D) & 1u;
    mbar_wait_bounded(mb + slot, par, a.err);
    const int t = wr0 + i;
    const SlotOut o =
        route_row<DT, SPEC ? 16 : 0, SPEC ? 4 : 0>(ring + slot * L::ROWB, bias_s, stab, a, wsp[w]);
    if (lane < a.k) {
      a.packed[size_t(t) * a.k + lane] = o.packed;
      if (a.ids) a.ids[size_t(t) * a.k + lane] = o.id;
      atomicAdd(&hist_s[o.lid], 1);
      if (i * a.k + lane < L::LID_ENTRIES) lid16[i * a.k + lane] = static_cast<uint16_t>(o.lid);
    }
    __syncwarp();
    if (lane == 0 && i + L::D < nw) {
      fence_proxy_async_smem();
      mbar_expect_tx(mb + slot, L::ROWB);
      bulk_g2s(ring + slot * L::ROWB, logits + size_t(t + L::D) * L::ROWB, L::ROWB, mb + slot);
    }
  }
  }
  __syncthreads();
  for (int e = tid; e < a.NE; e += NT) pw.hist[size_t(e) * pw.grid_max + cta] = hist_s[e];
  // CTA-local bin offsets of this CTA's entries (the ring and the scratch are free now)
  int* lbase_s = reinterpret_cast<int*>(smem + L::o3_lbase);
  block_scan_fast(hist_s, lbase_s, a.NE, tmp);

  int* flag_s = tmp + 32;
  if (!grid_barrier(pw.bar, grid, a.err, flag_s, a.barrier_wait_ns, a.barrier_skip_cta)) {
    grid_exit(pw.bar, grid);
    return;
  }

  // ---- column scan over CTAs (prefixes and bin totals)
  column_scan(pw, a.NE, grid, NW);

  if (!grid_barrier(pw.bar, grid, a.err, flag_s, a.barrier_wait_ns)) {
    grid_exit(pw.bar, grid);
    return;
  }

  // ---- phase 3: offsets, then this CTA's permutation entries (bin totals and this CTA's
  //      prefixes are loaded together: one round trip)
  int* cpre_s = reinterpret_cast<int*>(smem + L::o3_cpre);
  for (int e = tid; e < a.NE; e += NT) {
    const int c = __ldcg(pw.counts + e);
    const int p = __ldcg(pw.prefix + size_t(e) * pw.grid_max + cta);
    hist_s[e] = c;
    cpre_s[e] = p;
  }
  __syncthreads();
  block_scan_fast(hist_s, base_s, a.NE, tmp);
  if (cta == 0) {
    for (int e = tid; e < a.NE; e += NT) {
      a.counts[e] = hist_s[e];
      a.offsets[e] = base_s[e];
    }
    if (tid == 0) a.offsets[a.NE] = base_s[a.NE];
  }
  for (int e = tid; e < a.NE; e += NT) base_s[e] += cpre_s[e];

  // The ring and the routing scratch are free: warp counters [NW][kMaxBins], then a
  // staging buffer per warp for its packed ids, loaded a chunk of rows at a time with
  // all loads of a chunk in flight.
  int* wpre_all = reinterpret_cast<int*>(smem + L::o3_wpre);
  int* wpre = wpre_all + w * kMaxBins;
  int* stage = reinterpret_cast<int*>(smem + L::o3_stage) + w * L::STAGE_INTS;
  int* sval = reinterpret_cast<int*>(smem + L::o3_sval);
  uint16_t* sbin = reinterpret_cast<uint16_t*>(smem + L::o3_sbin);
  // the CTA's entries sorted by bin in shared memory, then written as runs (coalesced),
  // when they fit; otherwise each entry goes straight to its place
  const int nvalid = lbase_s[a.NE];
  const bool sorted = nvalid <= L::SORT_CAP;
  // this warp's ids: kept in shared memory by phase 1 when they fit, otherwise staged
  // from the packed values a chunk of rows at a time
  const bool keep = nw * a.k <= L::LID_ENTRIES;
  const int chunk_rows = keep ? max(nw, 1) : L::STAGE_INTS / a.k;
  const int nchunks = (nw + chunk_rows - 1) / chunk_rows;
  auto lid_of = [&](int c0, int r) -> int {
    return keep ? int(lid16[(c0 + r) * a.k + lane]) : int(uint32_t(stage[r * a.k + lane]) >> 16);
  };
  auto stage_chunk = [&](int c0) {
    const int n = min(chunk_rows, nw - c0) * a.k;
    const int32_t* src = pk + size_t(wr0 + c0) * a.k;
    for (int i0 = 0; i0 < n; i0 += 8 * 32) {
      int32_t v[8];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * 32 + lane;
        v[q] = (i < n) ? src[i] : 0;
      }
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int i = i0 + q * 32 + lane;
        if (i < n) stage[i] = v[q];
      }
    }
    __syncwarp();
  };
  __syncthreads();  // every warp is done with the ring and its scratch
  for (int e = lane; e < a.NE; e += 32) wpre[e] = 0;
  __syncwarp();
  // this warp's bin counts
  for (int c0 = 0; c0 < nw; c0 += chunk_rows) {
    if (!keep) stage_chunk(c0);
    const int nr = min(chunk_rows, nw - c0);
    if (lane < a.k)
      for (int r = 0; r < nr; ++r) {
        const int l = lid_of(c0, r);
        bool use = true;
        if constexpr (L::INDEX) {
          // kept ids carry phase 1's decision; staged ones are checked again
          // (keep is the same in every lane: either all lanes of kmask shuffle or none)
          const bool rep = keep ? false : repeated_in_row(l, kmask, a.k);
          use = l < a.NE && !rep;
        }
        if (use) atomicAdd(&wpre[l], 1);
      }
    __syncwarp();
  }
  __syncthreads();
  // warp prefixes per bin (from the CTA-local bin offset when sorting locally)
  for (int e = tid; e < a.NE; e += NT) {
    int run = sorted ? lbase_s[e] : 0;
    if (sorted) base_s[e] -= lbase_s[e];  // global place of local position 0 of bin e
#pragma unroll 4
    for (int w2 = 0; w2 < NW; ++w2) {
      const int v = wpre_all[w2 * kMaxBins + e];
      wpre_all[w2 * kMaxBins + e] = run;
      run += v;
    }
  }
  __syncthreads();
  // the walk: rows in order (the last chunk staged above is still in place)
  auto place = [&](int l, int rk, int x) {
    if (sorted) {
      sval[rk] = x;
      sbin[rk] = static_cast<uint16_t>(l);
    } else {
      a.perm[base_s[l] + rk] = x;
    }
    // entry x's place in perm; the walk visits entries in token order, so these stores
    // are coalesced row by row
    if (a.inv) a.inv[x] = base_s[l] + rk;
  };
  for (int c0 = 0; c0 < nw; c0 += chunk_rows) {
    if (!keep && nchunks > 1) stage_chunk(c0);
    const int nr = min(chunk_rows, nw - c0);
    if (lane < a.k) {
      for (int r = 0; r < nr; ++r) {
        const int l = lid_of(c0, r);
        bool use = true;
        if constexpr (L::INDEX) {
          // kept ids carry phase 1's decision; staged ones are checked again
          // (keep is the same in every lane: either all lanes of kmask shuffle or none)
          const bool rep = keep ? false : repeated_in_row(l, kmask, a.k);
          use = l < a.NE && !rep;
        }
        if (use) {
          const int rk = wpre[l];
          wpre[l] = rk + 1;
          place(l, rk, (wr0 + c0 + r) * a.k + lane);
        }
        __syncwarp(kmask);  // the next row may count the same bin in another lane
      }
    }
    __syncwarp();
  }
  if (sorted) {
    __syncthreads();
    for (int i = tid; i < nvalid; i += NT) a.perm[base_s[sbin[i]] + i] = sval[i];
  }
  grid_exit(pw.bar, grid);
}

template <int DT, bool SPEC>
static cudaError_t set_prefill_smem(int* bmin) {
  cudaError_t e = cudaFuncSetAttribute(k_route_prefill<DT, SPEC>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PrefillSmem<DT, SPEC>::total);
  if (e != cudaSuccess) return e;
  int b = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, k_route_prefill<DT, SPEC>,
                                                    PrefillSmem<DT, SPEC>::NW * 32,
                                                    PrefillSmem<DT, SPEC>::total);
  if (e != cudaSuccess) return e;
  *bmin = min(*bmin, b);
  return cudaSuccess;
}

cudaError_t setup_prefill_kernels(int* blocks_per_sm) {
  int b = 1 << 30;
  cudaError_t e;
  if ((e = set_prefill_smem<DT_F32, false>(&b)) != cudaSuccess) return e;
  if ((e = set_prefill_smem<DT_F32, true>(&b)) != cudaSuccess) return e;
  if ((e = set_prefill_smem<DT_BF16, false>(&b)) != cudaSuccess) return e;
  if ((e = set_prefill_smem<DT_BF16, true>(&b)) != cudaSuccess) return e;
  if ((e = set_prefill_smem<DT_PACKED, false>(&b)) != cudaSuccess) return e;
  *blocks_per_sm = b;
  return cudaSuccess;
}

bool prefill_fits(int T, int grid) { return T >= 0 && grid >= 1; }

template <int DT, bool SPEC>
static cudaError_t launch_t(const RouteArgs& a, const PrefillWS& ws, int grid, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(PrefillSmem<DT, SPEC>::NW * 32, 1, 1);
  cfg.dynamicSmemBytes = PrefillSmem<DT, SPEC>::total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_route_prefill<DT, SPEC>, a, ws);
}

cudaError_t launch_route_prefill(const RouteArgs& a, int dtype, const PrefillWS& ws, int grid,
                                 cudaStream_t st) {
  if (!prefill_fits(a.T, grid)) return cudaErrorInvalidValue;
  const bool spec = a.k == 16 && a.Kg == 4;
  if (dtype == DT_PACKED) return launch_t<DT_PACKED, false>(a, ws, grid, st);
  if (dtype == DT_BF16)
    return spec ? launch_t<DT_BF16, true>(a, ws, grid, st) : launch_t<DT_BF16, false>(a, ws, grid, st);
  return spec ? launch_t<DT_F32, true>(a, ws, grid, st) : launch_t<DT_F32, false>(a, ws, grid, st);
}

}  // namespace moe
