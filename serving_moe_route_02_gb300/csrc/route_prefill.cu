// route_prefill.cu -- prefill-size routing (thousands of rows) in one persistent,
// cooperative launch: one CTA of 16 warps per SM, contiguous row ranges per CTA.
//
// Phase 1 (the streaming part, bound by HBM and issue rate): every warp is its own row
//   engine.  Its lane 0 keeps D rows in flight with one-dimensional bulk copies
//   (cp.async.bulk, completion on a per-slot mbarrier) into a private ring in shared
//   memory; the warp routes each row (route_row), writes packed ids coalesced, and
//   counts the relabelled ids into the CTA's shared-memory histogram.
// Grid barrier 1, then a column scan: for each expert bin e, one warp scans the
//   per-CTA counts hist[e][0..grid) into prefix[e][c] and total counts[e].
// Grid barrier 2, then phase 3: every CTA scans counts into offsets (CTA 0 writes
//   counts and offsets), and walks its own rows in order, 32 rows at a time: a
//   per-bin 32-bit mask of the rows holding that bin gives each entry's stable rank,
//   so perm[offsets[e] + prefix[e][c] + rank] = t * k + j.
// Every wait (mbarrier, grid barrier) is bounded in time; a wait that runs out sets
// the device status word and the kernel returns.
#include <cooperative_groups.h>

#include "launch.h"

namespace moe {

constexpr int kPrefillWarps = 16;
constexpr int kPrefillThreads = 32 * kPrefillWarps;
constexpr int kChunkRows = 32;

__host__ __device__ constexpr int p_align(int x, int a) { return (x + a - 1) / a * a; }

template <int DT>
struct PrefillSmem {
  static constexpr int ROWB = (DT == DT_BF16) ? kE * 2 : kE * 4;
  static constexpr int D = (DT == DT_BF16) ? 3 : 2;  // rows in flight per warp
  static constexpr int STAB = (DT == DT_BF16) ? kSigTablePad * 4 : 0;
  static constexpr int o_stab = 0;
  static constexpr int o_ring = p_align(o_stab + STAB, 128);
  static constexpr int o_ws = p_align(o_ring + kPrefillWarps * D * ROWB, 128);
  static constexpr int o_hist = p_align(o_ws + kPrefillWarps * int(sizeof(WarpScratch)), 128);
  static constexpr int o_base = p_align(o_hist + (kMaxBins + 1) * 4, 128);
  static constexpr int o_mask = p_align(o_base + (kMaxBins + 1) * 4, 128);
  static constexpr int o_tmp = p_align(o_mask + kMaxBins * 4, 128);
  static constexpr int o_mbar = p_align(o_tmp + 33 * 4, 128);
  static constexpr int total = o_mbar + kPrefillWarps * D * 8 + 64;
};

static_assert(PrefillSmem<DT_F32>::total <= 227 * 1024, "prefill smem (f32) exceeds 227 KB");
static_assert(PrefillSmem<DT_BF16>::total <= 227 * 1024, "prefill smem (bf16) exceeds 227 KB");

// Grid-wide barrier for a cooperative launch; bounded in time.  bar[0] counts
// arrivals, bar[1] is the generation.  Returns false if the wait ran out.
__device__ bool grid_barrier(unsigned* bar, unsigned nblocks, int* err, int* flag_s) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned gen0;
    asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(gen0) : "l"(bar + 1) : "memory");
    __threadfence();
    const unsigned prev = atomicAdd(bar, 1u);
    int ok = 1;
    if (prev == nblocks - 1) {
      atomicExch(bar, 0u);
      __threadfence();
      atomicAdd(bar + 1, 1u);
    } else {
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        unsigned g;
        asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(g) : "l"(bar + 1) : "memory");
        if (g != gen0) break;
        if (globaltimer_ns() - t0 > kWaitLimitNs) {
          atomicExch(err, kErrTimeout);
          ok = 0;
          break;
        }
        __nanosleep(64);
      }
    }
    __threadfence();
    *flag_s = ok;
  }
  __syncthreads();
  return *flag_s != 0;
}

template <int DT>
__global__ void __launch_bounds__(kPrefillThreads, 1)
    k_route_prefill(RouteArgs a, PrefillWS pw) {
  using L = PrefillSmem<DT>;
  extern __shared__ __align__(128) uint8_t smem[];
  float* stab = reinterpret_cast<float*>(smem + L::o_stab);
  uint8_t* ring_all = smem + L::o_ring;
  WarpScratch* wsp = reinterpret_cast<WarpScratch*>(smem + L::o_ws);
  int* hist_s = reinterpret_cast<int*>(smem + L::o_hist);
  int* base_s = reinterpret_cast<int*>(smem + L::o_base);
  unsigned* mask_s = reinterpret_cast<unsigned*>(smem + L::o_mask);
  int* tmp = reinterpret_cast<int*>(smem + L::o_tmp);
  uint64_t* mbar_all = reinterpret_cast<uint64_t*>(smem + L::o_mbar);

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int grid = gridDim.x, cta = blockIdx.x;
  const int r0 = int((long long)a.T * cta / grid);
  const int r1 = int((long long)a.T * (cta + 1) / grid);
  const int nw = (r1 - r0 > w) ? (r1 - r0 - w + kPrefillWarps - 1) / kPrefillWarps : 0;
  uint8_t* ring = ring_all + w * L::D * L::ROWB;
  uint64_t* mb = mbar_all + w * L::D;
  const uint8_t* logits = static_cast<const uint8_t*>(a.logits);

  // ---- setup: mbarriers, sigmoid table, first rows in flight
  if (lane == 0) {
    for (int d = 0; d < L::D; ++d) mbar_init(mb + d, 1);
    fence_mbar_init();
  }
  uint64_t* tab_bar = mbar_all + kPrefillWarps * L::D;
  if (tid == 0 && L::STAB) {
    mbar_init(tab_bar, 1);
    fence_mbar_init();
  }
  for (int e = tid; e < a.NE; e += kPrefillThreads) hist_s[e] = 0;
  __syncthreads();
  if (tid == 0 && L::STAB) {
    mbar_expect_tx(tab_bar, L::STAB);
    bulk_g2s(stab, a.stab, L::STAB, tab_bar);
  }
  if (lane == 0) {
    for (int d = 0; d < L::D && d < nw; ++d) {
      const int t = r0 + w + d * kPrefillWarps;
      mbar_expect_tx(mb + d, L::ROWB);
      bulk_g2s(ring + d * L::ROWB, logits + size_t(t) * L::ROWB, L::ROWB, mb + d);
    }
  }
  float bl[kEPL];
  load_lane_bias(a.bias, bl);
  if (L::STAB) mbar_wait_bounded(tab_bar, 0, a.err);

  // ---- phase 1: route this warp's rows
  for (int i = 0; i < nw; ++i) {
    const int slot = i % L::D;
    const uint32_t par = uint32_t(i / L::D) & 1u;
    mbar_wait_bounded(mb + slot, par, a.err);
    const int t = r0 + w + i * kPrefillWarps;
    const SlotOut o = route_row<DT>(ring + slot * L::ROWB, bl, stab, a, wsp[w]);
    if (lane < a.k) {
      a.packed[size_t(t) * a.k + lane] = o.packed;
      if (a.ids) a.ids[size_t(t) * a.k + lane] = o.id;
      atomicAdd(&hist_s[o.lid], 1);
    }
    __syncwarp();
    if (lane == 0 && i + L::D < nw) {
      fence_proxy_async_smem();
      mbar_expect_tx(mb + slot, L::ROWB);
      bulk_g2s(ring + slot * L::ROWB, logits + size_t(t + L::D * kPrefillWarps) * L::ROWB,
               L::ROWB, mb + slot);
    }
  }
  __syncthreads();
  for (int e = tid; e < a.NE; e += kPrefillThreads) pw.hist[size_t(e) * pw.grid_max + cta] = hist_s[e];

  int* flag_s = tmp + 32;
  if (!grid_barrier(pw.bar, grid, a.err, flag_s)) return;

  // ---- column scan over CTAs, one warp per expert bin
  for (int e = cta * kPrefillWarps + w; e < a.NE; e += grid * kPrefillWarps) {
    const int* h = pw.hist + size_t(e) * pw.grid_max;
    int* p = pw.prefix + size_t(e) * pw.grid_max;
    int carry = 0;
    for (int c0 = 0; c0 < grid; c0 += 32) {
      const int c = c0 + lane;
      const int v = (c < grid) ? h[c] : 0;
      int incl = v;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      if (c < grid) p[c] = carry + incl - v;
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pw.counts[e] = carry;
  }

  if (!grid_barrier(pw.bar, grid, a.err, flag_s)) return;

  // ---- phase 3: offsets, then this CTA's permutation entries
  for (int e = tid; e < a.NE; e += kPrefillThreads) hist_s[e] = pw.counts[e];
  __syncthreads();
  block_exclusive_scan(hist_s, base_s, a.NE, tmp);
  if (cta == 0) {
    for (int e = tid; e < a.NE; e += kPrefillThreads) {
      a.counts[e] = hist_s[e];
      a.offsets[e] = base_s[e];
    }
    if (tid == 0) a.offsets[a.NE] = base_s[a.NE];
  }
  __syncthreads();
  for (int e = tid; e < a.NE; e += kPrefillThreads) {
    base_s[e] += pw.prefix[size_t(e) * pw.grid_max + cta];
    mask_s[e] = 0u;
  }
  __syncthreads();
  for (int cr = r0; cr < r1; cr += kChunkRows) {
    const int nr = min(kChunkRows, r1 - cr);
    const int ne = nr * a.k;
    const int32_t* pk = a.packed + size_t(cr) * a.k;
    for (int x = tid; x < ne; x += kPrefillThreads) {
      const int rr = x / a.k;
      const int l = int(uint32_t(pk[x]) >> 16);
      atomicOr(&mask_s[l], 1u << rr);
    }
    __syncthreads();
    for (int x = tid; x < ne; x += kPrefillThreads) {
      const int rr = x / a.k, j = x - rr * a.k;
      const int l = int(uint32_t(pk[x]) >> 16);
      const int pos = base_s[l] + __popc(mask_s[l] & ((1u << rr) - 1u));
      a.perm[pos] = (cr + rr) * a.k + j;
    }
    __syncthreads();
    for (int e = tid; e < a.NE; e += kPrefillThreads) {
      const unsigned m = mask_s[e];
      if (m) {
        base_s[e] += __popc(m);
        mask_s[e] = 0u;
      }
    }
    __syncthreads();
  }
}

cudaError_t setup_prefill_kernels(int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(k_route_prefill<DT_F32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       PrefillSmem<DT_F32>::total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_route_prefill<DT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           PrefillSmem<DT_BF16>::total);
  if (e != cudaSuccess) return e;
  int b0 = 0, b1 = 0;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b0, k_route_prefill<DT_F32>, kPrefillThreads,
                                                    PrefillSmem<DT_F32>::total);
  if (e != cudaSuccess) return e;
  e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b1, k_route_prefill<DT_BF16>, kPrefillThreads,
                                                    PrefillSmem<DT_BF16>::total);
  if (e != cudaSuccess) return e;
  *blocks_per_sm = min(b0, b1);
  return cudaSuccess;
}

cudaError_t launch_route_prefill(const RouteArgs& a, int dtype, const PrefillWS& ws, int grid,
                                 cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(kPrefillThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == DT_BF16) {
    cfg.dynamicSmemBytes = PrefillSmem<DT_BF16>::total;
    return cudaLaunchKernelEx(&cfg, k_route_prefill<DT_BF16>, a, ws);
  }
  cfg.dynamicSmemBytes = PrefillSmem<DT_F32>::total;
  return cudaLaunchKernelEx(&cfg, k_route_prefill<DT_F32>, a, ws);
}

}  // namespace moe
