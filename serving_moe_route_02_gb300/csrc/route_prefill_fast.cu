// route_prefill_fast.cu -- prefill-size routing of bf16 logits for the Kimi-K3 instance
// (E = 896 in 8 groups, k = 16, keep 4 groups) in one persistent, cooperative launch:
// one CTA of 16 warps per SM, a contiguous row range per CTA and per warp.
//
// Phase 1 (streaming): every warp keeps D rows in flight with one-dimensional bulk
//   copies into a private ring in shared memory and routes each row with route_row_fast
//   (approximate scores, exact table lookups only where a decision needs them).  Lanes
//   0..15 store the packed slots, then count their relabelled ids into the warp's own
//   16-bit counters (two per 32-bit word); the counter's old value is the entry's rank
//   among this warp's entries of the same id, in (token, slot) order, since a warp
//   routes its rows in order and ids are unique in a row.  (id, rank) is kept in shared
//   memory.
// CTA tail of phase 1: a column pass over the warps' counters gives each warp's prefix
//   per id and the CTA's histogram, which goes to the expert-major matrix hist[bin][cta];
//   a block scan gives the CTA-local bin offsets, and every entry is placed at its
//   CTA-local position (bin offset + warp prefix + rank) in a buffer that replaces the
//   ring: the CTA's entries sorted by (id, token, slot).
// Grid barrier 1, column scan over CTAs (prefixes and totals), grid barrier 2.
// Phase 3: offsets from the totals (CTA 0 writes counts and offsets); the sorted buffer
//   goes to perm in runs of consecutive addresses, one run per bin.
// Every wait is bounded in time; a wait that runs out sets the status word and the CTA
// leaves (through grid_exit, which restores the barrier words once all CTAs have left).
#include <cooperative_groups.h>

#include "persist.cuh"
#include "route_fast.cuh"

namespace moe {

namespace {

__host__ __device__ constexpr int f_align(int x, int a) { return (x + a - 1) / a * a; }

struct FastSmem {
  static constexpr int NW = 16;                    // warps per CTA
  static constexpr int D = 3;                      // rows in flight per warp
  static constexpr int ROWB = kE * 2;              // one bf16 row: 1,792 bytes
  static constexpr int WORDS = kMaxBins / 2;       // 16-bit counters, two per word
  static constexpr int o_stab = 0;
  static constexpr int o_bias = f_align(kSigTablePad * 4, 128);
  static constexpr int o_ring = f_align(o_bias + kE * 4, 128);
  static constexpr int o_wcnt = o_ring + NW * D * ROWB;
  static constexpr int o_ws = f_align(o_wcnt + NW * WORDS * 4, 128);
  static constexpr int o_hist = f_align(o_ws + NW * int(sizeof(FastScratch)), 128);
  static constexpr int o_lbase = f_align(o_hist + (kMaxBins + 1) * 4, 128);
  static constexpr int o_gbase = f_align(o_lbase + (kMaxBins + 1) * 4, 128);
  static constexpr int o_tmp = f_align(o_gbase + (kMaxBins + 1) * 4, 128);
  static constexpr int o_mbar = f_align(o_tmp + 64 * 4, 128);
  static constexpr int o_ent = f_align(o_mbar + (NW * D + 1) * 8, 128);
  // (id, rank) of each entry, per warp, in the room left
  static constexpr int ENT_PER_WARP = (227 * 1024 - o_ent) / (NW * 4) / 16 * 16;
  static constexpr int ROWS_PER_WARP = ENT_PER_WARP / 16;
  static constexpr int total = o_ent + NW * ENT_PER_WARP * 4;
  // the CTA's sorted entries, in the ring once phase 1 is over: values, then bins
  static constexpr int SORT_CAP = (NW * D * ROWB) / 6 / 8 * 8;
  static constexpr int o_sval = o_ring;
  static constexpr int o_sbin = o_ring + SORT_CAP * 4;
};

static_assert(FastSmem::total <= 227 * 1024, "fast prefill smem exceeds 227 KB");
static_assert(FastSmem::SORT_CAP >= FastSmem::NW * FastSmem::ENT_PER_WARP, "sorted entries fit the ring");
static_assert(FastSmem::ROWS_PER_WARP >= 32, "room for the entries of 32 rows per warp");
static_assert(FastSmem::ROWB % 128 == 0, "row slots keep 128-byte alignment");

}  // namespace

int fast_prefill_rows_per_warp() { return FastSmem::ROWS_PER_WARP; }
int fast_prefill_warps() { return FastSmem::NW; }

__global__ void __launch_bounds__(FastSmem::NW * 32, 1)
    k_route_prefill_fast(RouteArgs a, PrefillWS pw) {
  using L = FastSmem;
  constexpr int NW = L::NW;
  constexpr int NT = NW * 32;
  constexpr int K = 16;
  extern __shared__ __align__(128) uint8_t smem[];
  float* stab = reinterpret_cast<float*>(smem + L::o_stab);
  float* bias_s = reinterpret_cast<float*>(smem + L::o_bias);
  uint8_t* ring_all = smem + L::o_ring;
  uint32_t* wcnt_all = reinterpret_cast<uint32_t*>(smem + L::o_wcnt);
  FastScratch* wsp = reinterpret_cast<FastScratch*>(smem + L::o_ws);
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
  uint8_t* ring = ring_all + w * L::D * L::ROWB;
  uint64_t* mb = mbar_all + w * L::D;
  uint32_t* wcnt = wcnt_all + w * L::WORDS;
  uint32_t* ent = reinterpret_cast<uint32_t*>(smem + L::o_ent) + w * L::ENT_PER_WARP;
  const uint8_t* logits = static_cast<const uint8_t*>(a.logits);
  const int nwords = a.NE / 2;  // NE is a multiple of 4

  // ---- setup: mbarriers, counters, score table and bias, first rows in flight
  uint64_t* tab_bar = mbar_all + NW * L::D;
  if (lane == 0) {
    for (int d = 0; d < L::D; ++d) mbar_init(mb + d, 1);
    if (w == 0) mbar_init(tab_bar, 1);
    fence_mbar_init();
  }
  for (int i = tid; i < NW * L::WORDS; i += NT) wcnt_all[i] = 0u;
  __syncthreads();
  if (tid == 0) {
    mbar_expect_tx(tab_bar, uint32_t(kSigTablePad * 4 + kE * 4));
    bulk_g2s(stab, a.stab, kSigTablePad * 4, tab_bar);
    bulk_g2s(bias_s, a.bias, kE * 4, tab_bar);
  }
  if (lane == 0) {
    for (int d = 0; d < L::D && d < nw; ++d) {
      mbar_expect_tx(mb + d, L::ROWB);
      bulk_g2s(ring + d * L::ROWB, logits + size_t(wr0 + d) * L::ROWB, L::ROWB, mb + d);
    }
  }
  // first row whose wait ran out (-1: none); 0 also when the table never arrived
  int fail_at = mbar_wait_bounded(tab_bar, 0, a.err) ? -1 : 0;

  // error bounds of the approximate scores: B = max |bias| over the experts
  float bmax;
  {
    float m = 0.0f;
    for (int e = tid; e < kE; e += NT) m = fmaxf(m, fabsf(bias_s[e]));
    const uint32_t wm = __reduce_max_sync(0xffffffffu, __float_as_uint(m));
    if (lane == 0) tmp[w] = int(wm);
    __syncthreads();
    uint32_t bm = 0;
#pragma unroll
    for (int i = 0; i < NW; ++i) bm = max(bm, uint32_t(tmp[i]));
    bmax = __uint_as_float(bm);
  }
  const ApproxBounds bnd = approx_bounds(a.eps_half, bmax);
  // this lane's 0.5 + bias (registers for the whole launch)
  float c[kEPL];
  {
    const float4* bq = reinterpret_cast<const float4*>(bias_s + lane * kEPL);
#pragma unroll
    for (int q = 0; q < kEPL / 4; ++q) {
      const float4 v = bq[q];
      c[4 * q + 0] = __fadd_rn(0.5f, v.x);
      c[4 * q + 1] = __fadd_rn(0.5f, v.y);
      c[4 * q + 2] = __fadd_rn(0.5f, v.z);
      c[4 * q + 3] = __fadd_rn(0.5f, v.w);
    }
  }

  // ---- phase 1: route this warp's rows, rank their entries within the warp
  for (int i = 0; i < nw && fail_at < 0; ++i) {
    const int slot = i % L::D;
    const uint32_t par = uint32_t(i / L::D) & 1u;
    if (!mbar_wait_bounded(mb + slot, par, a.err)) {
      fail_at = i;
      break;
    }
    const int t = wr0 + i;
    const SlotOut o = route_row_fast(ring + slot * L::ROWB, bias_s, stab, c, bnd, a, wsp[w]);
    if (lane < K) {
      a.packed[size_t(t) * K + lane] = o.packed;
      if (a.ids) a.ids[size_t(t) * K + lane] = o.id;
      const uint32_t sh = uint32_t(o.lid & 1) * 16u;
      const uint32_t old = atomicAdd(wcnt + (o.lid >> 1), 1u << sh);
      ent[i * K + lane] = uint32_t(o.lid) | (((old >> sh) & 0xFFFFu) << 16);
    }
    __syncwarp();
    if (lane == 0 && i + L::D < nw) {
      fence_proxy_async_smem();
      mbar_expect_tx(mb + slot, L::ROWB);
      bulk_g2s(ring + slot * L::ROWB, logits + size_t(t + L::D) * L::ROWB, L::ROWB, mb + slot);
    }
  }
  // after a wait that ran out, the copies issued for rows fail_at .. fail_at + D - 1 may
  // still be owed to the ring: wait for them (bounded) before the ring is reused
  if (fail_at >= 0 && lane == 0) {
    if (w == 0) mbar_wait_bounded(tab_bar, 0, nullptr);
    for (int r = fail_at; r < nw && r < fail_at + L::D; ++r)
      mbar_wait_bounded(mb + r % L::D, uint32_t(r / L::D) & 1u, nullptr);
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
  block_scan_fast(hist_s, lbase_s, a.NE, tmp);
  // every routed entry to its CTA-local sorted position (the ring is free now); after a
  // wait that ran out only the rows before it were routed and counted
  const int nrouted = fail_at < 0 ? nw : fail_at;
  for (int x = lane; x < nrouted * K; x += 32) {
    const uint32_t v = ent[x];
    const int l = int(v & 0xFFFFu);
    const uint32_t wp = (wcnt[l >> 1] >> (uint32_t(l & 1) * 16u)) & 0xFFFFu;
    const int lp = lbase_s[l] + int(wp) + int(v >> 16);
    sval[lp] = (wr0 + x / K) * K + (x % K);
    sbin[lp] = static_cast<uint16_t>(l);
  }

  int* flag_s = tmp + 32;
  if (!grid_barrier(pw.bar, grid, a.err, flag_s, a.barrier_wait_ns, a.barrier_skip_cta)) {
    grid_exit(pw.bar, grid);
    return;
  }
  column_scan(pw, a.NE, grid, NW);
  if (!grid_barrier(pw.bar, grid, a.err, flag_s, a.barrier_wait_ns)) {
    grid_exit(pw.bar, grid);
    return;
  }

  // ---- phase 3: offsets, then the sorted entries to perm, one run per bin
  for (int e = tid; e < a.NE; e += NT) {
    hist_s[e] = __ldcg(pw.counts + e);
    gbase_s[e] = __ldcg(pw.prefix + size_t(e) * pw.grid_max + cta);
  }
  __syncthreads();
  int* off_s = reinterpret_cast<int*>(smem + L::o_ent);  // the entries are placed: reuse
  block_scan_fast(hist_s, off_s, a.NE, tmp);
  if (cta == 0) {
    for (int e = tid; e < a.NE; e += NT) {
      a.counts[e] = hist_s[e];
      a.offsets[e] = off_s[e];
    }
    if (tid == 0) a.offsets[a.NE] = off_s[a.NE];
  }
  // global place of CTA-local position 0 of bin e
  for (int e = tid; e < a.NE; e += NT) gbase_s[e] += off_s[e] - lbase_s[e];
  __syncthreads();
  const int nvalid = lbase_s[a.NE];
  for (int i = tid; i < nvalid; i += NT) a.perm[gbase_s[sbin[i]] + i] = sval[i];
  grid_exit(pw.bar, grid);
}

cudaError_t setup_prefill_fast(int* blocks_per_sm) {
  cudaError_t e = cudaFuncSetAttribute(k_route_prefill_fast, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       FastSmem::total);
  if (e != cudaSuccess) return e;
  return cudaOccupancyMaxActiveBlocksPerMultiprocessor(blocks_per_sm, k_route_prefill_fast,
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
  if (!prefill_fast_fits(a.T, grid) || a.k != 16 || a.Kg != 4) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(FastSmem::NW * 32, 1, 1);
  cfg.dynamicSmemBytes = FastSmem::total;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_route_prefill_fast, a, ws);
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
