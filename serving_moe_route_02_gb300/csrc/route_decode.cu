// route_decode.cu -- decode-size routing (T <= 64) in one launch of one thread-block
// cluster, plus the sigmoid table and elementwise score kernels.
//
// Decode rows are few (8-64 per step), so the kernel is latency-bound: CTAs of 8 warps
// holding up to 8 rows each (one CTA up to 4 rows, then 2..4 rows per CTA over up to 16
// CTAs, or up to 8 rows per CTA over 8 CTAs after the router contraction; see
// decode_ctas), all in one cluster.  Each warp routes one row (the prior art on the
// pages, FlashInfer's routingIndicesClusterKernel for Tier<896, 16>, also ran decode
// routing as one cluster -- sglang PR #37).  The histogram, scan and stable
// permutation need every row's ids.  After routing, each warp sends its row's
// relabelled ids into the id array of every other CTA of the cluster (one bulk copy
// per destination, from one lane each, through distributed shared memory, completion
// counted in bytes on the destination's mbarrier); once its mbarrier completes a CTA
// holds all rows' ids and builds, in its own shared memory, a mask of the rows holding
// each id (two 32-bit words per id).  Counts are the masks' popcounts, a block scan
// gives offsets, and since ids are unique within a row the stable rank of (t, j) is
// the number of earlier rows in its id's mask.  Each CTA writes the permutation
// entries of its own rows.  No global workspace and no atomics in global memory; every
// wait is bounded.
#include <cooperative_groups.h>
#include <cstring>

#include "launch.h"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kDecodeRowsPerCta = 8;
constexpr int kDecodeThreads = 32 * kDecodeRowsPerCta;
constexpr int kDecodeMaxCtas = 16;  // clusters of 16 where the GPU schedules them, else 8
constexpr int kDecodeMaxRows = 64;  // row masks are 64 bits
int g_decode_max_ctas = 8;

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int DT>
struct DecodeSmem {
  static constexpr int ROWB = (DT == DT_PACKED) ? 0 : (DT == DT_BF16) ? kE * 2 : kE * 4;
  static constexpr int STAB = (DT == DT_BF16) ? kSigTablePad * 4 : 0;
  static constexpr int BIASB = (DT == DT_PACKED) ? 0 : kE * 4;
  static constexpr int o_stab = 0;
  static constexpr int o_bias = align_up(o_stab + STAB, 128);  // (scores: no table)
  static constexpr int o_rows = align_up(o_bias + BIASB, 128);
  static constexpr int o_ws = align_up(o_rows + kDecodeRowsPerCta * ROWB, 128);
  static constexpr int o_lid = align_up(o_ws + kDecodeRowsPerCta * int(sizeof(WarpScratch)), 128);
  static constexpr int o_offs = align_up(o_lid + 64 * kMaxK * 4, 128);  // lid: [64 rows][32]
  static constexpr int o_mask = align_up(o_offs + (kMaxBins + 1) * 4, 128);
  static constexpr int o_tmp = align_up(o_mask + kMaxBins * 8, 128);
  static constexpr int o_mbar = align_up(o_tmp + 32 * 4, 128);
  static constexpr int used = o_mbar + 64;
  // at least 118 KB, more than half an SM's shared memory, so that the CTAs of the next
  // call (a programmatic dependent, launched early) never share an SM with this one's
  // (16 rows: 3.37 -> 3.29 us per call)
  static constexpr int total = used > 118 * 1024 ? used : 118 * 1024;
};

static_assert(DecodeSmem<DT_F32>::total <= 227 * 1024, "decode smem (f32) exceeds 227 KB");
static_assert(DecodeSmem<DT_BF16>::total <= 227 * 1024, "decode smem (bf16) exceeds 227 KB");
static_assert(DecodeSmem<DT_SCORE>::total <= 227 * 1024, "decode smem (scores) exceeds 227 KB");
static_assert(DecodeSmem<DT_PACKED>::total <= 227 * 1024, "decode smem (index) exceeds 227 KB");

// Exclusive scan over the bins of counts popc(mask[e]) into offs[0..n], offs[n] = total,
// by the whole block: thread i takes the bins [i per, i per + per), per = ceil(n / 256)
// (at most 5), with all its mask loads in flight; warp scans, then the warp totals
// through `wtot` (8 ints).  Ends with a block barrier.
// mask[e] holds rows 0..31 in its low word, 32..63 in its high word.
__device__ __forceinline__ void mask_count_scan(const unsigned long long* mask, int* offs, int n,
                                                int* wtot) {
  constexpr int kPer = (kMaxBins + kDecodeThreads - 1) / kDecodeThreads;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int per = (n + kDecodeThreads - 1) / kDecodeThreads;
  const int lo = tid * per;
  int c[kPer];
  int sum = 0;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    c[q] = (q < per && lo + q < n) ? __popcll(mask[lo + q]) : 0;
    sum += c[q];
  }
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) wtot[w] = incl;
  __syncthreads();
  int wpre = 0;
#pragma unroll
  for (int i = 0; i < kDecodeRowsPerCta; ++i) wpre += (i < w) ? wtot[i] : 0;
  int run = wpre + incl - sum;
#pragma unroll
  for (int q = 0; q < kPer; ++q) {
    if (q < per && lo + q < n) offs[lo + q] = run;
    run += c[q];
  }
  if (tid == kDecodeThreads - 1) offs[n] = run;
  __syncthreads();
}

// --------------------------------------------------------- MXFP4 quantisation
// The quant half of the fused route+quant decode launch: the batch's activations
// x [T, H] (bf16) become MXFP4 (OCP Microscaling v1.0 MXFP4, the format the routed MXFP4
// MoE consumes; sglang PR #37, description: route_quant_fused, decode batches up to 64
// tokens).  Per block of 32 consecutive elements of a row: scale exponent
// e = floor(log2 max |x|) - 2, clamped to [-127, 127] (-127 for a block of zeros), stored
// as the E8M0 byte e + 127; elements x / 2^e rounded to E2M1 to nearest, ties to even,
// saturating at 6, by the hardware conversion; two codes per byte, even element low.

// E2M1 codes of two floats: lo in bits 0-3, hi in bits 4-7.
__device__ __forceinline__ uint32_t e2m1x2(float lo, float hi) {
  uint32_t r;
  asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
      : "=r"(r)
      : "f"(hi), "f"(lo));
  return r;
}

// Quantises the batch's 32-element blocks (rows are contiguous, so block b starts at
// element 32 b): warp gw of GW takes warp steps gw, gw + GW, ... of 8 blocks each, lanes
// 4j..4j+3 block j of the step, 8 elements (16 bytes) per lane.  kQSteps steps' loads are
// issued before any is converted, so a warp keeps 8 KB in flight.
constexpr int kQSteps = 16;
__device__ __forceinline__ void mxfp4_quant_blocks(const RouteArgs& a, int gw, int GW) {
  constexpr unsigned FULL = 0xffffffffu;
  const int lane = threadIdx.x & 31;
  const int sub = lane & 3;
  const int nblk = a.T * (a.qH >> 5);
  const int nstep = (nblk + 7) >> 3;
  const uint4* xv = reinterpret_cast<const uint4*>(a.qx);
  uint32_t* qv = reinterpret_cast<uint32_t*>(a.qcodes);
  for (int s0 = gw; s0 < nstep; s0 += GW * kQSteps) {
    uint4 v[kQSteps];
#pragma unroll
    for (int u = 0; u < kQSteps; ++u) {
      const int b = (s0 + u * GW) * 8 + (lane >> 2);
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (b < nblk) v[u] = __ldg(xv + size_t(b) * 4 + sub);
    }
#pragma unroll
    for (int u = 0; u < kQSteps; ++u) {
      const int b = (s0 + u * GW) * 8 + (lane >> 2);
      // the block's largest magnitude, as bf16 magnitude bits (they order like the values)
      const uint32_t mm = __vmaxu2(__vmaxu2(v[u].x & 0x7FFF7FFFu, v[u].y & 0x7FFF7FFFu),
                                   __vmaxu2(v[u].z & 0x7FFF7FFFu, v[u].w & 0x7FFF7FFFu));
      uint32_t m = max(mm & 0xFFFFu, mm >> 16);
      m = max(m, __shfl_xor_sync(FULL, m, 1));
      m = max(m, __shfl_xor_sync(FULL, m, 2));
      int e = -127;
      if (m != 0u) {
        // floor(log2 amax): the exponent field, or for a subnormal the leading mantissa bit
        const int ex = int(m >> 7);
        const int fl = ex > 0 ? ex - 127 : -133 + (31 - __clz(int(m)));
        e = min(max(fl - 2, -127), 127);
      }
      const float inv = __int_as_float(uint32_t(127 - e) << 23);  // 2^-e (e <= 125 for bf16)
      const uint32_t w4[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
      uint32_t word = 0u;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const float lo = __fmul_rn(__uint_as_float(w4[i] << 16), inv);
        const float hi = __fmul_rn(__uint_as_float(w4[i] & 0xFFFF0000u), inv);
        word |= e2m1x2(lo, hi) << (8 * i);
      }
      if (b < nblk) {
        qv[size_t(b) * 4 + sub] = word;
        if (sub == 0) a.qscales[b] = static_cast<uint8_t>(e + 127);
      }
    }
  }
}

// SPEC: k = 16 and topk_group = 4 compiled in (the Kimi-K3 instance).  QUANT: the
// launch also quantises the activations a.qx (moe_route_quant).
template <int DT, bool SPEC, bool QUANT = false>
__global__ void __launch_bounds__(kDecodeThreads, 1) k_route_decode(RouteArgs a) {
  using L = DecodeSmem<DT>;
  extern __shared__ __align__(128) uint8_t smem[];
  cg::cluster_group cluster = cg::this_cluster();
  float* stab = reinterpret_cast<float*>(smem + L::o_stab);
  float* bias_s = reinterpret_cast<float*>(smem + L::o_bias);
  uint8_t* rows = smem + L::o_rows;
  WarpScratch* wsp = reinterpret_cast<WarpScratch*>(smem + L::o_ws);
  int* offs_s = reinterpret_cast<int*>(smem + L::o_offs);
  unsigned long long* mask_s = reinterpret_cast<unsigned long long*>(smem + L::o_mask);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L::o_mbar);
  uint64_t* xbar = mbar + 1;  // the other CTAs' rows of ids (bulk copies, counted in bytes)

  int32_t* lid_all = reinterpret_cast<int32_t*>(smem + L::o_lid);
  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int crank = static_cast<int>(cluster.block_rank());
  const int nctas = static_cast<int>(cluster.num_blocks());
  // rows split evenly over the cluster's CTAs (at most 8 each), so that for 9..63 rows
  // fewer warps share an SM's shared-memory bandwidth in the score phase
  const int rpc = (a.T + nctas - 1) / nctas;
  const int row0 = crank * rpc;
  const int nrows = max(0, min(rpc, a.T - row0));
  const uint32_t bytes = uint32_t(nrows) * L::ROWB + uint32_t(L::STAB) + uint32_t(L::BIASB);
  const bool have = DT != DT_PACKED && nrows > 0;  // CTAs without rows (T = 0) load nothing

  // a programmatic dependent launched after this kernel (the next routing call) may
  // start now: before its own griddepcontrol.wait it only loads the constant score
  // table, and that wait returns once this grid has completed and its writes are visible
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  if constexpr (QUANT) {
    // the activations' quantisation runs on the clusters after the first one, so that it
    // shares no SM with the routing; every warp of those CTAs takes a share
    if (blockIdx.x >= unsigned(nctas)) {
      asm volatile("griddepcontrol.wait;" ::: "memory");  // x is an input
      mxfp4_quant_blocks(a, (int(blockIdx.x) - nctas) * kDecodeRowsPerCta + w,
                         (int(gridDim.x) - nctas) * kDecodeRowsPerCta);
      return;
    }
  }
  // bytes of one row of ids as copied between CTAs (whole 16-byte chunks of the row slot)
  const uint32_t idrow = uint32_t((a.k + 3) / 4) * 16u;
  if (tid == 0) {
    mbar_init(mbar, 1);
    mbar_init(xbar, 1);
    fence_mbar_init();
    // every row that another CTA routes arrives here once
    if (nctas > 1) mbar_expect_tx(xbar, uint32_t(a.T - nrows) * idrow);
  }
  __syncthreads();
  if (tid == 0 && have) {
    mbar_expect_tx(mbar, bytes);
    // the score table is the library's own constant: it may be read before the
    // preceding kernel completes
    if (L::STAB) bulk_g2s(stab, a.stab, L::STAB, mbar);
  }
  // every CTA of the cluster must be running before another one stores into its shared
  // memory: arrive now (relaxed: nothing to publish, and no wait for the copies in
  // flight), wait after routing
  for (int e = tid; e < a.NE; e += kDecodeThreads) mask_s[e] = 0ull;
  if (nctas > 1) asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  // launched as a programmatic dependent: everything above overlaps the preceding
  // kernel; inputs are read and outputs written only after it has completed
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (tid == 0 && have) {
    bulk_g2s(bias_s, a.bias, kE * 4, mbar);
    bulk_g2s(rows, static_cast<const uint8_t*>(a.logits) + size_t(row0) * L::ROWB,
             uint32_t(nrows) * L::ROWB, mbar);
  }
  // only the routing warps need the rows; the others go on to the hardware barriers below
  // instead of polling this one
  if (have && w < nrows) mbar_wait_bounded(mbar, 0, a.err);

  SlotOut o = {};
  if constexpr (DT == DT_PACKED) {
    // index mode: the row's ids come from the given packed values; an id at or above
    // the bin count is reported and left out (-1)
    if (w < nrows && lane < a.k) {
      const int t = row0 + w;
      o.lid = int(uint32_t(static_cast<const int32_t*>(a.logits)[size_t(t) * a.k + lane]) >> 16);
      // ids must be distinct within a row (the ranks below count rows per id)
      const unsigned kmask = (a.k == 32) ? 0xffffffffu : ((1u << a.k) - 1u);
      const bool repeated = __popc(__match_any_sync(kmask, o.lid)) > 1;
      if (o.lid >= a.NE || repeated) {
        atomicExch(a.err, kErrBadId);
        o.lid = -1;
      }
      lid_all[t * kMaxK + lane] = o.lid;
    }
  } else if (w < nrows) {
    o = route_row<DT, SPEC ? 16 : 0, SPEC ? 4 : 0>(rows + w * L::ROWB, bias_s, stab, a, wsp[w]);
    const int t = row0 + w;
    if (lane < a.k) {
      a.packed[size_t(t) * a.k + lane] = o.packed;
      if (a.ids) a.ids[size_t(t) * a.k + lane] = o.id;
      lid_all[t * kMaxK + lane] = o.lid;
    }
  }
  if (nctas > 1) asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
  // ---- a9..a11: this warp's row of ids goes to every other CTA: lane c sends one bulk
  // copy into CTA c's id array, counted on that CTA's xbar (a cluster barrier after
  // remote stores cost more than these copies' round trip)
  if (nctas > 1 && w < nrows) {
    fence_proxy_async_smem();  // the row's ids (written above) visible to the copy engine
    __syncwarp();
    const uint32_t src = smem_addr(lid_all + (row0 + w) * kMaxK);
    if (lane < nctas && lane != crank) {
      uint32_t dst, bar;
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(dst) : "r"(src), "r"(lane));
      asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(bar) : "r"(smem_addr(xbar)), "r"(lane));
      asm volatile(
          "cp.async.bulk.shared::cluster.shared::cta.mbarrier::complete_tx::bytes [%0], [%1], %2, "
          "[%3];" ::"r"(dst),
          "r"(src), "r"(idrow), "r"(bar)
          : "memory");
      asm volatile("cp.async.bulk.commit_group;" ::: "memory");
    }
  }
  // this CTA's own rows (block barrier), then every other CTA's (their copies)
  __syncthreads();
  if (nctas > 1 && !mbar_wait_bounded(xbar, 0, a.err)) {
    // a copy into this CTA may still be on its way: every CTA sends its rows once its
    // own bounded row wait is over; wait that long again before going on
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(xbar, 0) && globaltimer_ns() - t0 < 2 * kWaitLimitNs) {
    }
  }
  uint32_t* mask32 = reinterpret_cast<uint32_t*>(mask_s);
  const int kk = SPEC ? 16 : a.k;
  for (int x = tid; x < a.T * kk; x += kDecodeThreads) {
    const int t = x / kk, j = x - t * kk;
    const int l = lid_all[t * kMaxK + j];
    if (DT != DT_PACKED || l >= 0) atomicOr(mask32 + 2 * l + (t >> 5), 1u << (t & 31));
  }
  __syncthreads();

  mask_count_scan(mask_s, offs_s, a.NE, reinterpret_cast<int*>(smem + L::o_tmp));
  if (crank == 0) {
    for (int e = tid; e < a.NE; e += kDecodeThreads) {
      a.counts[e] = __popcll(mask_s[e]);
      a.offsets[e] = offs_s[e];
    }
    if (tid == 0) a.offsets[a.NE] = offs_s[a.NE];
  }
  if (w < nrows && lane < a.k && (DT != DT_PACKED || o.lid >= 0)) {
    const int t = row0 + w;
    const int pos = offs_s[o.lid] + __popcll(mask_s[o.lid] & ((1ull << t) - 1ull));
    a.perm[pos] = t * a.k + lane;
    if (a.inv) a.inv[t * a.k + lane] = pos;
  }
  // the outgoing copies have read this CTA's id rows before it leaves
  if (nctas > 1 && w < nrows && lane < nctas && lane != crank)
    asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// --------------------------------------------------------------- sigmoid table
__global__ void k_sigmoid_table(float* tab, float2* etab) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i < kExpTable) {
    const double v = exp2(static_cast<double>(i) / kExpTable);
    const float hi = __double2float_rn(v);
    etab[i] = make_float2(hi, __double2float_rn(v - static_cast<double>(hi)));
  }
  if (i >= kSigTablePad) return;
  if (i >= kSigTable) {
    tab[i] = 0.0f;
    return;
  }
  const uint32_t sign = uint32_t(i / kSigN);
  const uint32_t h = (kSigLo + uint32_t(i % kSigN)) | (sign << 15);
  const float x = __uint_as_float(h << 16);
  const double e = exp(-static_cast<double>(x));
  const double s = 1.0 / (1.0 + e);
  tab[i] = __double2float_rn(s);
}

__global__ void k_sigmoid(const void* x, int dtype, const float* __restrict__ tab,
                          const float2* __restrict__ etab, float* s, int n) {
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x) {
    s[i] = (dtype == DT_BF16) ? sig_bf16(tab, static_cast<const uint16_t*>(x)[i])
                              : sig_f32(static_cast<const float*>(x)[i], etab);
  }
}

// E_f32 = max over every float32 x (not NaN) of |0.5 tanh.approx(x / 2) + 0.5 - sig_f32(x)|,
// the bound behind route_row's approximate float32 scores.  The difference is formed in
// float (fma(0.5, t, 0.5) rounded, then one subtraction), so the true value is at most
// the measured one times (1 + 2^-22) plus 2^-24, which the host adds.  For |x| > 80 the
// exact score is 1 (x > 0: sigmoid(x) > 1 - 2^-115 rounds to 1) or below 2^-115 (x < 0),
// so those are compared with 1 and 0 (an error of at most 2^-115, covered by the same
// 2^-24).  Written to *out as the bits of a non-negative float; *out must start at 0.
__global__ void k_approx_err_f32(const float2* __restrict__ etab, unsigned* out) {
  unsigned m = 0u;
  const uint64_t stride = uint64_t(gridDim.x) * blockDim.x;
  for (uint64_t u = uint64_t(blockIdx.x) * blockDim.x + threadIdx.x; u < (1ull << 32); u += stride) {
    const uint32_t bits = uint32_t(u);
    if ((bits & 0x7F800000u) == 0x7F800000u && (bits & 0x007FFFFFu) != 0u) continue;  // NaN
    const float x = __uint_as_float(bits);
    float t;
    asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(__fmul_rn(x, 0.5f)));
    const float s = fabsf(x) > 80.0f ? (x > 0.0f ? 1.0f : 0.0f) : sig_f32(x, etab);
    const float d = fabsf(__fsub_rn(__fmaf_rn(0.5f, t, 0.5f), s));
    m = max(m, __float_as_uint(d));
  }
  m = __reduce_max_sync(0xffffffffu, m);
  if ((threadIdx.x & 31) == 0 && m != 0u) atomicMax(out, m);
}

cudaError_t launch_approx_err_f32(const float2* etab, unsigned* out, cudaStream_t st) {
  k_approx_err_f32<<<152 * 8, 256, 0, st>>>(etab, out);
  return cudaGetLastError();
}

float approx_bound_f32(unsigned measured_bits) {
  float e;
  std::memcpy(&e, &measured_bits, sizeof(e));
  return e * (1.0f + 0x1p-22f) + 0x1p-24f;
}

cudaError_t launch_sigmoid_table(float* tab, float2* etab, cudaStream_t st) {
  k_sigmoid_table<<<(kSigTablePad + 255) / 256, 256, 0, st>>>(tab, etab);
  return cudaGetLastError();
}

cudaError_t launch_sigmoid(const void* x, int dtype, const float* tab, const float2* etab, float* s,
                           int n, cudaStream_t st) {
  if (n <= 0) return cudaSuccess;
  const int blocks = min((n + 255) / 256, 4096);
  k_sigmoid<<<blocks, 256, 0, st>>>(x, dtype, tab, etab, s, n);
  return cudaGetLastError();
}

// CTAs of a decode launch: one for up to 5 rows (no cluster barrier, which costs about
// 0.3 us); above that, the fewest CTAs that hold max(2, ceil(T / M)) rows each, M = 16
// where clusters of 16 can be scheduled, else 8 (8 rows: 4 CTAs of 2; 64 rows: 16 CTAs
// of 4, or 8 of 8).  Measured crossover: 6 rows.
int decode_ctas(int T, int max_ctas) {
  if (T <= 4) return 1;
  const int per = max(2, (T + max_ctas - 1) / max_ctas);
  return (T + per - 1) / per;
}

int decode_ctas(int T) { return decode_ctas(T, g_decode_max_ctas); }

__global__ void __launch_bounds__(kDecodeThreads, 1) k_empty() {}

// The floor kernel asks for the bf16 decode kernel's shared memory, so that both run in
// the same shared-memory configuration of the SM: with none asked for, an empty launch
// replayed after kernels that use most of the shared memory took 0.57 us instead of 0.38.
constexpr int kEmptySmem = DecodeSmem<DT_BF16>::total;

cudaError_t launch_empty(int ctas, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kDecodeThreads, 1, 1);
  cfg.dynamicSmemBytes = kEmptySmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // as the routing kernel
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, k_empty);
}

// Shared-memory size of one decode kernel; clears *wide if clusters of 16 are refused.
template <int DT, bool SPEC, bool QUANT = false>
static cudaError_t set_decode_smem(bool* wide) {
  cudaError_t e = cudaFuncSetAttribute(k_route_decode<DT, SPEC, QUANT>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, DecodeSmem<DT>::total);
  if (e != cudaSuccess) return e;
  if (cudaFuncSetAttribute(k_route_decode<DT, SPEC, QUANT>, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) !=
      cudaSuccess) {
    cudaGetLastError();
    *wide = false;
  }
  return cudaSuccess;
}

cudaError_t setup_decode_kernels() {
  cudaError_t e;
  bool wide = true;
  if ((e = set_decode_smem<DT_F32, false>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_F32, true>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_BF16, false>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_BF16, true>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_SCORE, false>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_SCORE, true>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_PACKED, false>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_F32, false, true>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_F32, true, true>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_BF16, false, true>(&wide)) != cudaSuccess) return e;
  if ((e = set_decode_smem<DT_BF16, true, true>(&wide)) != cudaSuccess) return e;
  if ((e = cudaFuncSetAttribute(k_empty, cudaFuncAttributeMaxDynamicSharedMemorySize, kEmptySmem)) != cudaSuccess)
    return e;
  if (cudaFuncSetAttribute(k_empty, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess) {
    cudaGetLastError();
    wide = false;
  }
  g_decode_max_ctas = wide ? 16 : 8;
  // clusters of 16 only where one can be resident (the largest shared-memory variant)
  if (g_decode_max_ctas == 16) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(16, 1, 1);
    cfg.blockDim = dim3(kDecodeThreads, 1, 1);
    cfg.dynamicSmemBytes = DecodeSmem<DT_BF16>::total;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 16;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, k_route_decode<DT_BF16, true>, &cfg) != cudaSuccess || n < 1)
      g_decode_max_ctas = 8;
    cudaGetLastError();  // clear a refused query
  }
  return cudaSuccess;
}

template <int DT, bool SPEC>
static cudaError_t launch_decode_t(cudaLaunchConfig_t& cfg, const RouteArgs& a) {
  cfg.dynamicSmemBytes = DecodeSmem<DT>::total;
  if constexpr (DT == DT_BF16 || DT == DT_F32) {
    if (a.qx != nullptr) {
      // route+quant: the routing cluster, then as many clusters of the same size as give
      // every quantising warp at most one pass of kQSteps steps (8 blocks a step)
      const int ctas = int(cfg.gridDim.x);
      const long long steps = (static_cast<long long>(a.T) * (a.qH >> 5) + 7) / 8;
      const long long per_cluster = static_cast<long long>(ctas) * kDecodeRowsPerCta * kQSteps;
      const long long q = steps > 0 ? (steps + per_cluster - 1) / per_cluster : 0;
      cfg.gridDim.x = unsigned(ctas * (1 + q));
      return cudaLaunchKernelEx(&cfg, k_route_decode<DT, SPEC, true>, a);
    }
  }
  return cudaLaunchKernelEx(&cfg, k_route_decode<DT, SPEC>, a);
}

cudaError_t launch_route_decode(const RouteArgs& a, int dtype, cudaStream_t st, int max_ctas) {
  if (a.T > kDecodeMaxRows) return cudaErrorInvalidValue;
  const int ctas = decode_ctas(a.T, max_ctas > 0 && max_ctas < g_decode_max_ctas ? max_ctas : g_decode_max_ctas);
  // a CTA's row buffer and warps hold at most kDecodeRowsPerCta rows
  if (ctas < 1 || (a.T + ctas - 1) / ctas > kDecodeRowsPerCta) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kDecodeThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  const bool spec = a.k == 16 && a.Kg == 4;
  if (dtype == DT_BF16) return spec ? launch_decode_t<DT_BF16, true>(cfg, a) : launch_decode_t<DT_BF16, false>(cfg, a);
  if (dtype == DT_SCORE) return spec ? launch_decode_t<DT_SCORE, true>(cfg, a) : launch_decode_t<DT_SCORE, false>(cfg, a);
  if (dtype == DT_PACKED) return launch_decode_t<DT_PACKED, false>(cfg, a);
  return spec ? launch_decode_t<DT_F32, true>(cfg, a) : launch_decode_t<DT_F32, false>(cfg, a);
}

}  // namespace moe
