// route_decode.cu -- decode-size routing (T <= 64) in one launch of one thread-block
// cluster, plus the sigmoid table and elementwise score kernels.
//
// Decode rows are few (8-64 per step), so the kernel is latency-bound: one CTA of 8
// warps per 8 rows, up to 8 CTAs in one cluster.  Each warp routes one row (the
// prior art on the pages, FlashInfer's routingIndicesClusterKernel for
// Tier<896, 16>, also ran decode routing as one cluster -- sglang PR #37).  The
// histogram, scan and stable permutation need every row's ids: after a cluster
// barrier each CTA reads all CTAs' relabelled ids through distributed shared memory,
// builds the histogram and a per-id bitmask of the rows containing it (ids are unique
// within a row, so the stable rank of (t, j) is the number of earlier rows holding the
// same id), scans, and writes the permutation entries of its own rows.  No global
// workspace, no atomics in global memory, no spin waits.
#include <cooperative_groups.h>

#include "launch.h"

namespace cg = cooperative_groups;

namespace moe {

constexpr int kDecodeRowsPerCta = 8;
constexpr int kDecodeThreads = 32 * kDecodeRowsPerCta;
constexpr int kDecodeMaxCtas = 8;

__host__ __device__ constexpr int align_up(int x, int a) { return (x + a - 1) / a * a; }

template <int DT>
struct DecodeSmem {
  static constexpr int ROWB = (DT == DT_BF16) ? kE * 2 : kE * 4;
  static constexpr int STAB = (DT == DT_BF16) ? kSigTablePad * 4 : 0;
  static constexpr int o_stab = 0;
  static constexpr int o_rows = align_up(o_stab + STAB, 128);  // (scores: no table)
  static constexpr int o_ws = align_up(o_rows + kDecodeRowsPerCta * ROWB, 128);
  static constexpr int o_lid = align_up(o_ws + kDecodeRowsPerCta * int(sizeof(WarpScratch)), 128);
  static constexpr int o_counts = align_up(o_lid + kDecodeRowsPerCta * 32 * 4, 128);
  static constexpr int o_offs = align_up(o_counts + kMaxBins * 4, 128);
  static constexpr int o_mask = align_up(o_offs + (kMaxBins + 1) * 4, 128);
  static constexpr int o_tmp = align_up(o_mask + kMaxBins * 8, 128);
  static constexpr int o_mbar = align_up(o_tmp + 32 * 4, 128);
  static constexpr int total = o_mbar + 64;
};

static_assert(DecodeSmem<DT_F32>::total <= 227 * 1024, "decode smem (f32) exceeds 227 KB");
static_assert(DecodeSmem<DT_BF16>::total <= 227 * 1024, "decode smem (bf16) exceeds 227 KB");
static_assert(DecodeSmem<DT_SCORE>::total <= 227 * 1024, "decode smem (scores) exceeds 227 KB");

template <int DT>
__global__ void __launch_bounds__(kDecodeThreads, 1) k_route_decode(RouteArgs a) {
  using L = DecodeSmem<DT>;
  extern __shared__ __align__(128) uint8_t smem[];
  cg::cluster_group cluster = cg::this_cluster();
  float* stab = reinterpret_cast<float*>(smem + L::o_stab);
  uint8_t* rows = smem + L::o_rows;
  WarpScratch* wsp = reinterpret_cast<WarpScratch*>(smem + L::o_ws);
  int32_t* lid_s = reinterpret_cast<int32_t*>(smem + L::o_lid);
  int* counts_s = reinterpret_cast<int*>(smem + L::o_counts);
  int* offs_s = reinterpret_cast<int*>(smem + L::o_offs);
  unsigned long long* mask_s = reinterpret_cast<unsigned long long*>(smem + L::o_mask);
  int* tmp = reinterpret_cast<int*>(smem + L::o_tmp);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + L::o_mbar);

  const int tid = threadIdx.x, w = tid >> 5, lane = tid & 31;
  const int crank = static_cast<int>(cluster.block_rank());
  const int row0 = crank * kDecodeRowsPerCta;
  const int nrows = max(0, min(kDecodeRowsPerCta, a.T - row0));
  const uint32_t bytes = uint32_t(nrows) * L::ROWB + uint32_t(L::STAB);
  const bool have = nrows > 0;  // CTAs without rows (T = 0) load nothing

  if (tid == 0) {
    mbar_init(mbar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0 && have) {
    mbar_expect_tx(mbar, bytes);
    if (L::STAB) bulk_g2s(stab, a.stab, L::STAB, mbar);
    bulk_g2s(rows, static_cast<const uint8_t*>(a.logits) + size_t(row0) * L::ROWB,
             uint32_t(nrows) * L::ROWB, mbar);
  }
  float bl[kEPL];
  load_lane_bias(a.bias, bl);
  if (have) mbar_wait_bounded(mbar, 0, a.err);

  if (w < nrows) {
    const SlotOut o = route_row<DT>(rows + w * L::ROWB, bl, stab, a, wsp[w]);
    const int t = row0 + w;
    if (lane < a.k) {
      a.packed[size_t(t) * a.k + lane] = o.packed;
      if (a.ids) a.ids[size_t(t) * a.k + lane] = o.id;
      lid_s[w * 32 + lane] = o.lid;
    }
  }
  cluster.sync();

  // ---- a9..a11 over all rows of the cluster
  for (int e = tid; e < a.NE; e += kDecodeThreads) {
    counts_s[e] = 0;
    mask_s[e] = 0ull;
  }
  __syncthreads();
  const int ntot = a.T * a.k;
  for (int x = tid; x < ntot; x += kDecodeThreads) {
    const int t = x / a.k, j = x - t * a.k;
    const int32_t* rl = cluster.map_shared_rank(lid_s, t / kDecodeRowsPerCta);
    const int l = rl[(t % kDecodeRowsPerCta) * 32 + j];
    atomicAdd(&counts_s[l], 1);
    atomicOr(&mask_s[l], 1ull << t);
  }
  __syncthreads();
  block_exclusive_scan(counts_s, offs_s, a.NE, tmp);
  if (crank == 0) {
    for (int e = tid; e < a.NE; e += kDecodeThreads) {
      a.counts[e] = counts_s[e];
      a.offsets[e] = offs_s[e];
    }
    if (tid == 0) a.offsets[a.NE] = offs_s[a.NE];
  }
  for (int x = tid; x < nrows * a.k; x += kDecodeThreads) {
    const int ww = x / a.k, j = x - ww * a.k;
    const int t = row0 + ww;
    const int l = lid_s[ww * 32 + j];
    const int pos = offs_s[l] + __popcll(mask_s[l] & ((1ull << t) - 1ull));
    a.perm[pos] = t * a.k + j;
  }
  cluster.sync();  // keep this CTA's shared memory alive for remote readers
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

__global__ void __launch_bounds__(kDecodeThreads, 1) k_empty() {}

cudaError_t launch_empty(int ctas, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kDecodeThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, k_empty);
}

cudaError_t setup_decode_kernels() {
  cudaError_t e = cudaFuncSetAttribute(k_route_decode<DT_F32>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DecodeSmem<DT_F32>::total);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(k_route_decode<DT_SCORE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           DecodeSmem<DT_SCORE>::total);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(k_route_decode<DT_BF16>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              DecodeSmem<DT_BF16>::total);
}

cudaError_t launch_route_decode(const RouteArgs& a, int dtype, cudaStream_t st) {
  const int ctas = max(1, (a.T + kDecodeRowsPerCta - 1) / kDecodeRowsPerCta);
  if (ctas > kDecodeMaxCtas) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(ctas, 1, 1);
  cfg.blockDim = dim3(kDecodeThreads, 1, 1);
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = ctas;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (dtype == DT_BF16) {
    cfg.dynamicSmemBytes = DecodeSmem<DT_BF16>::total;
    return cudaLaunchKernelEx(&cfg, k_route_decode<DT_BF16>, a);
  }
  if (dtype == DT_SCORE) {
    cfg.dynamicSmemBytes = DecodeSmem<DT_SCORE>::total;
    return cudaLaunchKernelEx(&cfg, k_route_decode<DT_SCORE>, a);
  }
  cfg.dynamicSmemBytes = DecodeSmem<DT_F32>::total;
  return cudaLaunchKernelEx(&cfg, k_route_decode<DT_F32>, a);
}

}  // namespace moe
