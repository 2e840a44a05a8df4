// api.cu -- the C ABI (include/moe_route.h): argument checks, per-device state and
// dispatch to the routing kernels.  No routing arithmetic happens on the host.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/moe_route.h"
#include "launch.h"

namespace {

using namespace moe;

struct DevState {
  std::atomic<bool> ready{false};  // set (release) once everything below is in place
  int nsm = 0;
  int blocks_per_sm = 0;
  int fast_blocks_per_sm = 0;  // the approximate-score persistent kernel
  float eps_half = 0.0f;       // its measured approximation bound (route_pair.cuh)
  float eps_f32 = -1.0f;       // route_row's float32 approximation bound
  float* stab = nullptr;  // sigmoid table for bf16 logits
  float2* etab = nullptr; // 2^(j/64) table for float32 logits
  int* err = nullptr;     // device status word
  PrefillWS pw = {};
  int* pw_block = nullptr;
  float* gscores = nullptr;  // [64][E] fp32 scores written by the fused contraction
};

constexpr int kMaxDevices = 64;
DevState g_dev[kMaxDevices];
std::mutex g_mu;
int g_path = 0;
// moe_route_arm_barrier_timeout: the next persistent launch's skipped CTA (-1: none) and
// grid-barrier wait limit
std::atomic<int> g_skip_cta{-1};
std::atomic<unsigned long long> g_skip_wait_ns{0};

bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return false;
  return cs != cudaStreamCaptureStatusNone;
}

// Creates the current device's state.  Must not run during stream capture.
int init_device(DevState& d) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (cudaDeviceGetAttribute(&d.nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  if (setup_decode_kernels() != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (setup_prefill_kernels(&d.blocks_per_sm) != cudaSuccess || d.blocks_per_sm < 1)
    return MOE_ROUTE_E_CUDA;
  if (setup_prefill_fast(&d.fast_blocks_per_sm) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  const int grid_max = d.nsm * d.blocks_per_sm;
  const size_t n_tab = size_t(kSigTablePad);
  const size_t n_hist = size_t(kMaxBins) * grid_max;
  if (setup_router_gemm() != cudaSuccess) return MOE_ROUTE_E_CUDA;
  // one block: [sigmoid table][exp table][hist][prefix][counts][bar x2, err, pad][logits]
  const size_t n_etab = size_t(2 * kExpTable);
  const size_t n_log = size_t(64) * kE;
  const size_t bytes = (n_tab + n_etab) * 4 + 2 * n_hist * 4 + size_t(kMaxBins) * 4 + 64 +
                       n_log * 4;
  int* blk = nullptr;
  if (cudaMalloc(&blk, bytes) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (cudaMemset(blk, 0, bytes) != cudaSuccess) {
    cudaFree(blk);
    return MOE_ROUTE_E_CUDA;
  }
  d.pw_block = blk;
  d.stab = reinterpret_cast<float*>(blk);
  d.etab = reinterpret_cast<float2*>(blk + n_tab);
  d.pw.hist = blk + n_tab + n_etab;
  d.pw.prefix = d.pw.hist + n_hist;
  d.pw.counts = d.pw.prefix + n_hist;
  d.pw.bar = reinterpret_cast<unsigned*>(d.pw.counts + kMaxBins);
  d.err = reinterpret_cast<int*>(d.pw.bar + 2);
  d.gscores = reinterpret_cast<float*>(d.pw.bar + 16);
  d.pw.grid_max = grid_max;
  if (launch_sigmoid_table(d.stab, d.etab, nullptr) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  // the approximation bound of the fast persistent kernel, measured into a spare word of
  // the zeroed workspace and read back (the word is zeroed again afterwards)
  unsigned* probe = d.pw.bar + 4;  // and probe + 1 for the float32 bound
  if (launch_approx_err(probe, nullptr) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (launch_approx_err_f32(d.etab, probe + 1, nullptr) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ROUTE_E_CUDA;
  unsigned bits[2] = {0, 0};
  if (cudaMemcpy(bits, probe, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (cudaMemset(probe, 0, sizeof(bits)) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  std::memcpy(&d.eps_half, &bits[0], sizeof(bits[0]));
  d.eps_f32 = approx_bound_f32(bits[1]);
  d.ready.store(true, std::memory_order_release);
  return MOE_ROUTE_OK;
}

// Returns the current device's state, creating it outside capture.
int get_state(cudaStream_t st, DevState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ROUTE_E_CUDA;
  DevState& d = g_dev[dev];
  if (!d.ready.load(std::memory_order_acquire)) {
    if (st != nullptr && capturing(st)) return MOE_ROUTE_E_WORKSPACE;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
      const int rc = init_device(d);
      if (rc != MOE_ROUTE_OK) return rc;
    }
  }
  *out = &d;
  return MOE_ROUTE_OK;
}

int bins(int E, int k, int cnt) { return cnt > 0 ? (cnt + k + 3) / 4 * 4 : E; }

int check_route_args(int T, int E, int k, int n_group, int topk_group, int off, int cnt) {
  if (T < 0 || E <= 0 || k <= 0 || n_group <= 0) return MOE_ROUTE_E_INVALID_ARG;
  if (E % n_group != 0 || E / n_group < 2) return MOE_ROUTE_E_INVALID_ARG;
  if (topk_group < 1 || topk_group > n_group) return MOE_ROUTE_E_INVALID_ARG;
  if (k > topk_group * (E / n_group)) return MOE_ROUTE_E_INVALID_ARG;
  if (cnt < 0 || off < 0 || off + cnt > E) return MOE_ROUTE_E_INVALID_ARG;
  if (E > 32767 || (cnt > 0 && cnt + k > 32767)) return MOE_ROUTE_E_INVALID_ARG;
  if (static_cast<long long>(T) * k >= (1ll << 31)) return MOE_ROUTE_E_INVALID_ARG;
  if (E != kE || n_group != kG || k > kMaxK) return MOE_ROUTE_E_UNSUPPORTED;
  if (bins(E, k, cnt) > kMaxBins) return MOE_ROUTE_E_UNSUPPORTED;
  return MOE_ROUTE_OK;
}

}  // namespace

namespace moe {
int route_args_status(int T, int E, int k, int n_group, int topk_group, int off, int cnt) {
  return check_route_args(T, E, k, n_group, topk_group, off, cnt);
}
}  // namespace moe

extern "C" {

int moe_route_bins(int E, int k, int local_count) { return bins(E, k, local_count); }

int moe_route_num_experts(int E, int k, int local_offset, int local_count) {
  (void)local_offset;
  if (local_count <= 0 || local_count >= E) return E;
  const int ne = bins(E, k, local_count);
  return ne < E ? ne : E;
}

int moe_route_reserve(void) {
  DevState* d = nullptr;
  return get_state(nullptr, &d);
}

int moe_route(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
              int n_group, int topk_group, float scale, int local_offset, int local_count,
              int32_t* packed, int32_t* counts, int32_t* offsets, int32_t* perm,
              int32_t* topk_ids, struct CUstream_st* stream) {
  return moe_route_ex(logits, logits_dtype, bias, T, E, k, n_group, topk_group, scale, local_offset,
                      local_count, packed, counts, offsets, perm, topk_ids, nullptr, stream);
}

namespace {

// The expert-GEMM layout asked of a routing call (moe_route_with_layout), validated.
struct LayoutReq {
  int tile, capacity;
  int32_t* padded_offsets;
  int32_t* padded_rows;
  int32_t* m_indices;
};

int route_impl(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
               int n_group, int topk_group, float scale, int local_offset, int local_count,
               int32_t* packed, int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* topk_ids,
               int32_t* inv_perm, const LayoutReq* lay, struct CUstream_st* stream) {
  int rc = check_route_args(T, E, k, n_group, topk_group, local_offset, local_count);
  if (rc != MOE_ROUTE_OK) return rc;
  if (logits_dtype != MOE_ROUTE_F32 && logits_dtype != MOE_ROUTE_BF16) return MOE_ROUTE_E_INVALID_ARG;
  if (!bias || !counts || !offsets) return MOE_ROUTE_E_INVALID_ARG;
  if (T > 0 && (!logits || !packed || !perm)) return MOE_ROUTE_E_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % 16 != 0 || reinterpret_cast<uintptr_t>(bias) % 16 != 0)
    return MOE_ROUTE_E_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DevState* d = nullptr;
  rc = get_state(st, &d);
  if (rc != MOE_ROUTE_OK) return rc;

  RouteArgs a = {};
  a.logits = logits;
  a.bias = bias;
  a.stab = d->stab;
  a.etab = d->etab;
  a.packed = packed;
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.ids = topk_ids;
  a.inv = inv_perm;
  a.err = d->err;
  a.T = T;
  a.k = k;
  a.Kg = topk_group;
  a.off = local_offset;
  a.cnt = local_count;
  a.NE = bins(E, k, local_count);
  a.scale = scale;
  a.eps_half = d->eps_half;
  // paths 3 and 4 compute every float32 score exactly (for comparisons)
  a.eps_f32 = (g_path == 3 || g_path == 4) ? -1.0f : d->eps_f32;
  const int dt = logits_dtype == MOE_ROUTE_BF16 ? DT_BF16 : DT_F32;

  const bool decode = (g_path == 1 || g_path == 4) || (g_path == 0 && T <= 64);
  cudaError_t ce;
  if (decode) {
    if (T > 64) return MOE_ROUTE_E_UNSUPPORTED;
    ce = launch_route_decode(a, dt, st);
  } else {
    if (T == 0) {
      ce = launch_route_decode(a, dt, st);
    } else {
      const int skip = g_skip_cta.exchange(-1);
      if (skip >= 0) {
        a.barrier_skip_cta = skip;
        a.barrier_wait_ns = g_skip_wait_ns.load();
      }
      // bf16 logits of the Kimi-K3 instance: the persistent kernel on approximate scores
      // (path 3 forces the exact-score kernel, for comparisons)
      int grid_fast = d->nsm * d->fast_blocks_per_sm;
      if (grid_fast > d->pw.grid_max) grid_fast = d->pw.grid_max;
      if (grid_fast > (T + 15) / 16) grid_fast = (T + 15) / 16;
      if (dt == DT_BF16 && k == 16 && topk_group == 4 && g_path != 3 && grid_fast >= 1 &&
          prefill_fast_fits(T, grid_fast)) {
        if (lay) {
          // this kernel writes the layout itself
          a.tile = lay->tile;
          a.capacity = lay->capacity;
          a.poffs = lay->padded_offsets;
          a.prows = lay->padded_rows;
          a.midx = lay->m_indices;
          lay = nullptr;
        }
        ce = launch_route_prefill_fast(a, d->pw, grid_fast, st);
      } else {
        const int grid_cap = d->pw.grid_max;
        int grid = (T + 15) / 16;
        if (grid > grid_cap) grid = grid_cap;
        if (!prefill_fits(T, grid)) return MOE_ROUTE_E_UNSUPPORTED;
        ce = launch_route_prefill(a, dt, d->pw, grid, st);
      }
    }
  }
  if (ce == cudaSuccess && lay) {
    // elsewhere the layout kernel follows the routing on the stream
    LayoutArgs g = {};
    g.counts = counts;
    g.offsets = offsets;
    g.perm = perm;
    g.n = T * k;
    g.NE = a.NE;
    g.tile = lay->tile;
    g.capacity = lay->capacity;
    g.padded_offsets = lay->padded_offsets;
    g.padded_rows = lay->padded_rows;
    g.m_indices = lay->m_indices;
    ce = launch_route_layout(g, d->nsm, st);
  }
  return ce == cudaSuccess ? MOE_ROUTE_OK : MOE_ROUTE_E_CUDA;
}

}  // namespace

int moe_route_ex(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
                 int n_group, int topk_group, float scale, int local_offset, int local_count,
                 int32_t* packed, int32_t* counts, int32_t* offsets, int32_t* perm,
                 int32_t* topk_ids, int32_t* inv_perm, struct CUstream_st* stream) {
  return route_impl(logits, logits_dtype, bias, T, E, k, n_group, topk_group, scale, local_offset,
                    local_count, packed, counts, offsets, perm, topk_ids, inv_perm, nullptr, stream);
}

int moe_route_with_layout(const void* logits, int logits_dtype, const float* bias, int T, int E,
                          int k, int n_group, int topk_group, float scale, int local_offset,
                          int local_count, int32_t* packed, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* topk_ids, int32_t* inv_perm, int tile,
                          int32_t* padded_offsets, int32_t* padded_rows, int32_t* m_indices,
                          int capacity, struct CUstream_st* stream) {
  int rc = check_route_args(T, E, k, n_group, topk_group, local_offset, local_count);
  if (rc != MOE_ROUTE_OK) return rc;
  const int NE = bins(E, k, local_count);
  const int need = moe_route_padded_capacity(T, k, NE, tile);
  if (need < 0) return MOE_ROUTE_E_INVALID_ARG;
  const bool padded = padded_rows || m_indices;
  if (padded && capacity < need) return MOE_ROUTE_E_INVALID_ARG;
  LayoutReq lay = {tile, padded ? capacity : 0, padded_offsets, padded_rows, m_indices};
  return route_impl(logits, logits_dtype, bias, T, E, k, n_group, topk_group, scale, local_offset,
                    local_count, packed, counts, offsets, perm, topk_ids, inv_perm,
                    (padded_offsets || padded) ? &lay : nullptr, stream);
}

int moe_route_quant(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
                    int n_group, int topk_group, float scale, int local_offset, int local_count,
                    const uint16_t* x, int H, uint8_t* x_q, uint8_t* x_scales, int32_t* packed,
                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* topk_ids,
                    struct CUstream_st* stream) {
  int rc = check_route_args(T, E, k, n_group, topk_group, local_offset, local_count);
  if (rc != MOE_ROUTE_OK) return rc;
  if (logits_dtype != MOE_ROUTE_F32 && logits_dtype != MOE_ROUTE_BF16) return MOE_ROUTE_E_INVALID_ARG;
  if (!bias || !counts || !offsets) return MOE_ROUTE_E_INVALID_ARG;
  if (T > 0 && (!logits || !packed || !perm || !x || !x_q || !x_scales)) return MOE_ROUTE_E_INVALID_ARG;
  if (H <= 0 || H % 32 != 0) return MOE_ROUTE_E_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % 16 != 0 || reinterpret_cast<uintptr_t>(bias) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(x) % 16 != 0 || reinterpret_cast<uintptr_t>(x_q) % 4 != 0)
    return MOE_ROUTE_E_INVALID_ARG;
  if (T > MOE_ROUTE_QUANT_MAX_TOKENS) return MOE_ROUTE_E_UNSUPPORTED;
  if (static_cast<long long>(T) * H >= (1ll << 31)) return MOE_ROUTE_E_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DevState* d = nullptr;
  rc = get_state(st, &d);
  if (rc != MOE_ROUTE_OK) return rc;
  RouteArgs a = {};
  a.logits = logits;
  a.bias = bias;
  a.stab = d->stab;
  a.etab = d->etab;
  a.packed = packed;
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.ids = topk_ids;
  a.err = d->err;
  a.T = T;
  a.k = k;
  a.Kg = topk_group;
  a.off = local_offset;
  a.cnt = local_count;
  a.NE = bins(E, k, local_count);
  a.scale = scale;
  a.qx = x;
  a.qcodes = x_q;
  a.qscales = x_scales;
  a.qH = H;
  a.eps_f32 = (g_path == 3 || g_path == 4) ? -1.0f : d->eps_f32;
  const int dt = logits_dtype == MOE_ROUTE_BF16 ? DT_BF16 : DT_F32;
  return launch_route_decode(a, dt, st) == cudaSuccess ? MOE_ROUTE_OK : MOE_ROUTE_E_CUDA;
}

int moe_router_gemm_route(const uint16_t* hidden, const uint16_t* w_router, const float* bias,
                          int T, int H, int E, int k, int n_group, int topk_group, float scale,
                          int local_offset, int local_count, float* logits_out, int32_t* packed,
                          int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* topk_ids,
                          struct CUstream_st* stream) {
  int rc = check_route_args(T, E, k, n_group, topk_group, local_offset, local_count);
  if (rc != MOE_ROUTE_OK) return rc;
  if (T < 1 || H <= 0) return MOE_ROUTE_E_INVALID_ARG;
  if (!hidden || !w_router || !bias || !packed || !counts || !offsets || !perm)
    return MOE_ROUTE_E_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(hidden) % 16 != 0 || reinterpret_cast<uintptr_t>(w_router) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(bias) % 16 != 0 || reinterpret_cast<uintptr_t>(logits_out) % 16 != 0)
    return MOE_ROUTE_E_INVALID_ARG;
  if (T > 64 || H % 64 != 0) return MOE_ROUTE_E_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DevState* d = nullptr;
  rc = get_state(st, &d);
  if (rc != MOE_ROUTE_OK) return rc;
  if ((H / 64) % router_gemm_cluster() != 0) return MOE_ROUTE_E_UNSUPPORTED;
  if (launch_router_gemm(hidden, w_router, logits_out, d->gscores, d->etab, T, H, E, d->err, st) !=
      cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  RouteArgs a = {};
  a.logits = d->gscores;
  a.bias = bias;
  a.stab = d->stab;
  a.etab = d->etab;
  a.packed = packed;
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.ids = topk_ids;
  a.err = d->err;
  a.T = T;
  a.k = k;
  a.Kg = topk_group;
  a.off = local_offset;
  a.cnt = local_count;
  a.NE = bins(E, k, local_count);
  a.scale = scale;
  // the routing's cluster launches while the contraction's 7 clusters of up to 16 CTAs
  // hold their SMs; a cluster of more than 8 CTAs found no room beside them and started
  // only as they left (about 2 us later at 32 rows)
  return launch_route_decode(a, DT_SCORE, st, 8) == cudaSuccess ? MOE_ROUTE_OK : MOE_ROUTE_E_CUDA;
}

int moe_route_index(const int32_t* packed, int T, int k, int NE, int32_t* counts,
                    int32_t* offsets, int32_t* perm, struct CUstream_st* stream) {
  if (T < 0 || k < 1 || NE < 1) return MOE_ROUTE_E_INVALID_ARG;
  if (static_cast<long long>(T) * k >= (1ll << 31)) return MOE_ROUTE_E_INVALID_ARG;
  if (!counts || !offsets || (T > 0 && (!packed || !perm))) return MOE_ROUTE_E_INVALID_ARG;
  if (k > kMaxK || NE > kMaxBins) return MOE_ROUTE_E_UNSUPPORTED;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DevState* d = nullptr;
  const int rc = get_state(st, &d);
  if (rc != MOE_ROUTE_OK) return rc;
  RouteArgs a = {};
  a.logits = packed;
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.err = d->err;
  a.T = T;
  a.k = k;
  a.Kg = 0;
  a.NE = NE;
  cudaError_t ce;
  if (T <= 64) {
    ce = launch_route_decode(a, DT_PACKED, st);
  } else {
    // k = 16 (the Kimi-K3 instance): the approximate-score kernel's ranking, placement
    // and barriers, reading the packed ids instead of routing (path 3 forces the other)
    int grid_fast = d->nsm * d->fast_blocks_per_sm;
    if (grid_fast > d->pw.grid_max) grid_fast = d->pw.grid_max;
    if (grid_fast > (T + 15) / 16) grid_fast = (T + 15) / 16;
    if (k == 16 && NE <= kFastBins && NE % 4 == 0 && reinterpret_cast<uintptr_t>(packed) % 16 == 0 &&
        g_path != 3 && grid_fast >= 1 && prefill_fast_fits(T, grid_fast)) {
      ce = launch_route_prefill_fast(a, d->pw, grid_fast, st);
    } else {
      int grid = (T + 15) / 16;
      if (grid > d->pw.grid_max) grid = d->pw.grid_max;
      ce = launch_route_prefill(a, DT_PACKED, d->pw, grid, st);
    }
  }
  return ce == cudaSuccess ? MOE_ROUTE_OK : MOE_ROUTE_E_CUDA;
}

int moe_route_dispatch_counts(const int32_t* offsets, int E, int num_ranks, int32_t* send_counts,
                              int32_t* send_offsets, struct CUstream_st* stream) {
  if (!offsets || E < 1 || num_ranks < 1 || E % num_ranks != 0) return MOE_ROUTE_E_INVALID_ARG;
  if (!send_counts && !send_offsets) return MOE_ROUTE_OK;
  return launch_dispatch_counts(offsets, E, num_ranks, send_counts, send_offsets,
                                reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_ROUTE_OK
             : MOE_ROUTE_E_CUDA;
}

int moe_route_alltoall_layout(const int32_t* matrix, int num_ranks, int rank, int32_t* send_displs,
                              int32_t* recv_counts, int32_t* recv_displs,
                              struct CUstream_st* stream) {
  if (!matrix || num_ranks < 1 || rank < 0 || rank >= num_ranks) return MOE_ROUTE_E_INVALID_ARG;
  if (num_ranks > 1024) return MOE_ROUTE_E_UNSUPPORTED;
  return launch_alltoall_layout(matrix, num_ranks, rank, send_displs, recv_counts, recv_displs,
                                reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_ROUTE_OK
             : MOE_ROUTE_E_CUDA;
}

int moe_route_padded_capacity(int T, int k, int NE, int tile) {
  if (T < 0 || k < 1 || NE < 1 || tile < 1) return MOE_ROUTE_E_INVALID_ARG;
  const long long cap = static_cast<long long>(T) * k + static_cast<long long>(NE) * (tile - 1);
  return cap < (1ll << 31) ? static_cast<int>(cap) : MOE_ROUTE_E_INVALID_ARG;
}

int moe_route_layout(const int32_t* counts, const int32_t* offsets, const int32_t* perm, int T,
                     int k, int NE, int tile, int32_t* inv_perm, int32_t* padded_offsets,
                     int32_t* padded_rows, int32_t* m_indices, int capacity,
                     struct CUstream_st* stream) {
  const int need = moe_route_padded_capacity(T, k, NE, tile);
  if (need < 0) return MOE_ROUTE_E_INVALID_ARG;
  if (NE > kMaxBins) return MOE_ROUTE_E_UNSUPPORTED;
  const int n = T * k;
  if (!counts || !offsets || (n > 0 && !perm)) return MOE_ROUTE_E_INVALID_ARG;
  const bool padded = padded_rows || m_indices;
  if (padded && capacity < need) return MOE_ROUTE_E_INVALID_ARG;
  if (!inv_perm && !padded_offsets && !padded) return MOE_ROUTE_OK;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DevState* d = nullptr;
  const int rc = get_state(st, &d);
  if (rc != MOE_ROUTE_OK) return rc;
  LayoutArgs g = {};
  g.counts = counts;
  g.offsets = offsets;
  g.perm = perm;
  g.n = n;
  g.NE = NE;
  g.tile = tile;
  g.capacity = padded ? capacity : 0;
  g.inv_perm = inv_perm;
  g.padded_offsets = padded_offsets;
  g.padded_rows = padded_rows;
  g.m_indices = m_indices;
  return launch_route_layout(g, d->nsm, st) == cudaSuccess ? MOE_ROUTE_OK : MOE_ROUTE_E_CUDA;
}

int moe_route_device_status(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ROUTE_E_CUDA;
  DevState& d = g_dev[dev];
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (!d.ready) return MOE_ROUTE_OK;
  int host = 0;
  if (cudaMemcpy(&host, d.err, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  if (host != 0) {
    // clear the status word and the grid barrier state left by the failed call
    if (cudaMemset(d.err, 0, sizeof(int)) != cudaSuccess) return MOE_ROUTE_E_CUDA;
    if (cudaMemset(d.pw.bar, 0, 2 * sizeof(unsigned)) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  }
  return host;
}

int moe_route_sigmoid(const void* x, int dtype, float* s, int n, struct CUstream_st* stream) {
  if (n < 0 || (n > 0 && (!x || !s))) return MOE_ROUTE_E_INVALID_ARG;
  if (dtype != MOE_ROUTE_F32 && dtype != MOE_ROUTE_BF16) return MOE_ROUTE_E_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  DevState* d = nullptr;
  const int rc = get_state(st, &d);
  if (rc != MOE_ROUTE_OK) return rc;
  return launch_sigmoid(x, dtype == MOE_ROUTE_BF16 ? DT_BF16 : DT_F32, d->stab, d->etab, s, n, st) ==
                 cudaSuccess
             ? MOE_ROUTE_OK
             : MOE_ROUTE_E_CUDA;
}

int moe_route_set_path(int path) {
  if (path < 0 || path > 4) return MOE_ROUTE_E_INVALID_ARG;
  const int prev = g_path;
  g_path = path;
  return prev;
}

int moe_route_arm_barrier_timeout(int cta, int wait_us) {
  if (cta < -1 || (cta >= 0 && (wait_us < 1 || wait_us > 2000000))) return MOE_ROUTE_E_INVALID_ARG;
  g_skip_wait_ns.store(static_cast<unsigned long long>(cta >= 0 ? wait_us : 0) * 1000ull);
  g_skip_cta.store(cta);
  return MOE_ROUTE_OK;
}

int moe_route_decode_ctas(int T) {
  if (T < 0 || T > 64) return MOE_ROUTE_E_INVALID_ARG;
  DevState* d = nullptr;
  const int rc = get_state(nullptr, &d);
  if (rc != MOE_ROUTE_OK) return rc;
  return decode_ctas(T);
}

int moe_route_empty(int ctas, struct CUstream_st* stream) {
  if (ctas < 1 || ctas > 16) return MOE_ROUTE_E_INVALID_ARG;
  DevState* d = nullptr;  // the kernel attributes (clusters above 8) are set with the state
  const int rc = get_state(reinterpret_cast<cudaStream_t>(stream), &d);
  if (rc != MOE_ROUTE_OK) return rc;
  return launch_empty(ctas, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess ? MOE_ROUTE_OK
                                                                                     : MOE_ROUTE_E_CUDA;
}

const char* moe_route_strerror(int status) {
  switch (status) {
    case MOE_ROUTE_OK: return "ok";
    case MOE_ROUTE_E_INVALID_ARG: return "invalid argument";
    case MOE_ROUTE_E_UNSUPPORTED: return "shape not supported by the kernels";
    case MOE_ROUTE_E_CUDA: return "CUDA runtime error";
    case MOE_ROUTE_E_WORKSPACE: return "library state missing during stream capture";
    case MOE_ROUTE_E_DEVICE_TIMEOUT: return "a bounded device-side wait ran out";
    case MOE_ROUTE_E_BAD_ID: return "a packed id is not below the number of bins or repeats in a row";
    default: return "unknown status";
  }
}

}  // extern "C"
