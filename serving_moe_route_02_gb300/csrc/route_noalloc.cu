// route_noalloc.cu -- moe_route_noalloc: the routing call for callers that cannot
// allocate device memory.
//
// moe_route keeps its per-CTA histograms, barrier words and score tables in a
// workspace it obtains with cudaMalloc on first use.  Some callers cannot allow that:
// a serving engine that reserves all free HBM for weights and KV cache at start-up and
// forbids later allocations, code that runs under a strict caching allocator or
// memory pool, or a plugin that may only touch the buffers it is handed.  This file
// gives them the same persistent routing kernel with its scratch in a fixed,
// file-scope device array instead.  Every GPU that loads the library holds the array
// (about 1.4 MB) until the process exits.
#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/moe_route.h"
#include "launch.h"

namespace moe {
namespace {

// Largest grid the static scratch covers; a device with more resident CTAs simply
// runs this many.
constexpr int kNoallocMaxCtas = 160;
constexpr size_t kTabBytes = size_t(kSigTablePad) * 4;
constexpr size_t kExpBytes = size_t(2 * kExpTable) * 4;
constexpr size_t kHistBytes = size_t(kMaxBins) * kNoallocMaxCtas * 4;
constexpr size_t o_tab = 0;
constexpr size_t o_exp = o_tab + kTabBytes;
constexpr size_t o_hist = (o_exp + kExpBytes + 255) / 256 * 256;
constexpr size_t o_prefix = o_hist + kHistBytes;
constexpr size_t o_counts = o_prefix + kHistBytes;
constexpr size_t o_bar = o_counts + size_t(kMaxBins) * 4;   // 2 words
constexpr size_t o_err = o_bar + 8;                          // 1 word
constexpr size_t o_probe = o_err + 4;                        // 2 words (set-up only)
constexpr size_t kNoallocBytes = (o_probe + 8 + 255) / 256 * 256;

// The scratch.  In host code this name is only a stand-in for the device object; the
// device address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocBytes];

struct NoallocDev {
  std::atomic<bool> ready{false};  // set (release) once the fields below are in place
  unsigned char* base = nullptr;   // device address of g_noalloc_scratch on this device
  int grid_max = 0;
  int grid_fast = 0;               // CTAs of the approximate-score persistent kernel
  float eps_half = 0.0f;           // its measured approximation bound
  float eps_f32 = -1.0f;           // route_row's float32 bound
};
NoallocDev g_na[64];
std::mutex g_na_mu;

// Once per device, with that device current: look up the array's device address,
// write the score tables into it and zero the barrier words.  Allocates nothing.
int noalloc_setup(int dev, NoallocDev& d) {
  void* p = nullptr;
  if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
    return MOE_ROUTE_E_CUDA;
  int nsm = 0, bpsm = 0, fbpsm = 0;
  if (cudaDeviceGetAttribute(&nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  if (setup_decode_kernels() != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (setup_prefill_kernels(&bpsm) != cudaSuccess || bpsm < 1) return MOE_ROUTE_E_CUDA;
  if (setup_prefill_fast(&fbpsm) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  unsigned char* base = static_cast<unsigned char*>(p);
  if (launch_sigmoid_table(reinterpret_cast<float*>(base + o_tab),
                           reinterpret_cast<float2*>(base + o_exp), nullptr) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  if (cudaMemset(base + o_bar, 0, o_probe + 8 - o_bar) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (launch_approx_err(reinterpret_cast<unsigned*>(base + o_probe), nullptr) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  if (launch_approx_err_f32(reinterpret_cast<const float2*>(base + o_exp),
                            reinterpret_cast<unsigned*>(base + o_probe + 4), nullptr) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ROUTE_E_CUDA;
  unsigned bits = 0;
  if (cudaMemcpy(&bits, base + o_probe, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  std::memcpy(&d.eps_half, &bits, sizeof(bits));
  if (cudaMemcpy(&bits, base + o_probe + 4, sizeof(bits), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  d.eps_f32 = approx_bound_f32(bits);
  d.base = base;
  d.grid_max = nsm * bpsm < kNoallocMaxCtas ? nsm * bpsm : kNoallocMaxCtas;
  d.grid_fast = nsm * fbpsm < kNoallocMaxCtas ? nsm * fbpsm : kNoallocMaxCtas;
  d.ready.store(true, std::memory_order_release);
  return MOE_ROUTE_OK;
}

}  // namespace
}  // namespace moe

extern "C" int moe_route_noalloc(const void* logits, int logits_dtype, const float* bias, int T,
                                 int E, int k, int n_group, int topk_group, float scale,
                                 int local_offset, int local_count, int32_t* packed,
                                 int32_t* counts, int32_t* offsets, int32_t* perm,
                                 int32_t* topk_ids, int32_t* status, struct CUstream_st* stream) {
  using namespace moe;
  // the same argument rules as moe_route
  if (T < 0 || E <= 0 || k <= 0 || n_group <= 0) return MOE_ROUTE_E_INVALID_ARG;
  if (E % n_group != 0 || E / n_group < 2) return MOE_ROUTE_E_INVALID_ARG;
  if (topk_group < 1 || topk_group > n_group) return MOE_ROUTE_E_INVALID_ARG;
  if (k > topk_group * (E / n_group)) return MOE_ROUTE_E_INVALID_ARG;
  if (local_count < 0 || local_offset < 0 || local_offset + local_count > E)
    return MOE_ROUTE_E_INVALID_ARG;
  if (E > 32767 || (local_count > 0 && local_count + k > 32767)) return MOE_ROUTE_E_INVALID_ARG;
  if (static_cast<long long>(T) * k >= (1ll << 31)) return MOE_ROUTE_E_INVALID_ARG;
  if (logits_dtype != MOE_ROUTE_F32 && logits_dtype != MOE_ROUTE_BF16) return MOE_ROUTE_E_INVALID_ARG;
  if (!bias || !counts || !offsets) return MOE_ROUTE_E_INVALID_ARG;
  if (T > 0 && (!logits || !packed || !perm)) return MOE_ROUTE_E_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(logits) % 16 != 0 || reinterpret_cast<uintptr_t>(bias) % 16 != 0)
    return MOE_ROUTE_E_INVALID_ARG;
  if (E != kE || n_group != kG || k > kMaxK) return MOE_ROUTE_E_UNSUPPORTED;
  const int NE = local_count > 0 ? (local_count + k + 3) / 4 * 4 : E;
  if (NE > kMaxBins) return MOE_ROUTE_E_UNSUPPORTED;  // beyond the static scratch

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return MOE_ROUTE_E_CUDA;
  NoallocDev& d = g_na[dev];
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (!d.ready.load(std::memory_order_acquire)) {
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (st != nullptr && cudaStreamIsCapturing(st, &cs) == cudaSuccess &&
        cs != cudaStreamCaptureStatusNone)
      return MOE_ROUTE_E_WORKSPACE;  // the first call on a device must not be captured
    std::lock_guard<std::mutex> lk(g_na_mu);
    if (!d.ready.load(std::memory_order_relaxed)) {
      const int rc = noalloc_setup(dev, d);
      if (rc != MOE_ROUTE_OK) return rc;
    }
  }

  RouteArgs a = {};
  a.logits = logits;
  a.bias = bias;
  a.stab = reinterpret_cast<const float*>(d.base + o_tab);
  a.etab = reinterpret_cast<const float2*>(d.base + o_exp);
  a.packed = packed;
  a.counts = counts;
  a.offsets = offsets;
  a.perm = perm;
  a.ids = topk_ids;
  a.err = status ? status : reinterpret_cast<int*>(d.base + o_err);
  a.T = T;
  a.k = k;
  a.Kg = topk_group;
  a.off = local_offset;
  a.cnt = local_count;
  a.NE = NE;
  a.scale = scale;
  a.eps_half = d.eps_half;
  a.eps_f32 = d.eps_f32;
  const int dt = logits_dtype == MOE_ROUTE_BF16 ? DT_BF16 : DT_F32;

  // words that must start at zero: the caller's status word and the grid barrier
  if (status && cudaMemsetAsync(status, 0, sizeof(int32_t), st) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  if (T == 0) return launch_route_decode(a, dt, st) == cudaSuccess ? MOE_ROUTE_OK : MOE_ROUTE_E_CUDA;
  if (cudaMemsetAsync(d.base + o_bar, 0, 8, st) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  PrefillWS ws = {};
  ws.hist = reinterpret_cast<int*>(d.base + o_hist);
  ws.prefix = reinterpret_cast<int*>(d.base + o_prefix);
  ws.counts = reinterpret_cast<int*>(d.base + o_counts);
  ws.bar = reinterpret_cast<unsigned*>(d.base + o_bar);
  ws.grid_max = kNoallocMaxCtas;
  // the same kernel choice as moe_route for T > 64 rows
  int grid_fast = d.grid_fast < (T + 15) / 16 ? d.grid_fast : (T + 15) / 16;
  if (dt == DT_BF16 && k == 16 && topk_group == 4 && grid_fast >= 1 && prefill_fast_fits(T, grid_fast))
    return launch_route_prefill_fast(a, ws, grid_fast, st) == cudaSuccess ? MOE_ROUTE_OK : MOE_ROUTE_E_CUDA;
  int grid = (T + 15) / 16;
  if (grid > d.grid_max) grid = d.grid_max;
  if (!prefill_fits(T, grid)) return MOE_ROUTE_E_UNSUPPORTED;
  return launch_route_prefill(a, dt, ws, grid, st) == cudaSuccess ? MOE_ROUTE_OK : MOE_ROUTE_E_CUDA;
}
