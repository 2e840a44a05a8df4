// route_host.cu -- moe_route_host: routing of a logit matrix held in host memory, with
// the results written back to host memory.  Host code only: the routing itself is
// moe_route on library-owned device staging.
//
// Two staging slots per device alternate between calls.  A call copies its logits
// host -> device on the library's copy stream, as soon as the slot's previous use (two
// calls back) has finished, so that call i + 1's input transfer overlaps call i's
// routing and its device -> host result copies on the caller's stream.
#include <cuda_runtime.h>

#include <cstdint>
#include <mutex>

#include "../../include/moe_route.h"
#include "launch.h"

namespace {

struct Slot {
  char* dev = nullptr;            // [logits | packed | counts | offsets | perm | ids]
  size_t cap = 0;
  cudaEvent_t loaded = nullptr;   // logits copied in (copy stream)
  cudaEvent_t free_ev = nullptr;  // routing and result copies done (caller's stream)
  bool used = false;
};

struct HostState {
  bool ready = false;
  cudaStream_t copy = nullptr;
  Slot slot[2];
  unsigned next = 0;
};

constexpr int kMaxDevices = 64;
HostState g_host[kMaxDevices];
std::mutex g_host_mu;

size_t align256(size_t n) { return (n + 255) & ~size_t(255); }

int init_host_state(HostState& h) {
  if (cudaStreamCreateWithFlags(&h.copy, cudaStreamNonBlocking) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  for (Slot& s : h.slot) {
    if (cudaEventCreateWithFlags(&s.loaded, cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&s.free_ev, cudaEventDisableTiming) != cudaSuccess)
      return MOE_ROUTE_E_CUDA;
  }
  h.ready = true;
  return MOE_ROUTE_OK;
}

bool capturing(cudaStream_t st) {
  cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return true;
  return cs != cudaStreamCaptureStatusNone;
}

}  // namespace

extern "C" {

int moe_route_host(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
                   int n_group, int topk_group, float scale, int local_offset, int local_count,
                   int32_t* packed, int32_t* counts, int32_t* offsets, int32_t* perm,
                   int32_t* topk_ids, struct CUstream_st* stream) {
  int rc = moe::route_args_status(T, E, k, n_group, topk_group, local_offset, local_count);
  if (rc != MOE_ROUTE_OK) return rc;
  if (logits_dtype != MOE_ROUTE_F32 && logits_dtype != MOE_ROUTE_BF16) return MOE_ROUTE_E_INVALID_ARG;
  if (!bias || !counts || !offsets) return MOE_ROUTE_E_INVALID_ARG;
  if (T > 0 && (!logits || !packed || !perm)) return MOE_ROUTE_E_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(bias) % 16 != 0) return MOE_ROUTE_E_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (capturing(st)) return MOE_ROUTE_E_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ROUTE_E_CUDA;
  // the device state (tables, workspace) before any copy is enqueued
  rc = moe_route_reserve();
  if (rc != MOE_ROUTE_OK) return rc;

  std::lock_guard<std::mutex> lk(g_host_mu);
  HostState& h = g_host[dev];
  if (!h.ready) {
    rc = init_host_state(h);
    if (rc != MOE_ROUTE_OK) return rc;
  }
  const int NE = moe_route_bins(E, k, local_count);
  const size_t tk = size_t(T) * size_t(k) * 4;
  const size_t b_log = size_t(T) * size_t(E) * (logits_dtype == MOE_ROUTE_BF16 ? 2 : 4);
  const size_t o_packed = align256(b_log);
  const size_t o_counts = o_packed + align256(tk);
  const size_t o_offsets = o_counts + align256(size_t(NE) * 4);
  const size_t o_perm = o_offsets + align256(size_t(NE + 1) * 4);
  const size_t o_ids = o_perm + align256(tk);
  const size_t need = o_ids + (topk_ids ? align256(tk) : 0);

  Slot& s = h.slot[h.next & 1u];
  if (s.cap < need) {
    // the slot's previous use must be over before its memory goes
    if (s.used && cudaEventSynchronize(s.free_ev) != cudaSuccess) return MOE_ROUTE_E_CUDA;
    if (s.dev) cudaFree(s.dev);
    s.dev = nullptr;
    s.cap = 0;
    s.used = false;
    const size_t cap = need + need / 4;
    if (cudaMalloc(&s.dev, cap) != cudaSuccess) return MOE_ROUTE_E_CUDA;
    s.cap = cap;
  }
  char* base = s.dev;

  // input: host -> staging on the copy stream, after the slot's previous use
  if (s.used && cudaStreamWaitEvent(h.copy, s.free_ev, 0) != cudaSuccess) return MOE_ROUTE_E_CUDA;
  if (b_log > 0 && cudaMemcpyAsync(base, logits, b_log, cudaMemcpyHostToDevice, h.copy) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  if (cudaEventRecord(s.loaded, h.copy) != cudaSuccess || cudaStreamWaitEvent(st, s.loaded, 0) != cudaSuccess)
    return MOE_ROUTE_E_CUDA;
  h.next++;
  s.used = true;

  int32_t* d_packed = reinterpret_cast<int32_t*>(base + o_packed);
  int32_t* d_counts = reinterpret_cast<int32_t*>(base + o_counts);
  int32_t* d_offsets = reinterpret_cast<int32_t*>(base + o_offsets);
  int32_t* d_perm = reinterpret_cast<int32_t*>(base + o_perm);
  int32_t* d_ids = topk_ids ? reinterpret_cast<int32_t*>(base + o_ids) : nullptr;
  rc = moe_route(base, logits_dtype, bias, T, E, k, n_group, topk_group, scale, local_offset,
                 local_count, d_packed, d_counts, d_offsets, d_perm, d_ids, stream);
  if (rc == MOE_ROUTE_OK) {
    // results: staging -> host on the caller's stream
    bool ok = true;
    if (tk > 0) {
      ok = ok && cudaMemcpyAsync(packed, d_packed, tk, cudaMemcpyDeviceToHost, st) == cudaSuccess;
      ok = ok && cudaMemcpyAsync(perm, d_perm, tk, cudaMemcpyDeviceToHost, st) == cudaSuccess;
      if (topk_ids)
        ok = ok && cudaMemcpyAsync(topk_ids, d_ids, tk, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    }
    ok = ok && cudaMemcpyAsync(counts, d_counts, size_t(NE) * 4, cudaMemcpyDeviceToHost, st) == cudaSuccess;
    ok = ok && cudaMemcpyAsync(offsets, d_offsets, size_t(NE + 1) * 4, cudaMemcpyDeviceToHost, st) ==
                   cudaSuccess;
    if (!ok) rc = MOE_ROUTE_E_CUDA;
  }
  // the slot is free once everything enqueued on the caller's stream so far is done
  if (cudaEventRecord(s.free_ev, st) != cudaSuccess && rc == MOE_ROUTE_OK) rc = MOE_ROUTE_E_CUDA;
  return rc;
}

int moe_route_host_release(void) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ROUTE_E_CUDA;
  std::lock_guard<std::mutex> lk(g_host_mu);
  HostState& h = g_host[dev];
  if (!h.ready) return MOE_ROUTE_OK;
  int rc = MOE_ROUTE_OK;
  for (Slot& s : h.slot) {
    if (s.used && cudaEventSynchronize(s.free_ev) != cudaSuccess) rc = MOE_ROUTE_E_CUDA;
    if (s.dev && cudaFree(s.dev) != cudaSuccess) rc = MOE_ROUTE_E_CUDA;
    s.dev = nullptr;
    s.cap = 0;
    s.used = false;
  }
  return rc;
}

}  // extern "C"
