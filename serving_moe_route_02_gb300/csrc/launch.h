// launch.h -- host-side launchers of the routing kernels (internal to the library).
#pragma once
#include <cstdint>
#include <cuda_runtime.h>

#include "route_row.cuh"

namespace moe {

// Per-device workspace of the persistent kernel (device memory, zeroed at creation).
struct PrefillWS {
  int* hist;       // [kMaxBins][grid_max] per-CTA histograms, expert-major
  int* prefix;     // [kMaxBins][grid_max] exclusive prefix over CTAs
  int* counts;     // [kMaxBins]
  unsigned* bar;   // [2]: arrival counter, exit counter
  int grid_max;
};

constexpr int kSigTablePad = (kSigTable + 3) / 4 * 4;  // table length rounded to 16 bytes

// Arguments of the expert-GEMM layout kernel (route_layout.cu).
struct LayoutArgs {
  const int32_t* counts;     // [NE]
  const int32_t* offsets;    // [NE + 1]
  const int32_t* perm;       // [n]
  int n, NE, tile, capacity;
  int32_t* inv_perm;         // [n] or nullptr
  int32_t* padded_offsets;   // [NE + 1] or nullptr
  int32_t* padded_rows;      // [capacity] or nullptr
  int32_t* m_indices;        // [capacity] or nullptr
};

cudaError_t launch_route_layout(const LayoutArgs& g, int nsm, cudaStream_t st);
cudaError_t launch_dispatch_counts(const int32_t* offsets, int E, int R, int32_t* send_counts,
                                   int32_t* send_offsets, cudaStream_t st);
cudaError_t launch_alltoall_layout(const int32_t* matrix, int R, int me, int32_t* send_displs,
                                   int32_t* recv_counts, int32_t* recv_displs, cudaStream_t st);
cudaError_t launch_sigmoid_table(float* tab, float2* etab, cudaStream_t st);
cudaError_t launch_sigmoid(const void* x, int dtype, const float* tab, const float2* etab, float* s,
                           int n, cudaStream_t st);
cudaError_t setup_decode_kernels();
// max_ctas > 0 caps the cluster below the default (16 where the GPU schedules it, else 8)
cudaError_t launch_route_decode(const RouteArgs& a, int dtype, cudaStream_t st, int max_ctas = 0);
int decode_ctas(int T);  // CTAs (one cluster) of a decode launch of T <= 64 rows
int decode_ctas(int T, int max_ctas);  // the same with at most max_ctas CTAs
cudaError_t launch_empty(int ctas, cudaStream_t st);
cudaError_t setup_router_gemm();
int router_gemm_cluster();
cudaError_t launch_router_gemm(const uint16_t* hidden, const uint16_t* w, float* logits,
                               float* scores, const float2* etab, int T, int H, int E, int* err,
                               cudaStream_t st);
cudaError_t setup_prefill_kernels(int* blocks_per_sm);
// True when the persistent kernel can take T rows on `grid` CTAs (T >= 0, grid >= 1).
bool prefill_fits(int T, int grid);
// The persistent kernel for bf16 logits with k = 16 and topk_group = 4, built on
// approximate scores (route_prefill_fast.cu).  prefill_fast_fits: T rows on `grid` CTAs
// fit its per-warp entry room.
cudaError_t setup_prefill_fast(int* blocks_per_sm);
// Bins it serves: 896 global ids, or at most 896 rank-local ids plus 16 for the other
// ranks' slots, rounded up to a multiple of 4.  Index mode (topk_group = 0 in the
// arguments) takes k = 16 and at most this many bins.
constexpr int kFastBins = kE + 16;
bool prefill_fast_fits(int T, int grid);
cudaError_t launch_route_prefill_fast(const RouteArgs& a, const PrefillWS& ws, int grid,
                                      cudaStream_t st);
// Writes the bits of E_half (route_pair.cuh) to *out, which must hold 0.
cudaError_t launch_approx_err(unsigned* out, cudaStream_t st);
// the float32 counterpart (route_row's approximate float32 scores), over all 2^32 inputs
cudaError_t launch_approx_err_f32(const float2* etab, unsigned* out, cudaStream_t st);
// eps_f32 from the measured maximum: the float-rounded differences' slack added
float approx_bound_f32(unsigned measured_bits);
// The argument checks of moe_route (status code; MOE_ROUTE_OK when the call is valid).
int route_args_status(int T, int E, int k, int n_group, int topk_group, int off, int cnt);
cudaError_t launch_route_prefill(const RouteArgs& a, int dtype, const PrefillWS& ws, int grid,
                                 cudaStream_t st);

}  // namespace moe
