// route_dispatch.cu -- layouts for expert-parallel dispatch and token-sharded routing.
//
// k_dispatch_counts: with global expert ids, R ranks owning contiguous ranges of E / R
//   experts, the entries each rank must receive are the perm segment between the expert
//   offsets at the range boundaries (perm is ordered by expert, then token, then slot),
//   so send_offsets[d] = offsets[d E / R] and send_counts[d] = its difference.
// k_alltoall_layout: from the gathered counts matrix [R][R] (row = source, column =
//   destination), rank `me`'s send displacements (scan of its row), receive counts (its
//   column) and receive displacements (scan of the column).
// Both are one small block: R <= 1,024.
#include "launch.h"

namespace moe {

__global__ void k_dispatch_counts(const int32_t* __restrict__ offsets, int E, int R,
                                  int32_t* send_counts, int32_t* send_offsets) {
  const int per = E / R;
  for (int d = threadIdx.x; d <= R; d += blockDim.x) {
    const int lo = offsets[d * per];
    if (send_offsets) send_offsets[d] = lo;
    if (d < R && send_counts) send_counts[d] = offsets[(d + 1) * per] - lo;
  }
}

// exclusive scan of up to 1,024 values held one per thread (blockDim.x = 1024)
__device__ __forceinline__ int block_excl_1024(int v, int* tmp, int& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) tmp[wid] = incl;
  __syncthreads();
  int base = 0;
  total = 0;
  for (int i = 0; i < 32; ++i) {
    const int t = tmp[i];
    if (i < wid) base += t;
    total += t;
  }
  __syncthreads();
  return base + incl - v;
}

__global__ void __launch_bounds__(1024) k_alltoall_layout(const int32_t* __restrict__ matrix, int R,
                                                          int me, int32_t* send_displs,
                                                          int32_t* recv_counts,
                                                          int32_t* recv_displs) {
  __shared__ int tmp[32];
  const int i = threadIdx.x;
  const int s = (i < R) ? matrix[size_t(me) * R + i] : 0;  // sent to rank i
  const int r = (i < R) ? matrix[size_t(i) * R + me] : 0;  // received from rank i
  int total = 0;
  const int sd = block_excl_1024(s, tmp, total);
  if (i < R && send_displs) send_displs[i] = sd;
  if (i == 0 && send_displs) send_displs[R] = total;
  const int rd = block_excl_1024(r, tmp, total);
  if (i < R) {
    if (recv_counts) recv_counts[i] = r;
    if (recv_displs) recv_displs[i] = rd;
  }
  if (i == 0 && recv_displs) recv_displs[R] = total;
}

cudaError_t launch_dispatch_counts(const int32_t* offsets, int E, int R, int32_t* send_counts,
                                   int32_t* send_offsets, cudaStream_t st) {
  k_dispatch_counts<<<1, 256, 0, st>>>(offsets, E, R, send_counts, send_offsets);
  return cudaGetLastError();
}

cudaError_t launch_alltoall_layout(const int32_t* matrix, int R, int me, int32_t* send_displs,
                                   int32_t* recv_counts, int32_t* recv_displs, cudaStream_t st) {
  k_alltoall_layout<<<1, 1024, 0, st>>>(matrix, R, me, send_displs, recv_counts, recv_displs);
  return cudaGetLastError();
}

}  // namespace moe
