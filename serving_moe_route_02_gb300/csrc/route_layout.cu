// route_layout.cu -- the layout of the routed entries that grouped expert GEMMs consume,
// built from the routing outputs (counts, offsets, perm):
//   inv_perm[perm[p]] = p                       inverse permutation (combine scatter)
//   padded_offsets[e + 1] = padded_offsets[e] + round_up(counts[e], tile)
//   padded row padded_offsets[e] + i (i < counts[e]): padded_rows = perm[offsets[e] + i],
//   m_indices = e; every other row below `capacity` holds -1 in both.
// One launch.  Every CTA scans the per-bin padded sizes itself (at most 1,056 bins), so
// no grid-wide synchronisation is needed.  The padded rows are cut into work items of
// one bin and at most 1,024 rows; a warp takes an item, finds its bin once (binary
// search over the items' prefix in shared memory) and copies the bin's perm entries with
// coalesced loads and stores.  Rows past the padded total are a coalesced -1 fill, and
// the inverse permutation a grid-stride loop over perm (coalesced reads, scattered
// writes).  Bound by HBM: about 4 B read and 12 B written per entry plus the padding.
#include "launch.h"

namespace moe {

constexpr int kLayoutThreads = 256;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kPieceShift = 10;  // rows per work item: 1,024

__global__ void __launch_bounds__(kLayoutThreads) k_route_layout(LayoutArgs g) {
  __shared__ int cnt_s[kMaxBins];
  __shared__ int off_s[kMaxBins];
  __shared__ int poff_s[kMaxBins + 1];  // padded offsets
  __shared__ int qoff_s[kMaxBins + 1];  // work-item offsets
  __shared__ int tmp_s[2 * kLayoutWarps];
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int NE = g.NE;

  // ---- per-bin padded size and item count, one exclusive scan of both (two barriers)
  const int per = (NE + kLayoutThreads - 1) / kLayoutThreads;
  const int lo = min(NE, tid * per), hi = min(NE, lo + per);
  int sp = 0, sq = 0;
  for (int e0 = lo; e0 < hi; e0 += 8) {
    int c[8], o[8];
#pragma unroll
    for (int u = 0; u < 8; ++u) {  // all loads of the group in flight
      c[u] = (e0 + u < hi) ? g.counts[e0 + u] : 0;
      o[u] = (e0 + u < hi) ? g.offsets[e0 + u] : 0;
    }
#pragma unroll
    for (int u = 0; u < 8; ++u) {
      const int e = e0 + u;
      if (e < hi) {
        const int psz = (c[u] + g.tile - 1) / g.tile * g.tile;
        cnt_s[e] = c[u];
        off_s[e] = o[u];
        poff_s[e] = psz;  // sizes for now, offsets after the scan
        qoff_s[e] = (psz + (1 << kPieceShift) - 1) >> kPieceShift;
        sp += psz;
        sq += qoff_s[e];
      }
    }
  }
  int ip = sp, iq = sq;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, ip, o);
    const int v = __shfl_up_sync(0xffffffffu, iq, o);
    if (lane >= o) {
      ip += u;
      iq += v;
    }
  }
  if (lane == 31) {
    tmp_s[wid] = ip;
    tmp_s[kLayoutWarps + wid] = iq;
  }
  __syncthreads();
  int rp = ip - sp, rq = iq - sq;
  for (int i = 0; i < wid; ++i) {
    rp += tmp_s[i];
    rq += tmp_s[kLayoutWarps + i];
  }
  for (int e = lo; e < hi; ++e) {
    const int a = poff_s[e], b = qoff_s[e];
    poff_s[e] = rp;
    qoff_s[e] = rq;
    rp += a;
    rq += b;
  }
  if (hi == NE && lo < hi) {
    poff_s[NE] = rp;
    qoff_s[NE] = rq;
  }
  __syncthreads();
  if (blockIdx.x == 0 && g.padded_offsets)
    for (int e = tid; e <= NE; e += kLayoutThreads) g.padded_offsets[e] = poff_s[e];

  const int total = poff_s[NE];
  const int nitems = qoff_s[NE];
  const int gwarp = blockIdx.x * kLayoutWarps + wid;
  const int nwarps = gridDim.x * kLayoutWarps;

  // ---- padded rows and m_indices: one bin and up to 1,024 rows per work item
  if (g.padded_rows || g.m_indices) {
    for (int it = gwarp; it < nitems; it += nwarps) {
      // largest e with qoff[e] <= it: item `it` belongs to bin e
      int a = 0, b = NE - 1;
      while (a < b) {
        const int mid = (a + b + 1) >> 1;
        if (qoff_s[mid] <= it) a = mid;
        else b = mid - 1;
      }
      const int e = a;
      const int i0 = (it - qoff_s[e]) << kPieceShift;
      const int i1 = min(i0 + (1 << kPieceShift), poff_s[e + 1] - poff_s[e]);
      const int c = cnt_s[e], src0 = off_s[e], dst0 = poff_s[e];
      // the item's 1,024 rows: 32 per lane, every load in flight at once
      constexpr int kRowsPerLane = (1 << kPieceShift) / 32;
      int row[kRowsPerLane];
#pragma unroll
      for (int u = 0; u < kRowsPerLane; ++u) {
        const int ii = i0 + lane + u * 32;
        row[u] = (ii < c && ii < i1) ? g.perm[src0 + ii] : -1;
      }
#pragma unroll
      for (int u = 0; u < kRowsPerLane; ++u) {
        const int ii = i0 + lane + u * 32;
        if (ii < i1) {
          if (g.padded_rows) g.padded_rows[dst0 + ii] = row[u];
          if (g.m_indices) g.m_indices[dst0 + ii] = (ii < c) ? e : -1;
        }
      }
    }
    // rows past the padded total
    const long long stride = (long long)gridDim.x * kLayoutThreads;
    for (long long r = total + (long long)blockIdx.x * kLayoutThreads + tid; r < g.capacity; r += stride) {
      if (g.padded_rows) g.padded_rows[r] = -1;
      if (g.m_indices) g.m_indices[r] = -1;
    }
  }

  // ---- inverse permutation, eight entries per thread in flight
  if (g.inv_perm) {
    const long long stride = (long long)gridDim.x * kLayoutThreads;
    for (long long p0 = (long long)blockIdx.x * kLayoutThreads + tid; p0 < g.n; p0 += 8 * stride) {
      int x[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const long long p = p0 + u * stride;
        x[u] = (p < g.n) ? g.perm[p] : -1;
      }
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (x[u] >= 0) g.inv_perm[x[u]] = int(p0 + u * stride);
    }
  }
}

cudaError_t launch_route_layout(const LayoutArgs& g, int nsm, cudaStream_t st) {
  // two CTAs per SM at most: each CTA repeats the per-bin scan
  const long long work = g.capacity > g.n ? g.capacity : g.n;
  long long blocks = (work + 16LL * kLayoutThreads - 1) / (16LL * kLayoutThreads);
  if (blocks > 2LL * nsm) blocks = 2LL * nsm;
  if (blocks < 1) blocks = 1;
  k_route_layout<<<int(blocks), kLayoutThreads, 0, st>>>(g);
  return cudaGetLastError();
}

}  // namespace moe
