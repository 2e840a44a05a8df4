// persist.cuh -- pieces shared by the persistent (cooperative, one CTA per SM) routing
// kernels: the bounded grid barrier and its reset, a block-wide exclusive scan, and the
// column scan that turns per-CTA bin counts into prefixes over CTAs.
#pragma once
#include "launch.h"

namespace moe {

// Grid-wide barrier for a cooperative launch, bounded in time.  One arrival counter
// (bar[0]): CTA 0 adds 2^31 - (nblocks - 1), every other CTA adds 1, so the counter's
// top bit flips exactly when all have arrived; two barriers bring it back to 0 (mod
// 2^32).  Each CTA waits at most limit_ns.  Returns false if the wait ran out (the
// status word then holds a timeout), or at once, without arriving, in CTA `skip_cta`
// (a test of the timeout path: the other CTAs' waits run out).
__device__ __forceinline__ bool grid_barrier(unsigned* bar, unsigned nblocks, int* err, int* flag_s,
                                             uint64_t limit_ns = kWaitLimitNs, int skip_cta = -1) {
  __syncthreads();
  if (threadIdx.x == 0) {
    int ok = 1;
    if (int(blockIdx.x) == skip_cta) {
      ok = 0;
    } else {
      const unsigned add = (blockIdx.x == 0) ? 0x80000000u - (nblocks - 1u) : 1u;
      unsigned old;
      // release: the CTA's writes ordered before it by the block barrier above
      asm volatile("atom.release.gpu.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(bar), "r"(add) : "memory");
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        unsigned cur;
        asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(cur) : "l"(bar) : "memory");
        if ((cur ^ old) & 0x80000000u) break;
        if (globaltimer_ns() - t0 > limit_ns) {
          atomicExch(err, kErrTimeout);
          ok = 0;
          break;
        }
      }
    }
    *flag_s = ok;
  }
  __syncthreads();
  return *flag_s != 0;
}

// The same barrier in two halves, so that a CTA can do work of its own between arriving
// and waiting.  grid_arrive: every thread calls it once the writes to publish are done;
// thread 0 returns the counter's value before its arrival (the others 0), which
// grid_wait needs.  CTA `skip_cta` does not arrive (the timeout test).
__device__ __forceinline__ unsigned grid_arrive(unsigned* bar, unsigned nblocks, int skip_cta = -1) {
  __syncthreads();
  unsigned old = 0u;
  if (threadIdx.x == 0 && int(blockIdx.x) != skip_cta) {
    const unsigned add = (blockIdx.x == 0) ? 0x80000000u - (nblocks - 1u) : 1u;
    // release: the CTA's writes ordered before it by the block barrier above
    asm volatile("atom.release.gpu.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(bar), "r"(add) : "memory");
  }
  return old;
}
// grid_wait: every thread calls it; true once every CTA has arrived, false if the wait ran
// out (the status word then holds a timeout) or at once in CTA `skip_cta`.
__device__ __forceinline__ bool grid_wait(unsigned* bar, unsigned old, int* err, int* flag_s,
                                          uint64_t limit_ns = kWaitLimitNs, int skip_cta = -1) {
  if (threadIdx.x == 0) {
    int ok = 1;
    if (int(blockIdx.x) == skip_cta) {
      ok = 0;
    } else {
      const uint64_t t0 = globaltimer_ns();
      for (;;) {
        unsigned cur;
        asm volatile("ld.acquire.gpu.u32 %0, [%1];" : "=r"(cur) : "l"(bar) : "memory");
        if ((cur ^ old) & 0x80000000u) break;
        if (globaltimer_ns() - t0 > limit_ns) {
          atomicExch(err, kErrTimeout);
          ok = 0;
          break;
        }
      }
    }
    *flag_s = ok;
  }
  __syncthreads();
  return *flag_s != 0;
}

// Every CTA calls this once on its way out, on every path (also after a wait that ran
// out).  The last CTA to leave puts the barrier words back to zero, so a call that gave
// up mid-barrier does not leave the next call a half-counted barrier.  bar[1] counts
// the CTAs that have left.
__device__ __forceinline__ void grid_exit(unsigned* bar, unsigned nblocks) {
  __syncthreads();
  if (threadIdx.x == 0) {
    unsigned old;
    asm volatile("atom.acq_rel.gpu.add.u32 %0, [%1], 1;" : "=r"(old) : "l"(bar + 1) : "memory");
    if (old == nblocks - 1u) {
      // every other CTA has left: nothing reads the words any more in this launch
      asm volatile("st.relaxed.gpu.u32 [%0], 0;" ::"l"(bar) : "memory");
      asm volatile("st.relaxed.gpu.u32 [%0], 0;" ::"l"(bar + 1) : "memory");
    }
  }
}

// Exclusive scan of in[0..n) into out[0..n], out[n] = total, with two block barriers.
// All threads of the block call it; `tmp` holds at least 32 ints.  in and out may alias.
__device__ __forceinline__ void block_scan_fast(const int* in, int* out, int n, int* tmp) {
  const int tid = threadIdx.x, nt = blockDim.x;
  const int lane = tid & 31, wid = tid >> 5;
  const int per = (n + nt - 1) / nt;
  const int lo = min(n, tid * per), hi = min(n, lo + per);
  int v[4];
  int sum = 0;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[i] = (lo + i < hi) ? in[lo + i] : 0;
    sum += v[i];
  }
  for (int i = lo + 4; i < hi; ++i) sum += in[i];  // only when n > 4 * blockDim.x
  int incl = sum;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += u;
  }
  if (lane == 31) tmp[wid] = incl;
  __syncthreads();
  // the warps before this one, summed in one warp reduction (at most 32 warps)
  int run = incl - sum + int(__reduce_add_sync(0xffffffffu, unsigned(lane < wid ? tmp[lane] : 0)));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    if (lo + i < hi) {
      out[lo + i] = run;
      run += v[i];
    }
  }
  for (int i = lo + 4; i < hi; ++i) {
    const int u = in[i];
    out[i] = run;
    run += u;
  }
  if (hi == n && lo < hi) out[n] = run;
  if (n == 0 && tid == 0) out[0] = 0;
  __syncthreads();
}

// Column scan over CTAs: for each bin e, prefix[e][c] = sum of hist[e][c'] over c' < c
// and counts[e] = the bin's total.  One warp per bin, lane l covering up to 8
// consecutive CTAs per pass of 256.  Called by every warp of every CTA between two
// grid barriers.
__device__ __forceinline__ void column_scan(const PrefillWS& pw, int NE, int grid, int nwarps) {
  const int w = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = blockIdx.x * nwarps + w; e < NE; e += grid * nwarps) {
    const int* h = pw.hist + size_t(e) * pw.grid_max;
    int* p = pw.prefix + size_t(e) * pw.grid_max;
    int carry = 0;
    for (int c0 = 0; c0 < grid; c0 += 256) {
      const int span = min(256, grid - c0);
      const int per = (span + 31) / 32;
      const int cl = c0 + lane * per;
      int v[8];
      int sum = 0;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        v[i] = (i < per && cl + i < c0 + span) ? __ldcg(h + cl + i) : 0;
        sum += v[i];
      }
      int incl = sum;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
      }
      int run = carry + incl - sum;
#pragma unroll
      for (int i = 0; i < 8; ++i) {
        if (i < per && cl + i < c0 + span) p[cl + i] = run;
        run += v[i];
      }
      carry += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) pw.counts[e] = carry;
  }
}

}  // namespace moe
