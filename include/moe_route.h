/*
 * moe_route.h -- C ABI of the GB300 (sm_103a) MoE token-to-expert routing library.
 *
 * One routing call, per token row t of a [T, E] logit matrix:
 *   s_e = sigmoid(logit_e); b_e = s_e + bias_e            (a1, a2)
 *     -- vLLM PR #59693 (ROCm token-sharded residual), description of its KimiMoE
 *        test: the router is a sigmoid with a correction bias and group-limited top-k.
 *   group score = sum of the two largest b of each group of E/n_group consecutive
 *   experts; keep the topk_group groups with the largest score (ties: lower group);
 *   choose the k largest b among the kept experts (ties: lower expert id); slot j
 *   of the row is the j-th of them in (b descending, id ascending) order   (a3-a5)
 *   w_j = bf16_rne(float(float(s_j / sum_slots s) * scale))                (a6)
 *   optional rank-local relabel: experts in [local_offset, local_offset +
 *   local_count) become 0..local_count-1, any other expert in slot j becomes
 *   local_count + j; num_experts NE = round_up(local_count + k, 4)         (a7)
 *   packed[t][j] = (id << 16) | bits(w_j)                                  (a8)
 *     -- sglang PR #37 (rank-local expert ids for the EP routed MoE), description:
 *        the fused route epilogue packs each slot as the expert id above the bf16
 *        weight bits; with a staged expert range the rank's own experts become
 *        0..count-1, every other expert takes count plus its slot index (so ids stay
 *        unique in a row), and the runner passes count + top_k rounded up to a
 *        multiple of 4 as the number of experts.
 * and over all rows:
 *   counts[e]  = number of entries with (relabelled) id e, e in [0, NE)     (a9)
 *   offsets    = exclusive scan of counts, offsets[NE] = T * k              (a10)
 *   perm[offsets[e] + r] = t * k + j for the r-th entry of id e in (t, j) order (a11)
 *     -- same passage: whichever ids are used, the expert GEMMs receive the same
 *        (token, local expert, weight) entries in the same order.
 * The Kimi-K3 instance is E = 896, k = 16, n_group = 8 (112 experts each),
 * topk_group = 4, scale = 2.5 (sglang PR #37: FlashInfer's Tier<896, 16> routing
 * specialisation; each of 8 expert-parallel ranks owns 112 of the 896 experts).
 *
 * Conventions for every entry point:
 *   - All array pointers are DEVICE pointers owned by the caller; the library never
 *     frees them.  Arrays are dense and row-major.  logits must be 16-byte aligned.
 *   - Work is enqueued on `stream` without host synchronisation, so calls can be
 *     captured in a CUDA graph once the library's per-device state exists (call
 *     moe_route_reserve() before capture).  Outputs are fully overwritten; no
 *     zeroing is needed.
 *   - Calls on one device share one workspace: calls must be ordered on the GPU
 *     (same stream, or otherwise serialised); concurrent calls race.
 *   - Routing of T <= 64 rows, the routing behind moe_router_gemm_route, and the
 *     bf16 routing of more rows for k = 16 and topk_group = 4 (also moe_route_index for
 *     k = 16) run as kernels launched with programmatic stream serialization that signal
 *     their dependents as they start.  A kernel launched after one on the same stream
 *     WITH that attribute may therefore start early and must execute
 *     griddepcontrol.wait (cudaGridDependencySynchronize) before it reads the outputs;
 *     kernels launched without it, and copies, start after the routing has completed,
 *     as usual.
 *   - Return value: MOE_ROUTE_OK or a negative moe_route_status.  A call that returns
 *     an error has enqueued nothing.  Errors detected on the device (a bounded wait
 *     that ran out) are reported by moe_route_device_status().
 *   - Supported shapes: E = 896 with n_group = 8 (the Kimi-K3 grouping), any
 *     topk_group in [1, 8], 1 <= k <= 32 with k <= topk_group * 112.  Other valid
 *     shapes return MOE_ROUTE_E_UNSUPPORTED.
 */
#ifndef MOE_ROUTE_H
#define MOE_ROUTE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st*`; NULL = legacy default stream */

typedef enum {
    MOE_ROUTE_OK = 0,
    MOE_ROUTE_E_INVALID_ARG = -1,    /* arguments violate the definition or a pointer is NULL */
    MOE_ROUTE_E_UNSUPPORTED = -2,    /* valid, but not a shape the kernels implement */
    MOE_ROUTE_E_CUDA = -3,           /* a CUDA runtime call failed (launch, allocation) */
    MOE_ROUTE_E_WORKSPACE = -4,      /* per-device state missing while the stream is capturing */
    MOE_ROUTE_E_DEVICE_TIMEOUT = -5, /* a bounded device-side wait ran out (see device_status) */
    MOE_ROUTE_E_BAD_ID = -6          /* moe_route_index: an id >= NE or repeated in a row (device_status) */
} moe_route_status;

typedef enum { MOE_ROUTE_F32 = 0, MOE_ROUTE_BF16 = 1 } moe_route_dtype;

/*
 * moe_route -- steps a1..a11 for a [T, E] matrix of router logits.
 *   logits        [T, E] float32 (dtype MOE_ROUTE_F32) or bfloat16 bits (MOE_ROUTE_BF16),
 *                 16-byte aligned.  Must be finite.
 *   bias          [E] float32 correction bias (selection only; weights use s).
 *   T >= 0; T = 0 writes zero counts and offsets only.
 *   E, k, n_group, topk_group, scale   as defined above; scale is routed_scaling_factor.
 *   local_offset, local_count  rank-local relabel range; local_count = 0 keeps global ids.
 *                 0 <= local_offset, local_offset + local_count <= E.
 *   packed        [T, k] int32 out: (id << 16) | bf16 weight bits (id relabelled if asked).
 *   counts        [NE] int32 out, offsets [NE + 1] int32 out, perm [T * k] int32 out,
 *                 NE = moe_route_bins(E, k, local_count).
 *   topk_ids      [T, k] int32 out, nullable: the GLOBAL expert ids in slot order.
 * Errors: INVALID_ARG when E % n_group != 0, E / n_group < 2, topk_group not in
 * [1, n_group], k < 1 or k > topk_group * E / n_group, T < 0, a required pointer is
 * NULL, logits not 16-byte aligned, local_count < 0, local_offset < 0,
 * local_offset + local_count > E, or an id would not fit 15 bits.
 */
int moe_route(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
              int n_group, int topk_group, float scale, int local_offset, int local_count,
              int32_t* packed, int32_t* counts, int32_t* offsets, int32_t* perm,
              int32_t* topk_ids, struct CUstream_st* stream);

/*
 * moe_route_ex -- moe_route with one more optional output:
 *   inv_perm  [T * k] int32 out, nullable: inv_perm[t * k + j] = the position of entry
 *             (t, j) in perm, i.e. perm[inv_perm[i]] = i (the inverse permutation).
 * The routing kernels know each entry's place when they write perm and store it here in
 * token order, so the stores are coalesced; moe_route_layout then need not build the
 * inverse map (pass its inv_perm as NULL).  The routed entries reach the expert GEMMs in
 * the routing's order (sglang PR #37, Rank-local expert ids for the EP routed MoE,
 * description), and the combine step that brings each entry's result back to its token
 * reads this map.  Everything else, including the errors, is as moe_route.
 */
int moe_route_ex(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
                 int n_group, int topk_group, float scale, int local_offset, int local_count,
                 int32_t* packed, int32_t* counts, int32_t* offsets, int32_t* perm,
                 int32_t* topk_ids, int32_t* inv_perm, struct CUstream_st* stream);

/*
 * moe_route_with_layout -- moe_route_ex and then moe_route_layout (without its inverse
 * map: inv_perm here is moe_route_ex's) in one call: the routing plus the expert-GEMM
 * layout that moe_route_layout defines, for a tile of `tile` rows.
 *   tile >= 1; padded_offsets [NE + 1] out, nullable; padded_rows [capacity] and
 *   m_indices [capacity] out, nullable, with capacity >= moe_route_padded_capacity(T, k,
 *   NE, tile) when either is given (all `capacity` rows are written).
 * Where the bf16 prefill kernel for k = 16 and topk_group = 4 routes the batch, that
 * kernel writes the layout itself in the same launch; otherwise the layout kernel
 * follows the routing on the stream.  The results are the same either way.
 * Errors: those of moe_route; INVALID_ARG for tile < 1, a capacity below the bound or a
 * bound beyond 2^31 - 1.  All layout outputs NULL: the same as moe_route_ex.
 */
int moe_route_with_layout(const void* logits, int logits_dtype, const float* bias, int T, int E,
                          int k, int n_group, int topk_group, float scale, int local_offset,
                          int local_count, int32_t* packed, int32_t* counts, int32_t* offsets,
                          int32_t* perm, int32_t* topk_ids, int32_t* inv_perm, int tile,
                          int32_t* padded_offsets, int32_t* padded_rows, int32_t* m_indices,
                          int capacity, struct CUstream_st* stream);

/*
 * moe_route_quant -- the fused route+quant decode launch: moe_route for a decode batch of
 * T <= MOE_ROUTE_QUANT_MAX_TOKENS rows and, in the same kernel launch, the MXFP4
 * quantisation of the batch's activations x that the routed MXFP4 MoE consumes.  The
 * page's fused launch (sglang PR #37, Rank-local expert ids for the EP routed MoE,
 * description: route_quant_fused handles decode batches up to MAX_TOKENS = 64 tokens
 * and writes the packed ids the MXFP4 routed MoE reads) does not define the activation
 * format; the reading taken is the MXFP4 format of the OCP Microscaling Formats (MX)
 * specification v1.0:
 *   per block of 32 consecutive elements of a row, e = floor(log2 max |x|) - 2 clamped
 *   to [-127, 127] (-127 for a block of zeros); x_scales holds the E8M0 byte e + 127;
 *   each element x / 2^e is rounded to E2M1 (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6) to
 *   nearest, ties to the code whose last bit is 0, magnitudes above 6 saturated, the
 *   sign kept (code bit 3); x_q holds two codes per byte, the even element in the low
 *   nibble.
 *   x         [T, H] bf16 bits, 16-byte aligned, finite; H % 32 == 0.
 *   x_q       [T, H / 2] bytes out, 4-byte aligned; x_scales [T, H / 32] bytes out.
 *   Routing arguments and outputs are those of moe_route (same results).
 * Errors: those of moe_route; INVALID_ARG for H <= 0, H % 32 != 0, NULL x / x_q /
 * x_scales with T > 0, or misaligned x / x_q; UNSUPPORTED for T > 64.  One kernel launch
 * (a programmatic dependent, like moe_route for T <= 64 rows): its first thread-block
 * cluster routes, the clusters after it quantise.
 */
#define MOE_ROUTE_QUANT_MAX_TOKENS 64
int moe_route_quant(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
                    int n_group, int topk_group, float scale, int local_offset, int local_count,
                    const uint16_t* x, int H, uint8_t* x_q, uint8_t* x_scales, int32_t* packed,
                    int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* topk_ids,
                    struct CUstream_st* stream);

/*
 * moe_router_gemm_route -- router contraction a0 fused in front of moe_route:
 *   logits[t][e] = sum_h hidden[t][h] * w_router[e][h], bf16 inputs, fp32 accumulate,
 * then steps a1..a11 on those fp32 logits.  The router weight is 896 x 7168 per layer
 * (HartsyInference PR #798, section Memory per GPU: 0.59 B router parameters over 92
 * layers).
 *   hidden      [T, H] bf16 bits, 16-byte aligned; w_router [E, H] bf16 bits (row e =
 *               expert e), 16-byte aligned.  H % 64 == 0.
 *   1 <= T <= 64 (decode batches).
 *   logits_out  [T, E] float32 out, nullable (the fp32 logits the routing used).
 *   other arguments as moe_route.  Supported: E = 896, n_group = 8, and H / 64 a
 *   multiple of the contraction's cluster size (16 K-splits where the GPU schedules
 *   seven clusters of 16 CTAs, as a GB300 does, else 8): H a multiple of 1024 on a
 *   GB300.  Other H return MOE_ROUTE_E_UNSUPPORTED.
 * w_router is read as a constant model weight: the contraction kernel is launched as a
 * programmatic dependent and starts loading the weight before the preceding kernel on
 * `stream` has completed (hidden, bias and all outputs wait for it).  The weight must
 * therefore not be written by work still pending on `stream` when the call is made
 * (write it, then synchronise, before the first call that reads it).
 */
int moe_router_gemm_route(const uint16_t* hidden, const uint16_t* w_router, const float* bias,
                          int T, int H, int E, int k, int n_group, int topk_group, float scale,
                          int local_offset, int local_count, float* logits_out, int32_t* packed,
                          int32_t* counts, int32_t* offsets, int32_t* perm, int32_t* topk_ids,
                          struct CUstream_st* stream);

/*
 * moe_route_layout -- the layout of the routed entries that grouped expert GEMMs consume,
 * built from the outputs of moe_route (or moe_router_gemm_route) on the same stream.
 * The pages name these structures without defining them: an expert-GEMM row index
 * built from the routing (InferenceX PR #2453, review summary of the MoonEP backend:
 * a kernel building DeepGEMM's m_indices) and the routed entries reaching the expert
 * GEMMs in the routing's order (sglang PR #37, description).  Definitions taken:
 *   inv_perm[perm[p]] = p                     (where entry t*k + j went; for the combine)
 *   padded_offsets[0] = 0,
 *   padded_offsets[e + 1] = padded_offsets[e] + round_up(counts[e], tile)
 *   padded row padded_offsets[e] + i, i < counts[e]:  padded_rows = perm[offsets[e] + i]
 *                                                      m_indices   = e
 *   every other row r < capacity:                     padded_rows = m_indices = -1
 * so each bin occupies whole tiles of `tile` rows, as a grouped GEMM with M-tiles of
 * that height expects (tile = 1 gives the unpadded layout).
 *   counts [NE], offsets [NE + 1], perm [T * k]: device, as moe_route wrote them
 *               (NE = moe_route_bins(E, k, local_count)); perm must be a permutation.
 *   tile >= 1.
 *   inv_perm [T * k], padded_offsets [NE + 1]: device outputs, nullable.
 *   padded_rows [capacity], m_indices [capacity]: device outputs, nullable; when either
 *               is given, capacity >= moe_route_padded_capacity(T, k, NE, tile), which
 *               bounds the padded total for any counts, so buffers sized once serve
 *               every call (CUDA graphs).  All `capacity` rows are written.
 * Errors: INVALID_ARG for T < 0, k < 1, NE < 1, tile < 1, a NULL counts/offsets (or
 * perm with T * k > 0), a capacity below the bound, or a bound beyond 2^31 - 1;
 * UNSUPPORTED for NE > 1,056.  All outputs NULL: returns OK and enqueues nothing.
 * One kernel launch; no allocation after the library's per-device state exists.
 * The inverse map costs one scattered 4-byte store per entry here; moe_route_ex writes
 * the same map from the routing kernels in token order, so a caller that routes with
 * moe_route_ex passes inv_perm = NULL here.
 */
int moe_route_layout(const int32_t* counts, const int32_t* offsets, const int32_t* perm, int T,
                     int k, int NE, int tile, int32_t* inv_perm, int32_t* padded_offsets,
                     int32_t* padded_rows, int32_t* m_indices, int capacity,
                     struct CUstream_st* stream);

/*
 * moe_route_index -- steps a9..a11 alone: counts, offsets and the stable (id, token, slot)
 * permutation of given packed values (id << 16 | weight).  For token-sharded routing:
 * each rank routes a contiguous slice of the tokens and the top-k results are gathered
 * (vLLM PR #59693, description of the token-sharded path); routing is row-independent,
 * so the gathered packed values are those of the whole batch, and this call gives every
 * rank the whole batch's counts, offsets and perm without routing the other slices.
 *   packed  [T, k] int32, device; ids must be < NE and distinct within each row (as every
 *           routing writes them; the ranks count the rows that hold an id).
 *   counts [NE], offsets [NE + 1], perm [T * k]: device outputs, as moe_route defines them.
 * Errors: INVALID_ARG for T < 0, k < 1, NE < 1, NULL pointers, T * k >= 2^31;
 * UNSUPPORTED for k > 32 or NE > 1,056.  An id >= NE, or an id repeated within a row, is
 * left out of every output and moe_route_device_status() then returns
 * MOE_ROUTE_E_BAD_ID (outputs unspecified, every write stays inside the arrays).
 */
int moe_route_index(const int32_t* packed, int T, int k, int NE, int32_t* counts,
                    int32_t* offsets, int32_t* perm, struct CUstream_st* stream);

/*
 * moe_route_dispatch_counts -- expert-parallel dispatch: num_ranks ranks own contiguous
 * ranges of E / num_ranks experts; from the offsets of a routing with GLOBAL ids
 * (local_count = 0, NE = E), send_offsets[d] = offsets[d * E / num_ranks] (num_ranks + 1)
 * and send_counts[d] = send_offsets[d + 1] - send_offsets[d].  The entries for rank d are
 * perm[send_offsets[d] .. send_offsets[d + 1]), already in (expert, token, slot) order.
 * The counts are one row of the counts matrix of a variable-size all-to-all (vLLM PR
 * #54606, description of its collectives).  Errors: INVALID_ARG for E % num_ranks != 0,
 * num_ranks < 1, NULL offsets.  Device pointers; one small kernel.
 */
int moe_route_dispatch_counts(const int32_t* offsets, int E, int num_ranks, int32_t* send_counts,
                              int32_t* send_offsets, struct CUstream_st* stream);

/*
 * moe_route_alltoall_layout -- rank `rank`'s view of the gathered counts matrix
 * matrix[num_ranks][num_ranks] (row = source rank, column = destination rank; device):
 *   send_displs [num_ranks + 1] = exclusive scan of row `rank`
 *   recv_counts [num_ranks]     = column `rank`
 *   recv_displs [num_ranks + 1] = exclusive scan of that column
 * Outputs nullable.  Errors: INVALID_ARG for rank outside [0, num_ranks), NULL matrix;
 * UNSUPPORTED for num_ranks > 1,024.  One small kernel.
 */
int moe_route_alltoall_layout(const int32_t* matrix, int num_ranks, int rank, int32_t* send_displs,
                              int32_t* recv_counts, int32_t* recv_displs,
                              struct CUstream_st* stream);

/* Rows the padded layout can need for any routing of T rows: T * k + NE * (tile - 1);
 * MOE_ROUTE_E_INVALID_ARG for invalid arguments or a bound beyond 2^31 - 1. */
int moe_route_padded_capacity(int T, int k, int NE, int tile);

/* Number of expert bins the outputs use: local_count > 0 ? round_up(local_count + k, 4) : E. */
int moe_route_bins(int E, int k, int local_count);

/*
 * Policy helper.  The page applies rank-local ids only when the rank's expert range is
 * strictly smaller than the whole set and relabelling makes the routing problem smaller
 * (sglang PR #37, Rank-local expert ids for the EP routed MoE, description).  Returns
 * round_up(local_count + k, 4) when 0 < local_count < E and that is smaller than E;
 * otherwise E, meaning the caller should pass local_count = 0 (global ids).
 */
int moe_route_num_experts(int E, int k, int local_offset, int local_count);

/*
 * Creates the current device's library state (workspace, sigmoid table for bf16
 * logits, kernel attributes).  Call once per device before capturing calls in a CUDA
 * graph; calls outside capture create it on first use.  Allocates with cudaMalloc.
 */
int moe_route_reserve(void);

/*
 * Waits for the current device, returns and clears the device-side error word
 * (MOE_ROUTE_OK, MOE_ROUTE_E_DEVICE_TIMEOUT or MOE_ROUTE_E_BAD_ID), and resets the
 * workspace's barrier state after an error.
 */
int moe_route_device_status(void);

/* Elementwise step a1 as the routing kernels compute it: s[i] = sigmoid(x[i]).
 * x: [n] float32 or bf16 bits (device), s: [n] float32 (device). */
int moe_route_sigmoid(const void* x, int dtype, float* s, int n, struct CUstream_st* stream);

/*
 * Kernel selection for moe_route: 0 = automatic (T <= 64: one-cluster decode kernel,
 * otherwise the persistent multi-CTA kernel), 1 = always the decode kernel (T <= 64
 * only), 2 = always the persistent kernel, 3 = always the persistent kernel and, for
 * bf16 logits with k = 16 and topk_group = 4, its variant that computes every score
 * from the exact table instead of the one that starts from approximate scores, 4 = the
 * decode kernel (T <= 64 only).  Paths 3 and 4 also compute every float32 score exactly
 * instead of starting from approximate ones (moe_route and moe_route_quant).  The
 * results are identical on every path; the choice is for comparisons.  Process-wide;
 * for tests and benchmarks.  Returns the previous setting, or MOE_ROUTE_E_INVALID_ARG.
 */
int moe_route_set_path(int path);

/*
 * Test hook for the failure path of the persistent kernel's grid barrier.  The pages
 * describe no counterpart.  Arms the next moe_route call on this process that launches
 * the persistent kernel: its CTA `cta` leaves before the first grid barrier without
 * arriving, and every grid-barrier wait of that launch is limited to wait_us
 * microseconds, so the other CTAs' waits run out, set MOE_ROUTE_E_DEVICE_TIMEOUT
 * (moe_route_device_status) and return; the last CTA out restores the barrier words,
 * so the following call runs normally.  Nothing waits without a bound.  The arming is
 * consumed by that one launch.  cta = -1 disarms.  INVALID_ARG for cta < -1, or
 * wait_us outside [1, 2000000] when cta >= 0.  A cta at or beyond the launch's CTA
 * count arms nothing that happens.
 */
int moe_route_arm_barrier_timeout(int cta, int wait_us);

/*
 * moe_route_noalloc -- moe_route for callers that cannot allocate device memory.
 * The pages describe no counterpart: this is a deployment variant of the same
 * routing kernels, not a step of the method.
 *
 * moe_route obtains its workspace with cudaMalloc on first use.  A caller that has
 * reserved all free HBM up front (a serving engine's weights and KV cache), runs under
 * a memory pool that forbids raw allocations, or may only touch the buffers it is
 * given, uses this entry point instead: it never calls cudaMalloc, cudaFree or any
 * allocating routine.  Its scratch is a fixed array in the library's device image,
 * about 1.4 MB, held by every GPU that loads the library until the process exits.
 *   - Arguments, outputs and results are those of moe_route.  It runs the persistent
 *     multi-CTA kernel for every T >= 1 (for bf16 logits with k = 16 and topk_group = 4
 *     the variant moe_route uses for such batches); T = 0 launches the decode kernel,
 *     which writes zero counts and offsets only.
 *   - status: nullable DEVICE pointer to one int32 the call sets to 0, then to
 *     MOE_ROUTE_E_DEVICE_TIMEOUT if a bounded device-side wait runs out.  With NULL,
 *     such an error is recorded only inside the library's array.
 *   - Limits: at most 1056 expert bins (any supported E, k and local_count fits) and
 *     at most 160 CTAs (a larger GPU runs 160); bins beyond the limit return
 *     MOE_ROUTE_E_UNSUPPORTED.
 *   - The first call on each device (with that device current) looks up the array's
 *     address, writes the score tables into it and waits for the device; make that
 *     first call before any stream capture (during capture it returns
 *     MOE_ROUTE_E_WORKSPACE and enqueues nothing).
 *   - Every call shares the one array and it keeps the last call's contents; each call
 *     zeroes the words that must start at zero.  Calls that overlap on the GPU (other
 *     streams, other threads) race on the array and must be serialised by the caller.
 */
int moe_route_noalloc(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
                      int n_group, int topk_group, float scale, int local_offset,
                      int local_count, int32_t* packed, int32_t* counts, int32_t* offsets,
                      int32_t* perm, int32_t* topk_ids, int32_t* status,
                      struct CUstream_st* stream);

/*
 * moe_route_host -- moe_route for a logit matrix in HOST memory, results to HOST memory.
 * The pages describe no counterpart: this is the end-to-end form of the same routing
 * (input transfer, the routing kernels, result transfer), not a step of the method.
 *   logits            [T, E] float32 or bfloat16 bits in host memory (any alignment).
 *   bias              [E] float32, DEVICE pointer, 16-byte aligned (a model parameter
 *                     that stays resident).
 *   packed, counts, offsets, perm, topk_ids   host memory, sizes as for moe_route
 *                     (topk_ids nullable).
 *   Other arguments, the results and the argument errors are those of moe_route.
 * Host buffers should be page-locked (cudaHostAlloc / cudaHostRegister); then the call
 * only enqueues work and returns, and the results are in place once `stream` has
 * completed the work enqueued so far (cudaStreamSynchronize).  Pageable buffers work
 * but make the copies synchronous with the host.
 * The library copies the logits into one of two device staging slots per device
 * (allocated on first use and grown with cudaMalloc; cudaFree when a slot grows),
 * on its own copy stream, routes them on `stream` and copies the results back on
 * `stream`.  Consecutive calls alternate between the slots, so call i + 1's input
 * transfer runs while call i routes and returns its results.  Consequences:
 *   - The logits are read at some point between the call and the completion of its
 *     routing, possibly before work enqueued earlier on `stream` has run: they must be
 *     complete when the call is made and unchanged until `stream` has finished the
 *     call's work; they must not be the target of work still pending on `stream`.
 *   - Calls on one device must come from one thread at a time or be serialised by the
 *     caller, and must be ordered on the GPU like moe_route calls (same stream).
 *   - Not capturable: during stream capture it returns MOE_ROUTE_E_UNSUPPORTED and
 *     enqueues nothing.
 *   - Argument errors enqueue nothing.  A CUDA error after the input copy has been
 *     enqueued returns MOE_ROUTE_E_CUDA with that copy still enqueued.
 */
int moe_route_host(const void* logits, int logits_dtype, const float* bias, int T, int E, int k,
                   int n_group, int topk_group, float scale, int local_offset, int local_count,
                   int32_t* packed, int32_t* counts, int32_t* offsets, int32_t* perm,
                   int32_t* topk_ids, struct CUstream_st* stream);

/* Frees the current device's moe_route_host staging slots, after waiting for the work
 * that uses them.  The next moe_route_host call allocates them again. */
int moe_route_host_release(void);

/*
 * Measurement helper: enqueues one launch of an empty kernel with the decode kernel's
 * launch shape and attributes (a cluster of `ctas` CTAs of 256 threads, 1 <= ctas <= 16,
 * the bf16 decode kernel's dynamic shared memory, programmatic stream serialization);
 * moe_route_decode_ctas(T) gives the shape of a
 * T-row routing launch.  A cluster of more than 8 CTAs may be refused (MOE_ROUTE_E_CUDA)
 * on a GPU that cannot schedule it; the library's own launches never ask for one there.  Replayed in a
 * CUDA graph it gives the launch-latency floor that decode routing is compared with.
 */
int moe_route_empty(int ctas, struct CUstream_st* stream);

/* CTAs (one thread-block cluster) of the routing kernel for T <= 64 rows: 1 for T <= 4;
 * otherwise the fewest that hold max(2, ceil(T / M)) rows each, M = 16 where the GPU can
 * schedule clusters of 16 CTAs (else 8).  Creates the device state like
 * moe_route_reserve.  INVALID_ARG for T outside [0, 64]. */
int moe_route_decode_ctas(int T);

/* Static description of a status code. */
const char* moe_route_strerror(int status);

#ifdef __cplusplus
}
#endif
#endif
