/*
 * oracle.h -- plain, slow, single-threaded CPU oracle for the MoE routing step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark may load this library.  It shares no code with
 * the CUDA path and the CUDA path never calls it.
 *
 * What it computes (per token row t, then over all rows):
 *   s_e  = sigmoid(logit_e)             sigmoid router (vLLM PR #59693, description)
 *   b_e  = s_e + bias_e                 correction bias (same passage)
 *   group-limited top-k over b          grouped top-k (same passage)
 *   weights = s of the chosen experts renormalised to `scale`, rounded to bf16
 *   packed  = (id << 16) | bf16 weight bits
 *                         (sglang PR #37, description: the packed format of the fused route)
 *   optional rank-local relabel (same passage: the rank's experts become
 *   0..count-1, any other expert in top-k slot k becomes count + k,
 *   num_experts = round_up(count + top_k, 4))
 *   histogram, exclusive-scan offsets and a stable (expert, token, slot) permutation
 *                         (same passage: "the same (token, local expert, weight)
 *                          entries reach the expert GEMMs in the same order")
 * Constants of the Kimi-K3 instance (896 experts, top_k 16, 8 groups of 112,
 * keep 4 groups, group score = sum of the top-2 biased scores, scale 2.5, ties to
 * the lower id, bf16 weights) are arguments here.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - sigmoid evaluated in double and rounded once to float; b is a float add.
 *   - slot order within a row: biased score descending, ties to the lower id.
 *   - group ties: the lower group index is kept first.
 *   - experts of dropped groups are excluded (never masked to 0).
 *   - top-2 counts equal values with multiplicity.
 *   - renormalisation: den = float sum of s over slots in slot order,
 *     w = float(float(s / den) * scale), then bf16 round-to-nearest-even; no epsilon.
 *   - perm holds the expanded index t*k + j; all T*k entries are included, so in
 *     rank-local mode bins count..count+k-1 hold the other ranks' slots.
 *   - logits and bias are finite.
 */
#ifndef MOE_ROUTE_ORACLE_H
#define MOE_ROUTE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_DT_F32 = 0, ORACLE_DT_BF16 = 1 };

/* sigma(x) = 1 / (1 + e^-x) evaluated in double, rounded once to float. */
float oracle_sigmoid(float x);

/* s[i] = oracle_sigmoid(x[i]) for i < n; x is float (dtype 0) or bf16 bits (dtype 1). */
void oracle_sigmoid_array(const void* x, int dtype, float* s, long n);

/* float -> bfloat16 bits, round to nearest, ties to even (finite inputs). */
uint16_t oracle_f32_to_bf16(float x);

/* Number of expert bins of the routed problem: count > 0 ? round_up(count + k, 4) : E. */
int oracle_num_experts(int E, int k, int local_offset, int local_count);

/* Full routing step.  logits: [T, E] row-major, float (dtype 0) or bf16 bits (dtype 1).
 * bias: [E].  Outputs: packed [T, k], counts [NE], offsets [NE + 1], perm [T * k],
 * ids_global [T, k] (nullable) = the chosen global expert ids in slot order.
 * Returns 0, or -1 for an invalid argument (same rules as the library). */
int oracle_route(const void* logits, int dtype, const float* bias, int T, int E, int k,
                 int n_group, int topk_group, float scale, int local_offset, int local_count,
                 int32_t* packed, int32_t* counts, int32_t* offsets, int32_t* perm,
                 int32_t* ids_global);

/* Router contraction: logits[t][e] = sum_h hidden[t][h] * w[e][h], bf16 inputs,
 * accumulated in double in index order; output double [T, E]. */
void oracle_router_gemm(const uint16_t* hidden, const uint16_t* w, int T, int H, int E,
                        double* logits);

/* Layout of the routed entries for grouped expert GEMMs, from the routing outputs
 * counts [NE], offsets [NE + 1] and perm [n] (n = T * k).  The pages only name these
 * structures (an expert-GEMM row index built from the routing -- InferenceX PR #2453,
 * review summary of the MoonEP backend; the entries reaching the expert GEMMs in the
 * routing's order -- sglang PR #37, description); the plainest reading is taken:
 *   inv_perm[perm[p]] = p                     (the inverse permutation)
 *   padded_offsets[0] = 0,
 *   padded_offsets[e + 1] = padded_offsets[e] + round_up(counts[e], tile)
 *   padded row padded_offsets[e] + i, i < counts[e]: padded_rows = perm[offsets[e] + i]
 *   and m_indices = e; every other row r < capacity holds -1 in both.
 * Any output may be NULL.  Returns padded_offsets[NE], or -1 for an invalid argument
 * (tile < 1, or capacity below the padded total when a padded array is asked for). */
int oracle_route_layout(const int32_t* counts, const int32_t* offsets, const int32_t* perm, int n,
                        int NE, int tile, int capacity, int32_t* inv_perm, int32_t* padded_offsets,
                        int32_t* padded_rows, int32_t* m_indices);

/* Steps 10-12 alone, from packed values (id << 16 | weight) of T rows of k slots, as
 * gathered from token-sharded routing (each rank routes a contiguous slice of the tokens
 * and the top-k results are gathered -- vLLM PR #59693, description of the sharded
 * path): counts [NE], offsets [NE + 1], perm [T * k] exactly as oracle_route defines
 * them.  Returns 0, or -1 for invalid arguments or an id >= NE. */
int oracle_route_index(const int32_t* packed, int T, int k, int NE, int32_t* counts,
                       int32_t* offsets, int32_t* perm);

/* Expert-parallel dispatch layout (vLLM PR #54606, description: a variable-size
 * all-to-all driven by a counts matrix).  R ranks own contiguous expert ranges of
 * E / R experts; for n global expert ids, send_counts[d] = entries whose expert rank d
 * owns, send_offsets = exclusive scan (R + 1).  Returns 0, or -1 for invalid arguments
 * (E % R != 0, an id outside [0, E)). */
int oracle_dispatch_counts(const int32_t* ids, int n, int E, int R, int32_t* send_counts,
                           int32_t* send_offsets);

/* All-to-all layout of rank `me` from the gathered counts matrix [R][R] (row = source,
 * column = destination): send_displs = exclusive scan of row me (R + 1), recv_counts =
 * column me, recv_displs = its exclusive scan (R + 1).  Returns 0 or -1. */
int oracle_alltoall_layout(const int32_t* matrix, int R, int me, int32_t* send_displs,
                           int32_t* recv_counts, int32_t* recv_displs);

/* MXFP4 quantisation of the decode batch's activations, the quant half of the fused
 * route+quant decode launch (sglang PR #37, description: route_quant_fused, decode
 * batches up to MAX_TOKENS = 64; the routed MoE is an MXFP4 MoE, Mxfp4MoEMethod).  The
 * pages do not define the activation format; the reading taken is the MXFP4 format of the
 * OCP Microscaling Formats (MX) specification v1.0:
 *   - a block is 32 consecutive elements of a row (H % 32 == 0);
 *   - shared scale X = 2^e with e = floor(log2(max_i |V_i|)) - 2 (2 is the exponent of
 *     the largest E2M1 normal, 6 = 1.5 * 2^2), e clamped to [-127, 127]; a block of
 *     zeros takes e = -127; the scale is stored as E8M0, the byte e + 127;
 *   - each element P_i = V_i / X rounded to E2M1 (magnitudes 0, 0.5, 1, 1.5, 2, 3, 4, 6;
 *     4-bit code sign | 2-bit exponent | 1-bit mantissa) to the nearest magnitude, ties to
 *     the code whose last bit is 0, magnitudes above 6 saturated to 6, the sign taken from
 *     V_i (so -0 and negative values that round to 0 give code 8);
 *   - storage: q [T, H / 2] bytes, byte i of a row holding element 2i in its low nibble
 *     and element 2i + 1 in its high nibble; scales [T, H / 32] bytes.
 * x: [T, H] bf16 bits.  Returns 0, or -1 when H % 32 != 0 or T < 0. */
int oracle_mxfp4_quant(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* scales);

/* E2M1 code (0..15) of an already scaled value, by the rule above. */
uint8_t oracle_e2m1_encode(double v);

#ifdef __cplusplus
}
#endif
#endif
