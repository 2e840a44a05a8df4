/*
 * oracle.c -- plain single-threaded CPU oracle for the MoE routing step.
 *
 * TEST INFRASTRUCTURE ONLY: loaded by the tests, the smoke check and the CPU
 * baseline of the benchmark; never by the library.  Each step follows the
 * definition in oracle.h literally, one row at a time, with no blocking or
 * reordering beyond what the definition states.
 *
 * Citations:
 *   sigmoid router, correction bias, grouped top-k:
 *       vLLM PR #59693 (ROCm token-sharded residual), description of the test
 *       KimiMoE (sigmoid scores, a correction bias, group-limited top-k).
 *   packed (id << 16 | bf16 weight), rank-local relabel, round_up(count+top_k, 4),
 *   same entries in the same order for the expert GEMMs:
 *       sglang PR #37 (rank-local expert ids for the EP routed MoE), description.
 *   router parameter count (896 x 7168 per layer):
 *       HartsyInference PR #798, section Memory per GPU (0.59 B router parameters).
 *   activation quantisation of the fused route+quant decode launch (MXFP4 MoE):
 *       sglang PR #37, description; format read from the OCP Microscaling Formats (MX)
 *       specification v1.0 (MXFP4: E2M1 elements, 32-element blocks, E8M0 scale).
 *
 * Built with -O2 -ffp-contract=off and without fast-math so that every float
 * operation is one IEEE operation in the order written.
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>

static float f32_from_bf16(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

uint16_t oracle_f32_to_bf16(float x) {
    uint32_t u;
    memcpy(&u, &x, sizeof u);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

float oracle_sigmoid(float x) {
    double e = exp(-(double)x);
    double s = 1.0 / (1.0 + e);
    return (float)s;
}

void oracle_sigmoid_array(const void* x, int dtype, float* s, long n) {
    for (long i = 0; i < n; ++i) {
        float v = (dtype == ORACLE_DT_F32) ? ((const float*)x)[i]
                                           : f32_from_bf16(((const uint16_t*)x)[i]);
        s[i] = oracle_sigmoid(v);
    }
}

int oracle_num_experts(int E, int k, int local_offset, int local_count) {
    (void)local_offset;
    if (local_count <= 0) return E;
    return ((local_count + k + 3) / 4) * 4;
}

static int args_valid(int T, int E, int k, int n_group, int topk_group, int local_offset,
                      int local_count) {
    if (T < 0 || E <= 0 || k <= 0 || n_group <= 0) return 0;
    if (E % n_group != 0) return 0;
    if (E / n_group < 2) return 0;
    if (topk_group < 1 || topk_group > n_group) return 0;
    if (k > topk_group * (E / n_group)) return 0;
    if (local_count < 0 || local_offset < 0) return 0;
    if (local_offset + local_count > E) return 0;
    if (E > 32767) return 0;
    if (local_count > 0 && local_count + k > 32767) return 0;
    return 1;
}

int oracle_route(const void* logits, int dtype, const float* bias, int T, int E, int k,
                 int n_group, int topk_group, float scale, int local_offset, int local_count,
                 int32_t* packed, int32_t* counts, int32_t* offsets, int32_t* perm,
                 int32_t* ids_global) {
    if (!args_valid(T, E, k, n_group, topk_group, local_offset, local_count)) return -1;
    if (dtype != ORACLE_DT_F32 && dtype != ORACLE_DT_BF16) return -1;
    const int gsize = E / n_group;
    const int NE = oracle_num_experts(E, k, local_offset, local_count);

    float* s = (float*)malloc(sizeof(float) * (size_t)E);
    float* b = (float*)malloc(sizeof(float) * (size_t)E);
    float* gs = (float*)malloc(sizeof(float) * (size_t)n_group);
    char* kept = (char*)malloc((size_t)n_group);
    char* taken = (char*)malloc((size_t)E);
    int* slot_id = (int*)malloc(sizeof(int) * (size_t)k);
    int32_t* lid = (int32_t*)malloc(sizeof(int32_t) * ((size_t)T * (size_t)k + 1));

    for (int t = 0; t < T; ++t) {
        /* 1-3: score and biased score */
        for (int e = 0; e < E; ++e) {
            float x;
            if (dtype == ORACLE_DT_F32)
                x = ((const float*)logits)[(size_t)t * E + e];
            else
                x = f32_from_bf16(((const uint16_t*)logits)[(size_t)t * E + e]);
            s[e] = oracle_sigmoid(x);
            b[e] = s[e] + bias[e];
        }
        /* 4: group score = sum of the two largest biased scores of the group */
        for (int g = 0; g < n_group; ++g) {
            float m1 = -INFINITY, m2 = -INFINITY;
            for (int e = g * gsize; e < (g + 1) * gsize; ++e) {
                if (b[e] > m1) {
                    m2 = m1;
                    m1 = b[e];
                } else if (b[e] > m2) {
                    m2 = b[e];
                }
            }
            gs[g] = m1 + m2;
        }
        /* 5: keep topk_group groups, largest score first, ties to the lower group */
        memset(kept, 0, (size_t)n_group);
        for (int r = 0; r < topk_group; ++r) {
            int best = -1;
            for (int g = 0; g < n_group; ++g) {
                if (kept[g]) continue;
                if (best < 0 || gs[g] > gs[best]) best = g;
            }
            kept[best] = 1;
        }
        /* 6: top-k among experts of kept groups; slot order = b descending, ties to lower id */
        memset(taken, 0, (size_t)E);
        for (int j = 0; j < k; ++j) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (!kept[e / gsize] || taken[e]) continue;
                if (best < 0 || b[e] > b[best]) best = e;
            }
            taken[best] = 1;
            slot_id[j] = best;
        }
        /* 7: renormalise the unbiased scores of the chosen experts to `scale`, bf16 */
        float den = 0.0f;
        for (int j = 0; j < k; ++j) den = den + s[slot_id[j]];
        for (int j = 0; j < k; ++j) {
            float q = s[slot_id[j]] / den;
            float w = q * scale;
            uint16_t wb = oracle_f32_to_bf16(w);
            /* 8: rank-local relabel of the packed id */
            int id = slot_id[j];
            int l;
            if (local_count > 0) {
                if (id >= local_offset && id < local_offset + local_count)
                    l = id - local_offset;
                else
                    l = local_count + j;
            } else {
                l = id;
            }
            /* 9: pack */
            packed[(size_t)t * k + j] = (int32_t)(((uint32_t)l << 16) | (uint32_t)wb);
            lid[(size_t)t * k + j] = l;
            if (ids_global) ids_global[(size_t)t * k + j] = id;
        }
    }

    /* 10: histogram of the (possibly relabelled) ids */
    for (int e = 0; e < NE; ++e) counts[e] = 0;
    for (size_t i = 0; i < (size_t)T * k; ++i) counts[lid[i]] += 1;
    /* 11: exclusive scan */
    offsets[0] = 0;
    for (int e = 0; e < NE; ++e) offsets[e + 1] = offsets[e] + counts[e];
    /* 12: stable permutation ordered by (expert, token, slot) */
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)(NE > 0 ? NE : 1));
    for (int e = 0; e < NE; ++e) cursor[e] = offsets[e];
    for (int t = 0; t < T; ++t)
        for (int j = 0; j < k; ++j) {
            int32_t l = lid[(size_t)t * k + j];
            perm[cursor[l]] = t * k + j;
            cursor[l] += 1;
        }

    free(cursor);
    free(lid);
    free(slot_id);
    free(taken);
    free(kept);
    free(gs);
    free(b);
    free(s);
    return 0;
}

void oracle_router_gemm(const uint16_t* hidden, const uint16_t* w, int T, int H, int E,
                        double* logits) {
    for (int t = 0; t < T; ++t)
        for (int e = 0; e < E; ++e) {
            double acc = 0.0;
            for (int h = 0; h < H; ++h)
                acc += (double)f32_from_bf16(hidden[(size_t)t * H + h]) *
                       (double)f32_from_bf16(w[(size_t)e * H + h]);
            logits[(size_t)t * E + e] = acc;
        }
}

int oracle_route_layout(const int32_t* counts, const int32_t* offsets, const int32_t* perm, int n,
                        int NE, int tile, int capacity, int32_t* inv_perm, int32_t* padded_offsets,
                        int32_t* padded_rows, int32_t* m_indices) {
    if (n < 0 || NE < 1 || tile < 1 || capacity < 0) return -1;
    /* inverse permutation: the entry perm[p] sits at position p */
    if (inv_perm)
        for (int p = 0; p < n; ++p) inv_perm[perm[p]] = p;
    /* padded offsets: each bin's block rounded up to a multiple of the tile */
    int32_t* poff = (int32_t*)malloc(sizeof(int32_t) * (size_t)(NE + 1));
    long long total = 0;
    poff[0] = 0;
    for (int e = 0; e < NE; ++e) {
        long long blocks = ((long long)counts[e] + tile - 1) / tile;
        total += blocks * tile;
        if (total > 0x7FFFFFFFLL) {
            free(poff);
            return -1;
        }
        poff[e + 1] = (int32_t)total;
    }
    if (padded_offsets)
        for (int e = 0; e <= NE; ++e) padded_offsets[e] = poff[e];
    if ((padded_rows || m_indices) && total > capacity) {
        free(poff);
        return -1;
    }
    /* padded rows: every row starts as padding, then each bin's entries in perm order */
    for (int r = 0; r < capacity; ++r) {
        if (padded_rows) padded_rows[r] = -1;
        if (m_indices) m_indices[r] = -1;
    }
    for (int e = 0; e < NE; ++e)
        for (int i = 0; i < counts[e]; ++i) {
            if (padded_rows) padded_rows[poff[e] + i] = perm[offsets[e] + i];
            if (m_indices) m_indices[poff[e] + i] = e;
        }
    free(poff);
    return (int)total;
}

int oracle_route_index(const int32_t* packed, int T, int k, int NE, int32_t* counts,
                       int32_t* offsets, int32_t* perm) {
    if (T < 0 || k < 1 || NE < 1) return -1;
    size_t n = (size_t)T * k;
    for (size_t i = 0; i < n; ++i)
        if ((int)((uint32_t)packed[i] >> 16) >= NE) return -1;
    /* histogram of the ids in the packed values */
    for (int e = 0; e < NE; ++e) counts[e] = 0;
    for (size_t i = 0; i < n; ++i) counts[(uint32_t)packed[i] >> 16] += 1;
    /* exclusive scan */
    offsets[0] = 0;
    for (int e = 0; e < NE; ++e) offsets[e + 1] = offsets[e] + counts[e];
    /* stable permutation ordered by (id, token, slot) */
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)NE);
    for (int e = 0; e < NE; ++e) cursor[e] = offsets[e];
    for (size_t i = 0; i < n; ++i) {
        int l = (int)((uint32_t)packed[i] >> 16);
        perm[cursor[l]] = (int32_t)i;
        cursor[l] += 1;
    }
    free(cursor);
    return 0;
}

int oracle_dispatch_counts(const int32_t* ids, int n, int E, int R, int32_t* send_counts,
                           int32_t* send_offsets) {
    if (n < 0 || E < 1 || R < 1 || E % R != 0) return -1;
    int per = E / R;
    for (int d = 0; d < R; ++d) send_counts[d] = 0;
    for (int i = 0; i < n; ++i) {
        if (ids[i] < 0 || ids[i] >= E) return -1;
        send_counts[ids[i] / per] += 1;
    }
    send_offsets[0] = 0;
    for (int d = 0; d < R; ++d) send_offsets[d + 1] = send_offsets[d] + send_counts[d];
    return 0;
}

int oracle_alltoall_layout(const int32_t* matrix, int R, int me, int32_t* send_displs,
                           int32_t* recv_counts, int32_t* recv_displs) {
    if (R < 1 || me < 0 || me >= R) return -1;
    send_displs[0] = 0;
    for (int d = 0; d < R; ++d) send_displs[d + 1] = send_displs[d] + matrix[(size_t)me * R + d];
    recv_displs[0] = 0;
    for (int s = 0; s < R; ++s) {
        recv_counts[s] = matrix[(size_t)s * R + me];
        recv_displs[s + 1] = recv_displs[s] + recv_counts[s];
    }
    return 0;
}

/* E2M1 magnitudes by code (code & 7): sign | exponent (2 bits, bias 1) | mantissa (1 bit);
 * exponent 0 is the subnormal range (0 and 0.5). */
static const double kE2M1[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

uint8_t oracle_e2m1_encode(double v) {
    int neg = signbit(v) ? 1 : 0;
    double a = fabs(v);
    if (a > 6.0) a = 6.0;  /* saturate to the largest magnitude */
    /* nearest magnitude; on an exact tie the code with last bit 0 */
    int best = 0;
    for (int c = 1; c < 8; ++c) {
        double dc = fabs(a - kE2M1[c]);
        double db = fabs(a - kE2M1[best]);
        if (dc < db || (dc == db && (c & 1) == 0)) best = c;
    }
    return (uint8_t)((neg << 3) | best);
}

int oracle_mxfp4_quant(const uint16_t* x, int T, int H, uint8_t* q, uint8_t* scales) {
    if (T < 0 || H <= 0 || H % 32 != 0) return -1;
    const int nb = H / 32;
    for (int t = 0; t < T; ++t) {
        for (int b = 0; b < nb; ++b) {
            const uint16_t* v = x + (size_t)t * H + (size_t)b * 32;
            /* shared exponent from the block's largest magnitude */
            double amax = 0.0;
            for (int i = 0; i < 32; ++i) {
                double a = fabs((double)f32_from_bf16(v[i]));
                if (a > amax) amax = a;
            }
            int e;
            if (amax == 0.0) {
                e = -127;
            } else {
                int ex;
                frexp(amax, &ex);   /* amax = m 2^ex, m in [0.5, 1): floor(log2) = ex - 1 */
                e = (ex - 1) - 2;
                if (e < -127) e = -127;
                if (e > 127) e = 127;
            }
            scales[(size_t)t * nb + b] = (uint8_t)(e + 127);
            /* elements: V / 2^e to E2M1, two per byte, the even element low */
            for (int i = 0; i < 32; i += 2) {
                uint8_t lo = oracle_e2m1_encode(ldexp((double)f32_from_bf16(v[i]), -e));
                uint8_t hi = oracle_e2m1_encode(ldexp((double)f32_from_bf16(v[i + 1]), -e));
                q[(size_t)t * (H / 2) + (size_t)b * 16 + i / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return 0;
}
