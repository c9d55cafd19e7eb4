/*
 * Plain fp64 CPU oracle for paged attention.  TEST INFRASTRUCTURE ONLY:
 * nothing in the product path calls, links or loads this file; only the tests,
 * the smoke check and the benchmark's CPU-baseline leg do.  It shares no code,
 * header or constant with the CUDA path.
 *
 * What it computes (the plain definition, nothing fused or reordered):
 *   for every sequence i, KV head h and query row (r, g) with g in h's group,
 *     1. gather the sequence's cache blocks in block-table order into one
 *        contiguous K_i / V_i of n rows ("The logical sequence remains ordered.
 *        The physical memory does not have to be." -- x321.org, "The serving
 *        bottleneck is not just FLOPs", section "PagedAttention borrows an
 *        operating-system trick"; chenhuiyu.github.io "A complete explanation
 *        from first principles", section "Logical continuity, physical
 *        flexibility");
 *     2. s_t = scale * sum_d q[d] * K_i[t][d]         (t < n)
 *        p   = softmax(s)                              (max subtracted)
 *        out = sum_t p_t * V_i[t]
 *      which is Attention(Q,K,V) = softmax(Q K^T / sqrt(d_head)) V from the
 *      same x321.org page, section "First understand what the KV cache is
 *      storing".
 *   Every value is widened from bf16 to fp64 exactly; all arithmetic is fp64.
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - cache layout [num_blocks][num_kv_heads][block_size][head_dim];
 *   - query head g reads KV head g / (num_q_heads / num_kv_heads)
 *     (contiguous grouped-query groups);
 *   - seq_len counts every cached token including the newest one;
 *   - a multi-token query chunk of q_len rows is causal inside the chunk:
 *     row r sees keys t <= seq_len - q_len + r, so n = seq_len - q_len + 1 + r;
 *   - n <= 0 gives an all-zero output row.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top 16 bits of an IEEE binary32; widening is exact. */
static double oracle_bf16_to_double(uint16_t bits) {
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int oracle_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
    return omp_get_max_threads();
#else
    (void)n;
    return 1;
#endif
}

/* Returns 0 on success, -1 on bad arguments, -3 when a needed block-table
 * entry lies outside [0, num_blocks) or a sequence needs more table entries
 * than max_blocks. */
int oracle_paged_attention(const uint16_t *q,        /* [B][q_len][Hq][d]      */
                           const uint16_t *k_cache,  /* [NB][Hkv][bs][d]       */
                           const uint16_t *v_cache,  /* [NB][Hkv][bs][d]       */
                           const int32_t *block_tables, /* [B][max_blocks]     */
                           int max_blocks,
                           const int32_t *seq_lens,  /* [B]                    */
                           int B, int q_len, int Hq, int Hkv, int d, int bs,
                           int NB, double scale,
                           double *out)              /* [B][q_len][Hq][d]      */
{
    if (B < 0 || q_len < 1 || Hq < 1 || Hkv < 1 || d < 1 || bs < 1 || NB < 0 ||
        Hq % Hkv != 0 || max_blocks < 0)
        return -1;
    const int G = Hq / Hkv;

    /* validate the tables first so that a bad entry is an error, not a crash */
    for (int i = 0; i < B; ++i) {
        int L = seq_lens[i];
        if (L < 0) return -1;
        int nblk = 0;
        while ((long long)nblk * bs < L) ++nblk; /* smallest count covering L */
        if (nblk > max_blocks) return -3;
        for (int j = 0; j < nblk; ++j) {
            int b = block_tables[(size_t)i * max_blocks + j];
            if (b < 0 || b >= NB) return -3;
        }
    }

    int status = 0;
#pragma omp parallel for collapse(2) schedule(dynamic, 1)
    for (int i = 0; i < B; ++i) {
        for (int h = 0; h < Hkv; ++h) {
            const int L = seq_lens[i];
            /* step 1: gather this (sequence, KV head) into contiguous rows */
            double *K = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * d);
            double *V = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1) * d);
            double *s = (double *)malloc(sizeof(double) * (size_t)(L > 0 ? L : 1));
            if (!K || !V || !s) {
#pragma omp atomic write
                status = -2;
                free(K); free(V); free(s);
                continue;
            }
            for (int t = 0; t < L; ++t) {
                int logical = t / bs, offset = t % bs;
                int phys = block_tables[(size_t)i * max_blocks + logical];
                size_t row = (((size_t)phys * Hkv + h) * bs + offset) * (size_t)d;
                for (int x = 0; x < d; ++x) {
                    K[(size_t)t * d + x] = oracle_bf16_to_double(k_cache[row + x]);
                    V[(size_t)t * d + x] = oracle_bf16_to_double(v_cache[row + x]);
                }
            }
            /* step 2: dense softmax attention for every query row of the group */
            for (int r = 0; r < q_len; ++r) {
                int n = L - q_len + 1 + r; /* keys visible to row r */
                for (int gg = 0; gg < G; ++gg) {
                    int g = h * G + gg;
                    const uint16_t *qrow = q + (((size_t)i * q_len + r) * Hq + g) * (size_t)d;
                    double *o = out + (((size_t)i * q_len + r) * Hq + g) * (size_t)d;
                    for (int x = 0; x < d; ++x) o[x] = 0.0;
                    if (n <= 0) continue;
                    double m = -INFINITY;
                    for (int t = 0; t < n; ++t) {
                        double acc = 0.0;
                        for (int x = 0; x < d; ++x)
                            acc += oracle_bf16_to_double(qrow[x]) * K[(size_t)t * d + x];
                        s[t] = scale * acc;
                        if (s[t] > m) m = s[t];
                    }
                    double denom = 0.0;
                    for (int t = 0; t < n; ++t) {
                        s[t] = exp(s[t] - m);
                        denom += s[t];
                    }
                    for (int t = 0; t < n; ++t) {
                        double p = s[t] / denom;
                        for (int x = 0; x < d; ++x) o[x] += p * V[(size_t)t * d + x];
                    }
                }
            }
            free(K); free(V); free(s);
        }
    }
    return status;
}
