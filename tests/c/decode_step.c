/*
 * decode_step.c -- one DSA decode step through libdsa's C ABI from a plain C program, on
 * the exact (integer-valued) workload shape: indexer scores, causal top-k and the
 * allocation-free sparse MLA, checked against the fp64 oracle linked in beside it.
 *
 * Two sequences (contexts 300 and 1000), one query each; indexer 4 heads of dim 32 with
 * weights in {0.5, 1, 2}; top-64; MLA with 4 heads, latent 64 + rope 16, scale 1/8.  Every
 * q and key value is an integer in [-4, 4] (exact in e4m3 and bf16), so the scores are
 * exact in fp32 and must equal the oracle's bit for bit, and so must the index sets; the
 * attention outputs must lie within one bf16 ulp of the oracle's plus the fp32 error of
 * forming the weighted mean (for |values| <= 4 and 64 keys: well under 0.05), and the
 * log-sum-exp within fp32 round-off (2^-16 + 2^-20 |lse|).
 *
 * Exit status 0 when everything matches, 1 on a mismatch, 2 when a call fails.
 * Test infrastructure only (it links the oracle).
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include <cuda_runtime_api.h>

#include "dsa.h"

/* the oracle's C entry points (test infrastructure) */
uint8_t orc_e4m3_encode(float x);
int orc_indexer_scores(const uint8_t *q8, const float *q_scale, const float *w,
                       const uint8_t *k8, const float *k_scale, const int32_t *seq_start,
                       const int32_t *block_table, int page_size, int pages_per_seq,
                       const int32_t *q_pos, int B, int T, int Hi, int Di, int Lmax,
                       double *scores, double *abs_terms);
int orc_topk(const double *scores, const int32_t *q_pos, int rows, int Lmax, int K,
             int32_t *idx);
int orc_sparse_mla(const uint16_t *q, const uint16_t *kv, const int32_t *seq_start,
                   const int32_t *block_table, int page_size, int pages_per_seq,
                   const int32_t *idx, const int32_t *q_pos, int B, int T, int H, int d, int r,
                   int K, double scale, double *out, double *lse);

enum { B = 2, HI = 4, DI = 32, H = 4, DL = 64, R = 16, K = 64 };
static const int lengths[B] = {300, 1000};

static uint32_t rng_state = 12345u;
static int small_int(void) { /* uniform in [-4, 4], seeded */
    rng_state = rng_state * 1664525u + 1013904223u;
    return (int)((rng_state >> 8) % 9u) - 4;
}

static uint16_t bf16_of_int(int v) { /* exact for small integers */
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(u >> 16);
}

static double bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

#define CK(x)                                                                         \
    do {                                                                              \
        cudaError_t e_ = (x);                                                         \
        if (e_ != cudaSuccess) {                                                      \
            fprintf(stderr, "%s: %s\n", #x, cudaGetErrorString(e_));                   \
            return 2;                                                                 \
        }                                                                             \
    } while (0)
#define DK(x)                                                                         \
    do {                                                                              \
        dsa_status_t s_ = (x);                                                        \
        if (s_ != DSA_OK) {                                                           \
            fprintf(stderr, "%s: %s\n", #x, dsa_status_string(s_));                    \
            return 2;                                                                 \
        }                                                                             \
    } while (0)

int main(void) {
    int Lmax = 0, n_rows = 0;
    int32_t seq_start[B], q_pos[B];
    for (int b = 0; b < B; ++b) {
        seq_start[b] = n_rows;
        n_rows += lengths[b];
        q_pos[b] = lengths[b] - 1;
        if (lengths[b] > Lmax) Lmax = lengths[b];
    }
    const int D = DL + R;
    /* host inputs */
    uint8_t *q8 = malloc((size_t)B * HI * DI), *k8 = malloc((size_t)n_rows * DI);
    float *q_scale = malloc(B * sizeof(float)), *k_scale = malloc((size_t)n_rows * sizeof(float));
    float *w = malloc((size_t)B * HI * sizeof(float));
    uint16_t *q = malloc((size_t)B * H * D * 2), *kv = malloc((size_t)n_rows * D * 2);
    for (int i = 0; i < B * HI * DI; ++i) q8[i] = orc_e4m3_encode((float)small_int());
    for (int i = 0; i < n_rows * DI; ++i) k8[i] = orc_e4m3_encode((float)small_int());
    for (int i = 0; i < B; ++i) q_scale[i] = 1.f;
    for (int i = 0; i < n_rows; ++i) k_scale[i] = 1.f;
    static const float wv[3] = {0.5f, 1.f, 2.f};
    for (int i = 0; i < B * HI; ++i) w[i] = wv[(small_int() + 4) % 3];
    for (int i = 0; i < B * H * D; ++i) q[i] = bf16_of_int(small_int());
    for (int i = 0; i < n_rows * D; ++i) kv[i] = bf16_of_int(small_int());

    /* device copies */
    uint8_t *d_q8, *d_k8;
    float *d_qs, *d_ks, *d_w, *d_scores, *d_lse;
    uint16_t *d_q, *d_kv, *d_out;
    int32_t *d_seq, *d_pos, *d_idx;
    CK(cudaMalloc((void **)&d_q8, (size_t)B * HI * DI));
    CK(cudaMalloc((void **)&d_k8, (size_t)n_rows * DI));
    CK(cudaMalloc((void **)&d_qs, B * sizeof(float)));
    CK(cudaMalloc((void **)&d_ks, (size_t)n_rows * sizeof(float)));
    CK(cudaMalloc((void **)&d_w, (size_t)B * HI * sizeof(float)));
    CK(cudaMalloc((void **)&d_scores, (size_t)B * Lmax * sizeof(float)));
    CK(cudaMalloc((void **)&d_lse, (size_t)B * H * sizeof(float)));
    CK(cudaMalloc((void **)&d_q, (size_t)B * H * D * 2));
    CK(cudaMalloc((void **)&d_kv, (size_t)n_rows * D * 2));
    CK(cudaMalloc((void **)&d_out, (size_t)B * H * DL * 2));
    CK(cudaMalloc((void **)&d_seq, B * sizeof(int32_t)));
    CK(cudaMalloc((void **)&d_pos, B * sizeof(int32_t)));
    CK(cudaMalloc((void **)&d_idx, (size_t)B * K * sizeof(int32_t)));
    CK(cudaMemcpy(d_q8, q8, (size_t)B * HI * DI, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_k8, k8, (size_t)n_rows * DI, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_qs, q_scale, B * sizeof(float), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_ks, k_scale, (size_t)n_rows * sizeof(float), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_w, w, (size_t)B * HI * sizeof(float), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_q, q, (size_t)B * H * D * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_kv, kv, (size_t)n_rows * D * 2, cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_seq, seq_start, B * sizeof(int32_t), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(d_pos, q_pos, B * sizeof(int32_t), cudaMemcpyHostToDevice));

    /* the step: indexer -> top-k -> sparse MLA (the allocation-free entry point) */
    const float scale = 0.125f;
    dsa_cache_layout_t layout = {d_seq, NULL, 0, 0, n_rows};
    DK(dsa_indexer_scores(d_q8, d_qs, d_w, d_k8, d_ks, &layout, d_pos, B, 1, HI, DI, Lmax,
                          d_scores, NULL));
    DK(dsa_topk(d_scores, d_pos, B, Lmax, K, d_idx, NULL));
    DK(dsa_sparse_mla_decode_noalloc(d_q, d_kv, &layout, d_idx, B, H, DL, R, K, scale, d_out,
                                     d_lse, NULL));
    CK(cudaDeviceSynchronize());
    uint32_t code = 0;
    DK(dsa_device_error(NULL, &code));

    float *scores = malloc((size_t)B * Lmax * sizeof(float));
    int32_t *idx = malloc((size_t)B * K * sizeof(int32_t));
    uint16_t *out = malloc((size_t)B * H * DL * 2);
    float *lse = malloc((size_t)B * H * sizeof(float));
    CK(cudaMemcpy(scores, d_scores, (size_t)B * Lmax * sizeof(float), cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(idx, d_idx, (size_t)B * K * sizeof(int32_t), cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(out, d_out, (size_t)B * H * DL * 2, cudaMemcpyDeviceToHost));
    CK(cudaMemcpy(lse, d_lse, (size_t)B * H * sizeof(float), cudaMemcpyDeviceToHost));

    /* the oracle */
    double *ref_scores = malloc((size_t)B * Lmax * sizeof(double));
    int32_t *ref_idx = malloc((size_t)B * K * sizeof(int32_t));
    double *ref_out = malloc((size_t)B * H * DL * sizeof(double));
    double *ref_lse = malloc((size_t)B * H * sizeof(double));
    if (orc_indexer_scores(q8, q_scale, w, k8, k_scale, seq_start, NULL, 0, 0, q_pos, B, 1, HI,
                           DI, Lmax, ref_scores, NULL) != 0 ||
        orc_topk(ref_scores, q_pos, B, Lmax, K, ref_idx) != 0 ||
        orc_sparse_mla(q, kv, seq_start, NULL, 0, 0, ref_idx, q_pos, B, 1, H, DL, R, K, scale,
                       ref_out, ref_lse) != 0) {
        fprintf(stderr, "oracle call failed\n");
        return 2;
    }

    int bad = 0;
    for (int b = 0; b < B; ++b)
        for (int s = 0; s <= q_pos[b]; ++s)
            if ((double)scores[b * Lmax + s] != ref_scores[b * Lmax + s]) ++bad;
    const int bad_scores = bad;
    for (int i = 0; i < B * K; ++i)
        if (idx[i] != ref_idx[i]) ++bad;
    const int bad_idx = bad - bad_scores;
    double max_out = 0.0, max_lse = 0.0;
    int bad_lse = 0;
    for (int i = 0; i < B * H * DL; ++i) {
        const double e = fabs(bf16_to_double(out[i]) - ref_out[i]);
        if (e > max_out) max_out = e;
    }
    for (int i = 0; i < B * H; ++i) { /* fp32 round-off of the log-sum-exp */
        const double e = fabs((double)lse[i] - ref_lse[i]);
        if (e > max_lse) max_lse = e;
        if (e > ldexp(1.0, -16) + ldexp(1.0, -20) * fabs(ref_lse[i])) ++bad_lse;
    }
    const int ok = bad == 0 && bad_lse == 0 && max_out <= 0.05 && code == 0;
    printf("%s: scores %d mismatches, indices %d mismatches, max |out - ref| %.3g, "
           "max |lse - ref| %.3g, device error word %#x\n",
           ok ? "ok" : "MISMATCH", bad_scores, bad_idx, max_out, max_lse, code);
    return ok ? 0 : 1;
}
