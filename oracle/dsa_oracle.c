/*
 * dsa_oracle.c -- plain, slow, fp64 CPU oracle of the DeepSeek Sparse Attention hot path.
 *
 * TEST INFRASTRUCTURE.  Only the test suite, the package smoke check and the benchmark's
 * CPU-baseline leg may load this code.  The CUDA library shares nothing with it: no
 * header, no helper, no table.
 *
 * Source pages (cited by title and section):
 *   [GLM53]  "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM"
 *            (SemiAnalysis, Chinese translation): §DeepSeek Sparse Attention,
 *            §Lightning Indexer, §Sparse MLA, §MLA changes, §IndexShare.
 *   [ES]     "La atención dispersa de GLM-5.3 reduce el cómputo, pero persiste la
 *            demanda de HBM" (remio.ai): the sections on what sparse attention changes
 *            and on IndexShare.
 *
 * What is computed, in the pages' order:
 *   1. Lightning indexer [GLM53 §Lightning Indexer]: queries and keys live in a low
 *      dimension; queries have several heads, the key has one; the per-head logit is the
 *      q.k dot product passed through ReLU; the token's indexer score is the weighted sum
 *      of those logits over the query heads.  No values, no softmax.
 *   2. Top-K [GLM53 §Lightning Indexer, §Sparse MLA; ES]: K = 2048; a query that attends
 *      fewer than K tokens stays dense, else the K best-scoring tokens are kept.  The one
 *      selection serves every attention head.
 *   3. Sparse MLA in MQA mode [GLM53 §Sparse MLA, §MLA changes]: attention over the
 *      selected tokens' cached latent rows only.
 *   4. IndexShare [GLM53 §IndexShare]: one indexer per group of 4 layers; the full layer
 *      caches its top-K indices and the shared layers reuse them (composed by the Python
 *      wrapper from steps 1-3).
 *
 * Readings taken where the pages are silent (formulas on [GLM53] were lost):
 *   - the weight is per query row and head, w[t,h], an input;
 *   - fp8 inputs are e4m3 codes with one positive fp32 scale per token; dequantised
 *     value = scale * e4m3(code);
 *   - causal: the query at position p sees tokens 0..p inclusive;
 *   - ties in the top-K go to the lower token index; the result is listed in ascending
 *     token order and padded with -1;
 *   - MQA mode: the key is the whole cached row (latent d + rope r), the value is the
 *     latent part (its first d entries); softmax scale is an input (1/sqrt(192+64) for
 *     the GLM-5 shapes of §MLA changes);
 *   - outputs: o[h,:] = sum_j p_j c_j[:d] / sum_j p_j, lse = m + ln(sum_j p_j) with
 *     p_j = exp(logit_j - m), m = max logit; a row with no valid index gives o = 0 and
 *     lse = -inf.
 *
 * Token addressing: token s of sequence b is physical row seq_start[b] + s, or, with a
 * block table, bt[b*pages_per_seq + s/page_size]*page_size + s%page_size.
 *
 * 0. Cache append, the step that feeds the path [GLM53 §Lightning Indexer: the indexer
 *    caches one key per token like the KV cache; §MLA changes: one latent row per token]:
 *    a new token's indexer key is stored as e4m3 codes with one fp32 scale per token and
 *    its latent row is copied.  Readings: the scale is an fp32 number (the per-token fp32
 *    scale of the cache), scale = max(amax, 1e-30) / 448 evaluated in fp32; the code is
 *    the e4m3 value nearest to the quotient x / scale itself (rounded once, ties to the
 *    even mantissa, saturating at +-448).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ---------- number formats ---------------------------------------------------------- */

/* OCP 8-bit floating point, E4M3 variant: 1 sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits, no infinities, S.1111.111 is NaN; exponent field 0 is subnormal
 * (value = mantissa/8 * 2^-6). */
double orc_e4m3_to_double(uint8_t code)
{
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
double orc_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int64_t phys_row(int b, int s, const int32_t *seq_start, const int32_t *bt,
                        int page_size, int pages_per_seq)
{
    if (bt)
        return (int64_t)bt[(int64_t)b * pages_per_seq + s / page_size] * page_size +
               s % page_size;
    return (int64_t)seq_start[b] + s;
}

/* ---------- 0. cache append ----------------------------------------------------------- */

/* e4m3 code of an fp32 value: the nearest e4m3 value, ties to the even mantissa, and
 * magnitudes from 448 up saturating to 448 (the largest finite e4m3 value).  Below 2^-6
 * the representable values are the multiples of 2^-9; in [2^E, 2^(E+1)) they are the
 * multiples of 2^(E-3).  Scaling by a power of two is exact, and rint() rounds half to
 * even in the default rounding mode. */
static uint8_t e4m3_encode_d(double x)
{
    const int sign = signbit(x) ? 1 : 0;
    const double a = fabs(x);
    uint8_t code;
    if (a >= 448.0) {
        code = 0x7E;
    } else if (a < ldexp(1.0, -6)) {
        code = (uint8_t)rint(ldexp(a, 9)); /* 0..8; 8 is 2^-6, the first normal code */
    } else {
        int e;
        frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
        int E = e - 1;
        double q = rint(ldexp(a, 3 - E)); /* 8..16 */
        if (q == 16.0) {
            q = 8.0;
            E += 1;
        }
        const int field = E + 7, mant = (int)q - 8;
        code = (field > 15 || (field == 15 && mant == 7)) ? 0x7E : (uint8_t)((field << 3) | mant);
    }
    return (uint8_t)(code | (sign << 7));
}

uint8_t orc_e4m3_encode(float x)
{
    return e4m3_encode_d((double)x);
}

/* Writes n new tokens into copies of the caches: token i of sequence seq[i] at position
 * pos[i] goes to its physical row (contiguous or paged addressing as above).  A token
 * whose row does not resolve is left out and counted; the count is returned. */
int orc_cache_append(const float *k_new, const uint16_t *c_new, const int32_t *seq,
                     const int32_t *pos, int n, int B, int Di, int D,
                     const int32_t *seq_start, const int32_t *bt, int page_size,
                     int pages_per_seq, int64_t num_rows, uint8_t *k8, float *k_scale,
                     uint16_t *kv)
{
    int skipped = 0;
    for (int i = 0; i < n; ++i) {
        const int b = seq[i], s = pos[i];
        int64_t row = -1;
        if (b >= 0 && b < B && s >= 0) {
            if (!bt || s / page_size < pages_per_seq) {
                if (!bt || bt[(int64_t)b * pages_per_seq + s / page_size] >= 0)
                    row = phys_row(b, s, seq_start, bt, page_size, pages_per_seq);
            }
        }
        if (row < 0 || row >= num_rows) {
            ++skipped;
            continue;
        }
        float amax = 0.0f;
        for (int c = 0; c < Di; ++c) {
            const float v = fabsf(k_new[(int64_t)i * Di + c]);
            if (v > amax)
                amax = v;
        }
        const float scale = (amax > 1e-30f ? amax : 1e-30f) / 448.0f;
        /* one rounding, of the quotient itself: the fp64 quotient of two fp32 values is
         * never within an fp64 half-ulp of an e4m3 rounding boundary it is not equal to */
        for (int c = 0; c < Di; ++c)
            k8[row * Di + c] = e4m3_encode_d((double)k_new[(int64_t)i * Di + c] / (double)scale);
        k_scale[row] = scale;
        if (c_new)
            memcpy(kv + row * D, c_new + (int64_t)i * D, (size_t)D * sizeof(uint16_t));
    }
    return skipped;
}

/* ---------- 1. lightning indexer ---------------------------------------------------- */

/*
 * scores[t, s] = sum_h w[t,h] * ReLU( q[t,h,:] . k[s,:] )        for s = 0..q_pos[t]
 * with q = q_scale[t] * e4m3(q8), k = k_scale[row(s)] * e4m3(k8)   [GLM53 §Lightning Indexer]
 * scores[t, s] = -inf for s > q_pos[t].  Rows t = b*T + i belong to sequence b.
 * abs_terms (may be NULL) receives sum_h |w[t,h]| * sum_c |q[t,h,c] * k[s,c]|, the sum of
 * the magnitudes of every term of the score: what the round-off of any evaluation of the
 * score in a shorter format is proportional to (0 past q_pos[t]).
 * Returns 0, or -1 on a bad argument.
 */
int orc_indexer_scores(const uint8_t *q8, const float *q_scale, const float *w,
                       const uint8_t *k8, const float *k_scale,
                       const int32_t *seq_start, const int32_t *block_table, int page_size,
                       int pages_per_seq, const int32_t *q_pos, int B, int T, int Hi, int Di,
                       int Lmax, double *scores, double *abs_terms)
{
    if (B <= 0 || T <= 0 || Hi <= 0 || Di <= 0 || Lmax <= 0)
        return -1;
    const int rows = B * T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int t = 0; t < rows; ++t) {
        const int b = t / T;
        const int p = q_pos[t];
        double *out = scores + (int64_t)t * Lmax;
        if (p < 0 || p >= Lmax) {
            bad |= 1;
            continue;
        }
        double *q = malloc(sizeof(double) * (size_t)Hi * Di);
        double *kk = malloc(sizeof(double) * (size_t)Di);
        for (int h = 0; h < Hi; ++h)
            for (int c = 0; c < Di; ++c)
                q[h * Di + c] = (double)q_scale[t] *
                                orc_e4m3_to_double(q8[((int64_t)t * Hi + h) * Di + c]);
        double *absrow = abs_terms ? abs_terms + (int64_t)t * Lmax : NULL;
        for (int s = 0; s < Lmax; ++s) {
            if (s > p) {
                out[s] = -INFINITY;
                if (absrow)
                    absrow[s] = 0.0;
                continue;
            }
            const int64_t row = phys_row(b, s, seq_start, block_table, page_size,
                                         pages_per_seq);
            for (int c = 0; c < Di; ++c)
                kk[c] = (double)k_scale[row] * orc_e4m3_to_double(k8[row * Di + c]);
            double score = 0.0, absum = 0.0;
            for (int h = 0; h < Hi; ++h) {
                double logit = 0.0, alogit = 0.0;
                for (int c = 0; c < Di; ++c) {
                    logit += q[h * Di + c] * kk[c];
                    alogit += fabs(q[h * Di + c] * kk[c]);
                }
                double relu = logit > 0.0 ? logit : 0.0;
                score += (double)w[(int64_t)t * Hi + h] * relu;
                absum += fabs((double)w[(int64_t)t * Hi + h]) * alogit;
            }
            out[s] = score;
            if (absrow)
                absrow[s] = absum;
        }
        free(q);
        free(kk);
    }
    return bad ? -1 : 0;
}

/* ---------- 2. causal top-K with the dense fallback ---------------------------------- */

typedef struct {
    double score;
    int32_t index;
} cand_t;

/* better first: higher score, then lower token index */
static int cand_cmp(const void *a, const void *b)
{
    const cand_t *x = a, *y = b;
    if (x->score > y->score)
        return -1;
    if (x->score < y->score)
        return 1;
    return (x->index > y->index) - (x->index < y->index);
}

static int int_cmp(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/*
 * For row t with n = q_pos[t] + 1 candidate tokens: if n <= K the row stays dense
 * (indices 0..n-1); otherwise the K tokens with the largest score, ties to the lower
 * index [GLM53 §Lightning Indexer].  Output idx[t, 0..K-1] in ascending token order,
 * -1 padded.  `scores` are doubles; an fp32 score array is widened exactly by the
 * caller, which keeps every comparison identical to one made in fp32.
 */
int orc_topk(const double *scores, const int32_t *q_pos, int rows, int Lmax, int K,
             int32_t *idx)
{
    if (rows < 0 || Lmax <= 0 || K <= 0)
        return -1;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int t = 0; t < rows; ++t) {
        const int n = q_pos[t] + 1;
        int32_t *out = idx + (int64_t)t * K;
        if (n <= 0 || n > Lmax) {
            bad |= 1;
            continue;
        }
        int taken;
        if (n <= K) {
            for (int s = 0; s < n; ++s)
                out[s] = s;
            taken = n;
        } else {
            cand_t *c = malloc(sizeof(cand_t) * (size_t)n);
            for (int s = 0; s < n; ++s) {
                c[s].score = scores[(int64_t)t * Lmax + s];
                c[s].index = s;
            }
            qsort(c, (size_t)n, sizeof(cand_t), cand_cmp);
            for (int j = 0; j < K; ++j)
                out[j] = c[j].index;
            free(c);
            qsort(out, (size_t)K, sizeof(int32_t), int_cmp);
            taken = K;
        }
        for (int j = taken; j < K; ++j)
            out[j] = -1;
    }
    return bad ? -1 : 0;
}

/* ---------- 3. sparse MLA, MQA (absorbed) mode --------------------------------------- */

/*
 * For row t (sequence b = t / T) and head h, over the valid entries j of idx[t, :]
 * (idx >= 0):  logit_j = scale * q[t,h,:] . c_j[:]   (all d + r entries)
 *              o[t,h,:] = sum_j exp(logit_j - m) c_j[:d] / sum_j exp(logit_j - m)
 *              lse[t,h] = m + ln sum_j exp(logit_j - m),   m = max_j logit_j
 * where c_j is the cached latent row of token idx[t, j]   [GLM53 §Sparse MLA, §MLA changes].
 * Returns 0, or -1 on a bad argument or an index outside 0..q_pos[t] (when q_pos given).
 */
int orc_sparse_mla(const uint16_t *q, const uint16_t *kv, const int32_t *seq_start,
                   const int32_t *block_table, int page_size, int pages_per_seq,
                   const int32_t *idx, const int32_t *q_pos, int B, int T, int H, int d, int r,
                   int K, double scale, double *out, double *lse)
{
    if (B <= 0 || T <= 0 || H <= 0 || d <= 0 || r < 0 || K <= 0 || d + r > 1024)
        return -1;
    const int D = d + r;
    const int rows = B * T;
    int bad = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : bad)
    for (int th = 0; th < rows * H; ++th) {
        const int t = th / H, h = th % H, b = t / T;
        const int32_t *sel = idx + (int64_t)t * K;
        double *o = out + ((int64_t)t * H + h) * d;
        double *logit = malloc(sizeof(double) * (size_t)K);
        double qh[1024];
        int n_valid = 0;
        double m = -INFINITY;
        for (int c = 0; c < D; ++c)
            qh[c] = orc_bf16_to_double(q[((int64_t)t * H + h) * D + c]);
        for (int j = 0; j < K; ++j) {
            logit[j] = -INFINITY;
            if (sel[j] < 0)
                continue;
            if (q_pos && sel[j] > q_pos[t]) {
                bad |= 1;
                continue;
            }
            const int64_t row = phys_row(b, sel[j], seq_start, block_table, page_size,
                                         pages_per_seq);
            double dot = 0.0;
            for (int c = 0; c < D; ++c)
                dot += qh[c] * orc_bf16_to_double(kv[row * D + c]);
            logit[j] = scale * dot;
            if (logit[j] > m)
                m = logit[j];
            ++n_valid;
        }
        for (int c = 0; c < d; ++c)
            o[c] = 0.0;
        if (n_valid == 0) {
            lse[(int64_t)t * H + h] = -INFINITY;
            free(logit);
            continue;
        }
        double l = 0.0;
        for (int j = 0; j < K; ++j) {
            if (sel[j] < 0 || (q_pos && sel[j] > q_pos[t]))
                continue;
            const double pj = exp(logit[j] - m);
            const int64_t row = phys_row(b, sel[j], seq_start, block_table, page_size,
                                         pages_per_seq);
            l += pj;
            for (int c = 0; c < d; ++c)
                o[c] += pj * orc_bf16_to_double(kv[row * D + c]);
        }
        for (int c = 0; c < d; ++c)
            o[c] /= l;
        lse[(int64_t)t * H + h] = m + log(l);
        free(logit);
    }
    return bad ? -1 : 0;
}

/*
 * Dense causal attention in the same MQA form, written without an index list: row t
 * attends to every token 0..q_pos[t].  Used to pin the sparse path (with K >= context the
 * two must agree).  Softmax as its textbook definition: P = exp(S) / sum(exp(S)) with the
 * row maximum subtracted from S first.
 */
int orc_dense_mla(const uint16_t *q, const uint16_t *kv, const int32_t *seq_start,
                  const int32_t *block_table, int page_size, int pages_per_seq,
                  const int32_t *q_pos, int B, int T, int H, int d, int r, double scale,
                  double *out, double *lse)
{
    if (B <= 0 || T <= 0 || H <= 0 || d <= 0 || r < 0)
        return -1;
    const int D = d + r;
    const int rows = B * T;
#pragma omp parallel for schedule(dynamic, 1)
    for (int th = 0; th < rows * H; ++th) {
        const int t = th / H, h = th % H, b = t / T;
        const int n = q_pos[t] + 1;
        double *S = malloc(sizeof(double) * (size_t)n);
        double rowmax = -INFINITY, denom = 0.0;
        for (int s = 0; s < n; ++s) {
            const int64_t row = phys_row(b, s, seq_start, block_table, page_size,
                                         pages_per_seq);
            double acc = 0.0;
            for (int c = 0; c < D; ++c)
                acc += orc_bf16_to_double(q[((int64_t)t * H + h) * D + c]) *
                       orc_bf16_to_double(kv[row * D + c]);
            S[s] = acc * scale;
            rowmax = S[s] > rowmax ? S[s] : rowmax;
        }
        for (int s = 0; s < n; ++s) {
            S[s] = exp(S[s] - rowmax);
            denom += S[s];
        }
        for (int c = 0; c < d; ++c) {
            double acc = 0.0;
            for (int s = 0; s < n; ++s) {
                const int64_t row = phys_row(b, s, seq_start, block_table, page_size,
                                             pages_per_seq);
                acc += (S[s] / denom) * orc_bf16_to_double(kv[row * D + c]);
            }
            out[((int64_t)t * H + h) * d + c] = acc;
        }
        lse[(int64_t)t * H + h] = rowmax + log(denom);
        free(S);
    }
    return 0;
}

/* ---------- accounting [GLM53 §MLA changes, §IndexShare] ------------------------------ */

/*
 * Decode SDPA in MQA mode, per cached token: the query of each of the H heads meets the
 * whole cached row once for the logit (2*H*(d+r) FLOP) and its latent part once for the
 * output (2*H*d FLOP); the row itself is read once, (d+r)*b bytes.  The formula on the
 * page was lost in extraction; this reading reproduces its printed results (the H=64
 * GLM-5 value, and H near 128 at the H800 ridge).
 */
double orc_mqa_decode_flops_per_token(int H, int d, int r)
{
    return 2.0 * H * (d + r) + 2.0 * H * d;
}

double orc_mqa_decode_bytes_per_token(int d, int r, int b)
{
    return (double)(d + r) * b;
}

double orc_mqa_decode_intensity(int H, int d, int r, int b)
{
    return orc_mqa_decode_flops_per_token(H, d, r) / orc_mqa_decode_bytes_per_token(d, r, b);
}

/* Heads H whose decode intensity equals a machine's ridge point (FLOP per byte). */
double orc_heads_at_ridge(double ridge, int d, int r, int b)
{
    return ridge * orc_mqa_decode_bytes_per_token(d, r, b) / (2.0 * (d + r) + 2.0 * d);
}

/* Attention-score FLOPs per (query, key) pair with H heads of dimension dh. */
double orc_sdpa_score_flops(int H, int dh)
{
    return 2.0 * H * dh;
}

/*
 * Indexer work over a group of G layers: without sharing every layer runs its own
 * indexer (G scans), with IndexShare one layer does and the others reuse its indices.
 * Returned: the fraction of indexer FLOPs (equally, of indexer key cache) removed.
 */
double orc_indexshare_indexer_cut(int G)
{
    const double unshared = (double)G, shared = 1.0;
    return (unshared - shared) / unshared;
}

/* Indexer FLOPs for one query row against n keys: Hi heads of dimension Di, one
 * multiply-add per element, plus the ReLU and weighted head sum (not counted). */
double orc_indexer_flops(int Hi, int Di, double n_keys)
{
    return 2.0 * Hi * Di * n_keys;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------- HiSparse host tier [ES, "HiSparse saca el historial completo de la GPU"] ---- */

/*
 * One decode step of a sequence's device working set: the full latent history stays in
 * host memory, the device keeps C slots, managed least recently used.  For the step's
 * index row idx[0..k-1] (-1 entries skipped; no token twice):
 *   - a selected token that is resident (res[t] = its slot) is a hit: its slot's last
 *     use becomes `step`;
 *   - the other selected tokens are misses, taken in their order in the row;
 *   - the victims are the m = #misses slots not used in this step (last use < step)
 *     that were used least recently: smallest last use first, the lower slot first
 *     among equal ones (never-used slots have last use 0);
 *   - the i-th miss (row order) goes to the i-th victim (ascending slot order): the
 *     victim's previous token stops being resident, the miss becomes resident there, the
 *     slot's last use becomes `step`, and loaded[i] records (token, slot).
 * res [Lmax] slot or -1, slot_tok [C] token or -1, slot_use [C] last use; step >= 1.
 * Returns the number of misses, or -1 if there are more misses than free candidates
 * or an index is out of range.
 */
typedef struct {
    uint32_t use;
    int32_t slot;
} lru_t;

static int lru_cmp(const void *a, const void *b)
{
    const lru_t *x = a, *y = b;
    if (x->use != y->use)
        return x->use < y->use ? -1 : 1;
    return (x->slot > y->slot) - (x->slot < y->slot);
}

int orc_hisparse_step(const int32_t *idx, int k, uint32_t step, int32_t *res, int Lmax,
                      int32_t *slot_tok, uint32_t *slot_use, int C, int32_t *loaded,
                      int *hits_out)
{
    int hits = 0, m = 0;
    int32_t *miss = malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
    for (int j = 0; j < k; ++j) {
        const int32_t t = idx[j];
        if (t < 0)
            continue;
        if (t >= Lmax) {
            free(miss);
            return -1;
        }
        if (res[t] >= 0) {
            slot_use[res[t]] = step;
            ++hits;
        } else {
            miss[m++] = t;
        }
    }
    lru_t *cand = malloc(sizeof(lru_t) * (size_t)C);
    int nc = 0;
    for (int s = 0; s < C; ++s)
        if (slot_use[s] < step) {
            cand[nc].use = slot_use[s];
            cand[nc].slot = s;
            ++nc;
        }
    if (m > nc) {
        free(miss);
        free(cand);
        return -1;
    }
    qsort(cand, (size_t)nc, sizeof(lru_t), lru_cmp); /* least recently used first */
    int32_t *victim = malloc(sizeof(int32_t) * (size_t)(m > 0 ? m : 1));
    for (int i = 0; i < m; ++i)
        victim[i] = cand[i].slot;
    qsort(victim, (size_t)m, sizeof(int32_t), int_cmp); /* ascending slot order */
    for (int i = 0; i < m; ++i) {
        const int32_t v = victim[i], t = miss[i];
        if (slot_tok[v] >= 0)
            res[slot_tok[v]] = -1;
        res[t] = v;
        slot_tok[v] = t;
        slot_use[v] = step;
        if (loaded) {
            loaded[2 * i] = t;
            loaded[2 * i + 1] = v;
        }
    }
    if (hits_out)
        *hits_out = hits;
    free(miss);
    free(cand);
    free(victim);
    return m;
}

/* ---------- MLA in MHA mode [GLM53 §Sparse MLA: MLA's two modes] --------------------- */

/*
 * MHA mode: the latent row c_j (d = 512 latent dims, then r = 64 rope dims) is projected up
 * per head h into a key of dn "nope" dims, w_uk[h] . c_j[:d], followed by the shared rope
 * dims c_j[d:d+r], and a value of vd dims, w_uv[h] . c_j[:d]; each query row t and head h
 * attends over the valid entries j of idx[t, :] with its own query q[t,h,:] (dn + r):
 *   logit_j = scale * (q[t,h,:dn] . (w_uk[h] c_j[:d]) + q[t,h,dn:] . c_j[d:d+r])
 *   o[t,h,:] = sum_j softmax(logit)_j (w_uv[h] c_j[:d])            (vd values)
 * w_uk [H, dn, d], w_uv [H, vd, d], q [rows, H, dn + r], all bf16 codes; no intermediate
 * value is rounded.  The n_rows cached rows are projected up first (per head), then each
 * row and head attends.  With w_uk folded into the query (the absorbed query w_uk[h]^T q_nope)
 * this is the MQA form of step 3 followed by w_uv: the two modes compute one attention.
 * Returns 0, or -1 on a bad argument.
 */
int orc_sparse_mha(const uint16_t *q, const uint16_t *kv, int64_t n_rows, const uint16_t *w_uk,
                   const uint16_t *w_uv, const int32_t *seq_start, const int32_t *block_table,
                   int page_size, int pages_per_seq, const int32_t *idx, int B, int T, int H,
                   int d, int r, int dn, int vd, int K, double scale, double *out, double *lse)
{
    if (B <= 0 || T <= 0 || H <= 0 || d <= 0 || r < 0 || dn <= 0 || vd <= 0 || K <= 0 ||
        n_rows <= 0)
        return -1;
    const int D = d + r, dq = dn + r;
    const int rows = B * T;
    /* 1. every cached row projected up, per head: kn[h][row] (dn), vv[h][row] (vd) */
    double *kn = malloc(sizeof(double) * (size_t)H * n_rows * dn);
    double *vv = malloc(sizeof(double) * (size_t)H * n_rows * vd);
    if (!kn || !vv) {
        free(kn);
        free(vv);
        return -1;
    }
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t hr = 0; hr < (int64_t)H * n_rows; ++hr) {
        const int h = (int)(hr / n_rows);
        const int64_t row = hr % n_rows;
        for (int i = 0; i < dn; ++i) {
            double acc = 0.0;
            for (int e = 0; e < d; ++e)
                acc += orc_bf16_to_double(w_uk[((int64_t)h * dn + i) * d + e]) *
                       orc_bf16_to_double(kv[row * D + e]);
            kn[hr * dn + i] = acc;
        }
        for (int i = 0; i < vd; ++i) {
            double acc = 0.0;
            for (int e = 0; e < d; ++e)
                acc += orc_bf16_to_double(w_uv[((int64_t)h * vd + i) * d + e]) *
                       orc_bf16_to_double(kv[row * D + e]);
            vv[hr * vd + i] = acc;
        }
    }
    /* 2. attention per query row and head over the selected tokens */
#pragma omp parallel for schedule(dynamic, 1)
    for (int th = 0; th < rows * H; ++th) {
        const int t = th / H, h = th % H, b = t / T;
        const int32_t *sel = idx + (int64_t)t * K;
        const uint16_t *qh = q + ((int64_t)t * H + h) * dq;
        double *o = out + ((int64_t)t * H + h) * vd;
        double *logit = malloc(sizeof(double) * (size_t)K);
        double m = -INFINITY;
        for (int e = 0; e < vd; ++e)
            o[e] = 0.0;
        for (int j = 0; j < K; ++j) {
            logit[j] = -INFINITY;
            if (sel[j] < 0)
                continue;
            const int64_t row = phys_row(b, sel[j], seq_start, block_table, page_size,
                                         pages_per_seq);
            const double *kr = kn + ((int64_t)h * n_rows + row) * dn;
            double dot = 0.0;
            for (int i = 0; i < dn; ++i)
                dot += orc_bf16_to_double(qh[i]) * kr[i];
            for (int i = 0; i < r; ++i)
                dot += orc_bf16_to_double(qh[dn + i]) * orc_bf16_to_double(kv[row * D + d + i]);
            logit[j] = scale * dot;
            if (logit[j] > m)
                m = logit[j];
        }
        double l = 0.0;
        if (m > -INFINITY) {
            for (int j = 0; j < K; ++j) {
                if (sel[j] < 0)
                    continue;
                const int64_t row = phys_row(b, sel[j], seq_start, block_table, page_size,
                                             pages_per_seq);
                const double pj = exp(logit[j] - m);
                const double *vr = vv + ((int64_t)h * n_rows + row) * vd;
                l += pj;
                for (int i = 0; i < vd; ++i)
                    o[i] += pj * vr[i];
            }
            for (int i = 0; i < vd; ++i)
                o[i] /= l;
            lse[(int64_t)t * H + h] = m + log(l);
        } else {
            lse[(int64_t)t * H + h] = -INFINITY;
        }
        free(logit);
    }
    free(kn);
    free(vv);
    return 0;
}
