/*
 * dsa.h -- libdsa: the DeepSeek Sparse Attention (DSA) hot path on one NVIDIA B300.
 *
 * The method (source page: "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory
 * TAM", SemiAnalysis, sections named below):
 *   1. lightning indexer (§Lightning Indexer): every cached token s gets the score
 *        I[t,s] = sum_h w[t,h] * ReLU( q_I[t,h,:] . k_I[s,:] )
 *      from a multi-head indexer query and the single-head indexer key cached for s;
 *   2. top-K (§Lightning Indexer, §Sparse MLA): the K = 2048 best tokens per query,
 *      or all of them when the query attends at most K tokens (dense);
 *   3. sparse MLA in MQA (absorbed) mode (§Sparse MLA, §MLA changes): attention over the
 *      selected tokens' cached latent rows only (latent d = 512 plus rope r = 64, bf16);
 *   4. IndexShare (§IndexShare): one indexer per 4 layers; the full layer's top-K index
 *      set is reused by the shared layers.
 *
 * Conventions for every entry point:
 *   - Array pointers are DEVICE pointers owned by the caller; libdsa allocates nothing.
 *     Scratch space, where an entry point needs some, is passed in by the caller and
 *     sized by dsa_workspace_bytes() (dsa_sparse_mla_decode_noalloc uses a fixed static
 *     array of the library instead).
 *   - Every call is asynchronous on `stream` (a cudaStream_t; NULL is the legacy default
 *     stream).  Argument errors are found on the host and returned before anything is
 *     launched; a failed launch returns DSA_ERR_CUDA.  No exception crosses the ABI.
 *   - Checks that need device data (an index out of range, a bad block-table entry, a
 *     position past the score row) are made on the device: the offending item is
 *     skipped and a device error word is set; dsa_device_error() reads and clears it.
 *     Every wait inside a kernel is bounded (about two seconds); a wait that runs out
 *     also sets the word and the kernel returns.
 *   - fp8 values are OCP e4m3 codes (uint8_t) with one positive fp32 scale per token;
 *     bf16 values are raw bfloat16 bits (uint16_t).  All arrays are dense row-major.
 *   - Query rows are grouped by sequence: with T rows per sequence, rows b*T .. b*T+T-1
 *     belong to sequence b.  Row t sits at position q_pos[t] and sees tokens
 *     0 .. q_pos[t] (causal; the query's own token is already cached).
 *   - Kernels launch with programmatic dependent launch: each may start while the
 *     previous kernel of the stream finishes.  Before it waits for that kernel
 *     (griddepcontrol.wait) a kernel reads only the call's per-step inputs -- queries,
 *     weights, positions, the cache layout -- never the caches, scores or index sets,
 *     which it reads after the wait.  So per-step inputs must be complete when the call
 *     is made: written by a copy, or by a kernel that does not trigger its dependents
 *     early (every kernel that does not use programmatic dependent launch).
 *   - The library holds no state beyond the device error word, the kernel attributes it
 *     sets once per device and the static scratch of dsa_sparse_mla_decode_noalloc;
 *     calls on different streams with different output and workspace buffers may run
 *     concurrently (dsa_sparse_mla_decode_noalloc excepted: see there).
 */
#ifndef DSA_H
#define DSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    DSA_OK = 0,
    DSA_ERR_INVALID_ARG = 1, /* null pointer, size out of range, misaligned pointer */
    DSA_ERR_UNSUPPORTED = 2, /* a shape this build does not implement */
    DSA_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    DSA_ERR_WORKSPACE = 4,   /* workspace missing or smaller than dsa_workspace_bytes() */
    DSA_ERR_DEVICE = 5,      /* dsa_device_error(): a device-side check fired */
    DSA_ERR_SCRATCH_LIMIT = 6 /* dsa_sparse_mla_decode_noalloc: shape needs more scratch
                                 than DSA_NOALLOC_SCRATCH_BYTES */
} dsa_status_t;

/*
 * Where token s of sequence b lives in a cache (the same for the indexer key cache and
 * every latent cache of an IndexShare group).  The pages mention page management for the
 * cache without a page size; libdsa supports both layouts:
 *   contiguous (block_table == NULL): physical row = seq_start[b] + s;
 *   paged      (block_table != NULL): physical row =
 *              block_table[b * pages_per_seq + s / page_size] * page_size + s % page_size.
 * num_rows is the number of physical rows in each cache (used for bounds checks).
 */
typedef struct {
    const int32_t *seq_start;   /* device [B], contiguous layout, else NULL */
    const int32_t *block_table; /* device [B, pages_per_seq], paged layout, else NULL */
    int32_t page_size;          /* tokens per page; the indexer needs a multiple of 64 */
    int32_t pages_per_seq;
    int64_t num_rows;           /* physical rows per cache */
} dsa_cache_layout_t;

/* Library version string. */
const char *dsa_version(void);

/* Static text for a status code. */
const char *dsa_status_string(dsa_status_t status);

/*
 * Lightning indexer scores (§Lightning Indexer).
 *   q8       [B*T, Hi, Di]  e4m3 indexer queries        q_scale [B*T] fp32 (> 0)
 *   w        [B*T, Hi]      fp32 weight per query head
 *   k8_cache [num_rows, Di] e4m3 indexer keys           k_scale [num_rows] fp32 (> 0)
 *   q_pos    [B*T]          position of each row (0 <= q_pos < Lmax)
 * Output scores [B*T, Lmax] fp32: scores[t, s] for s = 0..q_pos[t] is
 *   q_scale[t] * k_scale[s] * sum_h w[t,h] * ReLU(e4m3(q8[t,h,:]) . e4m3(k8[s,:])),
 * which equals the definition with dequantised q and k because the scales are
 * positive.  Entries past q_pos[t] are not written.
 * Supported: Di in {32, 64, 128}; Hi <= 256 with ceil(Hi/16)*16 <= 256; paged caches
 * need page_size % 64 == 0.  T == 1 is the decode form, T > 1 the prefill form (rows of
 * one sequence are scored together, up to 256/ceil16(Hi) rows per tensor-core tile).
 * k8_cache must be 16-byte aligned.
 */
dsa_status_t dsa_indexer_scores(const uint8_t *q8, const float *q_scale, const float *w,
                                const uint8_t *k8_cache, const float *k_scale,
                                const dsa_cache_layout_t *layout, const int32_t *q_pos,
                                int B, int T, int Hi, int Di, int Lmax, float *scores,
                                void *stream);

/*
 * Causal top-K with the dense fallback (§Lightning Indexer; top K = 2048 in §Sparse MLA).
 *   scores [rows, Lmax] fp32 (NaN not supported), q_pos [rows].
 * For row t with n = q_pos[t] + 1 candidates:
 *   n <= k : idx[t, :] = 0, 1, ..., n-1, then -1 up to k (the row stays dense);
 *   n >  k : the k tokens with the largest score, equal scores going to the lower token
 *            index (deterministic), listed in ascending token order.
 * Output idx [rows, k] int32.  1 <= k <= 8192; Lmax <= 375040 (a row's scores are split
 * over at most eight CTAs, each holding its slice in shared memory), else
 * DSA_ERR_UNSUPPORTED before any launch.
 */
dsa_status_t dsa_topk(const float *scores, const int32_t *q_pos, int rows, int Lmax, int k,
                      int32_t *idx, void *stream);

/*
 * Fused lightning indexer + causal top-K for chunked prefill (§Lightning Indexer; the
 * indexer "becomes the visible bottleneck" once attention is sparse: remio.ai, the
 * section on IndexShare).  Computes exactly what dsa_indexer_scores followed by dsa_topk
 * computes (same scores, same selection and tie rule, same output idx [B*T, k]), but the
 * [B*T, Lmax] score matrix never reaches memory: each query group's rows are scored and
 * selected on one SM, which keeps per row a coarse histogram of the scores it keeps and a
 * running threshold (the bin of the row's k-th best score so far), and appends to the
 * row's candidate list (in `workspace`) only scores at or above it; a second kernel
 * ranks the candidates of the row's final bin and writes the selection in ascending
 * token order.  Arguments as dsa_indexer_scores and dsa_topk.
 * workspace: at least dsa_indexer_topk_workspace_bytes(B, T, Lmax) bytes, 16-byte
 * aligned (candidate slots for every visible token of every row, and per-row counts);
 * typically a small part of it is written.
 * Supported: as dsa_indexer_scores with ceil(Hi/16)*16 == 64 (four query rows of 64
 * heads per tensor-core tile); 1 <= k <= 8192.  Meant for many query rows per sequence (each SM
 * owns whole query groups); decode batches are better served by the two separate calls.
 */
dsa_status_t dsa_indexer_topk(const uint8_t *q8, const float *q_scale, const float *w,
                              const uint8_t *k8_cache, const float *k_scale,
                              const dsa_cache_layout_t *layout, const int32_t *q_pos, int B,
                              int T, int Hi, int Di, int Lmax, int k, int32_t *idx,
                              void *workspace, size_t workspace_bytes, void *stream);

/* Workspace bytes of dsa_indexer_topk ((size_t)-1 for invalid sizes). */
size_t dsa_indexer_topk_workspace_bytes(int B, int T, int Lmax);

/*
 * Sparse MLA decode in MQA / absorbed mode (§Sparse MLA, §MLA changes), one query row per
 * sequence.  For sequence b and head h, over the valid entries j of idx[b, :] (-1 skips):
 *   logit_j = scale * q[b,h,:] . c_j[:]            (c_j = cached row of token idx[b,j],
 *                                                   all d + r entries)
 *   out[b,h,:] = sum_j softmax(logit)_j c_j[:d]    (bf16, round to nearest even)
 *   lse[b,h]   = ln sum_j exp(logit_j)             (fp32; -inf and out = 0 if no valid j)
 *   q [B, H, d+r] bf16, kv_cache [num_rows, d+r] bf16, idx [B, k] int32.
 * Supported: H <= 64, d % 64 == 0 (d <= 512), 0 <= r <= 64, (d + r) % 8 == 0,
 * 1 <= k <= 8192; q and kv_cache 16-byte aligned.  lse may be NULL.
 * workspace: at least dsa_workspace_bytes(DSA_OP_SPARSE_MLA, B, 1, H, d, k, 1) bytes
 * (may be NULL when that is 0).
 */
dsa_status_t dsa_sparse_mla_decode(const uint16_t *q, const uint16_t *kv_cache,
                                   const dsa_cache_layout_t *layout, const int32_t *idx,
                                   int B, int H, int d, int r, int k, float scale,
                                   uint16_t *out, float *lse, void *workspace,
                                   size_t workspace_bytes, void *stream);

/*
 * Top-K and sparse MLA decode in one call (§Lightning Indexer, §Sparse MLA): exactly
 * dsa_topk(scores, q_pos, B, Lmax, k, idx) followed by dsa_sparse_mla_decode(..., idx, ...)
 * -- same index set (written to idx), same outputs.  When a row's splits of the sparse
 * MLA form one thread-block cluster (or are one CTA) and its scores fit their shared
 * memory (about 26K scores per CTA at d = 512), one kernel does both: the cluster selects
 * the row's index set, then attends over it; otherwise the top-k runs as its own launch
 * first.  Arguments as the two calls; workspace as dsa_sparse_mla_decode.
 */
dsa_status_t dsa_topk_sparse_mla_decode(const float *scores, const int32_t *q_pos, int Lmax,
                                        const uint16_t *q, const uint16_t *kv_cache,
                                        const dsa_cache_layout_t *layout, int32_t *idx, int B,
                                        int H, int d, int r, int k, float scale, uint16_t *out,
                                        float *lse, void *workspace, size_t workspace_bytes,
                                        void *stream);

/* Size of the fixed device scratch behind dsa_sparse_mla_decode_noalloc (20 MiB). */
#define DSA_NOALLOC_SCRATCH_BYTES ((size_t)20 << 20)

/*
 * Sparse MLA decode that allocates nothing and takes no workspace.  The source page has
 * no counterpart to this entry point: it is a service of the library.  It computes what
 * dsa_sparse_mla_decode computes, with the same kernels and the same split of the keys,
 * but keeps the split-KV partial results in a fixed array of DSA_NOALLOC_SCRATCH_BYTES
 * that libdsa reserves statically on each device, instead of in caller memory.  It is
 * for callers that cannot allocate device memory on the decode path: a plain C host
 * program with no device allocator of its own, or a serving loop whose device memory is
 * all handed out up front, for which a per-call cudaMalloc/cudaFree would also
 * synchronise the device.
 *   - Set-up: the first call on each device (that device current) looks the array's
 *     address up with cudaGetSymbolAddress, which may load libdsa's device code, and
 *     returns DSA_ERR_CUDA if that fails.  Make this first call before any stream
 *     capture begins.  Later calls on the device reuse the address and do nothing but
 *     check the arguments and launch.  The address belongs to the context it was taken
 *     in (the device's primary context): if that context is replaced (a device reset),
 *     the next call looks it up again, so make that call before any capture too.
 *   - Limit: a shape for which dsa_workspace_bytes(DSA_OP_SPARSE_MLA, B, 1, H, d, k, 1)
 *     exceeds DSA_NOALLOC_SCRATCH_BYTES returns DSA_ERR_SCRATCH_LIMIT before anything is
 *     launched.  The split count keeps rows x splits within the SM count, so on a
 *     148-SM B300 every supported shape fits (at most 148 x 131,584 bytes).
 *   - Nothing in the array has to start at zero: each call writes every partial result
 *     before it reads it.
 *   - All calls on a device share the array: two calls whose executions overlap (on
 *     different streams, or from host threads that do not order their streams) race on
 *     it and their results are undefined.  Calls in order on one stream are safe.
 * Arguments, layouts and the other errors are those of dsa_sparse_mla_decode.
 */
dsa_status_t dsa_sparse_mla_decode_noalloc(const uint16_t *q, const uint16_t *kv_cache,
                                           const dsa_cache_layout_t *layout,
                                           const int32_t *idx, int B, int H, int d, int r,
                                           int k, float scale, uint16_t *out, float *lse,
                                           void *stream);

/*
 * Sparse MLA prefill: as dsa_sparse_mla_decode with T query rows per sequence, each row
 * with its own index set: q [B*T, H, d+r], idx [B*T, k], out [B*T, H, d], lse [B*T, H].
 * workspace: dsa_workspace_bytes(DSA_OP_SPARSE_MLA, B, T, H, d, k, 1).
 */
dsa_status_t dsa_sparse_mla_prefill(const uint16_t *q, const uint16_t *kv_cache,
                                    const dsa_cache_layout_t *layout, const int32_t *idx,
                                    int B, int T, int H, int d, int r, int k, float scale,
                                    uint16_t *out, float *lse, void *workspace,
                                    size_t workspace_bytes, void *stream);

/*
 * IndexShare (§IndexShare): the layers of one group attend over ONE index set, computed
 * by the group's full layer.  One launch runs the sparse MLA of all n_layers layers;
 * layer g reads q_layers[g] and kv_layers[g] and writes out_layers[g] / lse_layers[g]
 * (arrays of n_layers host-side pointers to device buffers; lse_layers or its entries may
 * be NULL).  Shapes as dsa_sparse_mla_prefill (T = 1 for decode); every layer's cache
 * uses `layout`.  1 <= n_layers <= 8.
 * workspace: dsa_workspace_bytes(DSA_OP_SPARSE_MLA, B, T, H, d, k, n_layers).
 */
dsa_status_t dsa_sparse_mla_shared(const uint16_t *const *q_layers,
                                   const uint16_t *const *kv_layers, int n_layers,
                                   const dsa_cache_layout_t *layout, const int32_t *idx,
                                   int B, int T, int H, int d, int r, int k, float scale,
                                   uint16_t *const *out_layers, float *const *lse_layers,
                                   void *workspace, size_t workspace_bytes, void *stream);

/*
 * Cache append, the step that feeds the path (§Lightning Indexer: the indexer keeps one
 * key per cached token, cached like the KV cache; §MLA changes: one latent row of d + r
 * bf16 values per token).  For each new token i of sequence seq[i] (0 <= seq[i] < B) at
 * position pos[i], with R its physical row under `layout`:
 *   scale      = max(max_c |k_new[i, c]|, 1e-30) / 448     (fp32)
 *   k8[R, c]   = e4m3(k_new[i, c] / scale), round to nearest even, saturating at 448
 *                (the exact quotient rounded once, not an fp32 quotient rounded again)
 *   k_scale[R] = scale
 *   kv[R, :]   = c_new[i, :]   (when c_new is not NULL)
 * so that the indexer then reads scale * e4m3(k8) = k_new to e4m3 precision.
 *   k_new [n, Di] fp32, c_new [n, D] bf16 or NULL, seq / pos [n] int32;
 *   k8_cache [num_rows, Di], k_scale [num_rows], kv_cache [num_rows, D] (NULL iff c_new is).
 * Supported: Di in {32, 64, 128}; D % 8 == 0; k_new, k8_cache, c_new and kv_cache
 * 16-byte aligned.  n == 0 does nothing (the arrays may then be NULL).  A token whose
 * row does not resolve (sequence out of range, page entry missing or negative, row past
 * num_rows) is skipped and sets the device error word.  Tokens that map to the same row
 * race.  The kernels that read the caches afterwards (indexer, sparse MLA) wait for the
 * append's completion (griddepcontrol.wait) before their first cache read.
 */
dsa_status_t dsa_cache_append(const float *k_new, const uint16_t *c_new, const int32_t *seq,
                              const int32_t *pos, int n, int B, int Di, int D,
                              const dsa_cache_layout_t *layout, uint8_t *k8_cache,
                              float *k_scale, uint16_t *kv_cache, void *stream);

/*
 * MLA in MHA mode for short contexts (§Sparse MLA: MLA's MHA mode has fewer FLOPs and much
 * more memory than its MQA mode, and below a context-length threshold it is the faster
 * one; vLLM uses it from 2K up to about 5K tokens with data-parallel attention).  For head
 * h and a cached latent row c (d latent dims, then r rope dims):
 *   key_h = [w_uk[h] . c[:d] (dn dims), c[d:d+r]],   value_h = w_uv[h] . c[:d] (vd dims).
 *
 * dsa_mla_up_project: out[i, :] = w . latent[i, :d] for the n rows of `latent` ([n, ld]
 * bf16, row pitch ld >= d elements), w [N, d] bf16 (w_uk as [H*dn, d], or w_uv as
 * [H*vd, d]), out [n, N] bf16 (fp32 accumulation, rounded to nearest even).  These are the
 * per-head keys and values of MHA mode, the memory its cache takes.
 * Supported: d % 64 == 0, N % 128 == 0, ld % 8 == 0; pointers 16-byte aligned.
 *
 * dsa_sparse_mha_prefill: for query row t (rows grouped by sequence as everywhere) and
 * head h, over the tokens of idx[t, :] (-1 skipped), with q [B*T, H, dn + r] bf16:
 *   logit_j = scale * q[t,h,:] . key_h(j),   out[t,h,:] = sum_j softmax(logit)_j value_h(j)
 * (bf16, vd values), lse[t,h] as in dsa_sparse_mla_decode (lse may be NULL).  k_up
 * [num_rows, H*dn] and v_up [num_rows, H*vd] are dsa_mla_up_project's outputs for the
 * rows of kv_cache [num_rows, d + r] (the rope dims are read from kv_cache); q_pos [B*T]
 * bounds the keys each row's tile visits.  The cache is contiguous (layout->seq_start;
 * no block table).  The selection is applied as a mask over dense 128-key tiles: at these
 * context lengths it covers much of the context.
 * workspace: dsa_mha_workspace_bytes(B, T, Lmax) bytes (selection bitmaps), 16-byte aligned.
 * Supported: dn % 64 == 0, r % 64 == 0, dn + r <= 256, vd in {128, 256}, d % 64 == 0,
 * Lmax <= 65536, k <= 8192; pointers 16-byte aligned.
 */
dsa_status_t dsa_mla_up_project(const uint16_t *latent, int64_t n, int ld, int d,
                                const uint16_t *w, int N, uint16_t *out, void *stream);

size_t dsa_mha_workspace_bytes(int B, int T, int Lmax);

dsa_status_t dsa_sparse_mha_prefill(const uint16_t *q, const uint16_t *k_up,
                                    const uint16_t *v_up, const uint16_t *kv_cache,
                                    const dsa_cache_layout_t *layout, const int32_t *idx,
                                    const int32_t *q_pos, int B, int T, int H, int d, int r,
                                    int dn, int vd, int k, int Lmax, float scale, uint16_t *out,
                                    float *lse, void *workspace, size_t workspace_bytes,
                                    void *stream);

/*
 * Host-tier working set of a latent cache (HiSparse, remio.ai: the section on HiSparse).
 * The full latent history of every sequence stays in pinned host memory; the device keeps
 * C slots per sequence, managed least recently used, and each decode step makes its
 * selected tokens resident before the sparse MLA reads them.  The result of the attention
 * does not change: the MLA reads the same rows through another layout.
 *   residency  [B, Lmax] int32: the pool row (b*C + slot) holding token t of sequence b,
 *              or -1.  It is a block table with one-token pages, so the step's MLA reads
 *              the working set through dsa_cache_layout_t{seq_start = NULL, block_table =
 *              residency, page_size = 1, pages_per_seq = Lmax, num_rows = B*C} and pool.
 *   slot_token [B, C] int32: the token in each slot, or -1.
 *   slot_use   [B, C] uint32: the last step that used each slot (0: never).
 *   pool       [B*C, D] bf16: the device working set.
 * dsa_hisparse_init sets residency and slot_token to -1 and slot_use to 0.
 * dsa_hisparse_fetch, for step `step` (>= 1, increasing from call to call) and the step's
 * selection idx [B, k] (-1 skipped; a token at most once per row):
 *   - a resident selected token is a hit: its slot's last use becomes `step`;
 *   - the others are misses, taken in index-row order; the victims are the slots of the
 *     sequence not used in this step, least recently used first (the lower slot first
 *     among equal last uses), listed in ascending slot order; miss i takes victim i: the
 *     victim's previous token stops being resident, the miss's row (host_kv row
 *     host_seq_start[b] + t, D bf16 values) is copied into the slot, and its last use
 *     becomes `step`;
 *   - stats [B, 2] (nullable) receives (hits, misses) per sequence.
 * host_kv is a device-accessible address of pinned host memory (cudaHostAlloc with
 * cudaHostAllocMapped, or any pinned allocation under unified addressing); the missed rows
 * are read from it directly by the kernel.  Supported: D % 8 == 0, k <= C <= 16384,
 * k <= 8192; host_kv and pool 16-byte aligned.  Steps out of order (fewer free slots than
 * misses) set the device error word (kernel id 6) and change nothing.
 */
dsa_status_t dsa_hisparse_init(int32_t *residency, int B, int Lmax, int32_t *slot_token,
                               uint32_t *slot_use, int C, void *stream);

dsa_status_t dsa_hisparse_fetch(const int32_t *idx, int B, int k, uint32_t step,
                                const uint16_t *host_kv, const int32_t *host_seq_start, int D,
                                int32_t *residency, int Lmax, int32_t *slot_token,
                                uint32_t *slot_use, int C, uint16_t *pool, int32_t *stats,
                                void *stream);

typedef enum {
    DSA_OP_INDEXER = 0,
    DSA_OP_TOPK = 1,
    DSA_OP_SPARSE_MLA = 2
} dsa_op_t;

/*
 * Scratch bytes an entry point needs on the current device for the given shape (rows =
 * B*T).  The indexer and top-k need none; the sparse MLA uses it for split-KV partial
 * results when there are too few rows to fill the GPU.  Returns 0 for a shape that
 * needs no scratch, and (size_t)-1 for invalid arguments.
 */
size_t dsa_workspace_bytes(dsa_op_t op, int B, int T, int H, int d, int k, int n_layers);

/*
 * Synchronises `stream`, then reads and clears the device error word.  Returns DSA_OK
 * if no device-side check fired since the last call, else DSA_ERR_DEVICE and, if `code`
 * is not NULL, the first recorded code (kernel id << 16 | reason; kernel ids: 1 indexer,
 * 2 top-k, 3 sparse MLA, 4 split combine, 5 cache append, 6 host-tier fetch, 7 MHA mode,
 * 8 wait probe; reasons: 1 a wait ran out, 2 a bad position, 3 a bad index, 4 a bad page,
 * 5 tensor memory unavailable).
 */
dsa_status_t dsa_device_error(void *stream, uint32_t *code);

/*
 * Diagnostics, not part of the method: checks on the device that a kernel's bounded wait
 * ends a broken pipeline instead of hanging it.  Launches one CTA whose two waiters wait,
 * through the same bounded wait every libdsa pipeline uses, on a barrier that nothing
 * completes: the first gives up after the time limit (about two seconds), records
 * (8 << 16 | 1) in the device error word and stops the other, which gives up at once.
 * `result` (device, 8-byte aligned, 4 x uint64_t, written by the kernel): per waiter
 * whether its barrier completed (expected 0), then how long each waited in nanoseconds.
 * Nothing faults; afterwards dsa_device_error() returns DSA_ERR_DEVICE with that code
 * and clears it, and the device is usable as before.
 */
dsa_status_t dsa_wait_probe(uint64_t *result, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* DSA_H */
