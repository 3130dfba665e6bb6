// internal.h -- launch parameters shared by the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>
#include <utility>

#include "dsa.h"

namespace dsa {

// Launch `kernel` with programmatic dependent launch enabled (see ptx.cuh) and the largest
// shared-memory carveout, so that consecutive kernels of a step overlap their launch.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kernel)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Kernel attributes: dynamic shared memory limit and carveout.
template <typename K>
cudaError_t set_smem_attrs(K kernel, int bytes) {
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
}

// Function attributes belong to a device, so what a kernel has been given is remembered
// per device (the largest request so far); the mutex makes concurrent first calls from
// several host threads safe.  One AttrCache per kernel (instantiation).
constexpr int kMaxDevices = 64;
struct AttrCache {
    std::mutex mu;
    int bytes[kMaxDevices] = {};
};

template <typename K>
cudaError_t ensure_smem_attrs(AttrCache &cache, K kernel, int bytes) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(cache.mu);
    if (cache.bytes[dev] >= bytes) return cudaSuccess;
    e = set_smem_attrs(kernel, bytes);
    if (e != cudaSuccess) return e;
    cache.bytes[dev] = bytes;
    return cudaSuccess;
}

// Read and clear the device error word of each kernel file (0: no error;
// 0xFFFFFFFF: the read itself failed).
uint32_t take_error_indexer();
uint32_t take_error_topk();
uint32_t take_error_mla();
uint32_t take_error_append();

// How token s of sequence b maps to a physical cache row (see dsa_cache_layout_t).
struct CacheLayout {
    const int32_t *seq_start;
    const int32_t *block_table;
    int32_t page_size;
    int32_t pages_per_seq;
    int64_t num_rows;
};

// ---- lightning indexer ------------------------------------------------------------
struct IndexerParams {
    const uint8_t *q8;
    const float *q_scale;
    const float *w;
    const float *k_scale;
    const int32_t *q_pos;
    float *scores;
    CacheLayout layout;
    int B, T, Hi, Di, Lmax;
    int HP;        // heads per query padded to a multiple of 16
    int G;         // query rows per tensor-core group (N = G * HP)
    int N;         // MMA N
    int groups_per_seq;
    int num_groups;
    int acc_cols;  // TMEM columns per accumulator buffer
    int num_acc;   // accumulator buffers
    int stages;    // key pipeline depth
    int q_tma;     // 1: query groups load by TMA (Hi == HP), 0: plain loads with padding
    // fused selection (dsa_indexer_topk): instead of storing scores, each row keeps the
    // candidates that can still be among its k best in cand[row * cap ..] as
    // (full key, token index), in four quarters of cap / 4 slots (one per epilogue warp),
    // and, at the end of its query group, meta[2 row] = the quarters' counts and
    // meta[2 row + 1] = {final coarse bin B0, count above B0, count in B0, 0}
    int sel;       // 1: fused selection
    int k;
    int64_t cap;   // candidate slots per row (>= Lmax)
    uint2 *cand;
    uint4 *meta;
};

// kmap: 64-row key boxes (any layout); kmap128: 128-row boxes (contiguous runs);
// qmap: query codes as [rows * Hi, Di] with N-row boxes (used when q_tma)
cudaError_t launch_indexer(const IndexerParams &p, const CUtensorMap &kmap,
                           const CUtensorMap &kmap128, const CUtensorMap &qmap, int num_sms,
                           cudaStream_t stream);

// ---- top-k ------------------------------------------------------------------------
struct TopkParams {
    const float *scores;
    const int32_t *q_pos;
    int32_t *idx;
    int rows, Lmax, k;
};

cudaError_t launch_topk(const TopkParams &p, int num_sms, cudaStream_t stream);
// Whether rows of Lmax scores fit the cluster top-k (the slices of a cluster of the largest
// size in shared memory): Lmax <= 375040.
bool topk_lmax_supported(int Lmax);

// The final selection of the fused indexer + top-k: per row, from the candidates and the
// counts the fused indexer left in cand / meta.
struct TopkCandParams {
    const uint2 *cand;
    const uint4 *meta;
    const int32_t *q_pos;
    int32_t *idx;
    int rows, Lmax, k;
    int64_t cap;
};
cudaError_t launch_topk_cand(const TopkCandParams &p, cudaStream_t stream);

// ---- sparse MLA -------------------------------------------------------------------
constexpr int kMaxLayers = 8;

struct MlaParams {
    const uint16_t *q[kMaxLayers];
    const uint16_t *kv[kMaxLayers];
    uint16_t *out[kMaxLayers];
    float *lse[kMaxLayers];
    const int32_t *idx;
    CacheLayout layout;
    float *partial;    // split-KV partials (workspace), or nullptr when splits == 1
    int layers, B, T, H, d, r, k;
    float scale_log2;  // softmax scale * log2(e)
    int splits;        // key splits per (row, layer)
    int tiles_per_split;
    int cluster;       // 1: the splits of a (row, layer) form a thread-block cluster and
                       // merge their partial results through the workspace
    // top-k in the same launch (decode): the splits of each row first select the row's
    // index set from `scores` (the row's cluster runs the cluster top-k, slices of
    // topk_slice scores) and write it to idx_out (= idx), then attend over it
    int topk;
    int topk_slice;
    const float *scores;
    const int32_t *q_pos;
    int Lmax;
    int32_t *idx_out;
};

// TMA descriptors of every layer: q viewed as [rows*H, d+r], kv as [num_rows, d+r] (bf16)
struct MlaMaps {
    CUtensorMap q[kMaxLayers];
    CUtensorMap kv[kMaxLayers];
};

int mla_tile_keys();  // keys per sparse MLA tile (the split unit)
// Key splits per (row, layer) and tiles per split for `rows` query rows of one layer.
void mla_split_plan(int rows, int k, int num_sms, int d, int *splits, int *tiles_per_split);
size_t mla_partial_bytes(int rows_times_layers, int splits, int d);
cudaError_t launch_sparse_mla(const MlaParams &p, const MlaMaps &maps, cudaStream_t stream);
// The slice size (scores per CTA) at which a row's top-k can run inside the sparse MLA
// kernel with `splits` CTAs per row for latent width d, or 0 when it cannot (no cluster
// for the splits, or the slice does not fit the kernel's tile buffers).
int mla_topk_slice(int Lmax, int splits, int d);

// ---- MLA in MHA mode -------------------------------------------------------------------
struct MhaParams {
    const int32_t *q_pos;      // [B*T]
    const int32_t *seq_start;  // [B] first cache row of each sequence (contiguous layout)
    uint32_t *bitmap;          // [B*T, words] selection bitmaps (workspace)
    uint16_t *out;             // [B*T, H, vd] bf16
    float *lse;                // [B*T, H] or nullptr
    int B, T, H, d, r, dn, dq, vd, k, Lmax, words;
    float scale_log2;
};
// out[n, N] = X[n, :d] . W[N, d]^T (xmap: X as [n, ld] with 64 x 128 boxes; wmap: W as [N, d])
cudaError_t launch_upproj(const CUtensorMap &xmap, const CUtensorMap &wmap, uint16_t *out, int n,
                          int N, int d, cudaStream_t stream);
// qmap: q as [B*T, H*dq]; kmap: k_up as [rows, H*dn]; rmap: the latent cache as [rows, d+r];
// vmap: v_up as [rows, H*vd]; all with 64 x 128 boxes, 128-byte swizzle
cudaError_t launch_mha(const MhaParams &p, const CUtensorMap &qmap, const CUtensorMap &kmap,
                       const CUtensorMap &rmap, const CUtensorMap &vmap, const int32_t *idx,
                       cudaStream_t stream);
uint32_t take_error_mha();

// ---- host-tier working set (HiSparse) ----------------------------------------------------
constexpr int kMaxHiSlots = 16384;  // device slots per sequence
constexpr int kMaxHiK = 8192;       // index-row length
struct HiParams {
    const int32_t *idx;             // [B, k] this step's selection (-1 skipped)
    const uint16_t *host_kv;        // device-accessible pointer to the host cache [rows, D]
    const int32_t *host_seq_start;  // [B] first host row of each sequence
    int32_t *residency;             // [B, Lmax] global pool row of each token, or -1
    int32_t *slot_token;            // [B, C] token in each slot, or -1
    uint32_t *slot_use;             // [B, C] last step each slot was used (0: never)
    uint16_t *pool;                 // [B * C, D] device working set
    int32_t *stats;                 // [B, 2] hits, misses (nullable)
    uint32_t step;
    int B, k, Lmax, C, D;
};
cudaError_t launch_hisparse_fetch(const HiParams &p, cudaStream_t stream);
cudaError_t launch_hisparse_init(int32_t *residency, int64_t n_res, int32_t *slot_token,
                                 uint32_t *slot_use, int64_t n_slots, cudaStream_t stream);
uint32_t take_error_hisparse();

// ---- cache append: new tokens' indexer keys (quantised) and latent rows into the caches
struct AppendParams {
    const float *k_new;     // [n, Di] fp32
    const uint16_t *c_new;  // [n, D] bf16, or nullptr: indexer keys only
    const int32_t *seq;     // [n] sequence of each token
    const int32_t *pos;     // [n] position of each token in its sequence
    CacheLayout layout;
    uint8_t *k8_cache;      // [num_rows, Di] e4m3 codes
    float *k_scale;         // [num_rows]
    uint16_t *kv_cache;     // [num_rows, D] bf16, or nullptr with c_new
    int n, B, Di, D;
};
cudaError_t launch_cache_append(const AppendParams &p, cudaStream_t stream);

// ---- diagnostics: a bounded wait that runs out on purpose ---------------------------------
cudaError_t launch_wait_probe(unsigned long long *out, cudaStream_t stream);
uint32_t take_error_probe();

}  // namespace dsa
