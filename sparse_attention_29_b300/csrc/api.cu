// api.cu -- the C ABI of libdsa: argument checks on the host, tensor-map set-up, launch.
//
// Every entry point validates its arguments before it launches anything and returns a
// dsa_status_t; no C++ exception crosses the ABI.
#include <cudaTypedefs.h>
#include <nvtx3/nvToolsExt.h>

#include <cstdio>
#include <cstring>
#include <mutex>

#include "internal.h"
#include "ptx.cuh"

using namespace dsa;

namespace {

#define DSA_VERSION_STRING "libdsa 0.1.0 (sm_103a)"

// One NVTX range per C-ABI call that launches work, named after the entry point, so that
// a timeline tool shows which call launched which kernels.  With no tool attached a range
// costs a check of a function pointer.
struct CallRange {
    explicit CallRange(const char *name) { nvtxRangePushA(name); }
    ~CallRange() { nvtxRangePop(); }
    CallRange(const CallRange &) = delete;
    CallRange &operator=(const CallRange &) = delete;
};
#define DSA_CALL_RANGE() const CallRange dsa_call_range_(__func__)

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

dsa_status_t from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return DSA_OK;
    (void)cudaGetLastError();
    return DSA_ERR_CUDA;
}

int current_sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

PFN_cuTensorMapEncodeTiled_v12000 get_encode_tiled() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

bool layout_ok(const dsa_cache_layout_t *L, int B, bool need_page64) {
    if (!L || L->num_rows <= 0) return false;
    if (L->block_table) {
        if (L->page_size <= 0 || L->pages_per_seq <= 0) return false;
        if (need_page64 && (L->page_size % 64) != 0) return false;
    } else if (!L->seq_start) {
        return false;
    }
    (void)B;
    return true;
}

CacheLayout to_layout(const dsa_cache_layout_t *L) {
    CacheLayout c;
    c.seq_start = L->seq_start;
    c.block_table = L->block_table;
    c.page_size = L->page_size;
    c.pages_per_seq = L->pages_per_seq;
    c.num_rows = L->num_rows;
    return c;
}

int pow2_at_least(int x) {
    int p = 32;
    while (p < x) p <<= 1;
    return p;
}

// fused top-k (decode): the row's scores, positions and score-row length; idx is written
struct FusedTopk {
    const float *scores;
    const int32_t *q_pos;
    int Lmax;
};

dsa_status_t mla_common(const uint16_t *const *q, const uint16_t *const *kv, int n_layers,
                        const dsa_cache_layout_t *layout, const int32_t *idx, int B, int T,
                        int H, int d, int r, int k, float scale, uint16_t *const *out,
                        float *const *lse, void *workspace, size_t workspace_bytes,
                        void *stream, const FusedTopk *ft = nullptr) {
    if (n_layers < 1 || n_layers > kMaxLayers) return DSA_ERR_INVALID_ARG;
    if (!q || !kv || !out || !idx || !layout) return DSA_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || H <= 0 || d <= 0 || r < 0 || k <= 0) return DSA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || scale != scale) return DSA_ERR_INVALID_ARG;
    if (H > 64 || d % 64 != 0 || d > 512 || r > 64 || (d + r) % 8 != 0 || k > 8192)
        return DSA_ERR_UNSUPPORTED;
    if ((int64_t)B * T * n_layers > (int64_t)1 << 30) return DSA_ERR_UNSUPPORTED;
    if ((int64_t)B * T * H >= ((int64_t)1 << 31) - 64) return DSA_ERR_UNSUPPORTED;
    if (layout && layout->num_rows >= ((int64_t)1 << 31) - 64) return DSA_ERR_UNSUPPORTED;
    if (!layout_ok(layout, B, false)) return DSA_ERR_INVALID_ARG;
    MlaParams p;
    std::memset(&p, 0, sizeof p);
    for (int g = 0; g < n_layers; ++g) {
        if (!q[g] || !kv[g] || !out[g]) return DSA_ERR_INVALID_ARG;
        if (!aligned16(q[g]) || !aligned16(kv[g]) || !aligned16(out[g])) return DSA_ERR_INVALID_ARG;
        p.q[g] = q[g];
        p.kv[g] = kv[g];
        p.out[g] = out[g];
        p.lse[g] = lse ? lse[g] : nullptr;
    }
    p.idx = idx;
    p.layout = to_layout(layout);
    p.layers = n_layers;
    p.B = B;
    p.T = T;
    p.H = H;
    p.d = d;
    p.r = r;
    p.k = k;
    p.scale_log2 = scale * 1.4426950408889634f;
    const int sms = current_sm_count();
    if (sms <= 0) return DSA_ERR_CUDA;
    const int units = B * T * n_layers;
    // the split of a row's keys is planned for the whole launch (every layer's rows), so an
    // IndexShare group fills the GPU as one launch: with few rows per layer its rows split
    // less than a single layer's would (its layers' outputs then differ from separate
    // per-layer calls by the rounding of the split merge)
    mla_split_plan(units, k, sms, d, &p.splits, &p.tiles_per_split);
    const size_t need = mla_partial_bytes(units, p.splits, d);
    if (need) {
        if (!workspace || workspace_bytes < need) return DSA_ERR_WORKSPACE;
        if (!aligned16(workspace)) return DSA_ERR_INVALID_ARG;
        p.partial = static_cast<float *>(workspace);
    }
    // TMA descriptors: q as [rows*H, D] (64-row x 64-column boxes), kv as [num_rows, D]
    // (one-row boxes for gather4), bf16, 128-byte swizzle
    if (ft) {
        // the row's splits select its index set first when they form one cluster (or are
        // one CTA) and the row's scores fit their tile buffers; otherwise a separate top-k
        // launch comes first
        const int slice = n_layers == 1 ? mla_topk_slice(ft->Lmax, p.splits, d) : 0;
        if (slice > 0) {
            p.topk = 1;
            p.topk_slice = slice;
            p.scores = ft->scores;
            p.q_pos = ft->q_pos;
            p.Lmax = ft->Lmax;
            p.idx_out = const_cast<int32_t *>(idx);
        } else {
            TopkParams tp;
            tp.scores = ft->scores;
            tp.q_pos = ft->q_pos;
            tp.idx = const_cast<int32_t *>(idx);
            tp.rows = B * T;
            tp.Lmax = ft->Lmax;
            tp.k = k;
            const cudaError_t e = launch_topk(tp, sms, static_cast<cudaStream_t>(stream));
            if (e != cudaSuccess) return from_cuda(e);
        }
    }
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_tiled();
    if (!encode) return DSA_ERR_CUDA;
    MlaMaps maps;
    std::memset(&maps, 0, sizeof maps);
    const int D = d + r;
    for (int g = 0; g < n_layers; ++g) {
        const cuuint64_t qdims[2] = {(cuuint64_t)D, (cuuint64_t)B * T * H};
        const cuuint64_t kdims[2] = {(cuuint64_t)D, (cuuint64_t)layout->num_rows};
        const cuuint64_t strides[1] = {(cuuint64_t)D * 2};
        const cuuint32_t qbox[2] = {64, 64};
        const cuuint32_t kbox[2] = {64, 1};
        const cuuint32_t estr[2] = {1, 1};
        CUresult c1 = encode(&maps.q[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                             const_cast<uint16_t *>(q[g]), qdims, strides, qbox, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        CUresult c2 = encode(&maps.kv[g], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2,
                             const_cast<uint16_t *>(kv[g]), kdims, strides, kbox, estr,
                             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (c1 != CUDA_SUCCESS || c2 != CUDA_SUCCESS) return DSA_ERR_CUDA;
    }
    return from_cuda(launch_sparse_mla(p, maps, static_cast<cudaStream_t>(stream)));
}

// ---- fixed scratch of dsa_sparse_mla_decode_noalloc ---------------------------------------
// Callers that cannot allocate device memory on the decode path (a plain C host with no
// device allocator, a serving loop whose memory is all handed out up front) get the
// split-KV partials from this array instead of a workspace.  It is part of the module's
// static storage: nothing here calls cudaMalloc or cudaFree.  The partials need no
// zeroing (each call writes every partial before the combine reads it); overlapping
// calls on one device share it and race.
static __device__ __align__(256) float g_noalloc_scratch[DSA_NOALLOC_SCRATCH_BYTES / sizeof(float)];

// per device: the array's address and the context it was looked up in
struct NoallocAddr {
    CUcontext ctx;
    void *addr;
};
NoallocAddr g_noalloc_addr[dsa::kMaxDevices];
std::mutex g_noalloc_mutex;

PFN_cuCtxGetCurrent_v4000 get_ctx_current() {
    static PFN_cuCtxGetCurrent_v4000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(p);
    });
    return fn;
}

// Address of the array on the current device.  The first call per device looks it up;
// the address belongs to the context it was taken in (the device's primary context), so
// it is looked up again if that context has been replaced (after a device reset).
dsa_status_t noalloc_scratch(void **ptr) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    if (dev < 0 || dev >= dsa::kMaxDevices) return DSA_ERR_UNSUPPORTED;
    PFN_cuCtxGetCurrent_v4000 ctx_current = get_ctx_current();
    if (!ctx_current) return DSA_ERR_CUDA;
    CUcontext ctx = nullptr;  // NULL until a runtime call has bound this thread's context
    if (ctx_current(&ctx) != CUDA_SUCCESS) return DSA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocAddr &a = g_noalloc_addr[dev];
    if (!a.addr || !ctx || a.ctx != ctx) {
        void *p = nullptr;
        // binds the device's primary context to this thread (and loads the module) if needed
        const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
        if (e != cudaSuccess || !p) return from_cuda(e != cudaSuccess ? e : cudaErrorUnknown);
        if (ctx_current(&ctx) != CUDA_SUCCESS || !ctx) return DSA_ERR_CUDA;
        a.addr = p;
        a.ctx = ctx;
    }
    *ptr = a.addr;
    return DSA_OK;
}

}  // namespace

extern "C" {

const char *dsa_version(void) { return DSA_VERSION_STRING; }

const char *dsa_status_string(dsa_status_t s) {
    switch (s) {
        case DSA_OK: return "ok";
        case DSA_ERR_INVALID_ARG: return "invalid argument";
        case DSA_ERR_UNSUPPORTED: return "unsupported shape";
        case DSA_ERR_CUDA: return "CUDA error";
        case DSA_ERR_WORKSPACE: return "workspace missing or too small";
        case DSA_ERR_DEVICE: return "device-side check failed";
        case DSA_ERR_SCRATCH_LIMIT: return "shape needs more than the fixed no-allocation scratch";
    }
    return "unknown status";
}

}  // extern "C"

namespace {

// Shared by the indexer entry points: checks, launch parameters and tensor maps, launch.
dsa_status_t indexer_common(const uint8_t *q8, const float *q_scale, const float *w,
                            const uint8_t *k8_cache, const float *k_scale,
                            const dsa_cache_layout_t *layout, const int32_t *q_pos, int B,
                            int T, int Hi, int Di, int Lmax, float *scores, int k,
                            uint2 *cand, int64_t cap, uint4 *meta, void *stream) {
    const bool sel = cand != nullptr;
    if (!q8 || !q_scale || !w || !k8_cache || !k_scale || !q_pos || (!sel && !scores))
        return DSA_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || Hi <= 0 || Di <= 0 || Lmax <= 0) return DSA_ERR_INVALID_ARG;
    if (Di != 32 && Di != 64 && Di != 128) return DSA_ERR_UNSUPPORTED;
    const int HP = (Hi + 15) / 16 * 16;
    if (HP > 256) return DSA_ERR_UNSUPPORTED;
    if (sel && HP != 64) return DSA_ERR_UNSUPPORTED;  // four 64-head rows per tile
    if (!aligned16(q8) || !aligned16(k8_cache)) return DSA_ERR_INVALID_ARG;
    if (!layout_ok(layout, B, true)) return DSA_ERR_INVALID_ARG;
    if ((int64_t)layout->num_rows >= ((int64_t)1 << 31) - 256) return DSA_ERR_UNSUPPORTED;
    IndexerParams p;
    std::memset(&p, 0, sizeof p);
    p.q8 = q8;
    p.q_scale = q_scale;
    p.w = w;
    p.k_scale = k_scale;
    p.q_pos = q_pos;
    p.scores = scores;
    p.layout = to_layout(layout);
    p.B = B;
    p.T = T;
    p.Hi = Hi;
    p.Di = Di;
    p.Lmax = Lmax;
    p.HP = HP;
    p.G = 256 / HP;
    if (p.G > T) p.G = T;
    if (p.G > 16) p.G = 16;
    p.N = p.G * HP;
    p.groups_per_seq = (T + p.G - 1) / p.G;
    const int64_t ng = (int64_t)B * p.groups_per_seq;
    if (ng > 16384) return DSA_ERR_UNSUPPORTED;
    p.num_groups = (int)ng;
    p.acc_cols = pow2_at_least(p.N);
    p.num_acc = 512 / p.acc_cols;  // every TMEM column: the MMA never waits on the epilogue
    if (p.num_acc > 8) p.num_acc = 8;
    p.sel = sel ? 1 : 0;
    p.k = k;
    p.cap = cap;
    p.cand = cand;
    p.meta = meta;

    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_tiled();
    if (!encode) return DSA_ERR_CUDA;
    CUtensorMap kmap, kmap128;
    const cuuint64_t dims[2] = {(cuuint64_t)Di, (cuuint64_t)layout->num_rows};
    const cuuint64_t strides[1] = {(cuuint64_t)Di};
    const cuuint32_t box[2] = {(cuuint32_t)Di, 64};
    const cuuint32_t box128[2] = {(cuuint32_t)Di, 128};
    const cuuint32_t estr[2] = {1, 1};
    const CUtensorMapSwizzle sw = Di == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                                  : Di == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                             : CU_TENSOR_MAP_SWIZZLE_32B;
    CUresult cr = encode(&kmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(k8_cache),
                         dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    CUresult cr2 = encode(&kmap128, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                          const_cast<uint8_t *>(k8_cache), dims, strides, box128, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (cr != CUDA_SUCCESS || cr2 != CUDA_SUCCESS) return DSA_ERR_CUDA;
    // query codes: one box of N rows = G query rows x Hi heads (needs Hi == HP)
    CUtensorMap qmap;
    std::memset(&qmap, 0, sizeof qmap);
    p.q_tma = (Hi == HP) ? 1 : 0;
    if (p.q_tma) {
        if ((int64_t)B * T * Hi >= ((int64_t)1 << 31) - 256) return DSA_ERR_UNSUPPORTED;
        const cuuint64_t qdims[2] = {(cuuint64_t)Di, (cuuint64_t)B * T * Hi};
        const cuuint32_t qbox[2] = {(cuuint32_t)Di, (cuuint32_t)p.N};
        CUresult cr3 = encode(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<uint8_t *>(q8),
                              qdims, strides, qbox, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
        if (cr3 != CUDA_SUCCESS) return DSA_ERR_CUDA;
    }
    const int sms = current_sm_count();
    if (sms <= 0) return DSA_ERR_CUDA;
    return from_cuda(launch_indexer(p, kmap, kmap128, qmap, sms, static_cast<cudaStream_t>(stream)));
}

// Workspace of dsa_indexer_topk: candidate lists (Lmax rounded up to a multiple of 128
// slots of 8 bytes per row: four quarters, one per epilogue warp, each holding the 32 of
// every 128 keys that warp scores), then per-row counts (32 bytes per row).
int64_t cand_slots(int Lmax) { return ((int64_t)Lmax + 127) / 128 * 128; }

}  // namespace

extern "C" {

dsa_status_t dsa_indexer_scores(const uint8_t *q8, const float *q_scale, const float *w,
                                const uint8_t *k8_cache, const float *k_scale,
                                const dsa_cache_layout_t *layout, const int32_t *q_pos,
                                int B, int T, int Hi, int Di, int Lmax, float *scores,
                                void *stream) {
    DSA_CALL_RANGE();
    return indexer_common(q8, q_scale, w, k8_cache, k_scale, layout, q_pos, B, T, Hi, Di, Lmax,
                          scores, 0, nullptr, 0, nullptr, stream);
}

size_t dsa_indexer_topk_workspace_bytes(int B, int T, int Lmax) {
    if (B <= 0 || T <= 0 || Lmax <= 0) return (size_t)-1;
    const int64_t rows = (int64_t)B * T;
    return (size_t)(rows * cand_slots(Lmax) * 8 + rows * 32);
}

dsa_status_t dsa_indexer_topk(const uint8_t *q8, const float *q_scale, const float *w,
                              const uint8_t *k8_cache, const float *k_scale,
                              const dsa_cache_layout_t *layout, const int32_t *q_pos, int B,
                              int T, int Hi, int Di, int Lmax, int k, int32_t *idx,
                              void *workspace, size_t workspace_bytes, void *stream) {
    DSA_CALL_RANGE();
    if (!idx || !workspace) return DSA_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || Lmax <= 0 || k <= 0) return DSA_ERR_INVALID_ARG;
    if (k > 8192) return DSA_ERR_UNSUPPORTED;
    const size_t need = dsa_indexer_topk_workspace_bytes(B, T, Lmax);
    if (workspace_bytes < need) return DSA_ERR_WORKSPACE;
    if (!aligned16(workspace)) return DSA_ERR_INVALID_ARG;
    const int64_t rows = (int64_t)B * T;
    const int64_t cap = cand_slots(Lmax);
    uint2 *cand = static_cast<uint2 *>(workspace);
    uint4 *meta = reinterpret_cast<uint4 *>(cand + rows * cap);
    dsa_status_t st = indexer_common(q8, q_scale, w, k8_cache, k_scale, layout, q_pos, B, T, Hi,
                                     Di, Lmax, nullptr, k, cand, cap, meta, stream);
    if (st != DSA_OK) return st;
    TopkCandParams tp;
    tp.cand = cand;
    tp.meta = meta;
    tp.q_pos = q_pos;
    tp.idx = idx;
    tp.rows = (int)rows;
    tp.Lmax = Lmax;
    tp.k = k;
    tp.cap = cap;
    return from_cuda(launch_topk_cand(tp, static_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_topk(const float *scores, const int32_t *q_pos, int rows, int Lmax, int k,
                      int32_t *idx, void *stream) {
    DSA_CALL_RANGE();
    if (!scores || !q_pos || !idx) return DSA_ERR_INVALID_ARG;
    if (rows <= 0 || Lmax <= 0 || k <= 0) return DSA_ERR_INVALID_ARG;
    if (k > 8192 || !topk_lmax_supported(Lmax)) return DSA_ERR_UNSUPPORTED;
    TopkParams p;
    p.scores = scores;
    p.q_pos = q_pos;
    p.idx = idx;
    p.rows = rows;
    p.Lmax = Lmax;
    p.k = k;
    const int sms = current_sm_count();
    if (sms <= 0) return DSA_ERR_CUDA;
    return from_cuda(launch_topk(p, sms, static_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_sparse_mla_decode(const uint16_t *q, const uint16_t *kv_cache,
                                   const dsa_cache_layout_t *layout, const int32_t *idx,
                                   int B, int H, int d, int r, int k, float scale,
                                   uint16_t *out, float *lse, void *workspace,
                                   size_t workspace_bytes, void *stream) {
    DSA_CALL_RANGE();
    return mla_common(&q, &kv_cache, 1, layout, idx, B, 1, H, d, r, k, scale, &out,
                      lse ? &lse : nullptr, workspace, workspace_bytes, stream);
}

dsa_status_t dsa_topk_sparse_mla_decode(const float *scores, const int32_t *q_pos, int Lmax,
                                        const uint16_t *q, const uint16_t *kv_cache,
                                        const dsa_cache_layout_t *layout, int32_t *idx, int B,
                                        int H, int d, int r, int k, float scale, uint16_t *out,
                                        float *lse, void *workspace, size_t workspace_bytes,
                                        void *stream) {
    DSA_CALL_RANGE();
    if (!scores || !q_pos || !idx) return DSA_ERR_INVALID_ARG;
    if (Lmax <= 0) return DSA_ERR_INVALID_ARG;
    if (!topk_lmax_supported(Lmax)) return DSA_ERR_UNSUPPORTED;
    FusedTopk ft;
    ft.scores = scores;
    ft.q_pos = q_pos;
    ft.Lmax = Lmax;
    return mla_common(&q, &kv_cache, 1, layout, idx, B, 1, H, d, r, k, scale, &out,
                      lse ? &lse : nullptr, workspace, workspace_bytes, stream, &ft);
}

dsa_status_t dsa_sparse_mla_decode_noalloc(const uint16_t *q, const uint16_t *kv_cache,
                                           const dsa_cache_layout_t *layout,
                                           const int32_t *idx, int B, int H, int d, int r,
                                           int k, float scale, uint16_t *out, float *lse,
                                           void *stream) {
    DSA_CALL_RANGE();
    void *scratch = nullptr;
    const dsa_status_t st = noalloc_scratch(&scratch);
    if (st != DSA_OK) return st;
    const size_t need = dsa_workspace_bytes(DSA_OP_SPARSE_MLA, B, 1, H, d, k, 1);
    if (need != (size_t)-1 && need > DSA_NOALLOC_SCRATCH_BYTES) return DSA_ERR_SCRATCH_LIMIT;
    // invalid shapes (need == -1) are rejected by the shared checks before any use
    return mla_common(&q, &kv_cache, 1, layout, idx, B, 1, H, d, r, k, scale, &out,
                      lse ? &lse : nullptr, scratch, DSA_NOALLOC_SCRATCH_BYTES, stream);
}

dsa_status_t dsa_sparse_mla_prefill(const uint16_t *q, const uint16_t *kv_cache,
                                    const dsa_cache_layout_t *layout, const int32_t *idx,
                                    int B, int T, int H, int d, int r, int k, float scale,
                                    uint16_t *out, float *lse, void *workspace,
                                    size_t workspace_bytes, void *stream) {
    DSA_CALL_RANGE();
    return mla_common(&q, &kv_cache, 1, layout, idx, B, T, H, d, r, k, scale, &out,
                      lse ? &lse : nullptr, workspace, workspace_bytes, stream);
}

dsa_status_t dsa_sparse_mla_shared(const uint16_t *const *q_layers,
                                   const uint16_t *const *kv_layers, int n_layers,
                                   const dsa_cache_layout_t *layout, const int32_t *idx,
                                   int B, int T, int H, int d, int r, int k, float scale,
                                   uint16_t *const *out_layers, float *const *lse_layers,
                                   void *workspace, size_t workspace_bytes, void *stream) {
    DSA_CALL_RANGE();
    return mla_common(q_layers, kv_layers, n_layers, layout, idx, B, T, H, d, r, k, scale,
                      out_layers, lse_layers, workspace, workspace_bytes, stream);
}

size_t dsa_workspace_bytes(dsa_op_t op, int B, int T, int H, int d, int k, int n_layers) {
    if (B <= 0 || T <= 0 || k <= 0) return (size_t)-1;
    if (op == DSA_OP_INDEXER || op == DSA_OP_TOPK) return 0;
    if (op != DSA_OP_SPARSE_MLA) return (size_t)-1;
    if (H <= 0 || H > 64 || d <= 0 || d % 64 != 0 || n_layers < 1 || n_layers > kMaxLayers)
        return (size_t)-1;
    const int sms = current_sm_count();
    if (sms <= 0) return (size_t)-1;
    const int units = B * T * n_layers;
    int splits = 1, tps = 1;
    mla_split_plan(units, k, sms, d, &splits, &tps);
    return mla_partial_bytes(units, splits, d);
}

dsa_status_t dsa_cache_append(const float *k_new, const uint16_t *c_new, const int32_t *seq,
                              const int32_t *pos, int n, int B, int Di, int D,
                              const dsa_cache_layout_t *layout, uint8_t *k8_cache,
                              float *k_scale, uint16_t *kv_cache, void *stream) {
    DSA_CALL_RANGE();
    if (n < 0 || B <= 0) return DSA_ERR_INVALID_ARG;
    if (Di != 32 && Di != 64 && Di != 128) return DSA_ERR_UNSUPPORTED;
    if (n == 0) return DSA_OK;  // nothing to append (the arrays may be NULL)
    if (!k_new || !seq || !pos || !k8_cache || !k_scale) return DSA_ERR_INVALID_ARG;
    if ((c_new == nullptr) != (kv_cache == nullptr)) return DSA_ERR_INVALID_ARG;
    if (c_new && (D <= 0 || D % 8 != 0)) return DSA_ERR_INVALID_ARG;
    if (!aligned16(k_new) || !aligned16(k8_cache)) return DSA_ERR_INVALID_ARG;
    if (c_new && (!aligned16(c_new) || !aligned16(kv_cache))) return DSA_ERR_INVALID_ARG;
    if (!layout_ok(layout, B, false)) return DSA_ERR_INVALID_ARG;
    AppendParams p;
    p.k_new = k_new;
    p.c_new = c_new;
    p.seq = seq;
    p.pos = pos;
    p.layout = to_layout(layout);
    p.k8_cache = k8_cache;
    p.k_scale = k_scale;
    p.kv_cache = kv_cache;
    p.n = n;
    p.B = B;
    p.Di = Di;
    p.D = c_new ? D : 0;
    return from_cuda(launch_cache_append(p, static_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_hisparse_init(int32_t *residency, int B, int Lmax, int32_t *slot_token,
                               uint32_t *slot_use, int C, void *stream) {
    DSA_CALL_RANGE();
    if (!residency || !slot_token || !slot_use) return DSA_ERR_INVALID_ARG;
    if (B <= 0 || Lmax <= 0 || C <= 0) return DSA_ERR_INVALID_ARG;
    if (C > kMaxHiSlots) return DSA_ERR_UNSUPPORTED;
    return from_cuda(launch_hisparse_init(residency, (int64_t)B * Lmax, slot_token, slot_use,
                                          (int64_t)B * C, static_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_hisparse_fetch(const int32_t *idx, int B, int k, uint32_t step,
                                const uint16_t *host_kv, const int32_t *host_seq_start, int D,
                                int32_t *residency, int Lmax, int32_t *slot_token,
                                uint32_t *slot_use, int C, uint16_t *pool, int32_t *stats,
                                void *stream) {
    DSA_CALL_RANGE();
    if (!idx || !host_kv || !host_seq_start || !residency || !slot_token || !slot_use || !pool)
        return DSA_ERR_INVALID_ARG;
    if (B <= 0 || k <= 0 || Lmax <= 0 || C <= 0 || D <= 0 || step == 0) return DSA_ERR_INVALID_ARG;
    if (D % 8 != 0 || !aligned16(host_kv) || !aligned16(pool)) return DSA_ERR_INVALID_ARG;
    if (k > kMaxHiK || C > kMaxHiSlots) return DSA_ERR_UNSUPPORTED;
    if (C < k) return DSA_ERR_INVALID_ARG;  // a step's selection must fit the working set
    if ((int64_t)B * C >= ((int64_t)1 << 31)) return DSA_ERR_UNSUPPORTED;
    // the kernel reads host_kv directly: it must be pinned host memory mapped at this very
    // address (or device memory); anything else is refused before a launch could fault
    cudaPointerAttributes pa;
    if (cudaPointerGetAttributes(&pa, host_kv) != cudaSuccess) {
        (void)cudaGetLastError();
        return DSA_ERR_INVALID_ARG;
    }
    const bool mapped_host = pa.type == cudaMemoryTypeHost && pa.devicePointer == host_kv;
    const bool on_device = pa.type == cudaMemoryTypeDevice || pa.type == cudaMemoryTypeManaged;
    if (!mapped_host && !on_device) return DSA_ERR_INVALID_ARG;
    HiParams p;
    p.idx = idx;
    p.host_kv = host_kv;
    p.host_seq_start = host_seq_start;
    p.residency = residency;
    p.slot_token = slot_token;
    p.slot_use = slot_use;
    p.pool = pool;
    p.stats = stats;
    p.step = step;
    p.B = B;
    p.k = k;
    p.Lmax = Lmax;
    p.C = C;
    p.D = D;
    return from_cuda(launch_hisparse_fetch(p, static_cast<cudaStream_t>(stream)));
}

static bool encode_bf16_2d(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows) {
    PFN_cuTensorMapEncodeTiled_v12000 encode = get_encode_tiled();
    if (!encode) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
    const cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
    const cuuint32_t box[2] = {64, 128};
    const cuuint32_t estr[2] = {1, 1};
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

dsa_status_t dsa_mla_up_project(const uint16_t *latent, int64_t n, int ld, int d,
                                const uint16_t *w, int N, uint16_t *out, void *stream) {
    DSA_CALL_RANGE();
    if (!latent || !w || !out) return DSA_ERR_INVALID_ARG;
    if (n <= 0 || ld <= 0 || d <= 0 || N <= 0 || d > ld) return DSA_ERR_INVALID_ARG;
    if (d % 64 != 0 || N % 128 != 0 || ld % 8 != 0) return DSA_ERR_UNSUPPORTED;
    if (n >= ((int64_t)1 << 31) - 128 || (int64_t)N * 2 >= ((int64_t)1 << 31)) return DSA_ERR_UNSUPPORTED;
    if (!aligned16(latent) || !aligned16(w) || !aligned16(out)) return DSA_ERR_INVALID_ARG;
    CUtensorMap xmap, wmap;
    if (!encode_bf16_2d(&xmap, latent, (uint64_t)ld, (uint64_t)n) ||
        !encode_bf16_2d(&wmap, w, (uint64_t)d, (uint64_t)N))
        return DSA_ERR_CUDA;
    return from_cuda(launch_upproj(xmap, wmap, out, (int)n, N, d, static_cast<cudaStream_t>(stream)));
}

size_t dsa_mha_workspace_bytes(int B, int T, int Lmax) {
    if (B <= 0 || T <= 0 || Lmax <= 0) return (size_t)-1;
    return (size_t)B * T * (size_t)((Lmax + 127) / 128 * 4) * 4;
}

dsa_status_t dsa_sparse_mha_prefill(const uint16_t *q, const uint16_t *k_up,
                                    const uint16_t *v_up, const uint16_t *kv_cache,
                                    const dsa_cache_layout_t *layout, const int32_t *idx,
                                    const int32_t *q_pos, int B, int T, int H, int d, int r,
                                    int dn, int vd, int k, int Lmax, float scale, uint16_t *out,
                                    float *lse, void *workspace, size_t workspace_bytes,
                                    void *stream) {
    DSA_CALL_RANGE();
    if (!q || !k_up || !v_up || !kv_cache || !layout || !idx || !q_pos || !out || !workspace)
        return DSA_ERR_INVALID_ARG;
    if (B <= 0 || T <= 0 || H <= 0 || d <= 0 || r <= 0 || dn <= 0 || vd <= 0 || k <= 0 || Lmax <= 0)
        return DSA_ERR_INVALID_ARG;
    if (!(scale > 0.f)) return DSA_ERR_INVALID_ARG;
    if (layout->block_table || !layout->seq_start || layout->num_rows <= 0) return DSA_ERR_UNSUPPORTED;
    if (dn % 64 != 0 || r % 64 != 0 || dn + r > 256 || (vd != 128 && vd != 256) || d % 64 != 0)
        return DSA_ERR_UNSUPPORTED;
    if (Lmax > 65536 || k > 8192) return DSA_ERR_UNSUPPORTED;
    if ((int64_t)B * T >= ((int64_t)1 << 30) || layout->num_rows >= ((int64_t)1 << 31) - 128)
        return DSA_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_up) || !aligned16(v_up) || !aligned16(kv_cache) ||
        !aligned16(out) || !aligned16(workspace))
        return DSA_ERR_INVALID_ARG;
    const size_t need = dsa_mha_workspace_bytes(B, T, Lmax);
    if (workspace_bytes < need) return DSA_ERR_WORKSPACE;
    MhaParams p;
    p.q_pos = q_pos;
    p.seq_start = layout->seq_start;
    p.bitmap = static_cast<uint32_t *>(workspace);
    p.out = out;
    p.lse = lse;
    p.B = B;
    p.T = T;
    p.H = H;
    p.d = d;
    p.r = r;
    p.dn = dn;
    p.dq = dn + r;
    p.vd = vd;
    p.k = k;
    p.Lmax = Lmax;
    p.words = (Lmax + 127) / 128 * 4;
    p.scale_log2 = scale * 1.4426950408889634f;
    const int64_t nr = layout->num_rows;
    CUtensorMap qmap, kmap, rmap, vmap;
    if (!encode_bf16_2d(&qmap, q, (uint64_t)H * p.dq, (uint64_t)B * T) ||
        !encode_bf16_2d(&kmap, k_up, (uint64_t)H * dn, (uint64_t)nr) ||
        !encode_bf16_2d(&rmap, kv_cache, (uint64_t)(d + r), (uint64_t)nr) ||
        !encode_bf16_2d(&vmap, v_up, (uint64_t)H * vd, (uint64_t)nr))
        return DSA_ERR_CUDA;
    return from_cuda(launch_mha(p, qmap, kmap, rmap, vmap, idx, static_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_wait_probe(uint64_t *result, void *stream) {
    DSA_CALL_RANGE();
    if (!result || (reinterpret_cast<uintptr_t>(result) & 7) != 0) return DSA_ERR_INVALID_ARG;
    return from_cuda(launch_wait_probe(reinterpret_cast<unsigned long long *>(result),
                                       static_cast<cudaStream_t>(stream)));
}

dsa_status_t dsa_device_error(void *stream, uint32_t *code) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(s) != cudaSuccess) return from_cuda(cudaErrorUnknown);
    const uint32_t words[7] = {take_error_indexer(), take_error_topk(), take_error_mla(),
                               take_error_append(), take_error_hisparse(), take_error_mha(),
                               take_error_probe()};
    uint32_t first = 0;
    for (uint32_t v : words) {
        if (v == 0xFFFFFFFFu) return DSA_ERR_CUDA;
        if (v && !first) first = v;
    }
    if (code) *code = first;
    return first ? DSA_ERR_DEVICE : DSA_OK;
}

}  // extern "C"
