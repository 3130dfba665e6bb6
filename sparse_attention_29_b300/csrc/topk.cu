// topk.cu -- causal top-k selection with the dense fallback.
//
// Source: "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM", §Lightning
// Indexer (keep the top-K tokens by indexer score; a query that attends fewer than K
// tokens stays dense) and §Sparse MLA (K = 2048).  Equal scores go to the lower token
// index, so the selection is deterministic; indices are written in ascending order.
//
// One thread-block cluster per query row runs the cluster top-k of topk_core.cuh (also run
// by the sparse MLA kernel when it selects its own rows); this file holds its launch shape
// and the final selection of the fused prefill indexer + top-k.
#include <cuda_fp16.h>

#include <mutex>

#include "internal.h"
#include "keys.cuh"
#include "ptx.cuh"
#include "topk_core.cuh"

namespace dsa {
namespace {

using namespace tk;

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const TopkParams p, int csize,
                                                            int slice_cap) {
    griddep_launch_dependents();
    griddep_wait();  // the scores come from the previous kernel
    extern __shared__ __align__(16) uint8_t smem_raw[];
    const uint32_t rank = csize > 1 ? cluster_rank() : 0u;
    topk_row(p, blockIdx.x / csize, csize, rank, slice_cap, smem_raw);
}

// ---- final selection of the fused indexer + top-k -------------------------------------
// One CTA per row.  The fused indexer kept, for every row that sees more than k tokens,
// every score whose coarse bin reached the row's running threshold, as (full key, token
// index); the final bin B0 holds the row's k-th best score, g candidates lie above it and
// c0 in it.  Selected: every candidate above B0, and the best r0 = k - g of the bin-B0
// candidates by (score, then lower index) -- ranked by direct comparison in shared memory
// when there are at most kRankCap of them, else by radix passes over their full keys and,
// among keys equal to the threshold, over their indices.  The selection goes to a bitmap
// of the row's tokens (kWinBits at a time) and is written in ascending token order.
constexpr int kRankCap = 4096;
constexpr int kWinBits = 65536;

struct CandSmem {
    uint32_t bitmap[kWinBits / 32];
    uint32_t key[kRankCap];
    int32_t idx[kRankCap];
    uint32_t hist[kBins];
    uint32_t warp_tot[kWarps];
    uint8_t chosen[kRankCap];
    int found_bin;
    uint32_t found_above;
    uint32_t n_cand;
};

// The bin of the `r`-th largest value (1-based) of the histogram `h` (kBins counts, all
// threads call): sets c.found_bin and c.found_above.
__device__ __forceinline__ void hist_crossing(const uint32_t *h, CandSmem &c, uint32_t r) {
    const int g = kThreads - 1 - (int)threadIdx.x;
    const uint4 v = reinterpret_cast<const uint4 *>(h)[g];
    const uint32_t cnt[4] = {v.w, v.z, v.y, v.x};  // bins 4g+3 down to 4g
    uint32_t above = block_excl_scan(v.x + v.y + v.z + v.w, c.warp_tot);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (above < r && above + cnt[i] >= r) {
            c.found_bin = 4 * g + 3 - i;
            c.found_above = above;
        }
        above += cnt[i];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1) topk_cand_kernel(const TopkCandParams p) {
    griddep_launch_dependents();
    griddep_wait();  // the candidates come from the previous kernel
    extern __shared__ __align__(16) uint8_t smem_raw[];
    CandSmem &S = *reinterpret_cast<CandSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x, k = p.k;
    int32_t *out = p.idx + (int64_t)row * k;
    int n_vis = p.q_pos[row] + 1;
    if (n_vis < 1 || n_vis > p.Lmax) {
        if (tid == 0) record_error(KID_TOPK, ERR_BAD_POSITION);
        n_vis = n_vis < 1 ? 0 : p.Lmax;
    }
    if (n_vis <= k) {  // dense: every visible token, then padding
        for (int i = tid; i < k; i += kThreads) out[i] = i < n_vis ? i : -1;
        return;
    }
    // the row's list: four quarters of seg slots, filled to the counts in meta[2 row]
    const uint4 mc = p.meta[2 * (int64_t)row], mb = p.meta[2 * (int64_t)row + 1];
    const uint32_t seg = p.cap / 4 < 0x7FFFFFFF ? (uint32_t)(p.cap / 4) : 0x7FFFFFFFu;
    const uint32_t n0 = min(mc.x, seg), n1 = min(mc.y, seg), n2 = min(mc.z, seg), n3 = min(mc.w, seg);
    const uint32_t o1 = n0, o2 = o1 + n1, o3 = o2 + n2, n = o3 + n3;
    const uint32_t B0 = mb.x, g = mb.y, c0 = mb.z;
    const uint2 *cl0 = p.cand + (int64_t)row * p.cap;
    auto entry = [&](uint32_t i) -> uint2 {  // i-th entry of the row, 0 <= i < n
        const uint32_t q = (i >= o1) + (i >= o2) + (i >= o3);
        const uint32_t base = q == 0 ? 0u : (q == 1 ? o1 : (q == 2 ? o2 : o3));
        return cl0[(int64_t)q * seg + (i - base)];
    };
    if (g >= (uint32_t)k || g + c0 < (uint32_t)k || B0 >= (uint32_t)kBins) {
        if (tid == 0) record_error(KID_TOPK, ERR_BAD_INDEX);
        for (int i = tid; i < k; i += kThreads) out[i] = -1;
        return;
    }
    const uint32_t r0 = (uint32_t)k - g;  // still needed from bin B0
    const bool all_bin = r0 == c0;
    const bool rank_path = !all_bin && c0 <= (uint32_t)kRankCap;
    uint32_t T = 0, I = 0;  // radix path: key threshold, and index threshold at key T
    if (tid == 0) S.n_cand = 0;
    __syncthreads();
    if (rank_path) {
        for (uint32_t i = tid; i < n; i += kThreads) {
            const uint2 e = entry(i);
            if (coarse_key(key_score(e.x)) == B0) {
                const uint32_t at = atomicAdd(&S.n_cand, 1u);
                if (at < (uint32_t)kRankCap) {
                    S.key[at] = e.x;
                    S.idx[at] = (int32_t)e.y;
                }
            }
        }
        __syncthreads();
        const uint32_t total = min(S.n_cand, (uint32_t)kRankCap);
        // a warp ranks four candidates at a time against every candidate of the bin
        for (uint32_t cb = (uint32_t)warp * 4; cb < total; cb += kWarps * 4) {
            uint32_t key[4], better[4];
            int32_t idx[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool v = cb + q < total;
                key[q] = v ? S.key[cb + q] : 0u;
                idx[q] = v ? S.idx[cb + q] : 0;
                better[q] = 0;
            }
            for (uint32_t j = lane; j < total; j += 32) {
                const uint32_t kj = S.key[j];
                const int32_t ij = S.idx[j];
#pragma unroll
                for (int q = 0; q < 4; ++q) better[q] += (kj > key[q]) || (kj == key[q] && ij < idx[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t bq = __reduce_add_sync(0xffffffffu, better[q]);
                if (lane == 0 && cb + q < total) S.chosen[cb + q] = bq < r0 ? 1 : 0;
            }
        }
        __syncthreads();
    } else if (!all_bin) {
        // many ties in the bin: radix passes over the bin's full keys (11, 11, 10 bits),
        // then over the indices of the keys equal to the threshold (11, 10, 10 bits)
        uint32_t r = r0, pref = 0;
#pragma unroll 1
        for (int pass = 0; pass < 6; ++pass) {
            const bool on_idx = pass >= 3;
            const int ps = on_idx ? pass - 3 : pass;
            const int sh = on_idx ? (ps == 0 ? 20 : (ps == 1 ? 10 : 0)) : (ps == 0 ? 21 : (ps == 1 ? 10 : 0));
            const uint32_t mask = (!on_idx && ps == 2) ? 0x3FFu : (on_idx && ps != 0 ? 0x3FFu : 0x7FFu);
            const int hsh = ps == 0 ? 32 : (on_idx ? (ps == 1 ? 20 : 10) : (ps == 1 ? 21 : 10));
            for (int b = tid; b < kBins; b += kThreads) S.hist[b] = 0;
            __syncthreads();
            for (uint32_t i = tid; i < n; i += kThreads) {
                const uint2 e = entry(i);
                if (coarse_key(key_score(e.x)) != B0) continue;
                uint32_t u;
                if (on_idx) {
                    if (e.x != T) continue;
                    u = e.y;
                } else {
                    u = e.x;
                }
                if (hsh < 32 && (u >> hsh) != (pref >> hsh)) continue;
                // indices: the smallest are wanted, so they count in reversed bin order
                const uint32_t bin = (u >> sh) & mask;
                atomicAdd(&S.hist[on_idx ? mask - bin : bin], 1u);
            }
            __syncthreads();
            hist_crossing(S.hist, S, r);
            const uint32_t bin = on_idx ? mask - (uint32_t)S.found_bin : (uint32_t)S.found_bin;
            pref |= bin << sh;
            r -= S.found_above;
            if (pass == 2) {
                T = pref;
                pref = 0;
            }
        }
        I = pref;
    }

    // ---- output: the selection as a bitmap of the row's tokens, written in order ----
    uint32_t base = 0;
    for (int w0 = 0; w0 < n_vis; w0 += kWinBits) {
        const int wn = min(kWinBits, n_vis - w0);
        const int nwords = (wn + 31) >> 5;
        for (int i = tid; i < nwords; i += kThreads) S.bitmap[i] = 0u;
        __syncthreads();
        for (uint32_t i = tid; i < n; i += kThreads) {
            const uint2 e = entry(i);
            const int s = (int)e.y - w0;
            if (s < 0 || s >= wn) continue;
            const uint32_t b = coarse_key(key_score(e.x));
            bool sel = b > B0;
            if (b == B0 && !rank_path) sel = all_bin || e.x > T || (e.x == T && e.y <= I);
            if (sel) atomicOr(&S.bitmap[s >> 5], 1u << (s & 31));
        }
        if (rank_path) {
            const uint32_t total = min(S.n_cand, (uint32_t)kRankCap);
            for (uint32_t j = tid; j < total; j += kThreads) {
                const int s = S.idx[j] - w0;
                if (S.chosen[j] && s >= 0 && s < wn) atomicOr(&S.bitmap[s >> 5], 1u << (s & 31));
            }
        }
        __syncthreads();
        // thread t owns words [t * per, (t + 1) * per): counts, scan, ordered write
        const int per = (nwords + kThreads - 1) / kThreads;
        const int lo = min(nwords, tid * per), hi = min(nwords, lo + per);
        uint32_t cnt = 0;
        for (int wd = lo; wd < hi; ++wd) cnt += __popc(S.bitmap[wd]);
        uint32_t at = base + block_excl_scan(cnt, S.warp_tot);
        for (int wd = lo; wd < hi; ++wd) {
            uint32_t bits = S.bitmap[wd];
            while (bits) {
                const int bit = __ffs(bits) - 1;
                if (at < (uint32_t)k) out[at] = w0 + wd * 32 + bit;
                ++at;
                bits &= bits - 1u;
            }
        }
        // the window's total: the last thread's end
        if (tid == kThreads - 1) S.warp_tot[0] = at;
        __syncthreads();
        base = S.warp_tot[0];
        __syncthreads();
    }
    if (tid == 0 && base != (uint32_t)k) record_error(KID_TOPK, ERR_BAD_INDEX);
}

}  // namespace

cudaError_t launch_topk_cand(const TopkCandParams &p, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    const size_t bytes = sizeof(CandSmem);
    static AttrCache attrs;
    cudaError_t e = ensure_smem_attrs(attrs, topk_cand_kernel, (int)bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(topk_cand_kernel, dim3(p.rows), dim3(kThreads), bytes, stream, p);
}

// Clusters of `cs` CTAs with `bytes` of shared memory each that the current device runs
// at once (0 if unknown); cached per device, cluster size and shared-memory size.
static int topk_max_clusters(int cs, int bytes) {
    constexpr int kDevs = 16, kSlots = 64;
    struct Entry { int cs, bytes, n; };
    static Entry cache[kDevs][kSlots];
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kDevs) return 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < kSlots; ++i) {
        Entry &e = cache[dev][i];
        if (e.cs == cs && e.bytes == bytes) return e.n;
        if (e.cs != 0) continue;
        if (set_smem_attrs(topk_kernel, 227 * 1024) != cudaSuccess) {
            (void)cudaGetLastError();
            return 0;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(cs);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = bytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = cs;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, topk_kernel, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        e = Entry{cs, bytes, n};
        return n;
    }
    return 0;
}

// Cluster size and slice capacity of a launch: enough CTAs per row to fill the GPU when
// rows are few, and to keep every slice within shared memory; a cluster size whose
// clusters would not all run at once (a second wave) is lowered while the slices still fit.
static void topk_shape(const TopkParams &p, int num_sms, int &csize, int &slice_cap) {
    constexpr int kSliceMax = 40960;
    const int by_fill = p.rows > 0 ? num_sms / p.rows : 1;
    int by_size = (p.Lmax + kSliceMax - 1) / kSliceMax;
    if (by_size < 1) by_size = 1;
    csize = by_fill > by_size ? by_fill : by_size;
    if (csize > kMaxCluster) csize = kMaxCluster;
    auto cap_of = [&](int cs) { return (((p.Lmax + cs - 1) / cs) + 31) & ~31; };
    while (csize > by_size && csize > 1) {
        const int n = topk_max_clusters(csize, (int)topk_layout(cap_of(csize)).total);
        if (n <= 0 || p.rows <= n) break;
        --csize;
    }
    slice_cap = cap_of(csize);
}

bool topk_lmax_supported(int Lmax) {
    if (Lmax <= 0) return false;
    const int cap = (((Lmax + kMaxCluster - 1) / kMaxCluster) + 31) & ~31;
    return topk_layout(cap).total <= 227 * 1024;
}

cudaError_t launch_topk(const TopkParams &p, int num_sms, cudaStream_t stream) {
    if (p.rows <= 0) return cudaSuccess;
    int csize, slice_cap;
    topk_shape(p, num_sms, csize, slice_cap);
    const size_t bytes = topk_layout(slice_cap).total;
    if (bytes > 227 * 1024) return cudaErrorInvalidValue;
    static AttrCache attrs;  // every slice size fits
    cudaError_t ea = ensure_smem_attrs(attrs, topk_kernel, 227 * 1024);
    if (ea != cudaSuccess) return ea;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(p.rows * csize);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = csize;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, topk_kernel, p, csize, slice_cap);
}

DSA_DEFINE_ERROR_READER(take_error_topk)

}  // namespace dsa
