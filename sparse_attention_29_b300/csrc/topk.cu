// topk.cu -- causal top-k selection with the dense fallback, one CTA per query row.
//
// Source: "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM", §Lightning
// Indexer (keep the top-K tokens by indexer score; a query that attends fewer than K
// tokens stays dense) and §Sparse MLA (K = 2048).  Equal scores go to the lower token
// index, so the selection is deterministic; indices are written in ascending order.
//
// Method: radix select on order-preserving integer keys of the fp32 scores.
//   1. coarse pass: a 2048-bin histogram of an 11-bit key taken from the score rounded to
//      fp16 (sign, 5 exponent bits, 5 mantissa bits).  Rounding to fp16 is monotone, so
//      the bins are ordered like the scores, and 32 bins per octave spread a realistic
//      score distribution far better than the top bits of the fp32 pattern would.  The
//      bin holding the k-th largest score is found by a suffix count.
//   2. refine: inside that bin only, three radix passes (11, 11, 10 bits) over the full
//      32-bit key find the k-th largest key T exactly, and how many elements equal to T
//      must still be taken.
//   3. one ordered pass writes every element above T and the lowest-index elements equal
//      to T, in ascending index order (block-wide prefix sums).
// Rows of up to 40960 candidates are staged in shared memory once; longer rows are read
// again from global memory (L2) by each pass.
#include <cuda_fp16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 1024;
constexpr int kWarps = kThreads / 32;
constexpr int kCacheCap = 40960;
constexpr int kCandCap = 4096;
constexpr int kBins = 2048;
constexpr int kItems = 8;  // consecutive elements per thread in the ordered pass

// Order-preserving map fp32 -> uint32 (larger score -> larger key); -0 and +0 are one key.
__device__ __forceinline__ uint32_t full_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (f == 0.f) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// 11-bit coarse key from the fp16 rounding of the score (monotone non-decreasing).
__device__ __forceinline__ uint32_t coarse_key(float f) {
    if (f == 0.f) f = 0.f;
    const uint16_t h = __half_as_ushort(__float2half_rn(f));
    const uint32_t u = (h & 0x8000u) ? (uint32_t)(~h & 0xFFFFu) : (uint32_t)(h | 0x8000u);
    return u >> 5;
}

struct TopkSmem {
    float cache[kCacheCap];
    uint32_t hist[kBins];
    uint32_t cand_key[kCandCap];
    uint32_t warp_tot[kWarps];
    uint32_t cand_count;
    int found_bin;
    uint32_t found_above;
};

// Block-wide exclusive scan of one uint32 per thread (all threads must call it).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_tot) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) warp_tot[warp] = x;
    __syncthreads();
    if (warp == 0) {
        const uint32_t t = warp_tot[lane];
        uint32_t s = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        warp_tot[lane] = s - t;  // exclusive prefix of the warp totals
    }
    __syncthreads();
    return warp_tot[warp] + x - v;
}

// Find the bin holding the r-th largest element (1-based r) of hist[0..kBins): sets
// sm.found_bin and sm.found_above = count of elements in higher bins.
__device__ __forceinline__ void find_crossing(TopkSmem &sm, uint32_t r) {
    const int t = threadIdx.x;
    const int b_hi = kBins - 1 - 2 * t;  // this thread's bins, descending: b_hi, b_hi - 1
    const uint32_t c0 = sm.hist[b_hi], c1 = sm.hist[b_hi - 1];
    const uint32_t above = block_excl_scan(c0 + c1, sm.warp_tot);
    if (above < r && above + c0 >= r) {
        sm.found_bin = b_hi;
        sm.found_above = above;
    } else if (above + c0 < r && above + c0 + c1 >= r) {
        sm.found_bin = b_hi - 1;
        sm.found_above = above + c0;
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1) topk_kernel(const TopkParams p) {
    extern __shared__ __align__(16) uint8_t smem_raw[];
    TopkSmem &sm = *reinterpret_cast<TopkSmem *>(smem_raw);
    griddep_launch_dependents();
    griddep_wait();  // the scores come from the previous kernel
    const int row = blockIdx.x;
    const int tid = threadIdx.x;
    const int k = p.k;
    int32_t *out = p.idx + (int64_t)row * k;
    int n = p.q_pos[row] + 1;
    if (n < 1 || n > p.Lmax) {
        if (tid == 0) record_error(KID_TOPK, ERR_BAD_POSITION);
        n = n < 1 ? 0 : p.Lmax;
    }
    if (n <= k) {  // dense: every visible token, then padding
        for (int i = tid; i < k; i += kThreads) out[i] = i < n ? i : -1;
        return;
    }
    const float *src = p.scores + (int64_t)row * p.Lmax;
    const bool cached = n <= kCacheCap;
    if (cached) {
        if ((reinterpret_cast<uintptr_t>(src) & 15) == 0) {
            const int n4 = n >> 2;
            for (int i = tid; i < n4; i += kThreads)
                reinterpret_cast<float4 *>(sm.cache)[i] = __ldg(reinterpret_cast<const float4 *>(src) + i);
            for (int i = (n4 << 2) + tid; i < n; i += kThreads) sm.cache[i] = __ldg(src + i);
        } else {
            for (int i = tid; i < n; i += kThreads) sm.cache[i] = __ldg(src + i);
        }
    }
    auto score = [&](int i) -> float { return cached ? sm.cache[i] : __ldg(src + i); };

    // ---- 1. coarse histogram ---------------------------------------------------------
    for (int b = tid; b < kBins; b += kThreads) sm.hist[b] = 0;
    if (tid == 0) sm.cand_count = 0;
    __syncthreads();
    for (int i = tid; i < n; i += kThreads) atomicAdd(&sm.hist[coarse_key(score(i))], 1u);
    __syncthreads();
    find_crossing(sm, (uint32_t)k);
    const uint32_t B0 = (uint32_t)sm.found_bin;
    uint32_t r = (uint32_t)k - sm.found_above;  // still to take from bin B0
    const uint32_t c0 = sm.hist[B0];
    __syncthreads();

    // ---- 2. exact threshold inside bin B0 ---------------------------------------------
    bool all_bin = (r == c0);
    uint32_t T = 0;
    if (!all_bin) {
        const bool use_cand = c0 <= (uint32_t)kCandCap;
        if (use_cand) {
            for (int i = tid; i < n; i += kThreads) {
                const float f = score(i);
                if (coarse_key(f) == B0) {
                    const uint32_t slot = atomicAdd(&sm.cand_count, 1u);
                    sm.cand_key[slot] = full_key(f);
                }
            }
            __syncthreads();
        }
        const int nc = use_cand ? (int)c0 : n;
        uint32_t pref = 0;  // key bits fixed so far
        const int shifts[3] = {21, 10, 0};
        const uint32_t masks[3] = {0x7FFu, 0x7FFu, 0x3FFu};
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = shifts[pass];
            for (int b = tid; b < kBins; b += kThreads) sm.hist[b] = 0;
            __syncthreads();
            const int hsh = pass == 0 ? 32 : shifts[pass - 1];  // bits above this digit
            for (int i = tid; i < nc; i += kThreads) {
                uint32_t u;
                if (use_cand) {
                    u = sm.cand_key[i];
                } else {
                    const float f = score(i);
                    if (coarse_key(f) != B0) continue;
                    u = full_key(f);
                }
                if (hsh < 32 && (u >> hsh) != (pref >> hsh)) continue;
                atomicAdd(&sm.hist[(u >> sh) & masks[pass]], 1u);
            }
            __syncthreads();
            find_crossing(sm, r);
            pref |= ((uint32_t)sm.found_bin) << sh;
            r -= sm.found_above;
            __syncthreads();
        }
        T = pref;  // the k-th largest key; r = how many keys equal to T to take
    }

    // ---- 3. ordered write --------------------------------------------------------------
    uint32_t sel_base = 0, eq_base = 0;
    const uint32_t r_eq = r;
    for (int base = 0; base < n; base += kThreads * kItems) {
        const int i0 = base + tid * kItems;
        uint32_t strict_mask = 0, eq_mask = 0;
#pragma unroll
        for (int e = 0; e < kItems; ++e) {
            const int i = i0 + e;
            if (i < n) {
                const float f = score(i);
                const uint32_t ck = coarse_key(f);
                if (ck > B0) {
                    strict_mask |= 1u << e;
                } else if (ck == B0) {
                    if (all_bin) {
                        strict_mask |= 1u << e;
                    } else {
                        const uint32_t u = full_key(f);
                        if (u > T) strict_mask |= 1u << e;
                        else if (u == T) eq_mask |= 1u << e;
                    }
                }
            }
        }
        const uint32_t eq_before = eq_base + block_excl_scan(__popc(eq_mask), sm.warp_tot);
        // the first r_eq equal keys in index order are taken
        uint32_t take_eq = 0, seen = eq_before;
#pragma unroll
        for (int e = 0; e < kItems; ++e) {
            if (eq_mask & (1u << e)) {
                if (seen < r_eq) take_eq |= 1u << e;
                ++seen;
            }
        }
        const uint32_t sel_mask = strict_mask | take_eq;
        uint32_t pos = sel_base + block_excl_scan(__popc(sel_mask), sm.warp_tot);
#pragma unroll
        for (int e = 0; e < kItems; ++e) {
            if (sel_mask & (1u << e)) {
                if (pos < (uint32_t)k) out[pos] = i0 + e;
                ++pos;
            }
        }
        // chunk totals: the last thread's end position
        __shared__ uint32_t chunk_end[2];
        if (tid == kThreads - 1) {
            chunk_end[0] = pos;
            chunk_end[1] = seen;
        }
        __syncthreads();
        sel_base = chunk_end[0];
        eq_base = chunk_end[1];
        __syncthreads();
    }
    if (tid == 0 && sel_base != (uint32_t)k) record_error(KID_TOPK, ERR_BAD_INDEX);
}

}  // namespace

cudaError_t launch_topk(const TopkParams &p, cudaStream_t stream) {
    const size_t bytes = sizeof(TopkSmem);
    static bool attr = false;
    if (!attr) {
        cudaError_t e = set_smem_attrs(topk_kernel, (int)bytes);
        if (e != cudaSuccess) return e;
        attr = true;
    }
    if (p.rows <= 0) return cudaSuccess;
    return launch_pdl(topk_kernel, dim3(p.rows), dim3(kThreads), bytes, stream, p);
}

DSA_DEFINE_ERROR_READER(take_error_topk)

}  // namespace dsa
