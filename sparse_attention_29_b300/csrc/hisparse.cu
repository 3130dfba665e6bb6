// hisparse.cu -- host-tier working set of the latent cache (HiSparse-style).
//
// Source: "La atención dispersa de GLM-5.3 reduce el cómputo, pero persiste la demanda de
// HBM" (remio.ai), the section on HiSparse: the full KV history stays in pinned host
// memory while the GPU keeps a small working set, managed least recently used; selected
// tokens missing from HBM are loaded from host memory and the least recently used entries
// are evicted, so that only the selection and a working buffer occupy HBM during decode.
// The placement changes nothing in the attention result.
//
// One CTA per sequence and decode step, before the sparse MLA of that step:
//   1. every selected token that is resident (residency[t] >= 0) is a hit, and its slot's
//      last use becomes `step`; the others are misses, ranked in their index-row order;
//   2. victims: the m = #misses slots whose last use is before `step`, least recently used
//      first and the lower slot first among equal last uses (never-used slots count as
//      used at 0) -- found by radix passes over the (inverted) last-use stamps in shared
//      memory, then listed in ascending slot order;
//   3. miss i takes victim i: the victim's previous token stops being resident, the miss's
//      row is copied from host memory into the slot (16-byte loads through the mapped
//      host pointer, one warp per row), and residency, slot token and last use are set.
// The residency table holds global pool rows (sequence b's slots are rows b*C .. b*C+C-1),
// so it is exactly a paged block table with one-token pages: the sparse MLA kernel reads
// the working set through dsa_cache_layout_t{block_table = residency, page_size = 1}.
#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr unsigned int KID_HISPARSE = 6;  // kernel id in the device error word
constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;

struct HiSmem {
    uint32_t key[kMaxHiSlots];     // inverted last use of every slot (0: used this step)
    int32_t miss[kMaxHiK];         // missed tokens, index-row order
    int32_t victim[kMaxHiK];       // victim slots, ascending
    uint32_t hist[kBins];
    uint32_t warp_tot[kWarps];
    int found_bin;
    uint32_t found_above;
    uint32_t hits;
};

__device__ __forceinline__ uint32_t excl_scan(uint32_t v, uint32_t *warp_tot) {
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
        const uint32_t t = lane < kWarps ? warp_tot[lane] : 0u;
        uint32_t s = t;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, s, o);
            if (lane >= o) s += y;
        }
        if (lane < kWarps) warp_tot[lane] = s - t;
    }
    __syncthreads();
    const uint32_t r = warp_tot[warp] + x - v;
    __syncthreads();
    return r;
}

// The bin of the r-th largest (1-based) of a kBins histogram: every thread owns 4 bins
// walked in descending order by a block scan.
static_assert(kBins == 4 * kThreads, "four bins per thread");
__device__ __forceinline__ void crossing(HiSmem &S, uint32_t r) {
    const int g = kThreads - 1 - (int)threadIdx.x;
    const uint4 v = reinterpret_cast<const uint4 *>(S.hist)[g];
    const uint32_t cnt[4] = {v.w, v.z, v.y, v.x};
    uint32_t above = excl_scan(v.x + v.y + v.z + v.w, S.warp_tot);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        if (above < r && above + cnt[i] >= r) {
            S.found_bin = 4 * g + 3 - i;
            S.found_above = above;
        }
        above += cnt[i];
    }
    __syncthreads();
}

__global__ void __launch_bounds__(kThreads, 1) hisparse_fetch_kernel(const HiParams p) {
    griddep_launch_dependents();
    griddep_wait();  // the index set (and the previous step's use of the pool) come first
    extern __shared__ __align__(16) uint8_t smem_raw[];
    HiSmem &S = *reinterpret_cast<HiSmem *>(smem_raw);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const int C = p.C;
    const int32_t *row = p.idx + (int64_t)b * p.k;
    int32_t *res = p.residency + (int64_t)b * p.Lmax;
    int32_t *stok = p.slot_token + (int64_t)b * C;
    uint32_t *use = p.slot_use + (int64_t)b * C;
    const int64_t pool0 = (int64_t)b * C;

    // ---- 1. hits and misses; misses ranked in index-row order ----
    if (tid == 0) S.hits = 0;
    __syncthreads();
    const int per = (p.k + kThreads - 1) / kThreads;
    const int j0 = min(p.k, tid * per), j1 = min(p.k, j0 + per);
    uint32_t nmiss = 0, nhit = 0;
    for (int j = j0; j < j1; ++j) {
        const int32_t t = row[j];
        if (t < 0) continue;
        if (t >= p.Lmax) {
            record_error(KID_HISPARSE, ERR_BAD_INDEX);
            continue;
        }
        const int32_t g = res[t];
        if (g >= 0) {
            const int64_t slot = g - pool0;
            if (slot >= 0 && slot < C) use[slot] = p.step;
            else record_error(KID_HISPARSE, ERR_BAD_PAGE);
            ++nhit;
        } else {
            ++nmiss;
        }
    }
    atomicAdd(&S.hits, nhit);
    uint32_t at = excl_scan(nmiss, S.warp_tot);
    for (int j = j0; j < j1; ++j) {
        const int32_t t = row[j];
        if (t >= 0 && t < p.Lmax && res[t] < 0) S.miss[at++] = t;
    }
    if (tid == kThreads - 1) S.warp_tot[0] = at;  // the total
    __syncthreads();
    const uint32_t m = S.warp_tot[0];
    __syncthreads();

    if (m > 0) {
        // ---- 2. victims: the m smallest last uses before `step` (ties: lower slot) ----
        // key = ~use for candidates (larger key = less recently used), 0 for slots used
        // in this step, so the m largest keys are the victims
        uint32_t nc = 0;
        for (int s = tid; s < C; s += kThreads) {
            const uint32_t u = use[s];
            S.key[s] = u < p.step ? ~u : 0u;
            nc += u < p.step;
        }
        for (int i = tid; i < kBins; i += kThreads) S.hist[i] = 0;
        const uint32_t ncand = excl_scan(nc, S.warp_tot) + nc;  // inclusive: the last thread's is the total
        if (tid == kThreads - 1) S.found_above = ncand;
        __syncthreads();
        if (S.found_above < m) {  // fewer free slots than misses (steps out of order)
            if (tid == 0) record_error(KID_HISPARSE, ERR_BAD_INDEX);
            return;
        }
        __syncthreads();
        uint32_t r = m, pref = 0;
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const uint32_t mask = pass == 2 ? 0x3FFu : 0x7FFu;
            const int hsh = pass == 0 ? 32 : (pass == 1 ? 21 : 10);
            if (pass > 0) {
                for (int i = tid; i < kBins; i += kThreads) S.hist[i] = 0;
                __syncthreads();
            }
            for (int s = tid; s < C; s += kThreads) {
                const uint32_t key = S.key[s];
                if (key == 0u) continue;
                if (hsh < 32 && (key >> hsh) != (pref >> hsh)) continue;
                atomicAdd(&S.hist[(key >> sh) & mask], 1u);
            }
            __syncthreads();
            crossing(S, r);
            pref |= ((uint32_t)S.found_bin) << sh;
            r -= S.found_above;
        }
        const uint32_t K = pref, r_eq = r;  // keys > K are victims, and the first r_eq == K
        // ascending slot order: thread t owns a contiguous range of slots
        const int ps = (C + kThreads - 1) / kThreads;
        const int s0 = min(C, tid * ps), s1 = min(C, s0 + ps);
        uint32_t ngt = 0, neq = 0;
        for (int s = s0; s < s1; ++s) {
            const uint32_t key = S.key[s];
            ngt += key > K && key != 0u;
            neq += key == K && key != 0u;
        }
        // a victim's position is the number of victims in lower slots: the strict victims
        // before it plus the equal-key victims before it (at most r_eq of those)
        uint32_t gt_b = excl_scan(ngt, S.warp_tot);
        uint32_t eq_b = excl_scan(neq, S.warp_tot);
        for (int s = s0; s < s1; ++s) {
            const uint32_t key = S.key[s];
            if (key == 0u) continue;
            if (key > K) {
                const uint32_t pos = gt_b + min(eq_b, r_eq);
                if (pos < m) S.victim[pos] = s;
                ++gt_b;
            } else if (key == K) {
                if (eq_b < r_eq) {
                    const uint32_t pos = gt_b + eq_b;
                    if (pos < m) S.victim[pos] = s;
                }
                ++eq_b;
            }
        }
        __syncthreads();

        // ---- 3. miss i takes victim i: bookkeeping, then the row copies ----
        for (uint32_t i = tid; i < m; i += kThreads) {
            const int32_t v = S.victim[i], t = S.miss[i];
            const int32_t old = stok[v];
            if (old >= 0 && old < p.Lmax) res[old] = -1;
            res[t] = (int32_t)(pool0 + v);
            stok[v] = t;
            use[v] = p.step;
        }
        const int nchunk = p.D / 8;  // 16-byte chunks of a row
        const int64_t hs = (int64_t)p.host_seq_start[b];
        for (uint32_t i = warp; i < m; i += kWarps) {
            const int32_t v = S.victim[i], t = S.miss[i];
            const uint4 *src = reinterpret_cast<const uint4 *>(p.host_kv + (hs + t) * p.D);
            uint4 *dst = reinterpret_cast<uint4 *>(p.pool + (pool0 + v) * p.D);
            for (int c = lane; c < nchunk; c += 32) dst[c] = src[c];
        }
    }
    if (tid == 0 && p.stats) {
        p.stats[2 * b] = (int32_t)S.hits;
        p.stats[2 * b + 1] = (int32_t)m;
    }
}

__global__ void hisparse_init_kernel(int32_t *residency, int64_t n_res, int32_t *slot_token,
                                     uint32_t *slot_use, int64_t n_slots) {
    griddep_launch_dependents();
    griddep_wait();
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_res; i += stride)
        residency[i] = -1;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n_slots; i += stride) {
        slot_token[i] = -1;
        slot_use[i] = 0u;
    }
}

}  // namespace

cudaError_t launch_hisparse_fetch(const HiParams &p, cudaStream_t stream) {
    if (p.B <= 0) return cudaSuccess;
    const size_t bytes = sizeof(HiSmem);
    static AttrCache attrs;
    cudaError_t e = ensure_smem_attrs(attrs, hisparse_fetch_kernel, (int)bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(hisparse_fetch_kernel, dim3(p.B), dim3(kThreads), bytes, stream, p);
}

cudaError_t launch_hisparse_init(int32_t *residency, int64_t n_res, int32_t *slot_token,
                                 uint32_t *slot_use, int64_t n_slots, cudaStream_t stream) {
    return launch_pdl(hisparse_init_kernel, dim3(148), dim3(256), 0, stream, residency, n_res,
                      slot_token, slot_use, n_slots);
}

DSA_DEFINE_ERROR_READER(take_error_hisparse)

}  // namespace dsa
