// topk_core.cuh -- the causal top-k of one row by one thread-block cluster: the body of
// the top-k kernel, shared with the sparse MLA kernel, which runs it for its own row
// before attending (decode: top-k and sparse MLA in one launch).
//
// Source: "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM", §Lightning
// Indexer (keep the top-K tokens by indexer score; a query that attends fewer than K
// tokens stays dense) and §Sparse MLA (K = 2048).  Equal scores go to the lower token
// index, so the selection is deterministic; indices are written in ascending order.
//
// CTA r of the cluster owns a contiguous slice of the row's candidates and keeps it in
// shared memory.  Keys are order-preserving integer images of the fp32 scores.
//   1. coarse: every CTA histograms an 11-bit key of its slice (the score rounded to
//      fp16: sign, 5 exponent and 5 mantissa bits -- monotone, and 32 bins per octave
//      spread realistic scores far better than the top bits of the fp32 pattern).  The
//      cluster sums the histograms through distributed shared memory and every CTA finds
//      the bin B0 that holds the k-th largest score, and how many it still needs from B0.
//   2. exact: the B0 candidates of all slices (typically a few hundred) are ranked by
//      (score, then lower index) by direct comparison; with more than kCandCap of them
//      (many exact ties) three distributed radix passes over the full 32-bit keys find
//      the k-th key instead, and ties are taken lowest index first across the slices.
//   3. output: CTAs exchange how many they select; each writes its selections, in index
//      order, at its offset.
// Rows that see at most k tokens skip all of this and write 0..n-1 then -1 padding.
#pragma once

#include "internal.h"
#include "keys.cuh"
#include "ptx.cuh"

namespace dsa {
namespace tk {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 2048;
constexpr int kCandCap = 1024;  // candidates ranked directly (per row, all slices)
constexpr int kMaxCluster = 8;

// ---- shared memory --------------------------------------------------------------------

struct Ctrl {
    uint64_t load_bar;
    uint32_t warp_tot[kWarps];
    uint32_t warp_st[kWarps], warp_eq[kWarps];  // per-warp counts (ordered pass)
    int found_bin;
    uint32_t found_above;
    uint32_t n_cand;      // B0 candidates in this slice (read by peers)
    uint32_t n_strict;    // surely selected in this slice
    uint32_t n_eq;        // keys equal to the threshold in this slice
    uint32_t peer_st[kMaxCluster], peer_eq[kMaxCluster];  // every slice's counts, pushed
};

struct Layout {
    uint32_t vals, masks, cand_key, cand_idx, hist, tot, ctrl, total;
};

__host__ __device__ inline Layout topk_layout(int slice_cap) {
    Layout L;
    uint32_t off = 0;
    L.vals = off;  // the slice starts at its global 16-byte phase: up to 3 floats in
    off += ((uint32_t)slice_cap + 4) * 4;
    L.masks = off;  // two ballots per 32 elements
    off += ((uint32_t)slice_cap + 31) / 32 * 8 + 16 * 8;
    off = (off + 15) & ~15u;
    L.cand_key = off;
    off += kCandCap * 4;
    L.cand_idx = off;
    off += kCandCap * 4;
    L.hist = off;
    off += 2 * kBins * 4;
    L.tot = off;
    off += kBins * 4;
    L.ctrl = off;
    off += sizeof(Ctrl);
    L.total = (off + 15) & ~15u;
    return L;
}

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
    const uint32_t res = warp_tot[warp] + x - v;
    __syncthreads();  // warp_tot is reused by the next call
    return res;
}

// Sum the cluster's histograms (`hist`, at the same offset in every CTA) into tot and
// find the bin holding the r-th largest element (1-based): sets c.found_bin and
// c.found_above (elements in higher bins).  Thread t owns the four bins of group
// kThreads-1-t, so a block scan in thread order walks the bins in descending order.
static_assert(kBins == 4 * kThreads, "four bins per thread");
__device__ __forceinline__ void cluster_crossing(const uint32_t *hist, uint32_t *tot, int csize,
                                                 Ctrl &c, uint32_t r) {
    const int g = kThreads - 1 - (int)threadIdx.x;
    uint4 s = reinterpret_cast<const uint4 *>(hist)[g];
    if (csize > 1) {
        s = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int rr = 0; rr < kMaxCluster; ++rr) {
            if (rr < csize) {
                const uint4 v = dsmem_ld4(hist + 4 * g, (uint32_t)rr);
                s.x += v.x;
                s.y += v.y;
                s.z += v.z;
                s.w += v.w;
            }
        }
    }
    reinterpret_cast<uint4 *>(tot)[g] = s;
    const uint32_t cnt[4] = {s.w, s.z, s.y, s.x};  // bins 4g+3 down to 4g
    uint32_t above = block_excl_scan(s.x + s.y + s.z + s.w, c.warp_tot);
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

// One row's top-k by the CTAs of a thread-block cluster (csize of them; this CTA has
// cluster rank `rank`), with `smem_raw` (16-byte aligned, topk_layout(slice_cap).total
// bytes) as its working space; all threads of every CTA of the cluster call it.  The
// selection goes to p.idx[row], in ascending token order.
__device__ __forceinline__ void topk_row(const TopkParams &p, int row, int csize, uint32_t rank,
                                         int slice_cap, uint8_t *smem_raw) {
    const Layout Ly = topk_layout(slice_cap);
    float *vals = reinterpret_cast<float *>(smem_raw + Ly.vals);
    uint32_t *cand_key = reinterpret_cast<uint32_t *>(smem_raw + Ly.cand_key);
    int32_t *cand_idx = reinterpret_cast<int32_t *>(smem_raw + Ly.cand_idx);
    uint32_t *hist = reinterpret_cast<uint32_t *>(smem_raw + Ly.hist);  // [2][kBins]
    uint32_t *tot = reinterpret_cast<uint32_t *>(smem_raw + Ly.tot);
    Ctrl &ctrl = *reinterpret_cast<Ctrl *>(smem_raw + Ly.ctrl);

    const int tid = threadIdx.x;
    const int k = p.k;
    int32_t *out = p.idx + (int64_t)row * k;
    int n = p.q_pos[row] + 1;
    if (n < 1 || n > p.Lmax) {
        if (tid == 0 && rank == 0) record_error(KID_TOPK, ERR_BAD_POSITION);
        n = n < 1 ? 0 : p.Lmax;
    }
    if (n <= k) {  // dense: every visible token, then padding (uniform for the cluster)
        const int per = (k + csize - 1) / csize;
        const int lo = (int)rank * per, hi = min(k, lo + per);
        for (int i = lo + tid; i < hi; i += kThreads) out[i] = i < n ? i : -1;
        return;
    }

    // ---- this CTA's slice [s_lo, s_hi) of the row, staged in shared memory ------------
    const int per = (n + csize - 1) / csize;
    const int s_lo = min(n, (int)rank * per), s_hi = min(n, s_lo + per);
    const int m = s_hi - s_lo;
    const float *src = p.scores + (int64_t)row * p.Lmax + s_lo;
    {
        // the 16-byte-aligned middle of the slice by bulk asynchronous copies (the slice
        // in shared memory starts at the same alignment phase), the ends by plain loads
        const int head = min(m, (int)(((16 - (reinterpret_cast<uintptr_t>(src) & 15)) & 15) / 4));
        const int mid = ((m - head) >> 2) << 2;
        float *dst = vals + ((reinterpret_cast<uintptr_t>(src) & 15) >> 2);  // same phase
        if (tid == 0) {
            mbar_init(&ctrl.load_bar, 1);
            fence_barrier_init();
        }
        __syncthreads();
        if (tid == 0) {
            mbar_arrive_expect_tx(&ctrl.load_bar, (uint32_t)mid * 4);
            for (int off = 0; off < mid; off += 8192) {
                const int len = min(8192, mid - off);
                asm volatile(
                    "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                        smem_u32(dst + head + off)),
                    "l"(src + head + off), "r"(len * 4), "r"(smem_u32(&ctrl.load_bar))
                    : "memory");
            }
        }
        for (int i = tid; i < head; i += kThreads) dst[i] = __ldg(src + i);
        for (int i = head + mid + tid; i < m; i += kThreads) dst[i] = __ldg(src + i);
        for (int b = tid; b < 2 * kBins; b += kThreads) hist[b] = 0;
        if (tid == 0) ctrl.n_cand = 0;
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(&ctrl.load_bar, 0)) {
            if (globaltimer_ns() - t0 > kWaitLimitNs) {
                record_error(KID_TOPK, ERR_WAIT_TIMEOUT);
                break;
            }
        }
        vals = dst;
    }
    __syncthreads();
    // the slice has landed: the barrier's memory may be reused (in the sparse MLA kernel the
    // whole region becomes tile buffers afterwards)
    if (tid == 0) mbar_inval(&ctrl.load_bar);
    // warp w owns the contiguous segment [w_lo, w_hi) of the slice and walks it in steps of
    // 32 consecutive elements (lane l takes element 32j + l): ballots give each step's
    // hits in index order without bank conflicts or atomics
    const int lane = tid & 31, warp = tid >> 5;
    const int seg = ((m + kWarps - 1) / kWarps + 31) & ~31;
    const int w_lo = min(m, warp * seg), w_hi = min(m, w_lo + seg);
    uint32_t *wmask = reinterpret_cast<uint32_t *>(smem_raw + Ly.masks) + 2 * (w_lo >> 5);

    // ---- 1. coarse histogram, summed over the cluster -------------------------------
#pragma unroll 4
    for (int i = tid; i < m; i += kThreads) atomicAdd(&hist[coarse_key(vals[i])], 1u);
    __syncthreads();
    if (csize > 1) cluster_sync();
    cluster_crossing(hist, tot, csize, ctrl, (uint32_t)k);
    const uint32_t B0 = (uint32_t)ctrl.found_bin;
    const uint32_t r0 = (uint32_t)k - ctrl.found_above;  // still needed from bin B0
    const uint32_t c0 = tot[B0];                          // B0 elements in the row

    // ---- 2. exact selection inside B0 -------------------------------------------------
    // afterwards: selected = coarse > B0, or coarse == B0 and
    //   (rank path)  it is among the r0 best B0 candidates of the row (its bit is OR-ed
    //                into the strict selection mask);
    //   (radix path) key > T, or key == T and among the first r_eq such keys of the row.
    const bool all_bin = (r0 == c0);
    const bool rank_path = !all_bin && c0 <= (uint32_t)kCandCap;
    uint32_t T = 0, r_eq = 0;
    uint32_t *masks_all = reinterpret_cast<uint32_t *>(smem_raw + Ly.masks);  // [m/32][2]
    if (rank_path) {
        // one pass: the strict selections (coarse key above B0) as bit masks in index
        // order, and this slice's few B0 candidates appended to a list.  Thread t takes
        // half (t & 1) of 32-element word (t >> 1), reading its 16 elements in an order
        // rotated by the word index so that a warp's reads hit 32 distinct banks; the two
        // halves of a word are merged with one shuffle.
        const int nwords = (m + 31) >> 5;
        for (int w0 = 0; w0 < nwords; w0 += kThreads / 2) {
            const int wd = w0 + (tid >> 1), hf = tid & 1;
            uint32_t st = 0;
            if (wd < nwords) {
                const int base = wd * 32 + hf * 16;
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int q = (e + wd) & 15;
                    const int i = base + q;
                    if (i < m) {
                        const float f = vals[i];
                        const uint32_t ck = coarse_key(f);
                        st |= (ck > B0 ? 1u : 0u) << (hf * 16 + q);
                        if (ck == B0) {
                            const uint32_t at = atomicAdd(&ctrl.n_cand, 1u);
                            cand_key[at] = full_key(f);
                            cand_idx[at] = s_lo + i;
                        }
                    }
                }
            }
            st |= __shfl_xor_sync(0xffffffffu, st, 1);
            if (wd < nwords && hf == 0) {
                masks_all[2 * wd] = st;
                masks_all[2 * wd + 1] = 0u;
            }
        }
        __syncthreads();
        const uint32_t mine = ctrl.n_cand;
        __syncthreads();
        if (csize > 1) cluster_sync();  // every slice's list is complete
        // gather every slice's candidates (tot and hist are free again)
        uint32_t *all_key = tot;                                   // kCandCap entries
        int32_t *all_idx = reinterpret_cast<int32_t *>(hist);      // kCandCap entries
        uint32_t total = mine;
        if (csize > 1) {
            uint32_t offs[kMaxCluster + 1];
            offs[0] = 0;
#pragma unroll
            for (int rr = 0; rr < kMaxCluster; ++rr)
                offs[rr + 1] = offs[rr] + (rr < csize ? dsmem_ld(&ctrl.n_cand, (uint32_t)rr) : 0u);
            total = offs[kMaxCluster];
            for (uint32_t j = tid; j < total; j += kThreads) {
                uint32_t rr = 0, base = 0;
#pragma unroll
                for (int q = 1; q < kMaxCluster; ++q)
                    if (j >= offs[q]) {
                        rr = (uint32_t)q;
                        base = offs[q];
                    }
                all_key[j] = dsmem_ld(cand_key + (j - base), rr);
                all_idx[j] = (int32_t)dsmem_ld(cand_idx + (j - base), rr);
            }
        } else {
            for (uint32_t j = tid; j < total; j += kThreads) {
                all_key[j] = cand_key[j];
                all_idx[j] = cand_idx[j];
            }
        }
        __syncthreads();
        // rank this slice's candidates against every candidate of the row: a warp takes
        // four candidates at a time, its lanes splitting the comparisons (each loaded
        // entry is compared with all four)
        for (uint32_t cb = (uint32_t)warp * 4; cb < mine; cb += kWarps * 4) {
            uint32_t key[4], better[4];
            int32_t idx[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const bool v = cb + q < mine;
                key[q] = v ? cand_key[cb + q] : 0u;
                idx[q] = v ? cand_idx[cb + q] : 0;
                better[q] = 0;
            }
#pragma unroll 2
            for (uint32_t j = lane; j < total; j += 32) {
                const uint32_t kj = all_key[j];
                const int32_t ij = all_idx[j];
#pragma unroll
                for (int q = 0; q < 4; ++q) better[q] += (kj > key[q]) || (kj == key[q] && ij < idx[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const uint32_t bq = __reduce_add_sync(0xffffffffu, better[q]);
                if (lane == 0 && cb + q < mine && bq < r0) {
                    const int li = idx[q] - s_lo;
                    atomicOr(&masks_all[2 * (li >> 5)], 1u << (li & 31));
                }
            }
        }
        __syncthreads();
    } else if (!all_bin) {
        // many exact ties: three radix passes (11, 11, 10 bits) over the full keys of B0,
        // histograms alternating between two buffers so that one cluster barrier per pass
        // separates a buffer's writes from its peers' reads
        uint32_t r = r0, pref = 0;
#pragma unroll 1
        for (int pass = 0; pass < 3; ++pass) {
            const int sh = pass == 0 ? 21 : (pass == 1 ? 10 : 0);
            const uint32_t mask = pass == 2 ? 0x3FFu : 0x7FFu;
            const int hsh = pass == 0 ? 32 : (pass == 1 ? 21 : 10);
            uint32_t *h = hist + ((pass + 1) & 1) * kBins;  // buffer 0 held the coarse pass
            for (int b = tid; b < kBins; b += kThreads) h[b] = 0;
            __syncthreads();
            for (int i = tid; i < m; i += kThreads) {
                const float f = vals[i];
                if (coarse_key(f) != B0) continue;
                const uint32_t u = full_key(f);
                if (hsh < 32 && (u >> hsh) != (pref >> hsh)) continue;
                atomicAdd(&h[(u >> sh) & mask], 1u);
            }
            __syncthreads();
            if (csize > 1) cluster_sync();
            cluster_crossing(h, tot, csize, ctrl, r);
            pref |= ((uint32_t)ctrl.found_bin) << sh;
            r -= ctrl.found_above;
        }
        T = pref;
        r_eq = r;
    }

    // ---- 3. counts, offsets, ordered write --------------------------------------------
    auto classify = [&](int i, bool &strict, bool &eq) {
        const float f = vals[i];
        const uint32_t ck = coarse_key(f);
        strict = false;
        eq = false;
        if (ck > B0) {
            strict = true;
        } else if (ck == B0) {
            if (all_bin) {
                strict = true;
            } else {
                const uint32_t u = full_key(f);
                if (u > T) strict = true;
                else if (u == T) eq = true;
            }
        }
    };
    // per warp segment: selection ballots (strict, equal to the threshold) in index order
    // (the rank path has them already: strict bits, selected candidates OR-ed in)
    const int nsteps = (w_hi - w_lo + 31) >> 5;
    uint32_t w_st = 0, w_eq = 0;
    if (!rank_path) {
#pragma unroll 4
        for (int j = 0; j < nsteps; ++j) {
            const int i = w_lo + 32 * j + lane;
            bool st = false, eq = false;
            if (i < w_hi) classify(i, st, eq);
            const uint32_t bst = __ballot_sync(0xffffffffu, st), beq = __ballot_sync(0xffffffffu, eq);
            if (lane == 0) {
                wmask[2 * j] = bst;
                wmask[2 * j + 1] = beq;
            }
            w_st += __popc(bst);
            w_eq += __popc(beq);
        }
    } else {
        for (int j = lane; j < nsteps; j += 32) w_st += __popc(wmask[2 * j]);
        w_st = __reduce_add_sync(0xffffffffu, w_st);
    }
    if (lane == 0) {
        ctrl.warp_st[warp] = w_st;
        ctrl.warp_eq[warp] = w_eq;
    }
    __syncthreads();
    if (warp == 0) {
        const uint32_t a = __reduce_add_sync(0xffffffffu, lane < kWarps ? ctrl.warp_st[lane] : 0u);
        const uint32_t b = __reduce_add_sync(0xffffffffu, lane < kWarps ? ctrl.warp_eq[lane] : 0u);
        if (lane == 0) {
            ctrl.n_strict = a;
            ctrl.n_eq = b;
        }
        // push this slice's counts into every CTA of the cluster (itself included; lane
        // rr to CTA rr), so that after the barrier all reads are local and no CTA reads a
        // peer that may already have finished
        if (lane < csize) {
            if (csize > 1) {
                dsmem_st(&ctrl.peer_st[rank], (uint32_t)lane, a);
                dsmem_st(&ctrl.peer_eq[rank], (uint32_t)lane, b);
            } else {
                ctrl.peer_st[0] = a;
                ctrl.peer_eq[0] = b;
            }
        }
    }
    __syncthreads();
    if (csize > 1) cluster_sync();
    // earlier slices' selections come first; equal keys are taken by ascending index
    uint32_t sel_before = 0, eq_before = 0;
    for (uint32_t rr = 0; rr < rank; ++rr) {
        const uint32_t s_r = ctrl.peer_st[rr];
        const uint32_t e_r = ctrl.peer_eq[rr];
        const uint32_t take = eq_before >= r_eq ? 0u : min(e_r, r_eq - eq_before);
        sel_before += s_r + take;
        eq_before += e_r;
    }
    uint32_t pos = sel_before;
    if (r_eq == 0) {
        // no equal keys to share out: this warp's offset is a scan over the warps' counts,
        // and lane l writes the selections of the warp's 32-element word l (+32, ...) on its
        // own, bit by bit, at that word's offset (a scan over the words' counts)
        const uint32_t wc = lane < kWarps ? ctrl.warp_st[lane] : 0u;
        uint32_t winc = wc;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, winc, o);
            if (lane >= o) winc += y;
        }
        pos += __shfl_sync(0xffffffffu, winc - wc, warp);
        for (int j0 = 0; j0 < nsteps; j0 += 32) {
            const int j = j0 + lane;
            uint32_t sel = j < nsteps ? wmask[2 * j] : 0u;
            const uint32_t cnt = __popc(sel);
            uint32_t incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            uint32_t at = pos + incl - cnt;
            const int ebase = s_lo + w_lo + 32 * j;
            while (sel) {
                const int bit = __ffs(sel) - 1;
                if (at < (uint32_t)k) out[at] = ebase + bit;
                ++at;
                sel &= sel - 1u;
            }
            pos += __shfl_sync(0xffffffffu, incl, 31);
        }
    } else {
        // this warp's offsets: earlier warps' strict selections and taken equal keys
        uint32_t eq_seen = eq_before;
        for (int w = 0; w < warp; ++w) {
            const uint32_t e_w = ctrl.warp_eq[w];
            const uint32_t take = eq_seen >= r_eq ? 0u : min(e_w, r_eq - eq_seen);
            pos += ctrl.warp_st[w] + take;
            eq_seen += e_w;
        }
        for (int j = 0; w_lo + 32 * j < w_hi; ++j) {
            const uint32_t bst = wmask[2 * j], beq = wmask[2 * j + 1];
            uint32_t take = 0;
            if (beq) {
                const uint32_t want = eq_seen >= r_eq ? 0u : r_eq - eq_seen;
                const uint32_t have = __popc(beq);
                if (want >= have) {
                    take = beq;
                } else if (want > 0) {
                    const uint32_t cut = __fns(beq, 0, (int)want + 1);  // position of the next one
                    take = beq & ((1u << cut) - 1u);
                }
                eq_seen += have;
            }
            const uint32_t sel = bst | take;
            if ((sel >> lane) & 1u) {
                const uint32_t at = pos + __popc(sel & ((1u << lane) - 1u));
                if (at < (uint32_t)k) out[at] = s_lo + w_lo + 32 * j + lane;
            }
            pos += __popc(sel);
        }
    }
    // the last warp of the last slice ends at k
    uint32_t sel_base = pos;
    sel_base = __shfl_sync(0xffffffffu, sel_base, 0);
    if (warp != kWarps - 1) sel_base = (uint32_t)k;
    if (rank == (uint32_t)csize - 1 && warp == kWarps - 1 && lane == 0 && sel_base != (uint32_t)k)
        record_error(KID_TOPK, ERR_BAD_INDEX);
}


}  // namespace tk
}  // namespace dsa
