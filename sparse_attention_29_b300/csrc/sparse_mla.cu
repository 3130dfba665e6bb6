// sparse_mla.cu -- sparse MLA in MQA (absorbed) mode over the selected tokens.
//
// Source: "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM", §Sparse MLA
// (DSA runs MLA in MQA mode over the top-K tokens only) and §MLA changes (latent d = 512,
// rope r = 64, 2 bytes per value; 64 query heads).  For a query row with heads h and the
// selected cached rows c_j (d + r wide):
//     logit[h, j] = scale * q[h, :] . c_j          (key = the whole row)
//     o[h, :]     = sum_j softmax_j(logit[h, :]) c_j[:d]   (value = the latent part)
//
// Mapping onto sm_103a.  The selected rows are gathered 128 at a time with cp.async
// (16-byte granules, issued by the softmax threads while they would otherwise wait for
// the next tile; a separate warp resolves row addresses two tiles ahead) into shared
// memory in the tensor cores' 128-byte-swizzled layout: chunk c of a tile holds dims
// 64c..64c+63 of the 128 rows.  (TMA gather4 issues at about one instruction per 65
// cycles per SM, which is ~10 us per 144 KB tile; cp.async from 128 threads is far
// cheaper to issue.)  That one layout serves both products:
//   S^T[key, head]  = C[key, :] . Q[head, :]      A = C (K-major), B = Q (K-major)
//   O^T[dim, head] += C[key, dim]^T P^T[key, head] A = C^T (MN-major), B = P^T (MN-major)
// so both run as M = 128 tcgen05 MMAs (keys resp. latent dims on M, the 64 heads on N)
// with fp32 accumulators in tensor memory (S: 64 columns, O: 4 x 64 columns).  After
// tcgen05.ld a softmax thread owns one key's 64 head logits; per-head maxima are
// reduced across the 128 keys of the tile with a transposing warp butterfly.  The
// probabilities are written (bf16) over the tile's rope chunk, which S no longer needs.
// One thread issues ~60-80 cycles per tcgen05.mma and a tile needs 68 of them (36 for S,
// 32 for O), so two issuer warps split the work: each accumulates half of the S chunks
// into its own S^T copy (the softmax adds the two) and runs half of the O M-blocks.
// Online softmax rescales O in tensor memory only when a head's running maximum grows
// by more than 2^8 (the result is the same; the unnormalised terms just stay < 2^8).
// The query (64 heads x 576 x 2 B = 72 KB) and one tile (144 KB) fill shared memory,
// so the next tile's gather is overlapped at chunk granularity: chunks are refilled as
// soon as the O product that reads them has completed.
//
// Rows with few keys are split over several CTAs (split-KV); each writes unnormalised
// partial results that a combine kernel merges with the log-sum-exp rule.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 224;      // warps 0-3 softmax + gather + epilogue, 4 and 6 MMA, 5 rows
constexpr int kSoftmaxThreads = 128;
constexpr int kMmaWarp = 4;        // MMA issuer 0 (also owns the tensor memory)
constexpr int kMmaWarp2 = 6;       // MMA issuer 1
constexpr int kProducerWarp = 5;
constexpr int kTileKeys = 128;
constexpr int kHeads = 64;         // heads padded to 64 (N of both products)
constexpr int kChunkBytes = kTileKeys * 128;  // 64 dims x 128 keys x 2 B
constexpr int kQChunkBytes = kHeads * 128;    // 64 dims x 64 heads x 2 B
constexpr float kRescaleLog2 = 8.f;           // lazy rescale threshold (log2 units)

struct MlaSmem {
    uint32_t q, tile, rows, red, rn, alpha, lsum, bars, total;
};

__host__ __device__ inline MlaSmem mla_smem(int nch) {
    MlaSmem s;
    uint32_t off = 0;
    s.q = off;
    off += (uint32_t)nch * kQChunkBytes;
    s.tile = off;
    off += (uint32_t)nch * kChunkBytes;
    s.rows = off;
    off += 2 * kTileKeys * 4;
    s.red = off;
    off += 4 * kHeads * 4;
    s.rn = off;
    off += kHeads * 4;
    s.alpha = off;
    off += kHeads * 4;
    s.lsum = off;
    off += kHeads * 4;
    s.bars = off;
    off += 20 * 8 + 16;
    s.total = off;
    return s;
}

__device__ __forceinline__ uint32_t swz128(int row, int gran) {
    const uint32_t lin = (uint32_t)row * 128 + (uint32_t)gran * 16;
    return lin ^ (((lin >> 7) & 7u) << 4);
}

// Physical cache row of token s of sequence b, or -1 if s or the layout entry is invalid.
__device__ __forceinline__ int64_t resolve_row(const CacheLayout &L, int b, int s) {
    if (s < 0) return -1;
    int64_t row;
    if (L.block_table) {
        const int lp = s / L.page_size;
        if (lp >= L.pages_per_seq) return -1;
        const int page = L.block_table[(int64_t)b * L.pages_per_seq + lp];
        if (page < 0) return -1;
        row = (int64_t)page * L.page_size + s % L.page_size;
    } else {
        row = (int64_t)L.seq_start[b] + s;
    }
    return (row >= 0 && row < L.num_rows) ? row : -1;
}

// Transposing butterfly over the 32 lanes of a warp: on entry x[0..63] are one key's
// values for heads 0..63; on exit x[0], x[1] hold heads 2*lane, 2*lane+1 combined over
// all 32 keys of the warp (max if kMax, else sum).
template <bool kMax>
__device__ __forceinline__ void warp_transpose_reduce(float (&x)[64], int lane) {
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int half = 32 >> step;
        const int off = 16 >> step;
        const bool upper = (lane & off) != 0;
#pragma unroll
        for (int i = 0; i < half; ++i) {
            const float send = upper ? x[i] : x[i + half];
            const float keep = upper ? x[i + half] : x[i];
            const float recv = __shfl_xor_sync(0xffffffffu, send, off);
            x[i] = kMax ? fmaxf(keep, recv) : keep + recv;
        }
    }
}

__device__ __forceinline__ void tmem_ld64(uint32_t taddr, float (&x)[64]) {
    uint32_t (&r)[64] = reinterpret_cast<uint32_t (&)[64]>(x);
    tmem_ld32(taddr, reinterpret_cast<uint32_t (&)[32]>(r[0]));
    tmem_ld32(taddr + 32, reinterpret_cast<uint32_t (&)[32]>(r[32]));
    tmem_ld_wait();
}

// S^T row of this thread's key: the sum of the two issuers' parts (columns 0-63, 64-127).
__device__ __forceinline__ void tmem_ld_s(uint32_t taddr, float (&x)[64]) {
    uint32_t (&r)[64] = reinterpret_cast<uint32_t (&)[64]>(x);
    tmem_ld32(taddr, reinterpret_cast<uint32_t (&)[32]>(r[0]));
    tmem_ld32(taddr + 32, reinterpret_cast<uint32_t (&)[32]>(r[32]));
    uint32_t y[32];
    tmem_ld32(taddr + 64, y);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] += __uint_as_float(y[i]);
    tmem_ld32(taddr + 96, y);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) x[32 + i] += __uint_as_float(y[i]);
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ MlaMaps maps, const MlaParams p) {
    const int nv = p.d / 64;             // latent (value) chunks
    const int nch = nv + 1;              // + the rope chunk
    const int nmb = (nv + 1) / 2;        // M-blocks of the O product (128 dims each)
    const int ngroups = nmb + 1;         // gather groups: V chunk pairs, then rope
    const int rope = nv;                 // index of the rope chunk (later: P)

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const MlaSmem L = mla_smem(nch);
    uint8_t *qs = smem + L.q;
    uint8_t *tile = smem + L.tile;
    uint8_t *pslot = tile + rope * kChunkBytes;
    int32_t *rows_sm = (int32_t *)(smem + L.rows);   // [2][128] physical rows, -1 invalid
    float *red = (float *)(smem + L.red);
    float *rn = (float *)(smem + L.rn);
    float *alpha = (float *)(smem + L.alpha);
    float *lsum = (float *)(smem + L.lsum);
    uint64_t *bars = (uint64_t *)(smem + L.bars);
    uint64_t *full = bars;           // [ngroups] chunk groups landed
    uint64_t *freeb = bars + 5;      // [ngroups] chunk groups free again
    uint64_t *s_full = bars + 10;    // S^T of the tile is in TMEM
    uint64_t *p_ready = bars + 11;   // P^T written (and O rescaled)
    uint64_t *o_done = bars + 12;    // O^T product of the tile complete
    uint64_t *drain = bars + 13;
    uint64_t *q_full = bars + 14;
    uint64_t *addr_ready = bars + 15;  // [2] row table of a tile written
    uint64_t *addr_empty = bars + 17;  // [2] row table of a tile no longer needed
    volatile int *abort_flag = (volatile int *)(bars + 20);
    uint32_t *tmem_base_sm = (uint32_t *)(bars + 20) + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    griddep_launch_dependents();
    griddep_wait();  // the index set comes from the previous kernel

    // work unit -> (row, layer, split)
    const int unit = blockIdx.x;
    const int split = unit % p.splits;
    const int rl = unit / p.splits;
    const int layer = rl % p.layers;
    const int row = rl / p.layers;
    const int b = row / p.T;
    const int ntiles_all = (p.k + kTileKeys - 1) / kTileKeys;
    const int t_begin = split * p.tiles_per_split;
    const int t_end = min(t_begin + p.tiles_per_split, ntiles_all);
    const int ntiles = max(0, t_end - t_begin);
    const int32_t *idx_row = p.idx + (int64_t)row * p.k;

    if (tid < kHeads) {
        rn[tid] = -INFINITY;
        alpha[tid] = 1.f;
    }
    if (p.r < 64) {
        // columns past d + r of the rope chunk: keep them zero in case the copy leaves
        // out-of-range columns untouched
        for (int e = tid; e < kTileKeys * 8; e += kThreads)
            *(uint4 *)(tile + rope * kChunkBytes + e * 16) = make_uint4(0, 0, 0, 0);
        fence_proxy_async();
    }
    if (tid == 0) {
        for (int g = 0; g < ngroups; ++g) {
            mbar_init(&full[g], kSoftmaxThreads);
            mbar_init(&freeb[g], g == ngroups - 1 ? 2 : 1);  // rope/P chunk: both issuers
        }
        mbar_init(s_full, 2);
        mbar_init(p_ready, kSoftmaxThreads);
        mbar_init(o_done, 2);
        mbar_init(drain, 2);
        mbar_init(q_full, 1);
        mbar_init(&addr_ready[0], 32);
        mbar_init(&addr_ready[1], 32);
        mbar_init(&addr_empty[0], kSoftmaxThreads);
        mbar_init(&addr_empty[1], kSoftmaxThreads);
        *abort_flag = 0;
        fence_barrier_init();
    }
    uint32_t tmem_cols = 32;
    while (tmem_cols < (uint32_t)(2 * kHeads + nmb * kHeads)) tmem_cols <<= 1;
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_base_sm, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_sm;
    const uint32_t tS = tmem;          // 2 x 64 columns: one S^T part per MMA issuer
    const uint32_t tO = tmem + 128;    // nmb x 64 columns

    if (warp == kProducerWarp) {
        // ===== query TMA, then the physical row of every selected key, 2 tiles ahead =====
        if (lane == 0) {
            const CUtensorMap *qmap = &maps.q[layer];
            prefetch_tmap(qmap);
            mbar_arrive_expect_tx(q_full, (uint32_t)(nch * kQChunkBytes));
            for (int c = 0; c < nch; ++c)
                tma_load_2d(qs + c * kQChunkBytes, qmap, q_full, c * 64, row * p.H);
        }
        for (int li = 0; li < ntiles; ++li) {
            const int buf = li & 1;
            if (li >= 2) {
                const bool got = mbar_wait(&addr_empty[buf], ((li - 2) >> 1) & 1, KID_MLA, abort_flag);
                if (!__all_sync(0xffffffffu, got)) break;
            }
            const int j0 = (t_begin + li) * kTileKeys + lane * 4;
            int y[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int j = j0 + e;
                int64_t r = -1;
                if (j < p.k) {
                    const int s = __ldg(idx_row + j);
                    if (s >= 0) {
                        r = resolve_row(p.layout, b, s);
                        if (r < 0) record_error(KID_MLA, ERR_BAD_INDEX);
                    }
                }
                y[e] = (int)r;
            }
            *(int4 *)(rows_sm + buf * kTileKeys + lane * 4) = make_int4(y[0], y[1], y[2], y[3]);
            mbar_arrive(&addr_ready[buf]);
        }
    } else if (warp == kMmaWarp || warp == kMmaWarp2) {
        // ================= MMA issuers =================
        // issuer r: S chunks [c_lo, c_hi) into its own S^T copy, O M-blocks [m_lo, m_hi)
        const int r = warp == kMmaWarp ? 0 : 1;
        const int nch_a = (nch + 1) / 2, nmb_a = (nmb + 1) / 2;
        const int c_lo = r == 0 ? 0 : nch_a, c_hi = r == 0 ? nch_a : nch;
        const int m_lo = r == 0 ? 0 : nmb_a, m_hi = r == 0 ? nmb_a : nmb;
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(128, kHeads, false, false);
            const uint32_t idO = idesc_bf16(128, kHeads, true, true);
            const uint32_t tile_a = smem_u32(tile), q_a = smem_u32(qs), p_a = smem_u32(pslot);
            const uint32_t tSr = tS + (uint32_t)(r * kHeads);
            bool ok = ntiles == 0 || mbar_wait(q_full, 0, KID_MLA, abort_flag);
            for (int li = 0; li < ntiles && ok; ++li) {
                // S^T part = C . Q^T over this issuer's chunks, as their gather groups land
                int waited = -1;
                for (int c = c_lo; c < c_hi && ok; ++c) {
                    const int g = c == rope ? ngroups - 1 : c / 2;
                    if (g != waited) {
                        ok = mbar_wait(&full[g], li & 1, KID_MLA, abort_flag);
                        if (!ok) break;
                        tc_fence_after();
                        fence_proxy_async();  // cp.async (generic proxy) data -> tensor cores
                        waited = g;
                    }
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = make_sdesc(tile_a + c * kChunkBytes + kk * 32, 16, 1024, kLayoutSW128);
                        const uint64_t bd = make_sdesc(q_a + c * kQChunkBytes + kk * 32, 16, 1024, kLayoutSW128);
                        mma_bf16(tSr, ad, bd, idS, (c > c_lo || kk > 0) ? 1u : 0u);
                    }
                }
                if (!ok) break;
                mma_commit(s_full);
                // O^T += C^T . P^T once the probabilities are in place
                if (!mbar_wait(p_ready, li & 1, KID_MLA, abort_flag)) break;
                tc_fence_after();
                for (int j = m_lo; j < m_hi; ++j) {
#pragma unroll
                    for (int ks = 0; ks < kTileKeys / 16; ++ks) {
                        const uint64_t ad = make_sdesc(tile_a + 2 * j * kChunkBytes + ks * 2048, kChunkBytes, 1024, kLayoutSW128);
                        const uint64_t bd = make_sdesc(p_a + ks * 2048, kChunkBytes, 1024, kLayoutSW128);
                        mma_bf16(tO + j * kHeads, ad, bd, idO, (li > 0 || ks > 0) ? 1u : 0u);
                    }
                    if (j < ngroups - 1) mma_commit(&freeb[j]);
                }
                mma_commit(&freeb[ngroups - 1]);
                mma_commit(o_done);
            }
            mma_commit(drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ================= softmax + epilogue (128 threads, one key each) ===============
        const int kl = warp * 32 + lane;          // key lane == TMEM lane
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        float lp[64];
#pragma unroll
        for (int h = 0; h < 64; ++h) lp[h] = 0.f;
        const uint16_t *kv = p.kv[layer];
        const int D = p.d + p.r;
        // Gather group g of tile li (its row table must be ready and the group free):
        // thread t owns one 16-byte column of the group and every 8th (or 16th) row, so
        // its swizzled destination advances by a constant 1 KB (or 2 KB) per step.
        auto gather_group = [&](int li, int g) {
            const int32_t *rows = rows_sm + (li & 1) * kTileKeys;
            const bool is_rope = (g == ngroups - 1);
            const int c0 = is_rope ? rope : 2 * g;
            const int nck = is_rope ? 1 : min(2, nv - 2 * g);
            if (nck == 2) {
                const int gc = kl & 15, rb = kl >> 4;
                const int c = c0 + (gc >> 3), gr = gc & 7;
                uint8_t *dst = tile + c * kChunkBytes + rb * 128 + ((gr ^ rb) << 4);
                const int col = c * 64 + gr * 8;
#pragma unroll 4
                for (int i = 0; i < 16; ++i) {
                    const int r = rows[rb + 8 * i];
                    cp_async_16(dst + i * 1024, r >= 0 ? kv + (int64_t)r * D + col : kv, r >= 0 ? 16u : 0u);
                }
            } else {
                const int gr = kl & 7, rb = kl >> 3;  // rows rb + 16 i
                uint8_t *dst = tile + c0 * kChunkBytes + (rb >> 3) * 1024 + (rb & 7) * 128 + ((gr ^ (rb & 7)) << 4);
                int col = c0 * 64 + gr * 8;
                bool in = true;
                if (is_rope) {
                    col = p.d + gr * 8;
                    in = gr * 8 < p.r;
                }
#pragma unroll 4
                for (int i = 0; i < 8; ++i) {
                    const int r = rows[rb + 16 * i];
                    const bool go = in && r >= 0;
                    cp_async_16(dst + i * 2048, go ? kv + (int64_t)r * D + col : kv, go ? 16u : 0u);
                }
            }
            cp_async_arrive(&full[g]);
        };
        bool ok = true;
        // tile 0: every group is free
        if (ntiles > 0) {
            const bool got = mbar_wait(&addr_ready[0], 0, KID_MLA, abort_flag);
            if (named_bar_or(2, kSoftmaxThreads, !got)) ok = false;
            else
                for (int g = 0; g < ngroups; ++g) gather_group(0, g);
        }
        for (int li = 0; li < ntiles && ok; ++li) {
            // every decision that guards a named barrier or a warp-collective TMEM access
            // is made uniform over the 128 threads first
            const bool got = mbar_wait(s_full, li & 1, KID_MLA, abort_flag);
            if (named_bar_or(2, kSoftmaxThreads, !got)) { ok = false; break; }
            tc_fence_after();
            const bool valid = rows_sm[(li & 1) * kTileKeys + kl] >= 0;
            float x[64];
            tmem_ld_s(tS + lane_addr, x);
#pragma unroll
            for (int h = 0; h < 64; ++h) x[h] = valid ? x[h] * p.scale_log2 : -INFINITY;
            warp_transpose_reduce<true>(x, lane);
            red[warp * 64 + 2 * lane] = x[0];
            red[warp * 64 + 2 * lane + 1] = x[1];
            named_bar_sync(1, kSoftmaxThreads);
            bool need = false;
            if (kl < kHeads) {
                const float m = fmaxf(fmaxf(red[kl], red[64 + kl]), fmaxf(red[128 + kl], red[192 + kl]));
                const float rold = rn[kl];
                need = m > rold + kRescaleLog2;
                const float rnew = need ? m : rold;
                alpha[kl] = need ? ex2_approx(rold - rnew) : 1.f;
                rn[kl] = rnew;
            }
            const bool any = named_bar_or(2, kSoftmaxThreads, need);
            // probabilities of this key for every head
            tmem_ld_s(tS + lane_addr, x);
            uint32_t pk[32];
#pragma unroll
            for (int h = 0; h < 64; h += 2) {
                float pr[2];
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const float rr = rn[h + e];
                    const float lg = x[h + e] * p.scale_log2;
                    pr[e] = (valid && rr != -INFINITY) ? ex2_approx(lg - rr) : 0.f;
                }
                const __nv_bfloat162 pb = __floats2bfloat162_rn(pr[0], pr[1]);
                const float2 pf = __bfloat1622float2(pb);
                lp[h] = fmaf(lp[h], alpha[h], pf.x);
                lp[h + 1] = fmaf(lp[h + 1], alpha[h + 1], pf.y);
                pk[h >> 1] = *reinterpret_cast<const uint32_t *>(&pb);
            }
#pragma unroll
            for (int gr = 0; gr < 8; ++gr)
                *(uint4 *)(pslot + swz128(kl, gr)) =
                    make_uint4(pk[gr * 4 + 0], pk[gr * 4 + 1], pk[gr * 4 + 2], pk[gr * 4 + 3]);
            fence_proxy_async();
            if (any && li > 0) {
                // rescale the running O (needs the previous tile's O product complete)
                const bool got_o = mbar_wait(o_done, (li - 1) & 1, KID_MLA, abort_flag);
                if (named_bar_or(2, kSoftmaxThreads, !got_o)) {
                    ok = false;
                } else {
                    tc_fence_after();
                    for (int mb = 0; mb < nmb; ++mb) {
                        uint32_t v[32];
#pragma unroll
                        for (int half = 0; half < 2; ++half) {
                            const uint32_t ta = tO + lane_addr + mb * kHeads + half * 32;
                            tmem_ld32(ta, v);
                            tmem_ld_wait();
#pragma unroll
                            for (int e = 0; e < 32; ++e)
                                v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha[half * 32 + e]);
                            tmem_st32(ta, v);
                        }
                    }
                    tmem_st_wait();
                }
            }
            tc_fence_before();
            mbar_arrive(p_ready);
            if (!ok) break;
            mbar_arrive(&addr_empty[li & 1]);  // row table of tile li fully used
            // gathers of the next tile, group by group as the O product frees them
            if (li + 1 < ntiles) {
                bool g_ok = mbar_wait(&addr_ready[(li + 1) & 1], ((li + 1) >> 1) & 1, KID_MLA, abort_flag);
                if (named_bar_or(2, kSoftmaxThreads, !g_ok)) { ok = false; break; }
                for (int g = 0; g < ngroups; ++g) {
                    g_ok = mbar_wait(&freeb[g], li & 1, KID_MLA, abort_flag);
                    if (named_bar_or(2, kSoftmaxThreads, !g_ok)) { ok = false; break; }
                    gather_group(li + 1, g);
                }
                if (!ok) break;
            }
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        // ---- epilogue ----
        named_bar_sync(1, kSoftmaxThreads);
        if (ntiles > 0) {
            const bool got = ok && mbar_wait(o_done, (ntiles - 1) & 1, KID_MLA, abort_flag);
            ok = !named_bar_or(2, kSoftmaxThreads, !got);
        }
        tc_fence_after();
        warp_transpose_reduce<false>(lp, lane);
        red[warp * 64 + 2 * lane] = lp[0];
        red[warp * 64 + 2 * lane + 1] = lp[1];
        named_bar_sync(1, kSoftmaxThreads);
        if (kl < kHeads) lsum[kl] = red[kl] + red[64 + kl] + red[128 + kl] + red[192 + kl];
        named_bar_sync(1, kSoftmaxThreads);
        const int unit_out = row * p.layers + layer;
        const bool have_o = ok && ntiles > 0;
        if (p.splits == 1) {
            uint16_t *out = p.out[layer] + (int64_t)row * p.H * p.d;
            for (int mb = 0; mb < nmb; ++mb) {
                const int dim = mb * 128 + kl;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    if (have_o) {
                        tmem_ld32(tO + lane_addr + mb * kHeads + half * 32, v);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0u;
                    }
                    if (dim < p.d) {
#pragma unroll
                        for (int e = 0; e < 32; ++e) {
                            const int h = half * 32 + e;
                            if (h < p.H) {
                                const float l = lsum[h];
                                const float o = l > 0.f ? __uint_as_float(v[e]) / l : 0.f;
                                out[(int64_t)h * p.d + dim] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
                            }
                        }
                    }
                }
            }
            if (kl < p.H && p.lse[layer]) {
                const float l = lsum[kl];
                p.lse[layer][(int64_t)row * p.H + kl] =
                    l > 0.f ? (rn[kl] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
        } else {
            // unnormalised partial: O [64][d], then R [64] (log2 domain), l [64]
            float *part = p.partial + ((int64_t)unit_out * p.splits + split) * (size_t)(kHeads * p.d + 2 * kHeads);
            for (int mb = 0; mb < nmb; ++mb) {
                const int dim = mb * 128 + kl;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    if (have_o) {
                        tmem_ld32(tO + lane_addr + mb * kHeads + half * 32, v);
                        tmem_ld_wait();
                    } else {
#pragma unroll
                        for (int e = 0; e < 32; ++e) v[e] = 0u;
                    }
                    if (dim < p.d) {
#pragma unroll
                        for (int e = 0; e < 32; ++e)
                            part[(int64_t)(half * 32 + e) * p.d + dim] = __uint_as_float(v[e]);
                    }
                }
            }
            if (kl < kHeads) {
                part[kHeads * p.d + kl] = rn[kl];
                part[kHeads * p.d + kHeads + kl] = lsum[kl];
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == kMmaWarp) tmem_dealloc(tmem, tmem_cols);
}

// Merge split-KV partials of one (row, layer, head): weights 2^(R_s - R_max) on the
// partial sums.  One CTA per (unit, head); each thread owns 4 consecutive dims.
constexpr int kCombineThreads = 128;

__global__ void __launch_bounds__(kCombineThreads) mla_combine_kernel(const MlaParams p) {
    griddep_launch_dependents();
    griddep_wait();  // the partials come from the previous kernel
    const int h = blockIdx.x % kHeads;
    const int unit = blockIdx.x / kHeads;  // row * layers + layer
    if (h >= p.H) return;
    const int layer = unit % p.layers;
    const int row = unit / p.layers;
    const size_t stride = (size_t)(kHeads * p.d + 2 * kHeads);
    const float *part = p.partial + (int64_t)unit * p.splits * stride;
    float rs[32], ws[32];
    float rmax = -INFINITY;
    for (int s = 0; s < p.splits; ++s) {
        rs[s] = __ldg(part + s * stride + kHeads * p.d + h);
        rmax = fmaxf(rmax, rs[s]);
    }
    float ltot = 0.f;
    for (int s = 0; s < p.splits; ++s) {
        ws[s] = (rmax == -INFINITY || rs[s] == -INFINITY) ? 0.f : ex2_approx(rs[s] - rmax);
        ltot = fmaf(ws[s], __ldg(part + s * stride + kHeads * p.d + kHeads + h), ltot);
    }
    const float inv = ltot > 0.f ? 1.f / ltot : 0.f;
    uint16_t *out = p.out[layer] + ((int64_t)row * p.H + h) * p.d;
    for (int d0 = threadIdx.x * 4; d0 < p.d; d0 += kCombineThreads * 4) {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int s = 0; s < p.splits; ++s) {
            const float4 v = __ldg(reinterpret_cast<const float4 *>(part + s * stride + (int64_t)h * p.d + d0));
            acc.x = fmaf(ws[s], v.x, acc.x);
            acc.y = fmaf(ws[s], v.y, acc.y);
            acc.z = fmaf(ws[s], v.z, acc.z);
            acc.w = fmaf(ws[s], v.w, acc.w);
        }
        const __nv_bfloat162 a = __floats2bfloat162_rn(acc.x * inv, acc.y * inv);
        const __nv_bfloat162 c = __floats2bfloat162_rn(acc.z * inv, acc.w * inv);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t *>(&a);
        pk.y = *reinterpret_cast<const uint32_t *>(&c);
        *reinterpret_cast<uint2 *>(out + d0) = pk;
    }
    if (threadIdx.x == 0 && p.lse[layer])
        p.lse[layer][(int64_t)row * p.H + h] =
            ltot > 0.f ? (rmax + __log2f(ltot)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

int mla_num_splits(int units, int k, int num_sms) {
    const int ntiles = (k + kTileKeys - 1) / kTileKeys;
    if (units <= 0) return 1;
    // one CTA per SM fits (shared memory); split rows only when there are too few
    int splits = num_sms / units;
    if (splits < 1) splits = 1;
    if (splits > ntiles) splits = ntiles;
    if (splits > 32) splits = 32;
    return splits;
}

size_t mla_partial_bytes(int units, int splits, int d) {
    if (splits <= 1) return 0;
    return (size_t)units * splits * (size_t)(kHeads * d + 2 * kHeads) * sizeof(float);
}

cudaError_t launch_sparse_mla(const MlaParams &p, const MlaMaps &maps, cudaStream_t stream) {
    const int nch = p.d / 64 + 1;
    const MlaSmem L = mla_smem(nch);
    const size_t bytes = L.total + 1024;
    static int attr_bytes = 0;
    if ((int)bytes > attr_bytes) {
        cudaError_t e = set_smem_attrs(sparse_mla_kernel, (int)bytes);
        if (e != cudaSuccess) return e;
        attr_bytes = (int)bytes;
    }
    const int units = p.B * p.T * p.layers;
    if (units <= 0) return cudaSuccess;
    cudaError_t e = launch_pdl(sparse_mla_kernel, dim3(units * p.splits), dim3(kThreads), bytes,
                               stream, maps, p);
    if (e != cudaSuccess || p.splits == 1) return e;
    return launch_pdl(mla_combine_kernel, dim3(units * kHeads), dim3(kCombineThreads), 0, stream, p);
}

DSA_DEFINE_ERROR_READER(take_error_mla)

}  // namespace dsa
