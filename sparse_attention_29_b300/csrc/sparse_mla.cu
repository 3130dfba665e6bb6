// sparse_mla.cu -- sparse MLA in MQA (absorbed) mode over the selected tokens.
//
// Source: "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM", §Sparse MLA
// (DSA runs MLA in MQA mode over the top-K tokens only) and §MLA changes (latent d = 512,
// rope r = 64, 2 bytes per value; 64 query heads).  For a query row with heads h and the
// selected cached rows c_j (d + r wide):
//     logit[h, j] = scale * q[h, :] . c_j          (key = the whole row)
//     o[h, :]     = sum_j softmax_j(logit[h, :]) c_j[:d]   (value = the latent part)
//
// Mapping onto sm_103a.  The selected rows are gathered 128 at a time (cp.async, 16-byte
// granules) into shared memory in the tensor cores' 128-byte-swizzled layout: chunk c of
// a tile holds dims 64c..64c+63 of the 128 rows.  That one layout serves both products:
//   S^T[key, head]  = C[key, :] . Q[head, :]      A = C (K-major), B = Q (K-major)
//   O^T[dim, head] += C[key, dim]^T P^T[key, head] A = C^T (MN-major), B = P^T (MN-major)
// so both run as M = 128 tcgen05 MMAs (keys resp. latent dims on M, the 64 heads on N)
// with fp32 accumulators in tensor memory (S: 64 columns, O: 4 x 64 columns).  After
// tcgen05.ld a softmax thread owns one key's 64 head logits; per-head maxima are
// reduced across the 128 keys of the tile with a transposing warp butterfly.  The
// probabilities are written (bf16) over the tile's rope chunk, which S no longer needs.
// Online softmax rescales O in tensor memory only when a head's running maximum grows
// by more than 2^8 (the result is the same; the unnormalised terms just stay < 2^8).
// The query (64 heads x 576 x 2 B = 72 KB) and one tile (144 KB) fill shared memory,
// so the next tile's gather is overlapped at chunk granularity: chunks are refilled as
// soon as the O product that reads them has completed.
//
// Rows with few keys are split over several CTAs (split-KV); each writes unnormalised
// partial results that a small combine kernel merges with the log-sum-exp rule.
#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 224;      // warps 0-3 softmax/epilogue, 4 MMA, 5-6 gather
constexpr int kSoftmaxThreads = 128;
constexpr int kProducerThreads = 64;
constexpr int kMmaWarp = 4;
constexpr int kTileKeys = 128;
constexpr int kHeads = 64;         // heads padded to 64 (N of both products)
constexpr int kChunkBytes = kTileKeys * 128;  // 64 dims x 128 keys x 2 B
constexpr int kQChunkBytes = kHeads * 128;    // 64 dims x 64 heads x 2 B
constexpr float kRescaleLog2 = 8.f;           // lazy rescale threshold (log2 units)

struct MlaSmem {
    uint32_t q, tile, rowaddr, red, rn, alpha, lsum, bars, total;
};

__host__ __device__ inline MlaSmem mla_smem(int nch) {
    MlaSmem s;
    uint32_t off = 0;
    s.q = off;
    off += (uint32_t)nch * kQChunkBytes;
    s.tile = off;
    off += (uint32_t)nch * kChunkBytes;
    s.rowaddr = off;
    off += kTileKeys * 8;
    s.red = off;
    off += 4 * kHeads * 4;
    s.rn = off;
    off += kHeads * 4;
    s.alpha = off;
    off += kHeads * 4;
    s.lsum = off;
    off += kHeads * 4;
    s.bars = off;
    off += 16 * 8 + 16;
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

__global__ void __launch_bounds__(kThreads, 1) sparse_mla_kernel(const MlaParams p) {
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
    int64_t *rowaddr = (int64_t *)(smem + L.rowaddr);
    float *red = (float *)(smem + L.red);
    float *rn = (float *)(smem + L.rn);
    float *alpha = (float *)(smem + L.alpha);
    float *lsum = (float *)(smem + L.lsum);
    uint64_t *bars = (uint64_t *)(smem + L.bars);
    uint64_t *full = bars;           // [ngroups]
    uint64_t *freeb = bars + 5;      // [ngroups]
    uint64_t *s_full = bars + 10;
    uint64_t *p_ready = bars + 11;
    uint64_t *o_done = bars + 12;
    uint64_t *drain = bars + 13;
    volatile int *abort_flag = (volatile int *)(bars + 16);
    uint32_t *tmem_base_sm = (uint32_t *)(bars + 16) + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

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
    const uint16_t *kv = p.kv[layer];
    const int D = p.d + p.r;

    // ---- query -> shared memory (zero-padded to 64 heads and to the rope chunk) -------
    {
        const uint16_t *q = p.q[layer] + (int64_t)row * p.H * D;
        for (int e = tid; e < kHeads * nch * 8; e += kThreads) {
            const int c = e / (kHeads * 8);
            const int rem = e - c * (kHeads * 8);
            const int h = rem >> 3, gr = rem & 7;
            uint4 v = make_uint4(0, 0, 0, 0);
            if (h < p.H) {
                int col = -1;
                if (c < nv) col = c * 64 + gr * 8;
                else if (gr * 8 < p.r) col = p.d + gr * 8;
                if (col >= 0) v = *(const uint4 *)(q + (int64_t)h * D + col);
            }
            *(uint4 *)(qs + c * kQChunkBytes + swz128(h, gr)) = v;
        }
        if (tid < kHeads) {
            rn[tid] = -INFINITY;
            alpha[tid] = 1.f;
        }
        fence_proxy_async();
    }
    if (tid == 0) {
        for (int g = 0; g < ngroups; ++g) {
            mbar_init(&full[g], kProducerThreads);
            mbar_init(&freeb[g], 1);
        }
        mbar_init(s_full, 1);
        mbar_init(p_ready, kSoftmaxThreads);
        mbar_init(o_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    uint32_t tmem_cols = 32;
    while (tmem_cols < (uint32_t)(kHeads + nmb * kHeads)) tmem_cols <<= 1;
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_base_sm, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_sm;
    const uint32_t tS = tmem;          // 64 columns
    const uint32_t tO = tmem + 64;     // nmb x 64 columns

    if (warp >= 5) {
        // ================= gather (2 warps; warp w owns tile rows 64w .. 64w+63) =======
        const int pw = warp - 5;
        const int row0 = pw * 64;
        bool ok = true;
        for (int li = 0; li < ntiles && ok; ++li) {
            const int tile_idx = t_begin + li;
            // element offsets of this warp's rows, -1 for padding / invalid entries
            for (int kk = row0 + lane; kk < row0 + 64; kk += 32) {
                const int j = tile_idx * kTileKeys + kk;
                int64_t a = -1;
                if (j < p.k) {
                    const int s = idx_row[j];
                    if (s >= 0) {
                        const int64_t r = resolve_row(p.layout, b, s);
                        if (r < 0) record_error(KID_MLA, ERR_BAD_INDEX);
                        else a = r * D;
                    }
                }
                rowaddr[kk] = a;
            }
            __syncwarp();
            for (int g = 0; g < ngroups; ++g) {
                if (li > 0) {
                    ok = mbar_wait(&freeb[g], (li - 1) & 1, KID_MLA, abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                }
                const bool is_rope = (g == ngroups - 1);
                const int c0 = is_rope ? rope : 2 * g;
                const int nck = is_rope ? 1 : min(2, nv - 2 * g);
                const int gpr = nck * 8;  // granules per row in this group
                for (int e = lane; e < 64 * gpr; e += 32) {
                    const int kr = row0 + e / gpr;
                    const int gg = e % gpr;
                    const int c = c0 + (gg >> 3), gr = gg & 7;
                    const int64_t a = rowaddr[kr];
                    int col;
                    uint32_t bytes = 16;
                    if (is_rope) {
                        col = p.d + gr * 8;
                        if (gr * 8 >= p.r) bytes = 0;
                    } else {
                        col = c * 64 + gr * 8;
                    }
                    if (a < 0) bytes = 0;
                    const uint16_t *src = bytes ? kv + a + col : kv;
                    cp_async_16(tile + c * kChunkBytes + swz128(kr, gr), src, bytes);
                }
                cp_async_arrive(&full[g]);
            }
            __syncwarp();
        }
        // drain: every issued copy lands before shared memory is released
        asm volatile("cp.async.wait_all;" ::: "memory");
    } else if (warp == kMmaWarp) {
        // ================= MMA issuer =================
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(128, kHeads, false, false);
            const uint32_t idO = idesc_bf16(128, kHeads, true, true);
            const uint32_t tile_a = smem_u32(tile), q_a = smem_u32(qs), p_a = smem_u32(pslot);
            for (int li = 0; li < ntiles; ++li) {
                bool ok = true;
                // S^T = C . Q^T over all chunks, group by group as the gathers land
                bool first = true;
                for (int g = 0; g < ngroups && ok; ++g) {
                    ok = mbar_wait(&full[g], li & 1, KID_MLA, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    fence_proxy_async();
                    const bool is_rope = (g == ngroups - 1);
                    const int c0 = is_rope ? rope : 2 * g;
                    const int nck = is_rope ? 1 : min(2, nv - 2 * g);
                    for (int c = c0; c < c0 + nck; ++c) {
#pragma unroll
                        for (int kk = 0; kk < 4; ++kk) {
                            const uint64_t ad = make_sdesc(tile_a + c * kChunkBytes + kk * 32, 16, 1024, kLayoutSW128);
                            const uint64_t bd = make_sdesc(q_a + c * kQChunkBytes + kk * 32, 16, 1024, kLayoutSW128);
                            mma_bf16(tS, ad, bd, idS, first ? 0u : 1u);
                            first = false;
                        }
                    }
                }
                if (!ok) break;
                mma_commit(s_full);
                // O^T += C^T . P^T once the probabilities are in place
                if (!mbar_wait(p_ready, li & 1, KID_MLA, abort_flag)) break;
                tc_fence_after();
                for (int j = 0; j < nmb; ++j) {
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
        bool ok = true;
        for (int li = 0; li < ntiles; ++li) {
            // every decision that guards a named barrier or a warp-collective TMEM access
            // is made uniform over the 128 threads first
            const bool got = mbar_wait(s_full, li & 1, KID_MLA, abort_flag);
            if (named_bar_or(2, kSoftmaxThreads, !got)) { ok = false; break; }
            tc_fence_after();
            const int j = (t_begin + li) * kTileKeys + kl;
            bool valid = false;
            if (j < p.k) valid = resolve_row(p.layout, b, idx_row[j]) >= 0;
            float x[64];
            tmem_ld64(tS + lane_addr, x);
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
            tmem_ld64(tS + lane_addr, x);
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
                if (named_bar_or(2, kSoftmaxThreads, !got_o)) { ok = false; }
                else {
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
        }
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
        if (p.splits == 1) {
            uint16_t *out = p.out[layer] + (int64_t)row * p.H * p.d;
            for (int mb = 0; mb < nmb; ++mb) {
                const int dim = mb * 128 + kl;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t v[32];
                    if (ok && ntiles > 0) {
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
                    if (ok && ntiles > 0) {
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

// Merge split-KV partials: per head, weights 2^(R_s - R_max) on the partial sums.
__global__ void __launch_bounds__(256) mla_combine_kernel(const MlaParams p) {
    const int unit = blockIdx.x;  // row * layers + layer
    const int layer = unit % p.layers;
    const int row = unit / p.layers;
    const size_t stride = (size_t)(kHeads * p.d + 2 * kHeads);
    const float *part = p.partial + (int64_t)unit * p.splits * stride;
    __shared__ float wsc[32][kHeads];  // splits <= 32
    __shared__ float rmax_s[kHeads], ltot_s[kHeads];
    const int tid = threadIdx.x;
    if (tid < kHeads) {
        float rmax = -INFINITY;
        for (int s = 0; s < p.splits; ++s) rmax = fmaxf(rmax, part[s * stride + kHeads * p.d + tid]);
        float ltot = 0.f;
        for (int s = 0; s < p.splits; ++s) {
            const float r = part[s * stride + kHeads * p.d + tid];
            const float w = (rmax == -INFINITY || r == -INFINITY) ? 0.f : ex2_approx(r - rmax);
            wsc[s][tid] = w;
            ltot += w * part[s * stride + kHeads * p.d + kHeads + tid];
        }
        rmax_s[tid] = rmax;
        ltot_s[tid] = ltot;
    }
    __syncthreads();
    uint16_t *out = p.out[layer] + (int64_t)row * p.H * p.d;
    for (int e = tid; e < p.H * p.d; e += blockDim.x) {
        const int h = e / p.d, dim = e - h * p.d;
        float acc = 0.f;
        for (int s = 0; s < p.splits; ++s) acc = fmaf(wsc[s][h], part[s * stride + (int64_t)h * p.d + dim], acc);
        const float l = ltot_s[h];
        out[e] = __bfloat16_as_ushort(__float2bfloat16_rn(l > 0.f ? acc / l : 0.f));
    }
    if (tid < p.H && p.lse[layer]) {
        const float l = ltot_s[tid];
        p.lse[layer][(int64_t)row * p.H + tid] =
            l > 0.f ? (rmax_s[tid] + __log2f(l)) * 0.69314718055994531f : -INFINITY;
    }
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

cudaError_t launch_sparse_mla(const MlaParams &p, cudaStream_t stream) {
    const int nch = p.d / 64 + 1;
    const MlaSmem L = mla_smem(nch);
    const size_t bytes = L.total + 1024;
    static int attr_bytes = 0;
    if ((int)bytes > attr_bytes) {
        cudaError_t e = cudaFuncSetAttribute(sparse_mla_kernel,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bytes);
        if (e != cudaSuccess) return e;
        attr_bytes = (int)bytes;
    }
    const int units = p.B * p.T * p.layers;
    if (units <= 0) return cudaSuccess;
    sparse_mla_kernel<<<units * p.splits, kThreads, bytes, stream>>>(p);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess || p.splits == 1) return e;
    mla_combine_kernel<<<units, 256, 0, stream>>>(p);
    return cudaGetLastError();
}

DSA_DEFINE_ERROR_READER(take_error_mla)

}  // namespace dsa
