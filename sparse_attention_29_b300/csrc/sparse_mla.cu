// sparse_mla.cu -- sparse MLA in MQA (absorbed) mode over the selected tokens.
//
// Source: "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM", §Sparse MLA
// (DSA runs MLA in MQA mode over the top-K tokens only) and §MLA changes (latent d = 512,
// rope r = 64, 2 bytes per value; 64 query heads).  For a query row with heads h and the
// selected cached rows c_j (d + r wide):
//     logit[h, j] = scale * q[h, :] . c_j          (key = the whole row)
//     o[h, :]     = sum_j softmax_j(logit[h, :]) c_j[:d]   (value = the latent part)
//
// Mapping onto sm_103a.  The selected rows are gathered 64 at a time (a tile) with
// cp.async in 16-byte granules into shared memory in the tensor cores' 128-byte-swizzled
// layout: chunk c of a tile holds dims 64c..64c+63 of its 64 rows.  That one layout
// serves both products:
//   S[head, key]    = Q[head, :] . C[key, :]       A = Q (K-major), B = C (K-major)
//   O^T[dim, head] += C[key, dim]^T P^T[key, head] A = C^T (MN-major), B = P (K-major)
// S runs as M = 64 tcgen05 MMAs (heads on M, keys on N), O^T as M = 128 MMAs (latent
// dims on M, heads on N), fp32 accumulators in tensor memory.
//
// The query (64 heads x 576 x 2 B = 72 KB) and two tiles (2 x 72 KB) fill shared memory,
// so tile i+1 is gathered while tile i is in the products and the softmax.  The gather
// is the pacing item: one SM moves about 35-40 GB/s of 16-byte cp.async only when many
// warps issue them from precomputed row addresses, so eight warps do nothing else
// (row addresses for the next tile are resolved while the current one is in flight).
// Four more warps issue the MMAs, one thread each (a thread issues a tcgen05.mma about
// every 55 cycles): two split the S chunks, each into its own accumulator (the softmax
// adds the two), and two split the O product's M-blocks, so that O of tile i never
// waits behind S of tile i+1.  S^T is double-buffered in tensor memory, so S of tile i+1 overlaps the
// softmax of tile i.
//
// Softmax: the M = 64 accumulator puts head 16w + i in TMEM lane 32w + i (w = warp,
// i < 16); a 16x32bx2 tcgen05.ld hands thread i < 16 of warp w keys 0-31 of that head
// and thread 16 + i keys 32-63, so all 128 softmax threads work and a head's maximum
// and sum over the tile are one thread's plus one shuffle.  A probability is
// p = 2^((S - m) * scale * log2 e) with S and the running maximum m in raw logit units,
// so the one rounded product sees the small difference, not the large logits.  Each p
// goes to the value product as two bf16 halves, hi = bf16(p) and lo = bf16(p - hi):
// the two MMAs over the same latent chunk (hi, then lo) weigh every value row with
// hi + lo, which is p to a relative 2^-16 instead of bf16's 2^-8, and the running sum
// adds exactly hi + lo.  hi is written (one 128-byte row of 64 keys per head) over the
// tile's rope chunk, which S no longer needs; lo goes to one separate buffer, reused
// once the previous tile's value product is done.  Online softmax rescales O in tensor
// memory only when a head's running maximum grows by more than 2^8 (the result is the
// same; the unnormalised terms just stay < 2^8).
//
// Rows with few keys are split over several CTAs (split-KV), merged with the log-sum-exp
// rule.  Up to kMaxClusterSplits splits of a row run as one thread-block cluster: each CTA
// writes its unnormalised O to the workspace and keeps its running maxima and sums in
// shared memory; after one cluster barrier every CTA finishes a slice of the latent dims
// from all splits (the partials come back from L2, the maxima and sums through
// distributed shared memory) -- no second kernel.  More splits than that write partial
// results for a combine kernel.
#include <cuda_bf16.h>

#include <mutex>

#include "internal.h"
#include "ptx.cuh"
#include "topk_core.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 512;       // 16 warps, roles below
constexpr int kSoftmaxThreads = 128;  // warps 0-3: softmax + epilogue
constexpr int kGatherWarp0 = 4;       // warps 4-11: gathers
constexpr int kGatherThreads = 256;
constexpr int kMmaWarp = 12;          // S issuer 0 (also owns the tensor memory)
constexpr int kMmaWarp2 = 13;         // S issuer 1
constexpr int kQWarp = 14;            // query TMA, then O issuer 1
constexpr int kOWarp = 15;            // O issuer 0
constexpr int kTileKeys = 64;
constexpr int kHeads = 64;            // heads padded to 64 (N of both products)
constexpr int kChunkBytes = kTileKeys * 128;  // 64 dims x 64 keys x 2 B
constexpr int kQChunkBytes = kHeads * 128;    // 64 dims x 64 heads x 2 B
constexpr float kRescaleLog2 = 8.f;           // lazy rescale threshold (log2 units)
constexpr int kMaxClusterSplits = 8;          // portable cluster size
static_assert(kMaxClusterSplits * kHeads * 4 <= kChunkBytes, "merge weights alias P_lo");

// named barriers: 1 softmax sync, 2 softmax OR
constexpr int kBarSm = 1, kBarSmOr = 2;

struct MlaSmem {
    uint32_t q, tile, plo, rn, alpha, lsum, wts, vm, bars, total;
};

__host__ __device__ inline MlaSmem mla_smem(int nch) {
    MlaSmem s;
    uint32_t off = 0;
    s.q = off;
    off += (uint32_t)nch * kQChunkBytes;
    s.tile = off;  // two tile buffers
    off += 2u * (uint32_t)nch * kChunkBytes;
    s.plo = off;   // low halves of a tile's probabilities (one buffer, 1024-aligned)
    s.wts = off;   // cluster merge, after the last tile: [split][head] weights
    off += kChunkBytes;
    s.rn = off;
    off += kHeads * 4;
    s.alpha = off;
    off += kHeads * 4;
    s.lsum = off;
    off += kHeads * 4;
    s.vm = off;  // [2 buffers][2] key-validity words of a tile
    off += 16;
    s.bars = off;
    off += 50 * 8 + 16;
    s.total = off;
    return s;
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

// 16x32bx2 load of 32 columns: thread i < 16 of the warp reads TMEM lane (base + i),
// columns [col, col + 32); thread 16 + i reads lane (base + i), columns [col + 32, col + 64).
__device__ __forceinline__ void tmem_ld_pair32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.16x32bx2.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32], 32;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

// This thread's key, 32 heads of S^T: the sum of the two issuers' parts (64 columns apart).
__device__ __forceinline__ void tmem_ld_s(uint32_t taddr, float (&x)[32]) {
    uint32_t c[32];
    tmem_ld_pair32(taddr, reinterpret_cast<uint32_t (&)[32]>(x));
    tmem_ld_pair32(taddr + 64, c);
    tmem_ld_wait();
#pragma unroll
    for (int i = 0; i < 32; ++i) x[i] += __uint_as_float(c[i]);
}

__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ MlaMaps maps, const MlaParams p) {
    const int nv = p.d / 64;             // latent (value) chunks
    const int nch = nv + 1;              // + the rope chunk
    const int nmb = (nv + 1) / 2;        // M-blocks of the O product (128 dims each)
    const int rope = nv;                 // index of the rope chunk (later: P)

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const MlaSmem L = mla_smem(nch);
    uint8_t *qs = smem + L.q;
    uint8_t *tiles = smem + L.tile;
    uint8_t *plo = smem + L.plo;
    uint32_t *vm = (uint32_t *)(smem + L.vm);
    float *rn = (float *)(smem + L.rn);
    float *alpha = (float *)(smem + L.alpha);
    float *lsum = (float *)(smem + L.lsum);
    uint64_t *bars = (uint64_t *)(smem + L.bars);
    // chunk-level pipeline: chunk c of a buffer is refilled as soon as the products that
    // read it are done (latent chunk pair j: O M-block j; rope chunk: P, all of O)
    uint64_t *full = bars;           // [2][9] chunk c of a buffer landed
    uint64_t *tfree = bars + 18;     // [2][4] O M-block j of the buffer's tile done
    uint64_t *tfree_p = bars + 26;   // [2] all of O done: the rope chunk (P) is free
    uint64_t *s_full = bars + 28;    // [2] S^T buffer written
    uint64_t *s_free = bars + 30;    // [2] S^T buffer read by the softmax
    uint64_t *p_ready = bars + 32;   // [2] P of the tile in its buffer (and O rescaled)
    uint64_t *o_done = bars + 34;    // O^T product of a tile complete
    uint64_t *q_full = bars + 35;
    uint64_t *drain = bars + 36;
    volatile int *abort_flag = (volatile int *)(bars + 48);
    uint32_t *tmem_base_sm = (uint32_t *)(bars + 48) + 1;
    int *have_o_sm = (int *)(bars + 49);  // cluster merge: this CTA's O is valid
    const size_t buf_bytes = (size_t)nch * kChunkBytes;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    griddep_launch_dependents();
    // Everything up to griddepcontrol.wait below reads only step inputs (the work unit,
    // the cache layout, the query), so it overlaps the end of the previous kernel.

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
    // Gather warp w (0-7) copies rows 4w..4w+3 and 32+4w..32+4w+3 of every tile; its
    // lanes 0-7 resolve those rows' addresses (lane l: row my_row).
    const int gw = warp - kGatherWarp0;
    const int my_row = (lane & 7) < 4 ? 4 * gw + (lane & 7) : 32 + 4 * gw + (lane & 7) - 4;
    const bool resolver = gw >= 0 && gw < kGatherThreads / 32 && lane < 8;
    const bool paged = p.layout.block_table != nullptr;
    const int64_t seq_base = (resolver && !paged) ? (int64_t)__ldg(p.layout.seq_start + b) : 0;

    if (tid < kHeads) {
        rn[tid] = -INFINITY;
        alpha[tid] = 1.f;
    }
    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            for (int c = 0; c < 9; ++c) mbar_init(&full[i * 9 + c], kGatherThreads);
            for (int j = 0; j < 4; ++j) mbar_init(&tfree[i * 4 + j], 1);
            mbar_init(&tfree_p[i], 2);
            mbar_init(&s_full[i], 2);
            mbar_init(&s_free[i], kSoftmaxThreads);
            mbar_init(&p_ready[i], kSoftmaxThreads);
        }
        mbar_init(o_done, 2);
        mbar_init(q_full, 1);
        mbar_init(drain, 4);
        *abort_flag = 0;
        fence_barrier_init();
    }
    uint32_t tmem_cols = 32;
    while (tmem_cols < (uint32_t)(4 * kHeads + nmb * kHeads)) tmem_cols <<= 1;
    if (warp == kMmaWarp) {
        tmem_alloc(tmem_base_sm, tmem_cols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_sm;
    if (warp == kQWarp && lane == 0 && ntiles > 0) {
        // the query (a step input) streams in while the previous kernel finishes
        const CUtensorMap *qmap = &maps.q[layer];
        prefetch_tmap(qmap);
        mbar_arrive_expect_tx(q_full, (uint32_t)(nch * kQChunkBytes));
        for (int c = 0; c < nch; ++c)
            tma_load_2d(qs + c * kQChunkBytes, qmap, q_full, c * 64, row * p.H);
    }
    griddep_wait();  // the index set (or the scores) come from the previous kernel
    if (p.topk) {
        // this row's top-k first, by the row's splits (the cluster), in the tile buffers
        // (free until the gathers start); the index set then comes back from L2
        TopkParams tp;
        tp.scores = p.scores;
        tp.q_pos = p.q_pos;
        tp.idx = p.idx_out;
        tp.rows = p.B * p.T;
        tp.Lmax = p.Lmax;
        tp.k = p.k;
        tk::topk_row(tp, row, p.splits, p.cluster ? cluster_rank() : 0u, p.topk_slice, tiles);
        // the barrier (arrive.release / wait.acquire at cluster scope, or the CTA barrier)
        // orders the index-set stores, global ones included, before the reads below
        if (p.cluster) cluster_sync();
        else __syncthreads();
    }
    // the resolving gather lanes fetch tile 0's token indices first (through L2: in one
    // launch with the top-k they were written by this cluster a moment ago)
    int s_pre = -1;
    if (resolver && ntiles > 0) {
        const int j = t_begin * kTileKeys + my_row;
        if (j < p.k) s_pre = ldcg_early(idx_row + j);
    }
    const uint32_t tS = tmem;          // [2 buffers][2 issuer parts] x 64 columns
    const uint32_t tO = tmem + 256;    // nmb x 64 columns

    // Roles by warpgroup, each with its register share: the softmax warpgroup holds a
    // key's logits, probabilities and running sums; the others need few.  Every
    // warpgroup returns to 128 before the common tail (the cluster merge).  512 threads
    // launch with 128 registers each (65536); after the adjustment 128 x 168 +
    // 384 x 88 = 55296 are in use.
    if (warp >= kMmaWarp) {
      asm volatile("setmaxnreg.dec.sync.aligned.u32 88;\n" ::: "memory");
      if (warp == kMmaWarp || warp == kMmaWarp2) {
        // ================= S issuers =================
        // issuer r: S chunks [c_lo, c_hi) into its own S^T part
        const int r = warp == kMmaWarp ? 0 : 1;
        const int nch_a = (nch + 1) / 2;
        const int c_lo = r == 0 ? 0 : nch_a, c_hi = r == 0 ? nch_a : nch;
        if (lane == 0) {
            const uint32_t idS = idesc_bf16(kHeads, kTileKeys, false, false);
            // descriptors of chunk 0; the address field (bytes >> 4) is advanced per MMA
            const uint64_t aq0 = make_sdesc(smem_u32(qs), 16, 1024, kLayoutSW128);
            const uint64_t bc0 = make_sdesc(smem_u32(tiles), 16, 1024, kLayoutSW128);
            bool ok = ntiles == 0 || mbar_wait(q_full, 0, KID_MLA, abort_flag);
            for (int li = 0; li < ntiles && ok; ++li) {
                const int bi = li & 1;
                if (li >= 2) ok = mbar_wait(&s_free[bi], ((li - 2) >> 1) & 1, KID_MLA, abort_flag);
                if (!ok) break;
                const uint64_t bct = bc0 + (uint64_t)((bi * buf_bytes) >> 4);
                const uint32_t tSr = tS + (uint32_t)(bi * 2 * kHeads + r * kHeads);
                for (int c = c_lo; c < c_hi && ok; ++c) {
                    ok = mbar_wait(&full[bi * 9 + c], (li >> 1) & 1, KID_MLA, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    fence_proxy_async();  // cp.async (generic proxy) data -> tensor cores
                    const uint64_t ad = aq0 + (uint64_t)(c * (kQChunkBytes >> 4));
                    const uint64_t bd = bct + (uint64_t)(c * (kChunkBytes >> 4));
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk)
                        mma_bf16(tSr, ad + 2 * kk, bd + 2 * kk, idS, (c > c_lo || kk > 0) ? 1u : 0u);
                }
                if (!ok) break;
                mma_commit(&s_full[bi]);
            }
            mma_commit(drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
      } else if (warp == kOWarp || warp == kQWarp) {
        // ============ O issuers: O^T += C^T . P^T once a tile's P is in place ============
        // issuer r: M-blocks [m_lo, m_hi)
        const int r = warp == kOWarp ? 0 : 1;
        const int nmb_a = (nmb + 1) / 2;
        const int m_lo = r == 0 ? 0 : nmb_a, m_hi = r == 0 ? nmb_a : nmb;
        if (lane == 0) {
            const uint32_t idO = idesc_bf16(128, kHeads, true, false);
            // descriptors of buffer 0 (A: M-block 0, K-step 0; B: P, K-step 0); the address
            // field (bytes >> 4) is advanced per MMA
            const uint64_t ac0 = make_sdesc(smem_u32(tiles), kChunkBytes, 1024, kLayoutSW128);
            const uint64_t bp0 = make_sdesc(smem_u32(tiles) + rope * kChunkBytes, 16, 1024, kLayoutSW128);
            const uint64_t bl0 = make_sdesc(smem_u32(plo), 16, 1024, kLayoutSW128);
            for (int li = 0; li < ntiles; ++li) {
                const int bi = li & 1;
                if (!mbar_wait(&p_ready[bi], (li >> 1) & 1, KID_MLA, abort_flag)) break;
                tc_fence_after();
                const uint64_t boff = (uint64_t)((bi * buf_bytes) >> 4);
                for (int j = m_lo; j < m_hi; ++j) {
                    const uint64_t ad = ac0 + boff + (uint64_t)(j * (2 * kChunkBytes >> 4));
                    const uint64_t bd = bp0 + boff;
                    // the same latent chunk pair weighed by the high, then the low halves
#pragma unroll
                    for (int ks = 0; ks < kTileKeys / 16; ++ks)
                        mma_bf16(tO + j * kHeads, ad + ks * (2048 >> 4), bd + 2 * ks, idO, (li > 0 || ks > 0) ? 1u : 0u);
#pragma unroll
                    for (int ks = 0; ks < kTileKeys / 16; ++ks)
                        mma_bf16(tO + j * kHeads, ad + ks * (2048 >> 4), bl0 + 2 * ks, idO, 1u);
                    mma_commit(&tfree[bi * 4 + j]);  // chunks 2j, 2j+1 are free again
                }
                mma_commit(&tfree_p[bi]);
                mma_commit(o_done);
            }
            mma_commit(drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
      }
      asm volatile("setmaxnreg.inc.sync.aligned.u32 128;\n" ::: "memory");
    } else if (warp >= kGatherWarp0) {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 88;\n" ::: "memory");
        // ================= gathers =================
        const int gt = tid - kGatherWarp0 * 32;
        const uint8_t *kv_bytes = reinterpret_cast<const uint8_t *>(p.kv[layer]);
        const int64_t row_bytes = (int64_t)(p.d + p.r) * 2;
        // Each warp resolves its own rows' addresses (lanes 0-7, one row each) ahead of
        // use: the token index of tile li + 2 and the page of tile li + 1 are loaded while
        // tile li is copied, and the addresses reach the copying lanes by shuffles, so the
        // warps never wait on a global load or on each other.  Same rule as resolve_row:
        // a valid token index that does not resolve is an error.
        auto idx_at = [&](int li) -> int {  // token index of this lane's row in tile li
            const int j = (t_begin + li) * kTileKeys + my_row;
            return (resolver && li < ntiles && j < p.k) ? ldcg_early(idx_row + j) : -1;
        };
        auto page_of = [&](int s) -> int {  // block-table entry of token s, or -1
            if (!paged || s < 0) return -1;
            const int lp = s / p.layout.page_size;
            return lp < p.layout.pages_per_seq
                       ? ldg_early(p.layout.block_table + (int64_t)b * p.layout.pages_per_seq + lp)
                       : -1;
        };
        auto finish = [&](int s, int page) -> const uint8_t * {
            if (s < 0) return nullptr;
            int64_t r;
            if (paged) r = page < 0 ? -1 : (int64_t)page * p.layout.page_size + s % p.layout.page_size;
            else r = seq_base + s;
            if (r < 0 || r >= p.layout.num_rows) {
                record_error(KID_MLA, ERR_BAD_INDEX);
                return nullptr;
            }
            return kv_bytes + r * row_bytes;
        };
        const uint8_t *cur = resolver && ntiles > 0 ? finish(s_pre, page_of(s_pre)) : nullptr;
        int s_nx = idx_at(1), pg_nx = -1;  // tile li + 1: token index, page
        // thread gt copies 16-byte granule (gt & 7) of chunk c for rows (gt >> 3) and
        // (gt >> 3) + 32, chunk by chunk, each chunk as soon as its space is free
        const int gi = gt & 7, ra = gt >> 3, rb = ra + 32;
        // decode (one query row per sequence): a selected row is read by this row only, so
        // the gathered rows are a stream read once, and L2 keeps them last; the query rows
        // of a prefill chunk select many of the same rows, which stay in L2 as usual
        const bool read_once = p.T == 1;
        const uint64_t rpol = policy_evict_first();
        // chunks go in the order their space is freed: the two O issuers' M-blocks
        // interleave (0, a, 1, a + 1, ...), the rope chunk (it held P) comes last; 4 bits
        // per position
        uint64_t corder = 0;
        {
            const int nmb_a = (nmb + 1) / 2;
            int pos = 0;
            for (int q = 0; q < nmb; ++q) {
                const int mb = (q & 1) ? nmb_a + (q >> 1) : (q >> 1);
                for (int w = 0; w < 2 && 2 * mb + w < nv; ++w) corder |= (uint64_t)(2 * mb + w) << (4 * pos++);
            }
            corder |= (uint64_t)rope << (4 * pos);
        }
        for (int li = 0; li < ntiles; ++li) {
            const int bi = li & 1;
            uint8_t *buf = tiles + bi * buf_bytes;
            const uint8_t *pa = reinterpret_cast<const uint8_t *>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(cur), lane >> 3));
            const uint8_t *pb = reinterpret_cast<const uint8_t *>(
                __shfl_sync(0xffffffffu, reinterpret_cast<uintptr_t>(cur), 4 + (lane >> 3)));
            pg_nx = page_of(s_nx);  // both loads complete while this tile is copied
            const int s_nn = idx_at(li + 2);
            bool fail = false;
            for (int cpos = 0; cpos < nch; ++cpos) {
                const int c = (int)((corder >> (4 * cpos)) & 15u);
                if (li >= 2 && !fail) {
                    const uint32_t par = ((li - 2) >> 1) & 1;
                    if (c == rope) fail = !mbar_wait(&tfree_p[bi], par, KID_MLA, abort_flag);
                    else if ((c & 1) == 0) fail = !mbar_wait(&tfree[bi * 4 + (c >> 1)], par, KID_MLA, abort_flag);
                }
                if (!fail) {
                    const bool in = c < nv || gi * 8 < p.r;
                    const int off = c * 128 + gi * 16;
                    uint8_t *dst = buf + c * kChunkBytes + ((gi ^ (ra & 7)) << 4);
                    const void *sa = (in && pa) ? pa + off : kv_bytes, *sb = (in && pb) ? pb + off : kv_bytes;
                    const uint32_t na = (in && pa) ? 16u : 0u, nb = (in && pb) ? 16u : 0u;
                    if (read_once) {
                        cp_async_16_hint(dst + ra * 128, sa, na, rpol);
                        cp_async_16_hint(dst + rb * 128, sb, nb, rpol);
                    } else {
                        cp_async_16(dst + ra * 128, sa, na);
                        cp_async_16(dst + rb * 128, sb, nb);
                    }
                }
                cp_async_arrive(&full[bi * 9 + c]);
            }
            cur = resolver && li + 1 < ntiles ? finish(s_nx, pg_nx) : nullptr;
            s_nx = s_nn;
            if (__any_sync(0xffffffffu, fail)) break;
        }
        asm volatile("cp.async.wait_all;" ::: "memory");
        asm volatile("setmaxnreg.inc.sync.aligned.u32 128;\n" ::: "memory");
    } else {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 168;\n" ::: "memory");
        // ================= softmax + epilogue (128 threads) ===============
        // The M = 64 accumulator of S puts head 16w + i in TMEM lane 32w + i (i < 16):
        // thread i < 16 of warp w takes head 16w + i, keys 0-31 of the tile, thread 16 + i
        // the same head, keys 32-63.  Maxima and sums are per thread plus one shuffle.
        const int hrow = warp * 16 + (lane & 15);
        const int kh = lane >> 4;
        const uint32_t lane_addr = (uint32_t)(warp * 32) << 16;
        const float c = p.scale_log2;  // softmax scale * log2 e
        float rmax = -INFINITY;  // running maximum of this head's raw logits q.c
        float lpart = 0.f;       // running sum of this thread's probabilities (hi + lo)
        // validity of key `key` of tile li (same rule as the gathers)
        auto key_valid = [&](int li, int key) -> bool {
            const int j = (t_begin + li) * kTileKeys + key;
            if (li >= ntiles || j >= p.k) return false;
            const int s = __ldcg(idx_row + j);
            return s >= 0 && resolve_row(p.layout, b, s) >= 0;
        };
        if (warp == 0) {
            const uint32_t m0 = __ballot_sync(0xffffffffu, key_valid(0, lane));
            const uint32_t m1 = __ballot_sync(0xffffffffu, key_valid(0, lane + 32));
            if (lane == 0) {
                vm[0] = m0;
                vm[1] = m1;
            }
        }
        named_bar_sync(kBarSm, kSoftmaxThreads);
        bool ok = true;
        for (int li = 0; li < ntiles && ok; ++li) {
            const int bi = li & 1;
            // warp 0 finds the next tile's valid keys (its loads overlap the wait below)
            bool vn0 = false, vn1 = false;
            if (warp == 0) {
                vn0 = key_valid(li + 1, lane);
                vn1 = key_valid(li + 1, lane + 32);
            }
            // every decision that guards a named barrier or a warp-collective TMEM access
            // is made uniform over the 128 threads first
            const bool got = mbar_wait(&s_full[bi], (li >> 1) & 1, KID_MLA, abort_flag);
            if (named_bar_or(kBarSmOr, kSoftmaxThreads, !got)) { ok = false; break; }
            tc_fence_after();
            const uint32_t taS = tS + lane_addr + (uint32_t)(bi * 2 * kTileKeys);
            float x[32];
            tmem_ld_s(taS, x);
            tc_fence_before();
            mbar_arrive(&s_free[bi]);
            const uint32_t vmask = vm[2 * bi + kh];
            float m = -INFINITY;
#pragma unroll
            for (int e = 0; e < 32; ++e) {
                x[e] = ((vmask >> e) & 1u) ? x[e] : -INFINITY;
                m = fmaxf(m, x[e]);
            }
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
            // (m - rmax) * c is +inf while nothing was valid yet, NaN (false) if still nothing is
            const bool need = (m - rmax) * c > kRescaleLog2;
            const float rnew = need ? m : rmax;
            const float al = need ? ex2_approx((rmax - rnew) * c) : 1.f;
            rmax = rnew;
            if (kh == 0) alpha[hrow] = al;
            if (warp == 0) {
                const uint32_t m0 = __ballot_sync(0xffffffffu, vn0);
                const uint32_t m1 = __ballot_sync(0xffffffffu, vn1);
                if (lane == 0) {
                    vm[2 * (bi ^ 1)] = m0;
                    vm[2 * (bi ^ 1) + 1] = m1;
                }
            }
            // the low halves' buffer and the running O are the previous tile's value
            // product's until it is complete
            bool got_o = true;
            if (li > 0) got_o = mbar_wait(o_done, (li - 1) & 1, KID_MLA, abort_flag);
            const bool any = named_bar_or(kBarSmOr, kSoftmaxThreads, need);
            if (named_bar_or(kBarSmOr, kSoftmaxThreads, !got_o)) {
                ok = false;
                break;
            }
            tc_fence_after();
            // probabilities of this head for its 32 keys, as hi + lo bf16 pairs; the sum
            // takes hi + lo (exact in fp32).  P^T goes K-major, head h's 64 keys in one
            // 128-byte row (128-byte swizzle), keys 8g..8g+7 in 16-byte granule g: hi over
            // the tile's rope chunk, lo into the low-halves buffer.
            uint8_t *prow = tiles + bi * buf_bytes + rope * kChunkBytes + hrow * 128;
            uint8_t *lrow = plo + hrow * 128;
            float ps = 0.f;
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint32_t pk[4], lk[4];
#pragma unroll
                for (int e = 0; e < 8; e += 2) {
                    const int i = 8 * q + e;
                    const float p0 = rmax != -INFINITY ? ex2_approx((x[i] - rmax) * c) : 0.f;
                    const float p1 = rmax != -INFINITY ? ex2_approx((x[i + 1] - rmax) * c) : 0.f;
                    const __nv_bfloat162 hb = __floats2bfloat162_rn(p0, p1);
                    const float2 hf = __bfloat1622float2(hb);
                    const __nv_bfloat162 lb = __floats2bfloat162_rn(p0 - hf.x, p1 - hf.y);
                    const float2 lf = __bfloat1622float2(lb);
                    ps += (hf.x + lf.x) + (hf.y + lf.y);
                    pk[e >> 1] = *reinterpret_cast<const uint32_t *>(&hb);
                    lk[e >> 1] = *reinterpret_cast<const uint32_t *>(&lb);
                }
                const int g = 4 * kh + q;
                *(uint4 *)(prow + ((g ^ (hrow & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *(uint4 *)(lrow + ((g ^ (hrow & 7)) << 4)) = make_uint4(lk[0], lk[1], lk[2], lk[3]);
            }
            lpart = fmaf(lpart, al, ps);
            fence_proxy_async();
            if (any && li > 0) {
                // rescale the running O (the previous tile's O product is complete, above);
                // here thread = TMEM lane = latent dim within each M-block; 16 heads at a
                // time (each step's scale factors come from shared memory)
#pragma unroll 1
                for (int mq = 0; mq < 4 * nmb; ++mq) {
                    const int hq = (mq & 3) * 16;
                    const uint32_t ta = tO + lane_addr + (mq >> 2) * kHeads + hq;
                    uint32_t v[16];
                    tmem_ld16(ta, v);
                    tmem_ld_wait();
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha[hq + e]);
                    tmem_st16(ta, v);
                }
                tmem_st_wait();
            }
            tc_fence_before();
            mbar_arrive(&p_ready[bi]);
        }
        // ---- epilogue ----
        named_bar_sync(kBarSm, kSoftmaxThreads);
        if (ntiles > 0) {
            const bool got = ok && mbar_wait(o_done, (ntiles - 1) & 1, KID_MLA, abort_flag);
            ok = !named_bar_or(kBarSmOr, kSoftmaxThreads, !got);
        }
        tc_fence_after();
        const float ltot = lpart + __shfl_xor_sync(0xffffffffu, lpart, 16);
        if (kh == 0) {
            rn[hrow] = rmax;
            lsum[hrow] = ltot;
        }
        named_bar_sync(kBarSm, kSoftmaxThreads);
        const int kl = tid;  // TMEM lane = latent dim within an M-block
        const int unit_out = row * p.layers + layer;
        const bool have_o = ok && ntiles > 0;
        if (p.cluster) {
            // O stays in tensor memory: all warps copy it out for the merge below
            if (tid == 0) *have_o_sm = have_o ? 1 : 0;
            tc_fence_before();
        } else if (p.splits == 1) {
            // the row is complete: its log-sum-exp and 1 / l (into alpha, free now) here,
            // the output below by all warps
            if (tid == 0) *have_o_sm = have_o ? 1 : 0;
            if (kl < kHeads) {
                const float l = lsum[kl];
                alpha[kl] = (have_o && l > 0.f) ? 1.f / l : 0.f;
                if (kl < p.H && p.lse[layer])
                    p.lse[layer][(int64_t)row * p.H + kl] =
                        l > 0.f ? (rn[kl] * c + __log2f(l)) * 0.69314718055994531f : -INFINITY;
            }
            tc_fence_before();
        } else {
            // unnormalised partial: O [64][d], then R [64] (raw logit units), l [64]
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
        asm volatile("setmaxnreg.dec.sync.aligned.u32 128;\n" ::: "memory");
    }

    if (!p.cluster && p.splits == 1) {
        // ===== one split: the output, O / l, from tensor memory by all 16 warps =====
        // warp w reads TMEM lanes 32 (w % 4) .. +31 (latent dims) and columns 16 (w / 4)
        // .. +15 (heads); consecutive threads store consecutive dims of a head
        __syncthreads();  // the softmax warps have seen O complete; 1 / l in alpha
        tc_fence_after();
        const bool valid_o = *have_o_sm != 0;
        const int q = warp & 3, cg = warp >> 2;
        const float *inv = alpha + 16 * cg;  // 1 / l of each head, 0 for an empty row
        uint16_t *out = p.out[layer] + (int64_t)row * p.H * p.d;
#pragma unroll 1
        for (int mb = 0; mb < nmb; ++mb) {
            uint32_t v[16];
            if (valid_o) {
                tmem_ld16(tO + ((uint32_t)(32 * q) << 16) + mb * kHeads + 16 * cg, v);
                tmem_ld_wait();
            } else {
#pragma unroll
                for (int e = 0; e < 16; ++e) v[e] = 0u;
            }
            const int dim = mb * 128 + 32 * q + lane;
            if (dim < p.d) {
#pragma unroll
                for (int e = 0; e < 16; ++e) {
                    const int h = 16 * cg + e;
                    const float o = __uint_as_float(v[e]) * inv[e];
                    if (h < p.H) out[(int64_t)h * p.d + dim] = __bfloat16_as_ushort(__float2bfloat16_rn(o));
                }
            }
        }
    }

    if (p.cluster) {
        // ===== merge the cluster's splits: CTA `split` finishes dims [d_lo, d_hi) =====
        // Every CTA writes its unnormalised O to its slot of the workspace as bf16 in
        // [head][dim] order (all 16 warps: warp w reads TMEM lanes 32 (w % 4) .. +31, the
        // latent dims, columns 16 (w / 4) .. +15, the heads; consecutive threads store
        // consecutive dims), then its running maxima and sums.  After one cluster barrier
        // each CTA reads its slice of every split's slot back from L2 (16-byte loads of 8
        // dims, issued before the weights are known), weighs and sums them in split order
        // and writes the output.  No CTA reads another's shared memory, so none waits for
        // the others once its slice is written.  The exchange moves bf16: one more
        // rounding (relative 2^-9) ahead of a weighted sum of at most eight terms whose
        // result is rounded to bf16 anyway.
        const size_t stride = (size_t)(kHeads * p.d + 2 * kHeads);  // floats per split slot
        const int unit_out = row * p.layers + layer;
        float *part_base = p.partial + (int64_t)unit_out * p.splits * stride;
        __syncthreads();  // the softmax warps have seen O complete; rn, lsum final
        tc_fence_after();
        {
            const bool valid_o = *have_o_sm != 0;
            float *slot = part_base + (size_t)split * stride;
            uint16_t *po = reinterpret_cast<uint16_t *>(slot);
            const int q = warp & 3, cg = warp >> 2;
            // every M-block's 16 columns are loaded before one wait
            uint32_t v[4][16];
#pragma unroll
            for (int mb = 0; mb < 4; ++mb)
                if (mb < nmb) tmem_ld16(tO + ((uint32_t)(32 * q) << 16) + mb * kHeads + 16 * cg, v[mb]);
            tmem_ld_wait();
#pragma unroll
            for (int mb = 0; mb < 4; ++mb) {
                const int dim = mb * 128 + 32 * q + lane;
                if (mb < nmb && dim < p.d) {
#pragma unroll
                    for (int e = 0; e < 16; ++e)
                        po[(int64_t)(16 * cg + e) * p.d + dim] =
                            valid_o ? __bfloat16_as_ushort(__float2bfloat16_rn(__uint_as_float(v[mb][e]))) : (uint16_t)0;
                }
            }
            if (tid < kHeads) {
                slot[kHeads * p.d + tid] = valid_o ? rn[tid] : -INFINITY;
                slot[kHeads * p.d + kHeads + tid] = valid_o ? lsum[tid] : 0.f;
            }
        }
        tc_fence_before();
        // release/acquire at cluster scope: the partials' global stores are visible to the
        // peers' reads after it
        cluster_sync();  // every split's O, maxima and sums are in the workspace
        float *wts = (float *)(smem + L.wts);  // [split][head] weights
        const int ds = ((p.d + p.splits - 1) / p.splits + 7) & ~7;
        const int d_lo = min(p.d, split * ds), d_hi = min(p.d, d_lo + ds);
        const int ng = (d_hi - d_lo) >> 3;  // groups of 8 dims
        const int n_items = ng * kHeads;    // (head, 8 dims); consecutive threads: dims
        const uint16_t *pbase = reinterpret_cast<const uint16_t *>(part_base);
        uint16_t *out = p.out[layer] + (int64_t)row * p.H * p.d;
        auto load_item = [&](int it, uint4 (&v)[kMaxClusterSplits]) {
            const int h = it / max(ng, 1), dim = d_lo + 8 * (it - h * ng);
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s)
                v[s] = (s < p.splits && it < n_items)
                           ? __ldcg(reinterpret_cast<const uint4 *>(pbase + (size_t)s * stride * 2 +
                                                                    (int64_t)h * p.d + dim))
                           : make_uint4(0u, 0u, 0u, 0u);
        };
        auto finish_item = [&](int it, const uint4 (&v)[kMaxClusterSplits]) {
            if (it >= n_items) return;
            const int h = it / ng, dim = d_lo + 8 * (it - h * ng);
            float acc[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s) {
                if (s >= p.splits) break;
                const float w = wts[s * kHeads + h];
                const uint32_t u[4] = {v[s].x, v[s].y, v[s].z, v[s].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    acc[2 * e] = fmaf(w, __uint_as_float(u[e] << 16), acc[2 * e]);
                    acc[2 * e + 1] = fmaf(w, __uint_as_float(u[e] & 0xFFFF0000u), acc[2 * e + 1]);
                }
            }
            if (h < p.H) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[2 * e], acc[2 * e + 1]);
                    pk[e] = *reinterpret_cast<const uint32_t *>(&b2);
                }
                *reinterpret_cast<uint4 *>(out + (int64_t)h * p.d + dim) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
        };
        // this thread's first two items: their loads go out before the weights are known
        uint4 va[kMaxClusterSplits], vb[kMaxClusterSplits];
        load_item(tid, va);
        load_item(tid + kThreads, vb);
        if (tid < kHeads) {
            // every split's maximum and sum for head h, all loads in flight at once
            const int h = tid;
            float rs[kMaxClusterSplits], ls[kMaxClusterSplits];
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s) {
                rs[s] = s < p.splits ? __ldcg(part_base + s * stride + kHeads * p.d + h) : -INFINITY;
                ls[s] = s < p.splits ? __ldcg(part_base + s * stride + kHeads * p.d + kHeads + h) : 0.f;
            }
            float R = -INFINITY;  // raw logit units, like every split's maximum
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s) R = fmaxf(R, rs[s]);
            float Lsum = 0.f;
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s) {
                rs[s] = (R == -INFINITY || rs[s] == -INFINITY) ? 0.f : ex2_approx((rs[s] - R) * p.scale_log2);
                Lsum = fmaf(rs[s], ls[s], Lsum);
            }
            const float inv = Lsum > 0.f ? 1.f / Lsum : 0.f;
#pragma unroll
            for (int s = 0; s < kMaxClusterSplits; ++s) wts[s * kHeads + h] = rs[s] * inv;
            if (split == 0 && h < p.H && p.lse[layer])
                p.lse[layer][(int64_t)row * p.H + h] =
                    Lsum > 0.f ? (R * p.scale_log2 + __log2f(Lsum)) * 0.69314718055994531f : -INFINITY;
        }
        __syncthreads();
        finish_item(tid, va);
        finish_item(tid + kThreads, vb);
        for (int it = tid + 2 * kThreads; it < n_items; it += 2 * kThreads) {
            load_item(it, va);
            load_item(it + kThreads, vb);
            finish_item(it, va);
            finish_item(it + kThreads, vb);
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
    for (int s = 0; s < p.splits; ++s) {  // maxima in raw logit units
        ws[s] = (rmax == -INFINITY || rs[s] == -INFINITY) ? 0.f : ex2_approx((rs[s] - rmax) * p.scale_log2);
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
            ltot > 0.f ? (rmax * p.scale_log2 + __log2f(ltot)) * 0.69314718055994531f : -INFINITY;
}

}  // namespace

int mla_tile_keys() { return kTileKeys; }

// Clusters of `cs` CTAs of the sparse MLA kernel (shared memory for latent width d) that
// the current device runs at once; cached per device, width and cluster size.
static int mla_max_clusters(int cs, int d) {
    constexpr int kDevs = 16;
    static int cache[kDevs][9][9];  // [device][d / 64][cs], 0: not queried yet
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    const int dd = d / 64;
    if (dev >= kDevs || dd < 1 || dd > 8 || cs < 1 || cs > kMaxClusterSplits) return 0;
    std::lock_guard<std::mutex> lock(mu);
    int &c = cache[dev][dd][cs];
    if (c == 0) {
        const size_t bytes = mla_smem(dd + 1).total + 1024;
        // the attribute is set to the largest width's need, so that it never drops below
        // what a launch for another width has already set
        if (set_smem_attrs(sparse_mla_kernel, (int)(mla_smem(9).total + 1024)) != cudaSuccess) {
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
        if (cudaOccupancyMaxActiveClusters(&n, sparse_mla_kernel, &cfg) != cudaSuccess) {
            (void)cudaGetLastError();
            n = 0;
        }
        c = n > 0 ? n : -1;
    }
    return c > 0 ? c : 0;
}

// Split plan of a launch: rows are split only when they are too few to fill the GPU, and
// when the splits of a row form a cluster, all rows' clusters must run at once (a second
// wave would double the time), so the split count comes down until they fit.  `units` is
// the rows of one layer: every layer of an IndexShare launch is split as a separate call
// would split it.
void mla_split_plan(int units, int k, int num_sms, int d, int *splits_out, int *tps_out) {
    const int ntiles = (k + kTileKeys - 1) / kTileKeys;
    int s = units > 0 ? num_sms / units : 1;
    if (s < 1) s = 1;
    if (s > ntiles) s = ntiles;
    if (s > 32) s = 32;
    for (;;) {
        const int tps = (ntiles + s - 1) / s;
        const int sf = (ntiles + tps - 1) / tps;
        if (sf <= 1 || sf > kMaxClusterSplits || units <= mla_max_clusters(sf, d)) {
            *splits_out = sf;
            *tps_out = tps;
            return;
        }
        s = sf - 1;
    }
}

bool mla_cluster_merge(int splits) { return splits > 1 && splits <= kMaxClusterSplits; }

int mla_topk_slice(int Lmax, int splits, int d) {
    if (splits < 1 || splits > kMaxClusterSplits || Lmax <= 0) return 0;
    const int slice = (((Lmax + splits - 1) / splits) + 31) & ~31;
    const uint32_t tile_bytes = 2u * (uint32_t)(d / 64 + 1) * kChunkBytes;
    return tk::topk_layout(slice).total <= tile_bytes ? slice : 0;
}

size_t mla_partial_bytes(int units, int splits, int d) {
    if (splits <= 1) return 0;
    return (size_t)units * splits * (size_t)(kHeads * d + 2 * kHeads) * sizeof(float);
}

cudaError_t launch_sparse_mla(const MlaParams &p, const MlaMaps &maps, cudaStream_t stream) {
    const int nch = p.d / 64 + 1;
    const MlaSmem L = mla_smem(nch);
    const size_t bytes = L.total + 1024;
    static AttrCache attrs;  // set to the largest width's need: every width fits
    cudaError_t ea = ensure_smem_attrs(attrs, sparse_mla_kernel, (int)(mla_smem(9).total + 1024));
    if (ea != cudaSuccess) return ea;
    const int units = p.B * p.T * p.layers;
    if (units <= 0) return cudaSuccess;
    MlaParams q = p;
    q.cluster = mla_cluster_merge(p.splits) ? 1 : 0;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(units * p.splits);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = bytes;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = q.cluster ? p.splits : 1;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    cudaError_t e = cudaLaunchKernelEx(&cfg, sparse_mla_kernel, maps, q);
    if (e != cudaSuccess || p.splits == 1 || q.cluster) return e;
    return launch_pdl(mla_combine_kernel, dim3(units * kHeads), dim3(kCombineThreads), 0, stream, p);
}

DSA_DEFINE_ERROR_READER(take_error_mla)

}  // namespace dsa
