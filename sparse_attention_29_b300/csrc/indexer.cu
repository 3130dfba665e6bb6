// indexer.cu -- lightning indexer scores on the tensor cores.
//
// Source: "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM", §Lightning
// Indexer: per query head the q.k dot product, ReLU, then a weighted sum over the query
// heads gives each cached token its score; keys are single-head, so one key row meets
// every head of the query.
//
// Mapping onto sm_103a.  One tensor-core tile is 128 keys (M) x N query-head columns
// (N = G query rows x HP padded heads) x Di (K), fp8 e4m3 in, fp32 out in tensor memory:
//   S[key, (row, head)] = k8[key, :] . q8[row, head, :]
// After tcgen05.ld each thread owns one key's N accumulators, so ReLU, the weighted
// head sum and both scales need no cross-thread traffic:
//   score[row, key] = k_scale[key] * sum_h (w[row, h] * q_scale[row]) * max(S, 0).
// The key cache streams through a TMA ring of 128-row tiles (HBM-bound for decode);
// the query group sits in shared memory (double-buffered across groups).
//
// Roles (192 threads): warp 0 loads (TMA for keys, plain loads for the query group),
// warp 1 issues the MMAs, warps 2-5 run the epilogue (warp w reads TMEM lanes
// 32*(w%4) .. +31).  CTAs are persistent: the tiles of all query groups form one list
// and each CTA takes a contiguous slice of it, so ragged contexts balance evenly.
#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr int kThreads = 192;
constexpr int kTileKeys = 128;
constexpr int kBoxRows = 64;

struct Smem {
    // offsets (bytes) from the 1024-aligned dynamic shared memory base
    uint32_t kstage, qbuf, qbuf_bytes, wbuf, gpos, prefix, bars, total;
};

__host__ __device__ inline Smem smem_layout(int Di, int N, int G, int stages, int num_groups,
                                            int num_acc) {
    Smem s;
    uint32_t off = 0;
    s.kstage = off;
    off += (uint32_t)stages * kTileKeys * Di;
    s.qbuf = off;
    s.qbuf_bytes = ((uint32_t)N * Di + 1023u) & ~1023u;
    off += 2 * s.qbuf_bytes;
    s.wbuf = off;
    off += 2 * (uint32_t)N * 4;
    s.gpos = off;
    off += 2 * 16 * 4;
    s.prefix = off;
    off += ((uint32_t)num_groups + 1 + 3) / 4 * 16;
    s.bars = off;
    off += (uint32_t)(2 * stages + 4 + 2 * num_acc + 1) * 8 + 16;  // + abort flag, tmem base
    s.total = off;
    (void)G;
    return s;
}

// Byte offset of (row, 16-byte granule) inside a K-major swizzled operand whose rows
// are `pitch` bytes (= the swizzle width, 32/64/128) -- the address-bit swizzle that
// both TMA and the tensor cores apply: bits [4, 4+log2(pitch/16)) ^= bits [7, ...).
__device__ __forceinline__ uint32_t swz_off(int row, int gran, int pitch) {
    const uint32_t lin = (uint32_t)row * pitch + (uint32_t)gran * 16;
    const uint32_t mask = (uint32_t)pitch / 16 - 1;
    return lin ^ (((lin >> 7) & mask) << 4);
}

struct TileCursor {
    const int *prefix;
    int num_groups;
    int g, j, t, te;
    __device__ void init(const int *pre, int ng, int tb, int te_) {
        prefix = pre;
        num_groups = ng;
        t = tb;
        te = te_;
        // the group holding tile tb: last g with prefix[g] <= tb (skipping empty groups)
        int lo = 0, hi = ng - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= tb) lo = mid;
            else hi = mid - 1;
        }
        g = lo;
        while (g < ng - 1 && pre[g + 1] <= tb) ++g;
        j = tb - pre[g];
    }
    __device__ bool valid() const { return t < te; }
    __device__ int tiles_in_group() const { return prefix[g + 1] - prefix[g]; }
    __device__ bool first_in_range(int tb) const { return j == 0 || t == tb; }
    __device__ bool last_in_range() const { return j == tiles_in_group() - 1 || t == te - 1; }
    __device__ void next() {
        ++t;
        ++j;
        while (g < num_groups && j >= prefix[g + 1] - prefix[g]) {
            ++g;
            j = 0;
        }
    }
};

template <int DI>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap kmap, const IndexerParams p) {
    constexpr int kTileBytes = kTileKeys * DI;
    constexpr uint32_t kLayout = DI == 128 ? kLayoutSW128 : (DI == 64 ? kLayoutSW64 : kLayoutSW32);
    constexpr uint32_t kSBO = 8 * DI;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Smem L = smem_layout(DI, p.N, p.G, p.stages, p.num_groups, p.num_acc);
    uint8_t *kstage = smem + L.kstage;
    uint8_t *qbuf = smem + L.qbuf;
    float *wbuf = (float *)(smem + L.wbuf);
    int *gpos = (int *)(smem + L.gpos);
    int *prefix = (int *)(smem + L.prefix);
    uint64_t *bars = (uint64_t *)(smem + L.bars);
    uint64_t *kfull = bars;
    uint64_t *kempty = kfull + p.stages;
    uint64_t *qfull = kempty + p.stages;
    uint64_t *qempty = qfull + 2;
    uint64_t *accfull = qempty + 2;
    uint64_t *accempty = accfull + p.num_acc;
    uint64_t *drain = accempty + p.num_acc;
    volatile int *abort_flag = (volatile int *)(drain + 1);
    uint32_t *tmem_base_sm = (uint32_t *)(drain + 1) + 1;

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;

    // ---- tile list: tiles of each query group, prefix-summed -------------------------
    {
        __shared__ int partial[kThreads];
        const int ng = p.num_groups;
        const int per = (ng + kThreads - 1) / kThreads;
        const int lo = min(tid * per, ng), hi = min(lo + per, ng);
        auto group_tiles = [&](int g) -> int {
            const int b = g / p.groups_per_seq;
            const int gi = g - b * p.groups_per_seq;
            const int r0 = b * p.T + gi * p.G;
            const int nr = min(p.G, p.T - gi * p.G);
            int maxpos = -1;
            for (int i = 0; i < nr; ++i) {
                const int pos = p.q_pos[r0 + i];
                if (pos < 0 || pos >= p.Lmax) {
                    if (blockIdx.x == 0) record_error(KID_INDEXER, ERR_BAD_POSITION);
                    continue;
                }
                maxpos = max(maxpos, pos);
            }
            return (maxpos + kTileKeys) / kTileKeys;
        };
        int local = 0;
        for (int g = lo; g < hi; ++g) local += group_tiles(g);
        partial[tid] = local;
        __syncthreads();
        if (tid == 0) {
            int run = 0;
            for (int i = 0; i < kThreads; ++i) {
                const int v = partial[i];
                partial[i] = run;
                run += v;
            }
            prefix[ng] = run;
        }
        __syncthreads();
        int run = partial[tid];
        for (int g = lo; g < hi; ++g) {
            prefix[g] = run;
            run += group_tiles(g);
        }
        __syncthreads();
    }
    const int total = prefix[p.num_groups];
    const int tb = (int)(((int64_t)total * blockIdx.x) / gridDim.x);
    const int te = (int)(((int64_t)total * (blockIdx.x + 1)) / gridDim.x);
    if (tb >= te) return;

    // ---- barriers, tensor memory -----------------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 1);
            mbar_init(&qempty[i], 1 + 4);
        }
        for (int i = 0; i < p.num_acc; ++i) {
            mbar_init(&accfull[i], 1);
            mbar_init(&accempty[i], 4);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {
        tmem_alloc(tmem_base_sm, (uint32_t)(p.acc_cols * p.num_acc));
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) prefetch_tmap(&kmap);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_sm;

    if (warp == 0) {
        // ================= producer =================
        TileCursor cur;
        cur.init(prefix, p.num_groups, tb, te);
        int it = 0, gcount = 0, issued = 0;
        bool ok = true;
        for (; cur.valid() && ok; cur.next(), ++it) {
            const int b = cur.g / p.groups_per_seq;
            if (cur.first_in_range(tb)) {
                const int slot = gcount & 1, use = gcount >> 1;
                if (use > 0) ok = mbar_wait(&qempty[slot], (use - 1) & 1, KID_INDEXER, abort_flag);
                ok = __all_sync(0xffffffffu, ok);
                if (!ok) break;
                // query group -> qbuf[slot]: row n = qi*HP + h, zero rows for padding
                const int gi = cur.g - b * p.groups_per_seq;
                const int r0 = b * p.T + gi * p.G;
                const int nr = min(p.G, p.T - gi * p.G);
                uint8_t *qdst = qbuf + slot * L.qbuf_bytes;
                const int grans = DI / 16;
                for (int e = lane; e < p.N * grans; e += 32) {
                    const int n = e / grans, gr = e - n * grans;
                    const int qi = n / p.HP, h = n - qi * p.HP;
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (qi < nr && h < p.Hi)
                        v = *(const uint4 *)(p.q8 + (((int64_t)(r0 + qi) * p.Hi + h) * DI) + gr * 16);
                    const int atom = n >> 3;
                    *(uint4 *)(qdst + atom * kSBO + swz_off(n & 7, gr, DI)) = v;
                }
                float *wdst = wbuf + slot * p.N;
                for (int n = lane; n < p.N; n += 32) {
                    const int qi = n / p.HP, h = n - qi * p.HP;
                    float v = 0.f;
                    if (qi < nr && h < p.Hi)
                        v = p.w[(int64_t)(r0 + qi) * p.Hi + h] * p.q_scale[r0 + qi];
                    wdst[n] = v;
                }
                if (lane < 16) {
                    int pos = -1;
                    if (lane < nr) {
                        pos = p.q_pos[r0 + lane];
                        if (pos < 0 || pos >= p.Lmax) pos = -1;
                    }
                    gpos[slot * 16 + lane] = pos;
                }
                fence_proxy_async();
                __syncwarp();
                if (lane == 0) mbar_arrive(&qfull[slot]);
                ++gcount;
            }
            if (lane == 0) {
                const int stage = it % p.stages, use = it / p.stages;
                if (use > 0) ok = mbar_wait(&kempty[stage], (use - 1) & 1, KID_INDEXER, abort_flag);
                if (ok) {
                    const int s0 = cur.j * kTileKeys;
                    const int maxpos = [&] {
                        int m = -1;
                        const int gi = cur.g - b * p.groups_per_seq;
                        const int r0 = b * p.T + gi * p.G;
                        const int nr = min(p.G, p.T - gi * p.G);
                        for (int i = 0; i < nr; ++i) m = max(m, p.q_pos[r0 + i]);
                        return m;
                    }();
                    int ys[2];
                    int nbox = 0;
                    for (int hb = 0; hb < 2; ++hb) {
                        const int s = s0 + hb * kBoxRows;
                        if (s > maxpos) break;
                        int64_t y;
                        if (p.layout.block_table) {
                            const int lp = s / p.layout.page_size;
                            const int page = lp < p.layout.pages_per_seq
                                ? p.layout.block_table[(int64_t)b * p.layout.pages_per_seq + lp] : -1;
                            if (page < 0 || (int64_t)page * p.layout.page_size >= p.layout.num_rows) {
                                record_error(KID_INDEXER, ERR_BAD_PAGE);
                                y = -2 * kBoxRows;  // wholly outside: TMA fills zeros
                            } else {
                                y = (int64_t)page * p.layout.page_size + s % p.layout.page_size;
                            }
                        } else {
                            y = (int64_t)p.layout.seq_start[b] + s;
                            if (y < 0 || y >= p.layout.num_rows) {
                                record_error(KID_INDEXER, ERR_BAD_INDEX);
                                y = -2 * kBoxRows;
                            }
                        }
                        ys[nbox++] = (int)y;
                    }
                    uint8_t *dst = kstage + stage * kTileBytes;
                    mbar_arrive_expect_tx(&kfull[stage], (uint32_t)(nbox * kBoxRows * DI));
                    for (int hb = 0; hb < nbox; ++hb)
                        tma_load_2d(dst + hb * kBoxRows * DI, &kmap, &kfull[stage], 0, ys[hb]);
                    issued = it + 1;
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
        }
        // drain: every issued key load must land before the CTA's shared memory goes away
        if (lane == 0) {
            for (int st = 0; st < p.stages && st < issued; ++st) {
                const int last_use = (issued - 1 - st) / p.stages;  // uses of stage st: 0..last_use
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&kfull[st], last_use & 1) &&
                       globaltimer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (warp == 1) {
        // ================= MMA issuer =================
        if (lane == 0) {
            TileCursor cur;
            cur.init(prefix, p.num_groups, tb, te);
            const uint32_t idesc = idesc_e4m3(128, p.N);
            int it = 0, gcount = 0, slot = 0;
            for (; cur.valid(); cur.next(), ++it) {
                if (cur.first_in_range(tb)) {
                    slot = gcount & 1;
                    if (!mbar_wait(&qfull[slot], (gcount >> 1) & 1, KID_INDEXER, abort_flag)) break;
                    ++gcount;
                }
                const int stage = it % p.stages;
                if (!mbar_wait(&kfull[stage], (it / p.stages) & 1, KID_INDEXER, abort_flag)) break;
                const int abuf = it % p.num_acc, ause = it / p.num_acc;
                if (ause > 0 &&
                    !mbar_wait(&accempty[abuf], (ause - 1) & 1, KID_INDEXER, abort_flag))
                    break;
                tc_fence_after();
                const uint32_t a0 = smem_u32(kstage + stage * kTileBytes);
                const uint32_t b0 = smem_u32(qbuf + slot * L.qbuf_bytes);
                const uint32_t d = tmem + (uint32_t)(abuf * p.acc_cols);
#pragma unroll
                for (int ks = 0; ks < DI / 32; ++ks) {
                    const uint64_t ad = make_sdesc(a0 + ks * 32, 16, kSBO, kLayout);
                    const uint64_t bd = make_sdesc(b0 + ks * 32, 16, kSBO, kLayout);
                    mma_e4m3(d, ad, bd, idesc, ks > 0 ? 1u : 0u);
                }
                mma_commit(&kempty[stage]);
                mma_commit(&accfull[abuf]);
                if (cur.last_in_range()) mma_commit(&qempty[slot]);
            }
            mma_commit(drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
    } else {
        // ================= epilogue =================
        const int quarter = warp & 3;
        const int key_in_tile = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        // this thread's key scale for the tile at cursor c (0 if the row is invalid); the
        // loads run two tiles ahead of their use, off the critical path
        auto key_scale = [&](const TileCursor &c) -> float {
            if (!c.valid()) return 0.f;
            const int bb = c.g / p.groups_per_seq;
            const int s = c.j * kTileKeys + key_in_tile;
            int64_t row;
            if (p.layout.block_table) {
                const int lp = s / p.layout.page_size;
                if (lp >= p.layout.pages_per_seq) return 0.f;
                const int page = p.layout.block_table[(int64_t)bb * p.layout.pages_per_seq + lp];
                if (page < 0) return 0.f;
                row = (int64_t)page * p.layout.page_size + s % p.layout.page_size;
            } else {
                row = (int64_t)p.layout.seq_start[bb] + s;
            }
            return (row >= 0 && row < p.layout.num_rows) ? __ldg(p.k_scale + row) : 0.f;
        };
        TileCursor cur;
        cur.init(prefix, p.num_groups, tb, te);
        TileCursor ahead = cur;
        float ksc_ring0 = key_scale(ahead);
        ahead.next();
        float ksc_ring1 = key_scale(ahead);
        ahead.next();
        int it = 0, gcount = 0, slot = 0;
        for (; cur.valid(); cur.next(), ++it) {
            const float ksc = ksc_ring0;
            ksc_ring0 = ksc_ring1;
            ksc_ring1 = key_scale(ahead);
            ahead.next();
            const int b = cur.g / p.groups_per_seq;
            if (cur.first_in_range(tb)) {
                slot = gcount & 1;
                const bool got = mbar_wait(&qfull[slot], (gcount >> 1) & 1, KID_INDEXER, abort_flag);
                if (!__all_sync(0xffffffffu, got)) break;  // warp-uniform: TMEM loads follow
                ++gcount;
            }
            const int abuf = it % p.num_acc;
            const bool got = mbar_wait(&accfull[abuf], (it / p.num_acc) & 1, KID_INDEXER, abort_flag);
            if (!__all_sync(0xffffffffu, got)) break;
            tc_fence_after();
            const int gi = cur.g - b * p.groups_per_seq;
            const int r0 = b * p.T + gi * p.G;
            const int nr = min(p.G, p.T - gi * p.G);
            const int s = cur.j * kTileKeys + key_in_tile;
            const int *pos = gpos + slot * 16;
            const float *wq = wbuf + slot * p.N;
            const uint32_t tacc = tmem + lane_addr + (uint32_t)(abuf * p.acc_cols);
            for (int qi = 0; qi < nr; ++qi) {
                float a0 = 0.f, a1 = 0.f, a2 = 0.f, a3 = 0.f;  // four independent chains
                for (int c0 = 0; c0 < p.HP; c0 += 64) {
                    uint32_t v[4][16];
                    const int nchunk = min(4, (p.HP - c0) / 16);
#pragma unroll
                    for (int c = 0; c < 4; ++c)
                        if (c < nchunk) tmem_ld16(tacc + (uint32_t)(qi * p.HP + c0 + c * 16), v[c]);
                    tmem_ld_wait();
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        if (c < nchunk) {
                            const float4 *w4 = (const float4 *)(wq + qi * p.HP + c0 + c * 16);
#pragma unroll
                            for (int e4 = 0; e4 < 4; ++e4) {
                                const float4 ww = w4[e4];
                                a0 = fmaf(ww.x, fmaxf(__uint_as_float(v[c][e4 * 4 + 0]), 0.f), a0);
                                a1 = fmaf(ww.y, fmaxf(__uint_as_float(v[c][e4 * 4 + 1]), 0.f), a1);
                                a2 = fmaf(ww.z, fmaxf(__uint_as_float(v[c][e4 * 4 + 2]), 0.f), a2);
                                a3 = fmaf(ww.w, fmaxf(__uint_as_float(v[c][e4 * 4 + 3]), 0.f), a3);
                            }
                        }
                    }
                }
                if (s <= pos[qi])
                    p.scores[(int64_t)(r0 + qi) * p.Lmax + s] = ((a0 + a1) + (a2 + a3)) * ksc;
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&accempty[abuf]);
                if (cur.last_in_range()) mbar_arrive(&qempty[slot]);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, (uint32_t)(p.acc_cols * p.num_acc));
}

template <int DI>
cudaError_t launch_di(const IndexerParams &p, const CUtensorMap &kmap, int grid,
                      cudaStream_t stream) {
    const Smem L = smem_layout(DI, p.N, p.G, p.stages, p.num_groups, p.num_acc);
    const size_t bytes = L.total + 1024;
    static int attr_set_bytes = 0;  // per process; max over calls
    if ((int)bytes > attr_set_bytes) {
        cudaError_t e = cudaFuncSetAttribute(indexer_kernel<DI>,
                                             cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)bytes);
        if (e != cudaSuccess) return e;
        attr_set_bytes = (int)bytes;
    }
    indexer_kernel<DI><<<grid, kThreads, bytes, stream>>>(kmap, p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_indexer(const IndexerParams &p_in, const CUtensorMap &kmap, int num_sms,
                           cudaStream_t stream) {
    IndexerParams p = p_in;
    // shared-memory budget: key ring takes what the query buffers and tile list leave
    const int budget = 227 * 1024 - 1024;
    const Smem base = smem_layout(p.Di, p.N, p.G, 0, p.num_groups, p.num_acc);
    const int per_stage = kTileKeys * p.Di + 16;
    p.stages = (budget - (int)base.total) / per_stage;
    if (p.stages > 12) p.stages = 12;
    if (p.stages < 2) return cudaErrorInvalidConfiguration;
    const int64_t max_tiles = (int64_t)p.num_groups * ((p.Lmax + kTileKeys - 1) / kTileKeys);
    const int grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
    if (grid <= 0) return cudaSuccess;
    switch (p.Di) {
        case 32: return launch_di<32>(p, kmap, grid, stream);
        case 64: return launch_di<64>(p, kmap, grid, stream);
        case 128: return launch_di<128>(p, kmap, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

DSA_DEFINE_ERROR_READER(take_error_indexer)

}  // namespace dsa
