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
// Roles (384 threads, three warpgroups): warp 0 produces (it resolves the cache rows of
// 32 tiles at a time, one lane per tile, then issues the TMA key loads, the query-group
// loads and cp.async copies of the key scales into a small ring), warps 1 and 2 issue
// the MMAs of alternate tiles (one elected thread each: the issue loop of one thread,
// ~1100 cycles per tile, would be slower than the 16 KB per ~750 cycles an SM's share of
// HBM delivers), warps 4-11 run the epilogue in two sets of four (warp w reads TMEM lanes
// 32*(w%4) .. +31): in decode the sets take alternate tiles, with several query rows
// per tile both sets take every tile and split its rows.  The epilogue warpgroups hold
// a tile's accumulators in registers, so setmaxnreg moves registers to them from the
// producer warpgroup.  Nothing on the per-tile path waits on a
// global load.  CTAs are persistent: the tiles of all query groups form one list and
// each CTA takes a contiguous slice of it, so ragged contexts balance evenly.
#include "internal.h"
#include "keys.cuh"
#include "ptx.cuh"

namespace dsa {
namespace {


constexpr int kMmaWarps = 2;                    // MMA issuers (alternate tiles): warps 1, 2
// Thread layout.  Warpgroup 0: producer, MMA, MMA, idle; then two epilogue sets of four
// warps.  Decode (one query row of 64 heads per group): the sets take alternate tiles
// (the weights stay in registers).  Several rows per group: both sets take every tile,
// query rows e, e + 2, ... for set e.  (Four sets of one row each were slower.)
// setmaxnreg moves registers from warpgroup 0 to the epilogue; the shares add up to the
// pool the block launches with (threads x the per-thread count ptxas gives the kernel).
template <bool kW64>
struct EpiCfg {
    static constexpr int kSets = 2;
    static constexpr int kWarps = 4 * kSets;
    static constexpr int kThreads = 32 * (4 + kWarps);
    static constexpr int kLaunchRegs = 168;  // 65536 / threads, rounded down to 8
    static constexpr int kRegsControl = 88;
    static constexpr int kRegsEpilogue = 208;
    static_assert(128 * kRegsControl + 32 * kWarps * kRegsEpilogue <= kThreads * kLaunchRegs,
                  "register split");
    static_assert(kThreads * kLaunchRegs <= 65536, "launch registers");
};
constexpr int kTileKeys = 128;
constexpr int kBoxRows = 64;

struct Smem {
    // offsets (bytes) from the 1024-aligned dynamic shared memory base
    uint32_t kstage, qbuf, qbuf_bytes, ksring, wbuf, gpos, prefix, gmax, sel, bars, total;
    int ring;
};

constexpr int kBatch = 32;  // tiles the producer resolves at once (one lane per tile)
constexpr int kStageSlots = 64;  // fused selection: staged candidates per (row, warp)

// Key-scale ring slots.  The producer fills a tile's slot when it issues the tile's key
// load, after the stage-free wait for tile (it - stages); by then the epilogue has
// finished every tile up to (it - stages - num_acc), so this many slots are never overrun.
__host__ __device__ inline int ks_ring_slots(int stages, int num_acc) {
    return stages + num_acc + 1;
}

// sel_rows: query rows per group whose fused selection state (a coarse histogram and
// three counters per row) the CTA keeps; 0 without fused selection.
__host__ __device__ inline Smem smem_layout(int Di, int N, int stages, int num_groups,
                                            int num_acc, int sel_rows) {
    Smem s;
    s.ring = ks_ring_slots(stages, num_acc);
    uint32_t off = 0;
    s.kstage = off;
    off += (uint32_t)stages * kTileKeys * Di;
    s.qbuf = off;
    s.qbuf_bytes = ((uint32_t)N * Di + 1023u) & ~1023u;
    off += 2 * s.qbuf_bytes;
    s.ksring = off;
    off += (uint32_t)s.ring * kTileKeys * 4;
    s.wbuf = off;
    off += 2 * (uint32_t)N * 4;
    s.gpos = off;
    off += 2 * 16 * 4;
    s.prefix = off;
    off += ((uint32_t)num_groups + 1 + 3) / 4 * 16;
    s.gmax = off;  // each group's largest valid position (from the tile list)
    off += ((uint32_t)num_groups + 3) / 4 * 16;
    s.sel = off;  // [rows][kCoarseBins] counts, [4][16] per-row counters, staging
    off += (uint32_t)sel_rows * kCoarseBins * 4 + (sel_rows ? 4 * 16 * 4 : 0);
    off = (off + 15) & ~15u;
    off += (uint32_t)sel_rows * 4 * kStageSlots * 8;  // [row][warp][kStageSlots] (key, index)
    s.bars = off;
    off += (uint32_t)(2 * stages + 4 + 2 * num_acc + 1 + s.ring + 1) * 8 + 16;  // + flag, tmem
    s.total = off;
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

// The query group and in-group index of tile t0 of the list of all (group, key tile) pairs.
struct TileCursor {
    int g, j, t;
    __device__ void init(const int *pre, int ng, int t0, int te) {
        t = t0;
        if (t0 >= te) {
            g = ng;
            j = 0;
            return;
        }
        // the group holding tile t0: last g with prefix[g] <= t0 (skipping empty groups)
        int lo = 0, hi = ng - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= t0) lo = mid;
            else hi = mid - 1;
        }
        g = lo;
        j = t0 - pre[g];
    }
    __device__ bool first_in_range(int tb) const { return j == 0 || t == tb; }
};

// Walks the groups of a CTA's tile range [tb, tb + n) in order: `g` is the group of the
// current tile; at_start/is_last say whether tile `it` (relative) starts or ends its group
// within the range.  One compare per tile; empty groups are skipped at boundaries.
struct GroupWalk {
    const int *prefix;
    int num_groups, tb, n, g, next_start;  // next_start: relative index of the next group
    __device__ void init(const int *pre, int ng, int tb_, int n_) {
        prefix = pre;
        num_groups = ng;
        tb = tb_;
        n = n_;
        int lo = 0, hi = ng - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (pre[mid] <= tb_) lo = mid;
            else hi = mid - 1;
        }
        g = lo;
        next_start = pre[g + 1] - tb_;
    }
    __device__ bool at_start(int it) const { return it == 0 || it == prev_end_; }
    __device__ bool is_last(int it) const { return it + 1 == next_start || it + 1 == n; }
    __device__ void step(int it) {
        if (it + 1 == next_start && it + 1 < n) {
            prev_end_ = it + 1;
            do {
                ++g;
                next_start = prefix[g + 1] - tb;
            } while (next_start == it + 1 && g + 1 < num_groups);
        }
    }
    int prev_end_ = -1;
};

// Largest valid position among the rows of query group g (-1 if none).
__device__ __forceinline__ int group_maxpos(const IndexerParams &p, int g, bool report) {
    const int b = g / p.groups_per_seq;
    const int gi = g - b * p.groups_per_seq;
    const int r0 = b * p.T + gi * p.G;
    const int nr = min(p.G, p.T - gi * p.G);
    int maxpos = -1;
    for (int i = 0; i < nr; ++i) {
        const int pos = __ldg(p.q_pos + r0 + i);
        if (pos < 0 || pos >= p.Lmax) {
            if (report) record_error(KID_INDEXER, ERR_BAD_POSITION);
            continue;
        }
        maxpos = max(maxpos, pos);
    }
    return maxpos;
}

// Packed fp32 pairs for the epilogue's weighted sum: fma.rn.f32x2 rounds each lane as
// fmaf does, so the pairs (even, odd head) reproduce the scalar chains bit for bit.
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ uint64_t fma2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ float sum2(uint64_t v) {
    float lo, hi;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
    return lo + hi;
}
// ReLU of two accumulator words, packed
__device__ __forceinline__ uint64_t relu2(uint32_t a, uint32_t b) {
    return pack2(fmaxf(__uint_as_float(a), 0.f), fmaxf(__uint_as_float(b), 0.f));
}

// Raise row q's selection threshold (a coarse bin) to the highest bin b whose count of
// candidates at or above b reaches k.  One warp; the bins are read from the top down, 32
// at a time.  Counts read while other warps still append are lower bounds, so the bin
// found never passes the row's true k-th best: no score that can still be selected is
// ever skipped.  With `exact` (no appends in flight) it returns the final bin and sets
// *above to the count strictly above it and *at to the count in it; -1 if fewer than k.
__device__ __forceinline__ int sel_scan(const volatile uint32_t *hist, int top, int floor_bin,
                                        uint32_t k, uint32_t *above, uint32_t *at) {
    const int lane = threadIdx.x & 31;
    uint32_t acc = 0;
    for (int b = top; b >= floor_bin; b -= 32) {
        const int bin = b - lane;
        const uint32_t c = bin >= floor_bin ? hist[bin] : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        const uint32_t hit = __ballot_sync(0xffffffffu, acc + incl >= k);
        if (hit) {
            const int f = __ffs(hit) - 1;
            const uint32_t inc_f = __shfl_sync(0xffffffffu, incl, f);
            const uint32_t c_f = __shfl_sync(0xffffffffu, c, f);
            if (above) *above = acc + inc_f - c_f;
            if (at) *at = c_f;
            return b - f;
        }
        acc += __shfl_sync(0xffffffffu, incl, 31);
    }
    return -1;
}

// kW64: decode form (one query row of 64 padded heads per group); its weights stay in
// registers.  Otherwise they are read from shared memory.
// kSel: fused selection (several rows per group only): every CTA owns whole query groups
// and keeps, per row, the candidates that can still be among the row's k best (see
// dsa_indexer_topk) instead of storing scores.
template <int DI, bool kW64, bool kSel>
__global__ void __launch_bounds__(EpiCfg<kW64>::kThreads, 1)
    indexer_kernel(const __grid_constant__ CUtensorMap kmap,
                   const __grid_constant__ CUtensorMap kmap128,
                   const __grid_constant__ CUtensorMap qmap, const IndexerParams p) {
    static_assert(!(kSel && kW64), "fused selection runs the several-rows epilogue");
    constexpr int kThreads = EpiCfg<kW64>::kThreads;
    constexpr int kEpiSets = EpiCfg<kW64>::kSets;
    constexpr int kEpiWarps = EpiCfg<kW64>::kWarps;
    constexpr int kTileBytes = kTileKeys * DI;
    constexpr uint32_t kLayout = DI == 128 ? kLayoutSW128 : (DI == 64 ? kLayoutSW64 : kLayoutSW32);
    constexpr uint32_t kSBO = 8 * DI;

    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = (uint8_t *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const Smem L = smem_layout(DI, p.N, p.stages, p.num_groups, p.num_acc, kSel ? p.G : 0);
    uint8_t *kstage = smem + L.kstage;
    uint8_t *qbuf = smem + L.qbuf;
    float *ksring = (float *)(smem + L.ksring);
    float *wbuf = (float *)(smem + L.wbuf);
    int *gpos = (int *)(smem + L.gpos);
    int *prefix = (int *)(smem + L.prefix);
    int *gmax = (int *)(smem + L.gmax);
    uint64_t *bars = (uint64_t *)(smem + L.bars);
    uint64_t *kfull = bars;
    uint64_t *kempty = kfull + p.stages;
    uint64_t *qfull = kempty + p.stages;
    uint64_t *qempty = qfull + 2;
    uint64_t *accfull = qempty + 2;
    uint64_t *accempty = accfull + p.num_acc;
    uint64_t *drain = accempty + p.num_acc;
    uint64_t *ksfull = drain + 1;
    uint64_t *gsync = ksfull + L.ring;  // fused selection: group-end rounds of the epilogue
    volatile int *abort_flag = (volatile int *)(gsync + 1);
    uint32_t *tmem_base_sm = (uint32_t *)(gsync + 1) + 1;
    // fused selection state of the current group's rows: coarse-bin counts of the
    // candidates kept, and per row the candidates kept, the threshold bin and the highest
    // bin seen
    uint32_t *hist = (uint32_t *)(smem + L.sel);
    uint32_t *sel_n = hist + (kSel ? p.G * kCoarseBins : 0);  // [row][quarter] counts
    int *sel_t = (int *)(sel_n + 16);   // threshold bin
    int *sel_top = sel_t + 16;          // highest bin kept
    float *sel_f = (float *)(sel_top + 16);  // coarse_floor(threshold bin)
    uint2 *stage = (uint2 *)(smem + ((L.sel + (uint32_t)(kSel ? p.G : 0) * kCoarseBins * 4 + 4 * 16 * 4 + 15) & ~15u));

    const int tid = threadIdx.x;
    const int warp = tid >> 5;
    const int lane = tid & 31;
    griddep_launch_dependents();
    // The tile list, the barriers and the tensor memory are set up while the previous
    // kernel of the stream finishes; the producer waits for it (griddepcontrol.wait)
    // before its first load, because that kernel may have written the key cache (a cache
    // append), and the epilogue waits before its first store (a previous top-k may still
    // read the scores).

    // ---- tile list: tiles of each query group, prefix-summed -------------------------
    {
        int *warp_sum = reinterpret_cast<int *>(kstage);  // scratch: the key ring is unused yet
        const int ng = p.num_groups;
        const int per = (ng + kThreads - 1) / kThreads;
        const int lo = min(tid * per, ng), hi = min(lo + per, ng);
        int local = 0;
        for (int g = lo; g < hi; ++g) {
            const int mp = group_maxpos(p, g, blockIdx.x == 0);
            gmax[g] = mp;
            const int n = (mp + kTileKeys) / kTileKeys;
            prefix[g] = n;  // counts first, offsets below
            local += n;
        }
        // block-wide exclusive scan of the per-thread sums
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) warp_sum[warp] = incl;
        __syncthreads();
        if (warp == 0) {
            const int v = lane < kThreads / 32 ? warp_sum[lane] : 0;
            int x = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            if (lane < kThreads / 32) warp_sum[lane] = x - v;
            if (lane == kThreads / 32 - 1) prefix[ng] = x;
        }
        __syncthreads();
        int run = warp_sum[warp] + incl - local;
        for (int g = lo; g < hi; ++g) {
            const int n = prefix[g];
            prefix[g] = run;
            run += n;
        }
        __syncthreads();
    }
    const int total = prefix[p.num_groups];
    int tb = (int)(((int64_t)total * blockIdx.x) / gridDim.x);
    int te = (int)(((int64_t)total * (blockIdx.x + 1)) / gridDim.x);
    if constexpr (kSel) {
        // whole groups: the groups whose first tile falls in this CTA's share of the list
        auto first_group_from = [&](int t) {  // first g with prefix[g] >= t
            int lo = 0, hi = p.num_groups;
            while (lo < hi) {
                const int mid = (lo + hi) >> 1;
                if (prefix[mid] < t) lo = mid + 1;
                else hi = mid;
            }
            return lo;
        };
        tb = prefix[first_group_from(tb)];
        te = prefix[first_group_from(te)];
    }
    if (tb >= te) return;
    const int ntile = te - tb;

    // ---- barriers, tensor memory -----------------------------------------------------
    if (tid == 0) {
        for (int i = 0; i < p.stages; ++i) {
            mbar_init(&kfull[i], 1);
            mbar_init(&kempty[i], 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(&qfull[i], 32);  // every producer lane (lane 0 also adds the TMA bytes)
            mbar_init(&qempty[i], kMmaWarps + kEpiWarps);  // every MMA issuer and epilogue warp
        }
        for (int i = 0; i < p.num_acc; ++i) {
            mbar_init(&accfull[i], 1);
            mbar_init(&accempty[i], kW64 ? 4 : kEpiWarps);  // the warps that read it
        }
        for (int i = 0; i < L.ring; ++i) mbar_init(&ksfull[i], 32);  // every producer lane
        mbar_init(drain, kMmaWarps);
        mbar_init(gsync, kEpiWarps);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 1) {  // allocates and frees the tensor memory
        tmem_alloc(tmem_base_sm, (uint32_t)(p.acc_cols * p.num_acc));
        tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&kmap);
        prefetch_tmap(&kmap128);
        if (p.q_tma) prefetch_tmap(&qmap);
    }
    if constexpr (kSel) {
        const int words = p.G * kCoarseBins + 3 * 16;
        for (int i = tid; i < words; i += kThreads) hist[i] = 0u;
        if (tid < 16) sel_f[tid] = -INFINITY;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_base_sm;

    const bool mma_warp = (warp == 1 || warp == 2);
    const int mma_rank = warp - 1;  // 0 .. kMmaWarps-1
    if (warp < 4) {
      if constexpr (EpiCfg<kW64>::kRegsControl < EpiCfg<kW64>::kLaunchRegs)
          asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(EpiCfg<kW64>::kRegsControl) : "memory");
      if (warp == 0) {
        // ================= producer =================
        // query group g -> slot: q codes by TMA (rows n = qi*HP + h) when the heads need no
        // padding, else plain loads with zero rows; weights * q_scale and positions by the
        // lanes.  Every lane arrives on qfull[slot]; lane 0 also adds the TMA bytes.
        auto load_group = [&](int g, int slot) {
            const int b = g / p.groups_per_seq;
            const int gi = g - b * p.groups_per_seq;
            const int r0 = b * p.T + gi * p.G;
            const int nr = min(p.G, p.T - gi * p.G);
            uint8_t *qdst = qbuf + slot * L.qbuf_bytes;
            if (p.q_tma) {
                if (lane == 0) {
                    mbar_expect_tx(&qfull[slot], (uint32_t)(p.N * DI));
                    tma_load_2d(qdst, &qmap, &qfull[slot], 0, r0 * p.Hi);
                }
            } else {
                constexpr int grans = DI / 16;
                for (int e = lane; e < p.N * grans; e += 32) {
                    const int n = e / grans, gr = e - n * grans;
                    const int qi = n / p.HP, h = n - qi * p.HP;
                    uint4 v = make_uint4(0, 0, 0, 0);
                    if (qi < nr && h < p.Hi)
                        v = __ldg((const uint4 *)(p.q8 + (((int64_t)(r0 + qi) * p.Hi + h) * DI) + gr * 16));
                    *(uint4 *)(qdst + (n >> 3) * kSBO + swz_off(n & 7, gr, DI)) = v;
                }
                fence_proxy_async();
            }
            // the position first, then two weights per lane, all in flight before any use
            const int pos = (lane < 16 && lane < nr) ? __ldg(p.q_pos + r0 + lane) : -1;
            float *wdst = wbuf + slot * p.N;
            for (int n0 = lane; n0 < p.N; n0 += 64) {
                float v[2], sc[2];
#pragma unroll
                for (int u = 0; u < 2; ++u) {
                    const int n = n0 + 32 * u;
                    const int qi = n / p.HP, h = n - qi * p.HP;
                    const bool in = n < p.N && qi < nr && h < p.Hi;
                    v[u] = in ? __ldg(p.w + (int64_t)(r0 + qi) * p.Hi + h) : 0.f;
                    sc[u] = in ? __ldg(p.q_scale + r0 + qi) : 0.f;
                }
#pragma unroll
                for (int u = 0; u < 2; ++u)
                    if (n0 + 32 * u < p.N) wdst[n0 + 32 * u] = v[u] * sc[u];
            }
            if (lane < 16) gpos[slot * 16 + lane] = (pos < 0 || pos >= p.Lmax) ? -1 : pos;
            __syncwarp();
            mbar_arrive(&qfull[slot]);
        };
        // the keys and their scales may have just been written by the previous kernel of
        // the stream (a cache append): the producer reads them only after
        // griddepcontrol.wait, which waits for that kernel's completion and memory flush
        griddep_wait();
        int it = 0, gcount = 1, issued = 0;
        // a sequence's keys are read by one query group only when its rows form one group
        // (decode): then they are a stream read once, and L2 keeps them last
        const bool read_once = p.groups_per_seq == 1;
        const uint64_t kpol = policy_evict_first();
        int pstage = 0, pslot = 0;
        uint32_t pphase = 0;
        bool ok = true;
        // ---- lane l resolves tile it0 + l of a batch in two phases: the raw loads (group,
        // cache page or sequence start, query positions) go out a whole batch ahead, and
        // the box rows are derived from them after the current batch has been issued ----
        // (fetch only moves loaded values into registers; finish() uses them, so nothing
        // here waits for a load in flight)
        int f_g = 0, f_newg = 0, f_s0 = 0, f_maxpos = -1, f_pg0 = -1, f_pg1 = -1, f_on = 0;
        int f_st = 0, f_lp = 0;
        auto fetch = [&](int it0) {
            const int nbf = min(kBatch, ntile - it0);
            f_on = lane < nbf;
            if (f_on) {
                TileCursor c;
                c.init(prefix, p.num_groups, tb + it0 + lane, te);
                f_g = c.g;
                f_newg = c.first_in_range(tb) && (it0 + lane > 0);  // the first is loaded
                const int b = c.g / p.groups_per_seq;
                f_s0 = c.j * kTileKeys;
                if (p.layout.block_table) {
                    const int lp0 = f_s0 / p.layout.page_size, lp1 = (f_s0 + kBoxRows) / p.layout.page_size;
                    const int *bt = p.layout.block_table + (int64_t)b * p.layout.pages_per_seq;
                    f_lp = (lp0 < p.layout.pages_per_seq ? 1 : 0) | (lp1 < p.layout.pages_per_seq ? 2 : 0);
                    f_pg0 = ldg_early(bt + ((f_lp & 1) ? lp0 : 0));
                    f_pg1 = ldg_early(bt + ((f_lp & 2) ? lp1 : 0));
                } else {
                    f_st = ldg_early(p.layout.seq_start + b);
                }
                f_maxpos = gmax[c.g];
            }
        };
        int l_g = 0, l_newg = 0, l_nbox = 0, l_y0 = 0, l_y1 = 0, l_r0 = -1, l_r1 = -1;
        auto finish = [&]() {
            l_g = f_g;
            l_newg = f_newg;
            l_nbox = 0;
            l_y0 = l_y1 = 0;
            l_r0 = l_r1 = -1;
            if (!f_on) return;
            int64_t yb[2];
            if (p.layout.block_table) {
                const int pg0 = (f_lp & 1) ? f_pg0 : -1, pg1 = (f_lp & 2) ? f_pg1 : -1;
                yb[0] = pg0 < 0 ? -1 : (int64_t)pg0 * p.layout.page_size + f_s0 % p.layout.page_size;
                yb[1] = pg1 < 0 ? -1 : (int64_t)pg1 * p.layout.page_size + (f_s0 + kBoxRows) % p.layout.page_size;
            } else {
                yb[0] = (int64_t)f_st + f_s0;
                yb[1] = (int64_t)f_st + f_s0 + kBoxRows;
            }
            int ys[2], rs[2];
            for (int hb = 0; hb < 2; ++hb) {
                ys[hb] = 0;
                rs[hb] = -1;
                if (f_s0 + hb * kBoxRows > f_maxpos) continue;
                const int64_t y = yb[hb];
                const bool good = y >= 0 && y < p.layout.num_rows;
                if (!good) record_error(KID_INDEXER, p.layout.block_table ? ERR_BAD_PAGE : ERR_BAD_INDEX);
                ys[hb] = good ? (int)y : -2 * kBoxRows;  // wholly outside: TMA fills zeros
                rs[hb] = good ? (int)y : -1;
                ++l_nbox;
            }
            l_y0 = ys[0];
            l_y1 = ys[1];
            l_r0 = rs[0];
            l_r1 = rs[1];
        };
        // the first batch's cache rows are fetched while the range's first group loads
        fetch(0);
        {
            TileCursor c0;
            c0.init(prefix, p.num_groups, tb, te);
            load_group(c0.g, 0);
        }
        finish();
        while (ok && it < ntile) {
            const int nb = min(kBatch, ntile - it);
            if (it + nb < ntile) fetch(it + nb);  // next batch's loads in flight meanwhile
            // ---- issue the batch in order ----
            for (int t = 0; t < nb; ++t, ++it) {
                const int g = __shfl_sync(0xffffffffu, l_g, t);
                if (__shfl_sync(0xffffffffu, l_newg, t)) {
                    const int slot = gcount & 1, use = gcount >> 1;
                    if (use > 0) ok = mbar_wait(&qempty[slot], (use - 1) & 1, KID_INDEXER, abort_flag);
                    ok = __all_sync(0xffffffffu, ok);
                    if (!ok) break;
                    load_group(g, slot);
                    ++gcount;
                }
                const int nbox = __shfl_sync(0xffffffffu, l_nbox, t);
                const int y0 = __shfl_sync(0xffffffffu, l_y0, t);
                const int y1 = __shfl_sync(0xffffffffu, l_y1, t);
                const int r0k = __shfl_sync(0xffffffffu, l_r0, t);
                const int r1k = __shfl_sync(0xffffffffu, l_r1, t);
                if (lane == 0) {
                    const int stage = pstage;
                    if (it >= p.stages) ok = mbar_wait(&kempty[stage], pphase ^ 1u, KID_INDEXER, abort_flag);
                    if (ok) {
                        uint8_t *dst = kstage + stage * kTileBytes;
                        mbar_arrive_expect_tx(&kfull[stage], (uint32_t)(nbox * kBoxRows * DI));
                        if (read_once) {  // keys no other query group reads: evict first
                            if (nbox == 2 && y1 == y0 + kBoxRows) {
                                tma_load_2d_hint(dst, &kmap128, &kfull[stage], 0, y0, kpol);  // one 128-row box
                            } else {
                                if (nbox > 0) tma_load_2d_hint(dst, &kmap, &kfull[stage], 0, y0, kpol);
                                if (nbox > 1) tma_load_2d_hint(dst + kBoxRows * DI, &kmap, &kfull[stage], 0, y1, kpol);
                            }
                        } else if (nbox == 2 && y1 == y0 + kBoxRows) {
                            tma_load_2d(dst, &kmap128, &kfull[stage], 0, y0);  // one 128-row box
                        } else {
                            if (nbox > 0) tma_load_2d(dst, &kmap, &kfull[stage], 0, y0);
                            if (nbox > 1) tma_load_2d(dst + kBoxRows * DI, &kmap, &kfull[stage], 0, y1);
                        }
                        issued = it + 1;
                    }
                }
                ok = __shfl_sync(0xffffffffu, ok, 0);
                if (!ok) break;
                if (++pstage == p.stages) { pstage = 0; pphase ^= 1u; }
                // this tile's key scales -> ring slot (free: see ks_ring_slots); 4 per lane
                {
                    const int slot = pslot;
                    if (++pslot == L.ring) pslot = 0;
                    float *ks = ksring + slot * kTileKeys + lane * 4;
                    const int k = lane * 4;
                    const int base = k < kBoxRows ? r0k : r1k;
                    const int64_t row = base < 0 ? -1 : (int64_t)base + (k & (kBoxRows - 1));
                    if (row >= 0 && row + 4 <= p.layout.num_rows &&
                        (reinterpret_cast<uintptr_t>(p.k_scale + row) & 15) == 0) {
                        cp_async_16(ks, p.k_scale + row, 16u);
                    } else {
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            const bool good = row >= 0 && row + e < p.layout.num_rows;
                            cp_async_4(ks + e, good ? p.k_scale + row + e : p.k_scale, good ? 4u : 0u);
                        }
                    }
                    cp_async_arrive(&ksfull[slot]);
                }
            }
            finish();
        }
        // drain: every issued copy must land before the CTA's shared memory goes away
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0) {
            for (int st = 0; st < p.stages && st < issued; ++st) {
                const int last_use = (issued - 1 - st) / p.stages;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_try_wait(&kfull[st], last_use & 1) &&
                       globaltimer_ns() - t0 < kWaitLimitNs) {
                }
            }
        }
    } else if (mma_warp) {
        // ================= MMA issuers =================
        // Per tile: stage, accumulator and phases advance by counters; the group changes
        // when the tile index reaches the next group's first tile (one compare per tile).
        if (lane == 0) {
            const uint32_t idesc = idesc_e4m3(128, p.N);
            const uint64_t adesc0 = make_sdesc(smem_u32(kstage), 16, kSBO, kLayout);
            const uint64_t bdesc0 = make_sdesc(smem_u32(qbuf), 16, kSBO, kLayout);
            GroupWalk gw;
            gw.init(prefix, p.num_groups, tb, ntile);
            int stage = 0, abuf = 0, gcount = 0, qslot = 0;
            uint32_t kphase = 0, aphase = 0;
            bool ok = true;
            for (int it = 0; it < ntile && ok; ++it) {
                if (gw.at_start(it)) {
                    qslot = gcount & 1;
                    ok = mbar_wait(&qfull[qslot], (gcount >> 1) & 1, KID_INDEXER, abort_flag);
                    ++gcount;
                    if (!ok) break;
                }
                if (it % kMmaWarps == mma_rank) {
                    ok = mbar_wait(&kfull[stage], kphase, KID_INDEXER, abort_flag);
                    if (ok && it >= p.num_acc)
                        ok = mbar_wait(&accempty[abuf], aphase ^ 1u, KID_INDEXER, abort_flag);
                    if (!ok) break;
                    tc_fence_after();
                    const uint32_t a_off = (uint32_t)(stage * kTileBytes) >> 4;
                    const uint32_t b_off = (uint32_t)(qslot * L.qbuf_bytes) >> 4;
                    const uint32_t d = tmem + (uint32_t)(abuf * p.acc_cols);
#pragma unroll
                    for (int ks = 0; ks < DI / 32; ++ks)
                        mma_e4m3(d, adesc0 + a_off + 2 * ks, bdesc0 + b_off + 2 * ks, idesc, ks > 0 ? 1u : 0u);
                    mma_commit(&kempty[stage]);
                    mma_commit(&accfull[abuf]);
                }
                // every issuer releases the query slot at the group's end (its own MMAs on
                // that slot, if any, are covered by the commit)
                if (gw.is_last(it)) mma_commit(&qempty[qslot]);
                gw.step(it);
                if (++stage == p.stages) { stage = 0; kphase ^= 1u; }
                if (++abuf == p.num_acc) { abuf = 0; aphase ^= 1u; }
            }
            mma_commit(drain);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait(drain, 0) && globaltimer_ns() - t0 < kWaitLimitNs) {
            }
        }
        __syncwarp();
      }
      // warp 3 has no role
    } else {
        if constexpr (EpiCfg<kW64>::kRegsEpilogue > EpiCfg<kW64>::kLaunchRegs)
            asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(EpiCfg<kW64>::kRegsEpilogue) : "memory");
        // ================= epilogue =================
        griddep_wait();  // earlier kernels in the stream are done with the scores
        const int quarter = warp & 3;
        const int eset = (warp - 4) / 4;  // set e: warps 4e+4 .. 4e+7
        const int key_in_tile = quarter * 32 + lane;
        const uint32_t lane_addr = (uint32_t)(quarter * 32) << 16;
        float wr[kW64 ? 64 : 1];
        GroupWalk gw;
        gw.init(prefix, p.num_groups, tb, ntile);
        int abuf = 0, kslot = 0, gcount = 0, slot = 0;
        uint32_t aphase = 0, ksphase = 0;
        int r0 = 0, nr = 0, gfirst = 0;  // current group: first row, rows, first tile (abs.)
        uint32_t grounds = 0;            // fused selection: group-end rounds completed
        const int ew = warp - 4;         // epilogue warp 0 .. kEpiWarps-1
        // fused selection: keep (key, index) of a visible score of row q (warp-wide call)
        // if its bin reaches the row's threshold `thr` (read once per tile: a threshold
        // one tile old is lower, which only keeps more); counts its bin, and the warp's
        // highest kept bin raises the row's highest bin
        // Each of the four warps serving a row appends to its own quarter of the row's list
        // (a warp sees 32 of every 128 keys, so a quarter of cap always holds them).  Kept
        // candidates are staged in shared memory and go out 32 at a time: one coalesced
        // 8-byte store per lane, and the 32 bin counts and the highest bin with every lane
        // active.  Counts in registers, for the j-th row of this set: sel_stg[j] staged,
        // sel_cnt[j] written to the list.
        uint32_t sel_cnt[kSel ? 2 : 1] = {}, sel_stg[kSel ? 2 : 1] = {};
        const int64_t seg = p.cap / 4;
        // write out `n` (<= 32) staged entries of row q (this set's row j), keep the rest
        auto sel_flush = [&](int q, int j, uint32_t n) {
            uint2 *st = stage + (q * 4 + quarter) * kStageSlots;
            const uint32_t cnt = j ? sel_cnt[1] : sel_cnt[0];
            const uint32_t stg = j ? sel_stg[1] : sel_stg[0];
            __syncwarp();
            uint32_t ck = 0;
            if ((uint32_t)lane < n) {
                const uint2 e = st[lane];
                ck = coarse_key(key_score(e.x));
                if (cnt + lane < seg) p.cand[(int64_t)(r0 + q) * p.cap + quarter * seg + cnt + lane] = e;
                atomicAdd(&hist[q * kCoarseBins + ck], 1u);
            }
            const uint32_t hi = __reduce_max_sync(0xffffffffu, ck);
            if (lane == 0 && n) atomicMax(&sel_top[q], (int)hi);
            __syncwarp();
            uint2 rest = make_uint2(0u, 0u);  // the staged entries past the first n move down
            const bool mv = (uint32_t)lane + n < stg;
            if (mv) rest = st[lane + n];
            __syncwarp();
            if (mv) st[lane] = rest;
            __syncwarp();
            if (j) { sel_cnt[1] = cnt + n; sel_stg[1] = stg - n; }
            else { sel_cnt[0] = cnt + n; sel_stg[0] = stg - n; }
        };
        auto sel_emit = [&](int q, int s, float sc, bool keep, float thr) {
            const bool pass = keep && sc >= thr;
            const uint32_t m = __ballot_sync(0xffffffffu, pass);
            if (!m) return;
            const int j = q >= kEpiSets ? 1 : 0;
            const uint32_t stg = j ? sel_stg[1] : sel_stg[0];
            if (pass) stage[(q * 4 + quarter) * kStageSlots + stg + __popc(m & ((1u << lane) - 1u))] =
                make_uint2(full_key(sc), (uint32_t)s);
            if (j) sel_stg[1] = stg + __popc(m);
            else sel_stg[0] = stg + __popc(m);
            if (stg + __popc(m) >= 32) sel_flush(q, j, 32);
        };
        // one group-end round: every epilogue warp arrives, then waits for all (bounded)
        auto sel_round = [&]() -> bool {
            __syncwarp();
            if (lane == 0) mbar_arrive(gsync);
            const bool ok = mbar_wait(gsync, grounds & 1u, KID_INDEXER, abort_flag);
            ++grounds;
            return __all_sync(0xffffffffu, ok);
        };
        for (int it = 0; it < ntile; ++it) {
            if (gw.at_start(it)) {
                slot = gcount & 1;
                const bool got = mbar_wait(&qfull[slot], (gcount >> 1) & 1, KID_INDEXER, abort_flag);
                if (!__all_sync(0xffffffffu, got)) break;  // warp-uniform: TMEM loads follow
                ++gcount;
                const int g = gw.g;
                const int b = g / p.groups_per_seq;
                const int gi = g - b * p.groups_per_seq;
                r0 = b * p.T + gi * p.G;
                nr = min(p.G, p.T - gi * p.G);
                gfirst = prefix[g];
                if constexpr (kW64) {
#pragma unroll
                    for (int h = 0; h < 64; h += 4) {
                        const float4 v = *(const float4 *)(wbuf + slot * p.N + h);
                        wr[h] = v.x;
                        wr[h + 1] = v.y;
                        wr[h + 2] = v.z;
                        wr[h + 3] = v.w;
                    }
                }
            }
            // decode: the two sets take alternate tiles; several query rows per tile: every
            // set takes every tile, query rows eset, eset + kEpiSets, ...
            if (!kW64 || (it & (kEpiSets - 1)) == eset) {
                const bool got = mbar_wait(&accfull[abuf], aphase, KID_INDEXER, abort_flag) &&
                                 mbar_wait(&ksfull[kslot], ksphase, KID_INDEXER, abort_flag);
                if (!__all_sync(0xffffffffu, got)) break;
                tc_fence_after();
                const float ksc = ksring[kslot * kTileKeys + key_in_tile];
                const int s = (tb + it - gfirst) * kTileKeys + key_in_tile;
                const int *pos = gpos + slot * 16;
                const uint32_t tacc = tmem + lane_addr + (uint32_t)(abuf * p.acc_cols);
                if constexpr (kW64) {
                    uint32_t v[64];
                    tmem_ld32(tacc, *reinterpret_cast<uint32_t (*)[32]>(&v[0]));
                    tmem_ld32(tacc + 32, *reinterpret_cast<uint32_t (*)[32]>(&v[32]));
                    tmem_ld_wait();
                    // four chains (heads h mod 4) as two packed pairs
                    uint64_t a01 = 0, a23 = 0;
#pragma unroll
                    for (int h = 0; h < 64; h += 4) {
                        a01 = fma2(pack2(wr[h + 0], wr[h + 1]), relu2(v[h + 0], v[h + 1]), a01);
                        a23 = fma2(pack2(wr[h + 2], wr[h + 3]), relu2(v[h + 2], v[h + 3]), a23);
                    }
                    if (s <= pos[0])
                        p.scores[(int64_t)r0 * p.Lmax + s] = (sum2(a01) + sum2(a23)) * ksc;
                } else {
                    // both sets work on every tile: set e takes query rows e, e + 2, ...
                    const float *wq = wbuf + slot * p.N;
                    if (!kSel && p.HP == 64 && eset + kEpiSets < nr) {
                        // this set's two rows (64 heads: at most 256 / 64 = 4 rows per group)
                        // together: both rows' 64-column loads, one wait, then the two rows'
                        // sums interleaved, each row's chains as in the one-row loop below
                        // (twice the independent work per wait: prefill_8k 7.41 -> 6.73 ms;
                        // with fused selection it spilled and was slower)
                        const int qa = eset, qb = eset + kEpiSets;
                        uint32_t va[64], vb[64];
                        tmem_ld32(tacc + (uint32_t)(qa * 64), *reinterpret_cast<uint32_t (*)[32]>(&va[0]));
                        tmem_ld32(tacc + (uint32_t)(qa * 64 + 32), *reinterpret_cast<uint32_t (*)[32]>(&va[32]));
                        tmem_ld32(tacc + (uint32_t)(qb * 64), *reinterpret_cast<uint32_t (*)[32]>(&vb[0]));
                        tmem_ld32(tacc + (uint32_t)(qb * 64 + 32), *reinterpret_cast<uint32_t (*)[32]>(&vb[32]));
                        tmem_ld_wait();
                        const ulonglong2 *wa = reinterpret_cast<const ulonglong2 *>(wq + qa * 64);
                        const ulonglong2 *wb = reinterpret_cast<const ulonglong2 *>(wq + qb * 64);
                        uint64_t a01 = 0, a23 = 0, b01 = 0, b23 = 0;
#pragma unroll
                        for (int h = 0; h < 64; h += 4) {
                            const ulonglong2 x = wa[h >> 2], y = wb[h >> 2];
                            a01 = fma2(x.x, relu2(va[h + 0], va[h + 1]), a01);
                            a23 = fma2(x.y, relu2(va[h + 2], va[h + 3]), a23);
                            b01 = fma2(y.x, relu2(vb[h + 0], vb[h + 1]), b01);
                            b23 = fma2(y.y, relu2(vb[h + 2], vb[h + 3]), b23);
                        }
                        const float sa = (sum2(a01) + sum2(a23)) * ksc;
                        const float sb = (sum2(b01) + sum2(b23)) * ksc;
                        if (s <= pos[qa]) p.scores[(int64_t)(r0 + qa) * p.Lmax + s] = sa;
                        if (s <= pos[qb]) p.scores[(int64_t)(r0 + qb) * p.Lmax + s] = sb;
                    } else if (kSel || p.HP == 64) {  // the fused selection runs 64-head rows only
                        // this set's rows one at a time: one 64-column load and wait each
                        for (int q = eset; q < nr; q += kEpiSets) {
                            // fused selection: this row's threshold for the tile, and whether
                            // the row selects at all (it sees more than k tokens)
                            const float thr = kSel ? *(volatile float *)&sel_f[q] : 0.f;
                            const bool keep_row = kSel && pos[q] + 1 > p.k;
                            uint32_t v0[64];
                            tmem_ld32(tacc + (uint32_t)(q * 64), *reinterpret_cast<uint32_t (*)[32]>(&v0[0]));
                            tmem_ld32(tacc + (uint32_t)(q * 64 + 32), *reinterpret_cast<uint32_t (*)[32]>(&v0[32]));
                            tmem_ld_wait();
                            const float4 *w0 = (const float4 *)(wq + q * 64);
                            uint64_t a01 = 0, a23 = 0;  // four chains as two packed pairs
#pragma unroll
                            for (int h = 0; h < 64; h += 4) {
                                const ulonglong2 ww = reinterpret_cast<const ulonglong2 *>(w0)[h >> 2];
                                a01 = fma2(ww.x, relu2(v0[h + 0], v0[h + 1]), a01);
                                a23 = fma2(ww.y, relu2(v0[h + 2], v0[h + 3]), a23);
                            }
                            const float sc = (sum2(a01) + sum2(a23)) * ksc;
                            if constexpr (kSel) sel_emit(q, s, sc, keep_row && s <= pos[q], thr);
                            else if (s <= pos[q]) p.scores[(int64_t)(r0 + q) * p.Lmax + s] = sc;
                        }
                    } else if constexpr (!kSel) {
                        // other head counts: this set's rows one at a time, 32 heads per
                        // load (then 16 for the rest; HP is a multiple of 16)
                        for (int q = eset; q < nr; q += kEpiSets) {
                            float a0 = 0.f, a1 = 0.f;
                            int c0 = 0;
                            for (; c0 + 32 <= p.HP; c0 += 32) {
                                uint32_t v[32];
                                tmem_ld32(tacc + (uint32_t)(q * p.HP + c0), v);
                                tmem_ld_wait();
                                const float *wr = wq + q * p.HP + c0;
#pragma unroll
                                for (int e = 0; e < 32; e += 2) {
                                    a0 = fmaf(wr[e], fmaxf(__uint_as_float(v[e]), 0.f), a0);
                                    a1 = fmaf(wr[e + 1], fmaxf(__uint_as_float(v[e + 1]), 0.f), a1);
                                }
                            }
                            if (c0 < p.HP) {
                                uint32_t v[16];
                                tmem_ld16(tacc + (uint32_t)(q * p.HP + c0), v);
                                tmem_ld_wait();
                                const float *wr = wq + q * p.HP + c0;
#pragma unroll
                                for (int e = 0; e < 16; e += 2) {
                                    a0 = fmaf(wr[e], fmaxf(__uint_as_float(v[e]), 0.f), a0);
                                    a1 = fmaf(wr[e + 1], fmaxf(__uint_as_float(v[e + 1]), 0.f), a1);
                                }
                            }
                            if (s <= pos[q]) p.scores[(int64_t)(r0 + q) * p.Lmax + s] = (a0 + a1) * ksc;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&accempty[abuf]);
                if constexpr (kSel) {
                    // every sixteenth tile one warp of the set (in turn) raises the set's
                    // rows' thresholds
                    if ((it & 15) == 15 && ((it >> 4) & 3) == quarter) {
                        for (int q = eset; q < nr; q += kEpiSets) {
                            const int t_cur = *(volatile int *)&sel_t[q];
                            const int tnew = sel_scan(hist + q * kCoarseBins,
                                                      *(volatile int *)&sel_top[q], t_cur,
                                                      (uint32_t)p.k, nullptr, nullptr);
                            if (lane == 0 && tnew > t_cur) {
                                *(volatile int *)&sel_t[q] = tnew;
                                *(volatile float *)&sel_f[q] = coarse_floor(tnew);
                            }
                        }
                    }
                }
            }
            if (gw.is_last(it)) {
                __syncwarp();
                if (lane == 0) mbar_arrive(&qempty[slot]);
                if constexpr (kSel) {
                    // the group's last tile: after every warp's appends, warp q finishes row q
                    // (its final bin and counts to meta), then the state is cleared for the
                    // next group; each step is a bounded round over all epilogue warps
                    // this warp writes out what it still stages, then its counts of its rows'
                    // list quarters go to shared memory for the finishing warp
                    if (eset < nr) sel_flush(eset, 0, sel_stg[0]);
                    if (eset + kEpiSets < nr) sel_flush(eset + kEpiSets, 1, sel_stg[1]);
                    if (lane == 0) {
                        if (eset < nr) sel_n[eset * 4 + quarter] = sel_cnt[0];
                        if (eset + kEpiSets < nr) sel_n[(eset + kEpiSets) * 4 + quarter] = sel_cnt[1];
                    }
                    sel_cnt[0] = sel_stg[0] = 0;
                    if constexpr (kSel) sel_cnt[1] = sel_stg[1] = 0;
                    if (!sel_round()) break;
                    if (ew < nr) {
                        const int pq = gpos[slot * 16 + ew];
                        if (pq >= 0 && pq + 1 > p.k) {
                            uint32_t above = 0, at = 0;
                            const int b0 = sel_scan(hist + ew * kCoarseBins, sel_top[ew], 0,
                                                    (uint32_t)p.k, &above, &at);
                            if (b0 < 0) record_error(KID_INDEXER, ERR_BAD_INDEX);
                            if (lane == 0) {
                                p.meta[2 * (r0 + ew)] = make_uint4(sel_n[ew * 4], sel_n[ew * 4 + 1],
                                                                   sel_n[ew * 4 + 2], sel_n[ew * 4 + 3]);
                                p.meta[2 * (r0 + ew) + 1] = make_uint4((uint32_t)max(b0, 0), above, at, 0u);
                            }
                        }
                    }
                    if (!sel_round()) break;
                    const int words = nr * kCoarseBins;
                    for (int i = ew * 32 + lane; i < words; i += kEpiWarps * 32) hist[i] = 0u;
                    if (ew == 0 && lane < 16) {
                        sel_t[lane] = 0;
                        sel_top[lane] = 0;
                        sel_f[lane] = -INFINITY;
                    }
                    if (!sel_round()) break;
                }
            }
            gw.step(it);
            if (++abuf == p.num_acc) { abuf = 0; aphase ^= 1u; }
            if (++kslot == L.ring) { kslot = 0; ksphase ^= 1u; }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, (uint32_t)(p.acc_cols * p.num_acc));
}

template <int DI, bool kW64, bool kSel>
cudaError_t launch_di(const IndexerParams &p, const CUtensorMap &kmap,
                      const CUtensorMap &kmap128, const CUtensorMap &qmap, int grid,
                      cudaStream_t stream) {
    const Smem L = smem_layout(DI, p.N, p.stages, p.num_groups, p.num_acc, kSel ? p.G : 0);
    const size_t bytes = L.total + 1024;
    static AttrCache attrs;
    cudaError_t e = ensure_smem_attrs(attrs, indexer_kernel<DI, kW64, kSel>, (int)bytes);
    if (e != cudaSuccess) return e;
    return launch_pdl(indexer_kernel<DI, kW64, kSel>, dim3(grid), dim3(EpiCfg<kW64>::kThreads),
                      bytes, stream, kmap, kmap128, qmap, p);
}

template <int DI>
cudaError_t launch_for_di(const IndexerParams &p, const CUtensorMap &kmap,
                          const CUtensorMap &kmap128, const CUtensorMap &qmap, int grid,
                          cudaStream_t stream) {
    if (p.sel) return launch_di<DI, false, true>(p, kmap, kmap128, qmap, grid, stream);
    if (p.N == 64 && p.G == 1) return launch_di<DI, true, false>(p, kmap, kmap128, qmap, grid, stream);
    return launch_di<DI, false, false>(p, kmap, kmap128, qmap, grid, stream);
}

}  // namespace

cudaError_t launch_indexer(const IndexerParams &p_in, const CUtensorMap &kmap,
                           const CUtensorMap &kmap128, const CUtensorMap &qmap, int num_sms,
                           cudaStream_t stream) {
    IndexerParams p = p_in;
    // shared-memory budget: the key ring takes what the rest leaves, up to 12 stages
    const int budget = 227 * 1024 - 1024;
    const int sel_rows = p.sel ? p.G : 0;
    p.stages = 12;  // ~192 KB in flight per SM keeps HBM busy across the ~3-6 us load latency
    while (p.stages >= 2 &&
           (int)smem_layout(p.Di, p.N, p.stages, p.num_groups, p.num_acc, sel_rows).total > budget)
        --p.stages;
    if (p.stages < 2) return cudaErrorInvalidConfiguration;
    const int64_t max_tiles = (int64_t)p.num_groups * ((p.Lmax + kTileKeys - 1) / kTileKeys);
    const int grid = (int)(max_tiles < num_sms ? max_tiles : num_sms);
    if (grid <= 0) return cudaSuccess;
    switch (p.Di) {
        case 32: return launch_for_di<32>(p, kmap, kmap128, qmap, grid, stream);
        case 64: return launch_for_di<64>(p, kmap, kmap128, qmap, grid, stream);
        case 128: return launch_for_di<128>(p, kmap, kmap128, qmap, grid, stream);
        default: return cudaErrorInvalidValue;
    }
}

DSA_DEFINE_ERROR_READER(take_error_indexer)

}  // namespace dsa
