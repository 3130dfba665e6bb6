// cache_append.cu -- the step before the path: new tokens into the caches.
//
// Source: "Inside GLM-5.3: How Sparse Attention Affects DRAM Memory TAM", §Lightning
// Indexer (the indexer keeps a key per cached token, cached like the KV cache) and §MLA
// changes (one 576-wide latent row per token, bf16).  For every new token i of sequence
// seq[i] at position pos[i], with physical row R(seq[i], pos[i]) of the cache layout:
//   scale      = max(amax_c |k_new[i, c]|, 1e-30) / 448           (fp32)
//   k8[R, c]   = e4m3_rne_satfinite(k_new[i, c] / scale)          (the quotient rounded once)
//   k_scale[R] = scale
//   kv[R, :]   = c_new[i, :]                                       (bf16 copy)
// so that scale * e4m3(k8[R, c]) is k_new[i, c] to e4m3 precision, the form the indexer
// reads.
//
// Mapping onto sm_103a.  Memory-bound (about 2.9 KB moved per token): one warp per token;
// a lane holds Di/32 consecutive key values (one vector load), the warp reduces their
// maximum by shuffles, each lane converts its values with the hardware e4m3 conversion
// (cvt.rn.satfinite.e4m3x2.f32: round to nearest even, saturating) and stores its codes
// as one word; the latent row moves as 16-byte loads and stores.  The code is the e4m3
// rounding of the exact quotient: the fp32 quotient is taken rounded toward zero and,
// when inexact (a non-zero fma remainder), its last bit is set ("round to odd"); an
// fp32 value rounded to odd carries enough bits (24 >= 4 + 2) for its rounding to the
// 4-bit e4m3 significand to equal the rounding of the exact quotient (Boldo and
// Melquiond, "Emulation of FMA and correctly rounded sums: proved algorithms using
// rounding to odd", IEEE Trans. Computers 2008).
//
// The kernel waits for its predecessor before touching memory and does not let its own
// successor start early; the indexer that follows reads the key cache only after its own
// griddepcontrol.wait, which waits for this kernel's completion and memory flush.
#include "internal.h"
#include "ptx.cuh"

namespace dsa {
namespace {

constexpr unsigned int KID_APPEND = 5;  // kernel id in the device error word (after KID_COMBINE)
constexpr int kTokensPerBlock = 8;      // one warp per token
constexpr float kE4m3Max = 448.f;
constexpr int kLatentAhead = 3;         // 16-byte latent chunks per lane loaded up front

// Two fp32 values to two e4m3 codes: `lo` in the low byte, `hi` in the high byte.
__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// x / s rounded to odd in fp32: the quotient rounded toward zero, with its last bit set
// when it is inexact (x - q s != 0; the fma gives that remainder's sign exactly).
__device__ __forceinline__ float div_round_odd(float x, float s) {
    const float q = __fdiv_rz(x, s);
    const float r = fmaf(-q, s, x);
    return r != 0.f ? __int_as_float(__float_as_int(q) | 1) : q;
}

template <int DI>
__global__ void __launch_bounds__(32 * kTokensPerBlock) cache_append_kernel(const AppendParams p) {
    griddep_wait();  // earlier kernels in the stream are done with these rows and inputs
    constexpr int kPer = DI / 32;  // key values per lane
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int i = blockIdx.x * kTokensPerBlock + warp;
    if (i >= p.n) return;
    // the loads that do not depend on the destination row go out first: the key, the
    // first 3 x 512 bytes of the latent row (all of a 576-wide bf16 row), the token's
    // sequence and position
    float x[kPer];
    const float *src = p.k_new + (int64_t)i * DI + kPer * lane;
    if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4 *>(src);
        x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
    } else if constexpr (kPer == 2) {
        const float2 v = *reinterpret_cast<const float2 *>(src);
        x[0] = v.x; x[1] = v.y;
    } else {
        x[0] = src[0];
    }
    const int nchunk = p.c_new ? p.D / 8 : 0;  // 16-byte chunks of the latent row
    const uint4 *csrc = reinterpret_cast<const uint4 *>(p.c_new + (int64_t)i * p.D);
    uint4 cb[kLatentAhead];
#pragma unroll
    for (int j = 0; j < kLatentAhead; ++j)
        if (lane + 32 * j < nchunk) cb[j] = csrc[lane + 32 * j];
    const int b = p.seq[i], s = p.pos[i];
    int64_t row = -1;
    if (b >= 0 && b < p.B && s >= 0) {
        if (p.layout.block_table) {
            const int lp = s / p.layout.page_size;
            if (lp < p.layout.pages_per_seq) {
                const int page = p.layout.block_table[(int64_t)b * p.layout.pages_per_seq + lp];
                if (page >= 0) row = (int64_t)page * p.layout.page_size + s % p.layout.page_size;
            }
        } else {
            row = (int64_t)p.layout.seq_start[b] + s;
        }
    }
    if (row < 0 || row >= p.layout.num_rows) {
        if (lane == 0) record_error(KID_APPEND, p.layout.block_table ? ERR_BAD_PAGE : ERR_BAD_INDEX);
        return;
    }

    // ---- indexer key: per-token scale, e4m3 codes ----
    float amax = 0.f;
#pragma unroll
    for (int e = 0; e < kPer; ++e) amax = fmaxf(amax, fabsf(x[e]));
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float scale = fmaxf(amax, 1e-30f) / kE4m3Max;
    uint8_t *dst = p.k8_cache + row * DI + kPer * lane;
#pragma unroll
    for (int e = 0; e < kPer; ++e) x[e] = div_round_odd(x[e], scale);
    if constexpr (kPer == 4) {
        const uint32_t c = (uint32_t)e4m3x2(x[0], x[1]) | ((uint32_t)e4m3x2(x[2], x[3]) << 16);
        *reinterpret_cast<uint32_t *>(dst) = c;
    } else if constexpr (kPer == 2) {
        *reinterpret_cast<uint16_t *>(dst) = e4m3x2(x[0], x[1]);
    } else {
        *dst = (uint8_t)(e4m3x2(x[0], 0.f) & 0xFFu);
    }
    if (lane == 0) p.k_scale[row] = scale;

    // ---- latent row: a plain copy, 16 bytes per lane and step ----
    if (nchunk) {
        uint4 *cdst = reinterpret_cast<uint4 *>(p.kv_cache + row * p.D);
#pragma unroll
        for (int j = 0; j < kLatentAhead; ++j)
            if (lane + 32 * j < nchunk) cdst[lane + 32 * j] = cb[j];
        for (int g = lane + 32 * kLatentAhead; g < nchunk; g += 32) cdst[g] = csrc[g];
    }
}

}  // namespace

cudaError_t launch_cache_append(const AppendParams &p, cudaStream_t stream) {
    if (p.n <= 0) return cudaSuccess;
    const dim3 grid((p.n + kTokensPerBlock - 1) / kTokensPerBlock), block(32 * kTokensPerBlock);
    switch (p.Di) {
        case 32: return launch_pdl(cache_append_kernel<32>, grid, block, 0, stream, p);
        case 64: return launch_pdl(cache_append_kernel<64>, grid, block, 0, stream, p);
        case 128: return launch_pdl(cache_append_kernel<128>, grid, block, 0, stream, p);
        default: return cudaErrorInvalidValue;
    }
}

DSA_DEFINE_ERROR_READER(take_error_append)

}  // namespace dsa
