// keys.cuh -- order-preserving integer images of fp32 scores, shared by the top-k
// selections.
//
// full_key: a bijection from fp32 scores (one key for -0 and +0; NaN unsupported) onto
// uint32 that preserves order: a larger score has a larger key.
// coarse_key: an 11-bit, order-preserving (non-decreasing) bin of the score, taken from
// its rounding to fp16 (sign, 5 exponent and 5 mantissa bits: 32 bins per octave), so
// realistic score distributions spread over many bins.  full_key refines coarse_key:
// a higher bin always holds strictly larger scores.
#pragma once

#include <cuda_fp16.h>

#include <cstdint>

namespace dsa {

__device__ __forceinline__ uint32_t full_key(float f) {
    uint32_t u = __float_as_uint(f);
    if (f == 0.f) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// The score a full key stands for (+0 for the key of both zeros).
__device__ __forceinline__ float key_score(uint32_t key) {
    const uint32_t u = (key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key;
    return __uint_as_float(u);
}

__device__ __forceinline__ uint32_t coarse_key(float f) {
    if (f == 0.f) f = 0.f;
    const uint16_t h = __half_as_ushort(__float2half_rn(f));
    const uint32_t u = (h & 0x8000u) ? (uint32_t)(~h & 0xFFFFu) : (uint32_t)(h | 0x8000u);
    return u >> 5;
}

constexpr int kCoarseBins = 2048;

// A float below every score whose coarse bin is at least `bin`: the fp16 value ordered
// just before the bin's lowest one (a score that rounds into the bin or above exceeds
// it), or -inf when there is none.  Comparing scores with it keeps all of the bin and
// above, and at most the scores that round to that one fp16 value besides.
__device__ __forceinline__ float coarse_floor(int bin) {
    const uint32_t u = (uint32_t)bin << 5;  // lowest ordered fp16 image in the bin
    if (u == 0u) return -INFINITY;
    const uint32_t v = u - 1u;               // the one ordered just before it
    const uint16_t h = (v & 0x8000u) ? (uint16_t)(v & 0x7FFFu) : (uint16_t)(~v & 0xFFFFu);
    const float f = __half2float(__ushort_as_half(h));
    return (f != f) ? -INFINITY : f;         // below the bottom: negative NaN images
}

}  // namespace dsa
