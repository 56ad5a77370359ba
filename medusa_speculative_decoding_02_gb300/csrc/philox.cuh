// philox.cuh -- counter-based random numbers for the sampling paths.
//
// Philox4x64-10 as published by Salmon, Moraes, Dror and Shaw ("Parallel
// random numbers: as easy as 1, 2, 3", SC 2011): ten rounds of two 64x64
// multiplies on a four-word counter, a two-word key bumped by Weyl
// increments between rounds.  Stream layout used by every sampling kernel:
// counter = (v / 4, row, b, purpose), key = (seed, step); the uniform for
// index v is word v % 4 of the block, as ((w >> 41) + 0.5) * 2^-23, which is
// exact in float32 and never 0 or 1.
#pragma once

#include <stdint.h>

namespace medusa {

enum { kRngDraft = 1, kRngAccept = 2, kRngResample = 3 };

struct Philox4x64 {
    uint64_t w[4];
};

__device__ __forceinline__ Philox4x64 philox4x64(uint64_t c0, uint64_t c1, uint64_t c2,
                                                 uint64_t c3, uint64_t k0, uint64_t k1) {
    constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
    constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        if (r > 0) {
            k0 += kW0;
            k1 += kW1;
        }
        const uint64_t hi0 = __umul64hi(kM0, c0), lo0 = kM0 * c0;
        const uint64_t hi1 = __umul64hi(kM1, c2), lo1 = kM1 * c2;
        const uint64_t y0 = hi1 ^ c1 ^ k0, y2 = hi0 ^ c3 ^ k1;
        c0 = y0;
        c1 = lo1;
        c2 = y2;
        c3 = lo0;
    }
    Philox4x64 o;
    o.w[0] = c0;
    o.w[1] = c1;
    o.w[2] = c2;
    o.w[3] = c3;
    return o;
}

// word j (0..3) of a block, without a dynamically indexed local array
__device__ __forceinline__ uint64_t philox_word(const Philox4x64 &r, int j) {
    return j == 0 ? r.w[0] : j == 1 ? r.w[1] : j == 2 ? r.w[2] : r.w[3];
}

// uniform in (0, 1) from one 64-bit word (exact in float32)
__device__ __forceinline__ float word_uniform(uint64_t w) {
    return ((float)(uint32_t)(w >> 41) + 0.5f) * 1.1920928955078125e-7f;  // 2^-23
}

// Gumbel noise -log(-log u) for the uniform of index v in stream
// (purpose, b, row) under (seed, step)
__device__ __forceinline__ float gumbel_at(uint64_t seed, uint64_t step, int purpose, int b,
                                           int row, int v) {
    const Philox4x64 r = philox4x64((uint64_t)(v >> 2), (uint64_t)row, (uint64_t)b,
                                    (uint64_t)purpose, seed, step);
    return -logf(-logf(word_uniform(philox_word(r, v & 3))));
}

__device__ __forceinline__ float uniform_at(uint64_t seed, uint64_t step, int purpose, int b,
                                            int row, int v) {
    const Philox4x64 r = philox4x64((uint64_t)(v >> 2), (uint64_t)row, (uint64_t)b,
                                    (uint64_t)purpose, seed, step);
    return word_uniform(philox_word(r, v & 3));
}

}  // namespace medusa
