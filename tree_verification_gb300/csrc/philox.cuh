// Philox-4x32-10, the counter-based generator of Salmon, Moraes, Dror and
// Shaw ("Parallel random numbers: as easy as 1, 2, 3", SC 2011), and the
// Gumbel noise the sampling kernels draw from it.
//
// Noise for request b, sampled position pos and token v: counter
// (v / 4, pos, b, 0), key (seed low, seed high); output word v % 4 is the
// 32-bit draw x, u = ((x >> 9) + 1/2) / 2^23 (exact in float32) and the noise
// is -log(-log(u)).  Keying by position makes every node at a position, and
// autoregressive sampling at that position, see the same noise.
#pragma once

#include <stdint.h>

namespace graft {

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, uint2 k) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x), lo0 = 0xD2511F53u * c.x;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z), lo1 = 0xCD9E8D57u * c.z;
        c = make_uint4(hi1 ^ c.y ^ k.x, lo1, hi0 ^ c.w ^ k.y, lo0);
        k.x += 0x9E3779B9u;
        k.y += 0xBB67AE85u;
    }
    return c;
}

// Gumbel(0, 1) noise from one 32-bit draw.
__device__ __forceinline__ float gumbel_of(uint32_t x) {
    const float u = (static_cast<float>(x >> 9) + 0.5f) * (1.0f / 8388608.0f);
    return -logf(-logf(u));
}

// The four draws for tokens 4q .. 4q + 3.
__device__ __forceinline__ uint4 noise_draws(unsigned long long seed, uint32_t b, uint32_t pos, uint32_t q) {
    return philox4x32_10(make_uint4(q, pos, b, 0u),
                         make_uint2((uint32_t)(seed & 0xffffffffull), (uint32_t)(seed >> 32)));
}

}  // namespace graft
