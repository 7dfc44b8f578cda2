// philox.cuh -- device Philox4x32-10 and the two variates the verify step draws from it.
//
// Philox4x32-10 is the counter-based generator of Salmon, Moraes, Dror and Shaw,
// "Parallel Random Numbers: As Easy as 1, 2, 3" (SC'11), section 4: ten rounds, each
// multiplying words 0 and 2 of the counter by two fixed odd constants (32x32 -> 64 bits),
// mixing the high halves with words 1 and 3 and the key, and bumping the key by a Weyl
// sequence between rounds.
//
// The random-number contract (shared with every caller through the public header):
//   acceptance uniform of draft position i of sequence b:
//       counter (0, i, b, 0), word 0 w,        u = (w >> 8) * 2^-24 (exact in fp32)
//   exponential of token x in the race at row r of sequence b:
//       counter (x >> 2, r, b, 1), word (x & 3) w,  E = -log1p(-(w + 0.5) * 2^-32)
#pragma once

#include <cstdint>

namespace specverify {

struct PhiloxKey {
    uint32_t k0, k1;
};

__host__ __device__ __forceinline__ PhiloxKey philox_key(uint64_t seed) {
    return PhiloxKey{static_cast<uint32_t>(seed & 0xffffffffu), static_cast<uint32_t>(seed >> 32)};
}

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key) {
    uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
    for (int round = 0; round < 10; ++round) {
        if (round > 0) {
            k0 += 0x9E3779B9u;  // Weyl increments: golden ratio and sqrt(3) - 1
            k1 += 0xBB67AE85u;
        }
        const uint32_t lo0 = 0xD2511F53u * c.x;
        const uint32_t hi0 = __umulhi(0xD2511F53u, c.x);
        const uint32_t lo1 = 0xCD9E8D57u * c.z;
        const uint32_t hi1 = __umulhi(0xCD9E8D57u, c.z);
        c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    }
    return c;
}

// Acceptance uniform u in [0, 1) with 24 random bits.
__device__ __forceinline__ float accept_uniform(PhiloxKey key, uint32_t b, uint32_t i) {
    const uint4 w = philox4x32_10(make_uint4(0u, i, b, 0u), key);
    return static_cast<float>(w.x >> 8) * 0x1p-24f;
}

// Counter of the race block holding tokens 4k .. 4k+3 at row r of sequence b.
__device__ __forceinline__ uint4 race_block(PhiloxKey key, uint32_t b, uint32_t r, uint32_t k) {
    return philox4x32_10(make_uint4(k, r, b, 1u), key);
}

__device__ __forceinline__ uint32_t word_of(uint4 v, uint32_t k) {
    return k == 0 ? v.x : (k == 1 ? v.y : (k == 2 ? v.z : v.w));
}

// ln E for the race exponential E = -log1p(-U), U = (w + 0.5) 2^-32, in fp32.
// Below U = 1/2 the log1p form is accurate; above it, 1 - U = (~w + 0.5) 2^-32 is formed
// from the complement word so that no precision is lost where U rounds towards 1.
__device__ __forceinline__ float race_log_exponential(uint32_t w) {
    float E;
    if (w < 0x80000000u) {
        const float U = (static_cast<float>(w) + 0.5f) * 0x1p-32f;
        E = -log1pf(-U);
    } else {
        const float one_minus_U = (static_cast<float>(~w) + 0.5f) * 0x1p-32f;
        E = -logf(one_minus_U);
    }
    return logf(E);
}

}  // namespace specverify
