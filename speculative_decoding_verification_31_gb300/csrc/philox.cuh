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

// Round keys of one launch: key k_r = key + r * (Weyl increment), r = 0..9.  Passed in the
// kernel parameters so that every round reads its key as a constant operand.
struct PhiloxRoundKeys {
    uint32_t k0[10], k1[10];
};

__host__ __device__ __forceinline__ PhiloxRoundKeys philox_round_keys(PhiloxKey key) {
    PhiloxRoundKeys rk;
    for (int r = 0; r < 10; ++r) {
        rk.k0[r] = key.k0 + static_cast<uint32_t>(r) * 0x9E3779B9u;
        rk.k1[r] = key.k1 + static_cast<uint32_t>(r) * 0xBB67AE85u;
    }
    return rk;
}

// One 32x32 -> 64-bit product (PTX mul.wide.u32) split into its halves.
__device__ __forceinline__ void mul_wide(uint32_t a, uint32_t b, uint32_t& hi, uint32_t& lo) {
    asm("{.reg .b64 t; mul.wide.u32 t, %2, %3; mov.b64 {%0, %1}, t;}"
        : "=r"(lo), "=r"(hi)
        : "r"(a), "r"(b));
}

__device__ __forceinline__ void philox_round(uint4& c, uint32_t k0, uint32_t k1) {
    uint32_t hi0, lo0, hi1, lo1;
    mul_wide(0xD2511F53u, c.x, hi0, lo0);
    mul_wide(0xCD9E8D57u, c.z, hi1, lo1);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
}

// The race counters of one row, (k, r, b, 1), differ only in word 0.  Of the first round's
// two products, the one of word 2 (= b) is then the same for every k, and so is the second
// round's product of word 0; both are computed once per row.
struct RaceRowRng {
    uint32_t c0_1, c1_1;    // words 0 and 1 after round 1
    uint32_t hi_2, lo_2;    // 0xD2511F53 * c0_1 (round 2)
};

__device__ __forceinline__ RaceRowRng race_row_rng(const PhiloxRoundKeys& rk, uint32_t b,
                                                   uint32_t r) {
    RaceRowRng q;
    q.c0_1 = __umulhi(0xCD9E8D57u, b) ^ r ^ rk.k0[0];
    q.c1_1 = 0xCD9E8D57u * b;
    q.hi_2 = __umulhi(0xD2511F53u, q.c0_1);
    q.lo_2 = 0xD2511F53u * q.c0_1;
    return q;
}

// Philox4x32-10 of counter (k, r, b, 1): the same four words as race_block(), with the
// per-row parts of rounds 1 and 2 taken from `q`.
__device__ __forceinline__ uint4 race_block_fast(const RaceRowRng& q, const PhiloxRoundKeys& rk,
                                                 uint32_t k) {
    // round 1
    uint32_t h, c3;
    mul_wide(0xD2511F53u, k, h, c3);
    const uint32_t c2 = h ^ 1u ^ rk.k1[0];
    // round 2
    uint32_t h2, l2;
    mul_wide(0xCD9E8D57u, c2, h2, l2);
    uint4 c = make_uint4(h2 ^ q.c1_1 ^ rk.k0[1], l2, q.hi_2 ^ c3 ^ rk.k1[1], q.lo_2);
#pragma unroll
    for (int round = 2; round < 10; ++round) philox_round(c, rk.k0[round], rk.k1[round]);
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
