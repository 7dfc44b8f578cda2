// device_common.cuh -- element types, streaming loads and small reductions shared by the
// verify kernels.
#pragma once

#include <cfloat>
#include <cstdint>

namespace specverify {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

// 2^x on the special-function unit (PTX ex2.approx.ftz.f32: relative error about 2^-22,
// results below 2^-126 flush to zero, which is negligible in a sum whose largest term is 1).
__device__ __forceinline__ float ex2_fast(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// 16-byte streaming load through the non-coherent path without L1 allocation: every logit
// is read once by the row-statistics pass.
__device__ __forceinline__ uint4 ld_stream16(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

// Element traits: how 16 bytes of logits widen to fp32.
struct Bf16Elem {
    using storage = uint16_t;
    static constexpr int kVec = 8;                      // elements per 16-byte load
    static constexpr uint32_t kNegInfWord = 0xFF80FF80u;  // two bf16 -inf
    __device__ __forceinline__ static float load1(const storage* p) {
        const uint16_t h = __ldg(reinterpret_cast<const unsigned short*>(p));
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    __device__ __forceinline__ static void widen(const uint4& v, float (&f)[kVec]) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            f[2 * k] = __uint_as_float(w[k] << 16);              // lower address first
            f[2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u);
        }
    }
    // Eight values from an address that is only 2-byte aligned, packed as a 16-byte load of
    // them packs them (the lower address in the lower half of each word), with the widest
    // loads the address allows.  (Rows of an odd vocabulary start off 16-byte boundaries.)
    __device__ __forceinline__ static uint4 load_vec_unaligned(const storage* p) {
        const uintptr_t a = reinterpret_cast<uintptr_t>(p);
        if ((a & 7u) == 0) {
            const uint2* q = reinterpret_cast<const uint2*>(p);
            const uint2 lo = __ldg(q), hi = __ldg(q + 1);
            return make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
        if ((a & 3u) == 0) {
            const unsigned int* q = reinterpret_cast<const unsigned int*>(p);
            return make_uint4(__ldg(q), __ldg(q + 1), __ldg(q + 2), __ldg(q + 3));
        }
        const unsigned short* q = reinterpret_cast<const unsigned short*>(p);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k)
            w[k] = static_cast<uint32_t>(__ldg(q + 2 * k)) | (static_cast<uint32_t>(__ldg(q + 2 * k + 1)) << 16);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
    // The largest of the vector's eight values (exact: a maximum of bf16 values is one of
    // them), on packed pairs before widening.
    __device__ __forceinline__ static float vmax(const uint4& v) {
        uint32_t a, b;
        asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(v.x), "r"(v.y));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(b) : "r"(v.z), "r"(v.w));
        asm("max.bf16x2 %0, %1, %2;" : "=r"(a) : "r"(a), "r"(b));
        return fmaxf(__uint_as_float(a << 16), __uint_as_float(a & 0xFFFF0000u));
    }
};

struct F32Elem {
    using storage = float;
    static constexpr int kVec = 4;
    static constexpr uint32_t kNegInfWord = 0xFF800000u;
    __device__ __forceinline__ static float load1(const storage* p) { return __ldg(p); }
    __device__ __forceinline__ static void widen(const uint4& v, float (&f)[kVec]) {
        f[0] = __uint_as_float(v.x);
        f[1] = __uint_as_float(v.y);
        f[2] = __uint_as_float(v.z);
        f[3] = __uint_as_float(v.w);
    }
    __device__ __forceinline__ static float vmax(const uint4& v) {
        return fmaxf(fmaxf(__uint_as_float(v.x), __uint_as_float(v.y)),
                     fmaxf(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    // Four values from an address that is only 4-byte aligned (see Bf16Elem).
    __device__ __forceinline__ static uint4 load_vec_unaligned(const storage* p) {
        if ((reinterpret_cast<uintptr_t>(p) & 7u) == 0) {
            const uint2* q = reinterpret_cast<const uint2*>(p);
            const uint2 lo = __ldg(q), hi = __ldg(q + 1);
            return make_uint4(lo.x, lo.y, hi.x, hi.y);
        }
        const unsigned int* q = reinterpret_cast<const unsigned int*>(p);
        return make_uint4(__ldg(q), __ldg(q + 1), __ldg(q + 2), __ldg(q + 3));
    }
};

// Split [x0, x1) of a row into a scalar head (until 16-byte alignment), a body of whole
// 16-byte vectors and a scalar tail.
template <class ET>
struct RowSpan {
    const typename ET::storage* base;  // row + x0
    int head;                          // scalar elements before the first aligned vector
    int nvec;                          // whole vectors
    int tail;                          // scalar elements after the vectors
    __device__ __forceinline__ RowSpan(const typename ET::storage* row, int x0, int x1) {
        base = row + x0;
        const int n = x1 - x0;
        const uintptr_t addr = reinterpret_cast<uintptr_t>(base);
        int h = static_cast<int>(((16u - (addr & 15u)) & 15u) / sizeof(typename ET::storage));
        head = h < n ? h : n;
        nvec = (n - head) / ET::kVec;
        tail = n - head - nvec * ET::kVec;
    }
    __device__ __forceinline__ const uint4* vec() const {
        return reinterpret_cast<const uint4*>(base + head);
    }
};

// Online softmax statistics in base 2: m is the running maximum of x*c (c = log2(e)/T),
// clamped to >= -FLT_MAX so that -inf logits never meet -inf - (-inf); s is the running
// sum of 2^(x*c - m).
struct SoftmaxStat {
    float m, s;
};

// Symmetric in a and b, with every rounding explicit (no contraction into an FMA, whose
// choice of product could differ between call sites): every lane of a butterfly ends with the
// same bits, and so does every kernel that merges the same partials in the same order.
__device__ __forceinline__ SoftmaxStat merge_stat(SoftmaxStat a, SoftmaxStat b) {
    const float M = fmaxf(a.m, b.m);
    return SoftmaxStat{M, __fadd_rn(__fmul_rn(a.s, ex2_fast(a.m - M)), __fmul_rn(b.s, ex2_fast(b.m - M)))};
}

__device__ __forceinline__ SoftmaxStat warp_merge_stat(SoftmaxStat v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        SoftmaxStat o{__shfl_xor_sync(0xffffffffu, v.m, off), __shfl_xor_sync(0xffffffffu, v.s, off)};
        v = merge_stat(v, o);
    }
    return v;
}

// (value, index) argmax with the lowest index winning equal values.
struct ArgMax {
    float v;
    int i;
};

__device__ __forceinline__ bool argmax_better(ArgMax a, ArgMax b) {
    return a.v > b.v || (a.v == b.v && a.i < b.i);
}

__device__ __forceinline__ ArgMax warp_argmax(ArgMax a) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        ArgMax o{__shfl_xor_sync(0xffffffffu, a.v, off), __shfl_xor_sync(0xffffffffu, a.i, off)};
        if (argmax_better(o, a)) a = o;
    }
    return a;
}


// Shared-memory address of a CTA-local pointer, and the mbarrier operations that the
// TMA-fed kernels use (one thread arms a barrier with the bytes it expects, the copy engine
// completes them, every waiting thread polls the phase parity).
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_test(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

}  // namespace specverify
