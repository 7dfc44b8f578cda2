// lmhead.cuh -- the LM head on the tensor cores (sm_103a tcgen05), with the verify step's
// row statistics as its epilogue.
//
// Logits are L = H W^T: hidden states H [rows, d] and head weights W [V, d], both bf16 and
// row-major (so both operands are K-major), accumulated in fp32.  A CTA owns one tile of
// 128 rows and a contiguous run of 256-wide vocabulary tiles; per tile it streams K in
// 64-element slices:
//   warp 0     one elected thread issues TMA loads (cp.async.bulk.tensor, 128-byte swizzle)
//              of the A and B slices into a 4-stage shared-memory ring;
//   warp 1     allocates 512 TMEM columns (two 128 x 256 fp32 accumulators) and one
//              elected thread issues tcgen05.mma (M = 128, N = 256, K = 16; bf16 x bf16 ->
//              fp32), committing each stage back to the producer and each finished tile
//              to the epilogue;
//   warps 2-5  the epilogue: each reads its 32 TMEM lanes (one row per thread) with
//              tcgen05.ld and either writes the logits (spec_lmhead_logits) or folds them
//              into the row's online softmax statistics -- max and sum of 2^(x c - m) in
//              base 2, c = log2(e) / T of the row -- and keeps the logit at the row's draft
//              token, and, when asked, the largest logit of every 8-token block of the row
//              rounded up to bf16 (the verify from hidden states bounds its race with them).
// The two accumulators let the tensor cores run the next tile while the epilogue drains the
// last.  Every mbarrier wait is bounded (kWaitLimitNs): on a timeout the kernel records
// SPEC_ETIMEOUT, stops issuing, waits (bounded) for its loads in flight and frees its TMEM.
// This is a dense contraction (2 rows * V * d flops per row), the one place of the verify
// pipeline where tensor cores apply.
#pragma once

#include <cuda.h>
#include <cstdint>

namespace specverify {

constexpr int kGemmBM = 128;      // rows per tile (TMEM lanes)
constexpr int kGemmBN = 256;      // vocabulary entries per tile (TMEM columns per accumulator)
constexpr int kGemmBK = 64;       // K per stage: one 128-byte swizzle row of bf16
constexpr int kGemmStages = 4;
constexpr int kGemmThreads = 192; // 6 warps
constexpr uint32_t kGemmStageA = kGemmBM * kGemmBK * 2;  // 16 KB
constexpr uint32_t kGemmStageB = kGemmBN * kGemmBK * 2;  // 32 KB
constexpr uint32_t kGemmTmemCols = 512;
// Logits leave through a per-warp 32 x 32 staging block (rows padded to 36 floats: 16-byte
// aligned, and the transposed float4 accesses fall in distinct banks), so that each
// quarter-warp writes 128 contiguous bytes of one row.
constexpr int kStageStride = 36;
constexpr uint32_t kGemmStageOut = 4 * 32 * kStageStride * 4;  // four epilogue warps
// dynamic shared memory: 1024-byte alignment slack, the ring, the barriers, the staging
constexpr uint32_t kGemmSmem = 1024 + kGemmStages * (kGemmStageA + kGemmStageB) + 256 + kGemmStageOut;

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1), A and B bf16
// (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0), N >> 3 at bits 17-22,
// M >> 4 at bits 24-28.
constexpr uint32_t kGemmIdesc = (1u << 4) | (1u << 7) | (1u << 10) |
                                (static_cast<uint32_t>(kGemmBN >> 3) << 17) |
                                (static_cast<uint32_t>(kGemmBM >> 4) << 24);

// Shared-memory matrix descriptor of a K-major tile stored as TMA writes it with the
// 128-byte swizzle: rows of 128 bytes, 8-row (1024-byte) swizzle atoms.  Start address
// >> 4 in bits 0-13, leading-byte offset (unused by this layout) 1 in bits 16-29, stride
// byte offset 1024 >> 4 in bits 32-45, descriptor version 1 in bits 46-47, layout
// SWIZZLE_128B = 2 in bits 61-63.  The stage buffers are 1024-byte aligned.
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    return static_cast<uint64_t>((saddr >> 4) & 0x3FFFu) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

// Bounded wait for the phase of the given parity to complete; false after kWaitLimitNs or
// once *abort is set by another thread of the CTA.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, volatile int* abort) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_time_ns();
    while (!mbar_test(bar, parity)) {
        if (*abort) return false;
        if (global_time_ns() - t0 > kWaitLimitNs) return false;
    }
    return true;
}

__device__ __forceinline__ void tma_load_2d(const CUtensorMap* map, uint64_t* bar, void* dst, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_addr(bar)), "r"(x), "r"(y)
        : "memory");
}

__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(kGemmIdesc), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void umma_commit(uint64_t* bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void tmem_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void tmem_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane (the warp's 32-lane slice).
__device__ __forceinline__ void tmem_load32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32"
        " {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15,"
        " %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]),
          "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]),
          "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr)
        : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// One product of a launch: rows of H against W, with its epilogue outputs.
struct LmHeadPart {
    int rows;                     // rows of H (0: the part is absent)
    float* logits;                // [rows, V] fp32 output (logits epilogue)
    uint16_t* block_max;          // [rows, lm_block_stride(V)] bf16 bits: the largest logit of
                                  // each 8-token block, rounded up (statistics epilogue), or nullptr
    const float* T_row;           // [rows] temperature of each row (statistics epilogue)
    const int32_t* token_row;     // [rows] token whose logit to keep (-1: none), or nullptr
    float2* stat_parts;           // [rows][nchunks] (scaled max, sum) in base 2
    float* token_logit;           // [rows] logit at token_row (raw, before 1/T)
};

// A launch computes up to two products with the same V and d (the target rows against the
// target head and the draft rows against the draft head): grid rows [0, m_tiles0) are
// part 0's row tiles, the rest part 1's, so both share one wave of CTAs.
struct LmHeadParams {
    int V, d;
    int tiles_per_cta;            // vocabulary tiles of one CTA (its chunk)
    int nchunks;                  // chunks per row: ceil(V / (kGemmBN * tiles_per_cta))
    int m_tiles0;                 // row tiles of part 0
    LmHeadPart part[2];
    int32_t* status;
    // single-part views used by the merge kernel
    int rows;
    const float* T_row;
    const int32_t* token_row;
    float2* stat_parts;
    float* token_logit;
};

constexpr int kLmBlock = 8;  // tokens per block maximum

// Row stride (bf16 elements) of the block maxima: ceil(V / 8) rounded up to a multiple of 4,
// so that the four maxima of 32 columns are one aligned 8-byte word.
__host__ __device__ __forceinline__ int lm_block_stride(int V) { return ((V + kLmBlock - 1) / kLmBlock + 3) & ~3; }

// bf16 bits of the smallest bf16 value >= f (f not NaN): truncation rounds a negative value up
// already; a positive value with dropped bits moves up one bf16 step (+inf stays +inf).
__device__ __forceinline__ uint32_t bf16_round_up(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u >> 16) + (((u & 0xFFFFu) != 0u && !(u >> 31)) ? 1u : 0u);
}

// Columns [col0, col0 + 32) of one row's logits, v, to dst = row + col0 (16-byte stores where
// the run is whole and aligned).
__device__ __forceinline__ void store_logits32(float* dst, const float (&v)[32], int col0, int V) {
    if (col0 + 32 <= V && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0) {
#pragma unroll
        for (int i = 0; i < 32; i += 4)
            *reinterpret_cast<float4*>(dst + i) = make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (col0 + i < V) dst[i] = v[i];
    }
}

// kLogits: write the logits; otherwise the statistics epilogue.
template <bool kLogits>
__global__ void __launch_bounds__(kGemmThreads, 1)
lmhead_kernel(const __grid_constant__ CUtensorMap map_h0, const __grid_constant__ CUtensorMap map_w0,
              const __grid_constant__ CUtensorMap map_h1, const __grid_constant__ CUtensorMap map_w1,
              LmHeadParams p) {
    extern __shared__ uint8_t gemm_smem_raw[];
    uint8_t* base = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(gemm_smem_raw) + 1023) &
                                               ~static_cast<uintptr_t>(1023));
    uint8_t* stage_a = base;
    uint8_t* stage_b = base + kGemmStages * kGemmStageA;
    uint64_t* bars = reinterpret_cast<uint64_t*>(stage_b + kGemmStages * kGemmStageB);
    uint64_t* full = bars;                     // [stages] TMA -> MMA
    uint64_t* empty = bars + kGemmStages;      // [stages] MMA -> TMA
    uint64_t* tfull = bars + 2 * kGemmStages;  // [2] MMA -> epilogue
    uint64_t* tempty = tfull + 2;              // [2] epilogue -> MMA
    uint64_t* tdrain = tempty + 2;             // every MMA of this CTA is done
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tdrain + 1);
    volatile int* abort = reinterpret_cast<volatile int*>(tmem_slot + 1);
    float* stage_out = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(bars) + 256);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const bool second = static_cast<int>(blockIdx.y) >= p.m_tiles0;
    const LmHeadPart& part = p.part[second ? 1 : 0];
    const CUtensorMap* map_h = second ? &map_h1 : &map_h0;
    const CUtensorMap* map_w = second ? &map_w1 : &map_w0;
    const int m_tile = second ? static_cast<int>(blockIdx.y) - p.m_tiles0 : static_cast<int>(blockIdx.y);
    const int chunk = blockIdx.x;
    const int n_tiles_total = (p.V + kGemmBN - 1) / kGemmBN;
    const int t_begin = chunk * p.tiles_per_cta;
    const int t_end = min(n_tiles_total, t_begin + p.tiles_per_cta);
    const int ntiles = max(0, t_end - t_begin);
    const int kb_count = p.d / kGemmBK;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGemmStages; ++s) {
            mbar_init(full + s, 1);
            mbar_init(empty + s, 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(tfull + a, 1);
            mbar_init(tempty + a, 4);  // one arrival per epilogue warp
        }
        mbar_init(tdrain, 1);
        *abort = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 1) {  // TMEM: two 256-column accumulators
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_addr(tmem_slot)),
                     "r"(kGemmTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    tmem_fence_before();
    __syncthreads();
    tmem_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ---- TMA producer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0;
            for (int t = 0; t < ntiles && !*abort; ++t) {
                const int n0 = (t_begin + t) * kGemmBN;
                for (int kb = 0; kb < kb_count; ++kb) {
                    if (!mbar_wait(empty + stage, phase ^ 1u, abort)) {
                        *abort = 1;
                        break;
                    }
                    mbar_expect_tx(full + stage, kGemmStageA + kGemmStageB);
                    tma_load_2d(map_h, full + stage, stage_a + stage * kGemmStageA, kb * kGemmBK,
                                m_tile * kGemmBM);
                    tma_load_2d(map_w, full + stage, stage_b + stage * kGemmStageB, kb * kGemmBK, n0);
                    ++issued;
                    if (++stage == kGemmStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (*abort) {
                // let the loads in flight land before the CTA's shared memory goes away
                const int pending = min(issued, kGemmStages);
                for (int k = 0; k < pending; ++k) {
                    if (--stage < 0) {
                        stage = kGemmStages - 1;
                        phase ^= 1u;
                    }
                    volatile int never = 0;
                    mbar_wait(full + stage, phase, &never);
                }
                set_status(p.status, 4 /* SPEC_ETIMEOUT */);
            }
        }
    } else if (warp == 1) {
        // ---- MMA issuer ----
        if (lane == 0) {
            int stage = 0;
            uint32_t phase = 0;
            for (int t = 0; t < ntiles && !*abort; ++t) {
                const int acc = t & 1;
                const uint32_t acc_phase = (t >> 1) & 1u;
                if (!mbar_wait(tempty + acc, acc_phase ^ 1u, abort)) {
                    *abort = 1;
                    break;
                }
                tmem_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * kGemmBN);
                for (int kb = 0; kb < kb_count; ++kb) {
                    if (!mbar_wait(full + stage, phase, abort)) {
                        *abort = 1;
                        break;
                    }
                    tmem_fence_after();
                    const uint64_t adesc = sw128_kmajor_desc(smem_addr(stage_a + stage * kGemmStageA));
                    const uint64_t bdesc = sw128_kmajor_desc(smem_addr(stage_b + stage * kGemmStageB));
#pragma unroll
                    for (int kk = 0; kk < kGemmBK / 16; ++kk)  // +32 bytes of K per step
                        umma_bf16(d_tmem, adesc + 2 * kk, bdesc + 2 * kk, (kb | kk) != 0);
                    umma_commit(empty + stage);  // the stage is free once these MMAs are done
                    if (++stage == kGemmStages) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (*abort) break;
                umma_commit(tfull + acc);  // the tile's accumulator is complete
            }
            // whatever happened, no MMA may still write TMEM when it is freed
            umma_commit(tdrain);
            volatile int never = 0;
            if (!mbar_wait(tdrain, 0, &never)) set_status(p.status, 4 /* SPEC_ETIMEOUT */);
        }
    } else {
        // ---- epilogue: warps 2..5, TMEM lane slice (warp % 4) * 32 ----
        const int slice = warp & 3;
        const int row = m_tile * kGemmBM + slice * 32 + lane;
        const bool row_ok = row < part.rows;
        float c = 1.0f;
        int tok = -1;
        if (!kLogits && row_ok) {
            c = kLog2e / part.T_row[row];
            if (part.token_row) tok = part.token_row[row];
        }
        // logits output (logits epilogue): staged and written row by row where the rows are
        // 16-byte aligned
        float* const lout = kLogits ? part.logits : nullptr;
        const bool staged = lout && p.V % 4 == 0 && (reinterpret_cast<uintptr_t>(lout) & 15u) == 0;
        float* const stg = stage_out + slice * 32 * kStageStride;
        const int row0 = m_tile * kGemmBM + slice * 32;
        uint16_t* const bmrow = (!kLogits && row_ok && part.block_max)
                                    ? part.block_max + static_cast<long long>(row) * lm_block_stride(p.V)
                                    : nullptr;
        float m = -FLT_MAX, s = 0.0f, xtok = 0.0f;
        for (int t = 0; t < ntiles; ++t) {
            const int acc = t & 1;
            const uint32_t acc_phase = (t >> 1) & 1u;
            // lane 0 waits (bounded) and the warp follows it, so that the warp stays converged
            // for the .sync.aligned TMEM loads; then every lane observes the completed phase
            int ok = 0;
            if (lane == 0) ok = mbar_wait(tfull + acc, acc_phase, abort);
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) {
                if (lane == 0) *abort = 1;
                break;
            }
            volatile int never = 0;
            mbar_wait(tfull + acc, acc_phase, &never);  // completed: returns at once
            __syncwarp();
            tmem_fence_after();
            const int n0 = (t_begin + t) * kGemmBN;
#pragma unroll 1
            for (int c32 = 0; c32 < kGemmBN / 32; ++c32) {
                float v[32];
                tmem_load32(tmem_base + (static_cast<uint32_t>(slice * 32) << 16) +
                                static_cast<uint32_t>(acc * kGemmBN + c32 * 32),
                            v);
                const int col0 = n0 + c32 * 32;
                if (lout) {
                    if (staged && col0 + 32 <= p.V) {  // (uniform over the warp)
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            *reinterpret_cast<float4*>(stg + lane * kStageStride + i) =
                                make_float4(v[i], v[i + 1], v[i + 2], v[i + 3]);
                        __syncwarp();
                        const int cq = 4 * (lane & 7);
#pragma unroll
                        for (int r0 = 0; r0 < 32; r0 += 4) {
                            const int r = r0 + (lane >> 3);
                            if (row0 + r < part.rows)  // streaming stores: keep the heads' tiles in L2
                                __stcs(reinterpret_cast<float4*>(lout + static_cast<long long>(row0 + r) * p.V + col0 + cq),
                                       *reinterpret_cast<const float4*>(stg + r * kStageStride + cq));
                        }
                        __syncwarp();
                    } else if (row_ok) {
                        store_logits32(lout + static_cast<long long>(row) * p.V + col0, v, col0, p.V);
                    }
                }
                if (!kLogits) {
                    float bmax = -INFINITY;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (col0 + i < p.V) bmax = fmaxf(bmax, v[i]);
                    if (bmrow && col0 < p.V) {  // the four 8-token block maxima, rounded up
                        uint32_t h[4];
#pragma unroll
                        for (int k = 0; k < 4; ++k) {
                            float mk = -INFINITY;
#pragma unroll
                            for (int i = 8 * k; i < 8 * k + 8; ++i)
                                if (col0 + i < p.V) mk = fmaxf(mk, v[i]);
                            h[k] = bf16_round_up(mk);
                        }
                        *reinterpret_cast<uint2*>(bmrow + (col0 >> 3)) = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
                    }
                    const float mn = fmaxf(m, fmaxf(bmax * c, -FLT_MAX));
                    float part = 0.0f;
#pragma unroll
                    for (int i = 0; i < 32; ++i)
                        if (col0 + i < p.V) part += ex2_fast(fmaf(v[i], c, -mn));
                    s = fmaf(s, ex2_fast(m - mn), part);
                    m = mn;
                    if (tok >= col0 && tok < col0 + 32) {
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            if (tok == col0 + i) xtok = v[i];
                    }
                }
            }
            tmem_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty + acc);
        }
        if (!kLogits && row_ok && !*abort) {
            store_stat(part.stat_parts + static_cast<long long>(row) * p.nchunks + chunk, m, s);
            if (tok >= t_begin * kGemmBN && tok < t_end * kGemmBN && tok < p.V && part.token_logit)
                part.token_logit[row] = xtok;
        }
        if (*abort && lane == 0) set_status(p.status, 4 /* SPEC_ETIMEOUT */);
    }
    tmem_fence_before();
    __syncthreads();
    if (warp == 1) {
        __syncwarp();
        tmem_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem_base),
                     "r"(kGemmTmemCols)
                     : "memory");
    }
}

// ----------------------------------------------------------------------------------------
// The verify step from hidden states (spec_verify_lmhead): the statistics kernel above runs
// on the target rows (T) and the draft rows (T_d) with each row's draft token, keeping the
// largest logit of every 8-token block of the target rows (rounded up to bf16: 1/4 byte per
// logit); then
//   lmhead_scan   one warp per sequence: the accept test of every position from ln p(d_i),
//                 ln q(d_i) and u_i (the same rule and random numbers as the logits path) and
//                 the sequence's outputs;
//   lmhead_race   races each sequence's row j without its logits: every token's Philox word
//                 is drawn, a token whose block maximum cannot reach the best score so far
//                 is dropped on its word alone (one integer compare), and the few that remain
//                 get their exact logits h . w_x (target, and draft for a residual) from a
//                 warp's dot product over d, most promising first.  The heads are read once
//                 by the statistics pass, plus one row of each head per candidate.
// ----------------------------------------------------------------------------------------

struct LmVerifyParams {
    int B, gamma, V, d;
    const uint16_t* h_target;    // [B, gamma+1, d] bf16 bits
    const uint16_t* h_draft;     // [B, gamma, d]
    const int32_t* tokens;       // [B, gamma]
    const float* logZ_t;         // [B, gamma+1] nats
    const float* logp_t;         // [B, gamma+1] ln p_i(d_i) (NaN at row gamma)
    const float* logZ_d;         // [B, gamma]
    const float* logq_d;         // [B, gamma]
    SeqInfo* seq;                // [B]
    float T, Td;
    const float* T_seq;
    const float* Td_seq;
    PhiloxKey key;
    uint32_t seq_base;
    int32_t* out_tokens;         // [B, gamma+1]
    int32_t* out_n;              // [B]
    int32_t* status;
};

__global__ void __launch_bounds__(256) lmhead_scan_kernel(LmVerifyParams q) {
    const int lane = threadIdx.x & 31;
    const int b = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (b >= q.B) return;
    const float Tb = q.T_seq ? q.T_seq[b] : q.T, Tdb = q.Td_seq ? q.Td_seq[b] : q.Td;
    const uint32_t bg = q.seq_base + static_cast<uint32_t>(b);
    const int32_t* tok = q.tokens + static_cast<long long>(b) * q.gamma;
    bool bad = false;
    int j = q.gamma;
    for (int i0 = 0; i0 < q.gamma; i0 += 32) {
        const int i = i0 + lane;
        bool reject = false;
        if (i < q.gamma) {
            const int d = tok[i];
            if (d < 0 || d >= q.V) {
                bad = true;
            } else {
                const float u = accept_uniform(q.key, bg, static_cast<uint32_t>(i));
                const float lp = q.logp_t[static_cast<long long>(b) * (q.gamma + 1) + i];
                const float lq = q.logq_d[static_cast<long long>(b) * q.gamma + i];
                // accept iff u < min(1, p/q); p(d) = 0 rejects, q(d) = 0 < p(d) accepts
                reject = !((lp > -INFINITY) && (u < expf(lp - lq)));
            }
        }
        const uint32_t rej = __ballot_sync(0xffffffffu, reject);
        if (rej && j == q.gamma) j = i0 + __ffs(rej) - 1;
    }
    if (__any_sync(0xffffffffu, bad)) j = -1;
    int32_t* out = q.out_tokens + static_cast<long long>(b) * (q.gamma + 1);
    for (int t = lane; t <= q.gamma; t += 32)
        if (t != j || j < 0) out[t] = (j >= 0 && t < j) ? tok[t] : -1;
    const bool residual = j >= 0 && j < q.gamma;
    if (lane == 0) {
        q.out_n[b] = j;
        SeqInfo si;
        si.j = j;
        si.cp = kLog2e / Tb;
        si.cq = kLog2e / Tdb;
        // log2 p(x) = x cp - mp - l2sp with mp = log2 Z (the row statistics as one number)
        si.mp = j >= 0 ? q.logZ_t[static_cast<long long>(b) * (q.gamma + 1) + j] * kLog2e : 0.0f;
        si.l2sp = 0.0f;
        si.mq = residual ? q.logZ_d[static_cast<long long>(b) * q.gamma + j] * kLog2e : 0.0f;
        si.l2sq = 0.0f;
        si.pad = 0;
        q.seq[b] = si;
        if (j < 0) set_status(q.status, 3 /* SPEC_EBADTOKEN */);
    }
}

// Per-row temperature and draft token of the target rows (b, i <= gamma; no token at
// i = gamma) and the draft rows (b, i < gamma).
__global__ void lmhead_rows_kernel(LmVerifyParams q, float* T_t, int32_t* tok_t, float* T_d, int32_t* tok_d) {
    const long long k = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    const long long rows_t = static_cast<long long>(q.B) * (q.gamma + 1);
    if (k < rows_t) {
        const int b = static_cast<int>(k / (q.gamma + 1)), i = static_cast<int>(k % (q.gamma + 1));
        T_t[k] = q.T_seq ? q.T_seq[b] : q.T;
        tok_t[k] = i < q.gamma ? q.tokens[static_cast<long long>(b) * q.gamma + i] : -1;
    }
    if (k < static_cast<long long>(q.B) * q.gamma) {
        const int b = static_cast<int>(k / q.gamma);
        T_d[k] = q.Td_seq ? q.Td_seq[b] : q.Td;
        tok_d[k] = q.tokens[k];
    }
}

// ---- the race from block maxima ----

constexpr int kLmMaxD = 32768;  // hidden size limit of the verify from hidden states (the race
                                // holds two bf16 hidden states in shared memory: 4 d bytes)

struct LmRaceParams {
    const uint16_t* h_target;   // [B, gamma+1, d] bf16 bits
    const uint16_t* h_draft;    // [B, gamma, d]
    const uint16_t* w_target;   // [V, d]
    const uint16_t* w_draft;    // [V, d]
    const uint16_t* block_max;  // [B (gamma+1), nbm] bf16 bits: each 8-token block's largest
                                // logit, rounded up
    const float* logp_t;        // [B, gamma+1] ln p_i(d_i) (the scan's inputs)
    const float* logq_d;        // [B, gamma] ln q_i(d_i)
    int d, nbm;                 // nbm = lm_block_stride(V)
};

// A score the race's winner reaches with near certainty, used as every warp's starting
// threshold; if the winner turns out lower, the sequence is raced again without it, so the
// outcome never depends on it.  The winning score is ln N + G with N the total weight and G
// a standard Gumbel variable (the largest ln w(x) - ln E_x, E_x unit exponentials), and
// P(G < -2) = exp(-e^2) < 7e-4.  Bonus row: N = 1.  Residual at a rejected position j:
// N = sum max(0, p - q) = sum max(0, q - p) >= q(d_j) - p(d_j) > 0 (a rejection needs q > p).
__device__ __forceinline__ float lm_race_guess(const LmRaceParams& q, const VerifyParams& p, int b, int j) {
    if (j >= p.gamma) return -2.0f;
    const float lp = q.logp_t[static_cast<long long>(b) * (p.gamma + 1) + j];
    const float lq = q.logq_d[static_cast<long long>(b) * p.gamma + j];
    if (!(lq > lp)) return -INFINITY;
    // ln(q - p) = ln q + ln(1 - p/q)
    return lq + log1pf(-expf(lp - lq)) - 2.0f;
}

// The logits h . w_x of one token against one or two heads, by a warp: lane l takes the
// 16-byte groups l, l + 32, ... of d (h from shared memory), products and sums in fp32, then
// a butterfly sum (every lane adds the same two partial sums at each level, so all lanes
// end with the same value).  xd is computed only when `two`.
__device__ __forceinline__ void warp_logits(const uint16_t* hs_t, const uint16_t* wt, const uint16_t* hs_d,
                                            const uint16_t* wd, bool two, int d, int lane, float& xt,
                                            float& xd) {
    float at = 0.0f, ad = 0.0f;
    const uint4* wt4 = reinterpret_cast<const uint4*>(wt);
    const uint4* wd4 = reinterpret_cast<const uint4*>(wd);
    const uint4* ht4 = reinterpret_cast<const uint4*>(hs_t);
    const uint4* hd4 = reinterpret_cast<const uint4*>(hs_d);
#pragma unroll 8
    for (int k = lane; k < d / 8; k += 32) {
        float fw[8], fh[8];
        Bf16Elem::widen(__ldg(wt4 + k), fw);
        Bf16Elem::widen(ht4[k], fh);
#pragma unroll
        for (int e = 0; e < 8; ++e) at = fmaf(fw[e], fh[e], at);
        if (two) {
            Bf16Elem::widen(__ldg(wd4 + k), fw);
            Bf16Elem::widen(hd4[k], fh);
#pragma unroll
            for (int e = 0; e < 8; ++e) ad = fmaf(fw[e], fh[e], ad);
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        at += __shfl_xor_sync(0xffffffffu, at, off);
        ad += __shfl_xor_sync(0xffffffffu, ad, off);
    }
    xt = at;
    xd = ad;
}

// Largest Philox word a token of a block whose largest target logit is bm can have and still
// reach the score thr.  With U >= w 2^-32 and E = -log1p(-U) >= U, a token's score is at most
// ln p(x) + (32 - log2 w) ln 2, and ln p(x) <= ((bm + delta) cp - mp) ln 2 (the residual's
// weight max(0, p - q) never exceeds p), so it can reach thr only if
//     log2 w <= R = (bm + delta) cp - mp + 32 - thr log2(e).
// delta = 1e-3 (1 + |bm|) covers the gap between the GEMM's block maximum and a token's logit
// recomputed by warp_logits, and R gets a further 1e-3 for exp2f's rounding; w = 0 (whose
// bound is infinite) always passes.
__device__ __forceinline__ uint32_t lm_word_bound(float bm, float thr, const SeqInfo& si) {
    if (!(thr > -INFINITY)) return 0xffffffffu;
    const float R = fmaf(bm + 1e-3f * (1.0f + fabsf(bm)), si.cp, 32.0f - si.mp - thr * kLog2e) + 1e-3f;
    if (!(R < 31.99f)) return 0xffffffffu;
    if (!(R > 0.0f)) return 0u;
    return static_cast<uint32_t>(exp2f(R));
}

// Warps of one group race chunks cb + wib, cb = cb_begin, cb_begin + cb_step, ... (< nch) of
// 1024 tokens of the raced row (lane l: tokens x0 = 1024 (cb + wib) + 32 l .. x0 + 31, four
// 8-token blocks whose maxima are bm_row[x0 / 8 ..]); best / best_idx / thr are the warp's
// (the same in every lane).
__device__ __forceinline__ void lm_race_chunks(const VerifyParams& p, const LmRaceParams& q, const SeqInfo& si,
                                               bool residual, uint32_t bg, const uint16_t* bm_row,
                                               const uint16_t* hs_t, const uint16_t* hs_d,
                                               const uint16_t* wt_base, const uint16_t* wd_base, int cb_begin,
                                               int cb_step, int wib, int lane, volatile float* s_thr, int nw,
                                               float& best, int& best_idx, float& thr) {
    const RaceRowRng rr = race_row_rng(p.rk, bg, static_cast<uint32_t>(si.j));
    const int nch = (p.V + 1023) >> 10;
    for (int cb = cb_begin; cb < nch; cb += cb_step) {
        const int ch = cb + wib;
        const int x0 = ch * 1024 + 32 * lane;
        const int nvalid = ch < nch ? max(0, min(32, p.V - x0)) : 0;
        float bm[4];
        {
            const uint2 h = nvalid > 0 ? __ldg(reinterpret_cast<const uint2*>(bm_row + (x0 >> 3))) : make_uint2(0xFF80FF80u, 0xFF80FF80u);
            bm[0] = __uint_as_float(h.x << 16);
            bm[1] = __uint_as_float(h.x & 0xFFFF0000u);
            bm[2] = __uint_as_float(h.y << 16);
            bm[3] = __uint_as_float(h.y & 0xFFFF0000u);
        }
        uint32_t w[32];
#pragma unroll
        for (int k = 0; k < 8; ++k) {
            const uint4 v = race_block_fast(rr, p.rk, static_cast<uint32_t>(x0 >> 2) + static_cast<uint32_t>(k));
            w[4 * k] = v.x;
            w[4 * k + 1] = v.y;
            w[4 * k + 2] = v.z;
            w[4 * k + 3] = v.w;
        }
        const uint32_t valid = nvalid >= 32 ? 0xffffffffu : ((1u << nvalid) - 1u);
        // the tokens of this lane's four blocks that can still reach thr
        auto candidates = [&](float t) -> uint32_t {
            uint32_t m = 0;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                if (!(bm[k] > -INFINITY)) continue;  // every weight of the block is zero
                const uint32_t wb = lm_word_bound(bm[k], t, si);
#pragma unroll
                for (int e = 8 * k; e < 8 * k + 8; ++e) m |= (w[e] <= wb ? 1u : 0u) << e;
            }
            return m & valid;
        };
        uint32_t cand = candidates(thr);
        while (true) {
            const uint32_t lanes = __ballot_sync(0xffffffffu, cand != 0u);
            if (!lanes) break;
            // the most promising candidate of the warp: the largest bound bm cp - log2 w of
            // each lane's candidates, then of the lanes
            float key = -INFINITY;
            int el = 0;
#pragma unroll
            for (int e = 0; e < 32; ++e)
                if ((cand >> e) & 1u) {
                    const float ke = fmaf(bm[e >> 3], si.cp, -__log2f(static_cast<float>(w[e]) + 0.5f));
                    if (ke > key) {
                        key = ke;
                        el = e;
                    }
                }
            uint32_t wl = 0;
#pragma unroll
            for (int e = 0; e < 32; ++e) wl = e == el ? w[e] : wl;
            int src = lane;
#pragma unroll
            for (int off = 16; off > 0; off >>= 1) {
                const float ok = __shfl_xor_sync(0xffffffffu, key, off);
                const int os = __shfl_xor_sync(0xffffffffu, src, off);
                if (ok > key || (ok == key && os < src)) {
                    key = ok;
                    src = os;
                }
            }
            const int e = __shfl_sync(0xffffffffu, el, src);
            const uint32_t wx = __shfl_sync(0xffffffffu, wl, src);
            if (lane == src) cand &= ~(1u << e);
            const int x = ch * 1024 + 32 * src + e;
            float xt, xd;
            warp_logits(hs_t, wt_base + static_cast<long long>(x) * q.d, hs_d,
                        residual ? wd_base + static_cast<long long>(x) * q.d : wt_base, residual, q.d, lane, xt, xd);
            const float lw = race_log_weight(xt, xd, si, residual);
            const float sc = lw > -INFINITY ? lw - race_log_exponential(wx) : -INFINITY;
            if (sc > -INFINITY && (sc > best || (sc == best && x < best_idx))) {
                best = sc;
                best_idx = x;
            }
            if (best > thr) {
                thr = best;
                cand &= candidates(thr);
            }
        }
        // every warp's best so far bounds the sequence's best from below: share them through
        // shared memory without a barrier (an old or a new value is such a bound either way)
        if (lane == 0) s_thr[wib] = thr;
        const float t = lane < nw ? s_thr[lane] : -INFINITY;
        thr = fmaxf(thr, float_unorder(__reduce_max_sync(0xffffffffu, float_order(t))));
    }
}

// G blocks per sequence (8 warps each) race its row j from the block maxima: block g takes
// the chunks 8 g + w, 8 g + w + 8 G, ... (warp w); the blocks' winners meet in the race
// partial slots, and the sequence's last block writes the token.  Dynamic shared memory: the
// raced rows' hidden states (target, and draft for a residual), 2 d bf16.
__global__ void __launch_bounds__(256, SPECVERIFY_RACE_MINBLOCKS) lmhead_race_kernel(VerifyParams p, LmRaceParams q) {
    extern __shared__ uint4 lm_h_smem[];
    __shared__ float s_thr[8];
    __shared__ RaceState s_best[8];
    __shared__ int s_last;
    constexpr int NW = 8;
    const int G = p.rgroups;
    const int b = blockIdx.x / G, g = blockIdx.x % G;
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const SeqInfo si = p.seq[b];
    if (si.j < 0) return;
    const bool residual = si.j < p.gamma;
    uint16_t* hs_t = reinterpret_cast<uint16_t*>(lm_h_smem);
    uint16_t* hs_d = hs_t + q.d;
    {
        const uint4* src_t = reinterpret_cast<const uint4*>(q.h_target + (static_cast<long long>(b) * (p.gamma + 1) + si.j) * q.d);
        const uint4* src_d = residual ? reinterpret_cast<const uint4*>(q.h_draft + (static_cast<long long>(b) * p.gamma + si.j) * q.d)
                                      : nullptr;
        for (int k = threadIdx.x; k < q.d / 8; k += blockDim.x) {
            lm_h_smem[k] = __ldg(src_t + k);
            lm_h_smem[q.d / 8 + k] = residual ? __ldg(src_d + k) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    if (threadIdx.x < NW) s_thr[threadIdx.x] = -INFINITY;
    __syncthreads();
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    const uint16_t* bm_row = q.block_max + (static_cast<long long>(b) * (p.gamma + 1) + si.j) * q.nbm;
    const float guess = (p.debug_flags & kDebugRaceAgain) ? INFINITY : lm_race_guess(q, p, b, si.j);
    float best = -INFINITY, thr = guess;
    int best_idx = INT_MAX;
    lm_race_chunks(p, q, si, residual, bg, bm_row, hs_t, hs_d, q.w_target, q.w_draft, g * NW, G * NW, wib, lane,
                   s_thr, NW, best, best_idx, thr);
    if (lane == 0) s_best[wib] = RaceState{best, best_idx, -INFINITY};
    __syncthreads();
    RacePart* parts = p.race_parts + static_cast<long long>(b) * race_slots(p.rpieces);
    if (threadIdx.x == 0) {
        RaceState m = s_best[0];
        for (int k = 1; k < NW; ++k) m = race_merge(m, s_best[k]);
        const long long ps = static_cast<long long>(b) * race_slots(p.rpieces) + g;
        if (g < race_slots(p.rpieces) && sv_in_range(p, ps, p.caps.race))
            *reinterpret_cast<unsigned long long*>(parts + g) = pack_race(m.best, m.idx);
        s_last = (atomicAdd(p.tickets + b, 1) == G - 1);
    }
    __syncthreads();
    if (!s_last) return;
    // last block of this sequence: merge every block's winner, waiting (bounded) for each
    RaceState m{-INFINITY, INT_MAX, -INFINITY};
    if (wib == 0) {
        for (int k = lane; k < G; k += 32) {
            unsigned long long v = ld_relaxed_u64g(parts + k);
            if (v == 0ull) {
                const unsigned long long t0 = global_time_ns();
                while ((v = ld_relaxed_u64g(parts + k)) == 0ull) {
                    if (global_time_ns() - t0 > kWaitLimitNs) break;
                    __nanosleep(64);
                }
                if (v == 0ull) set_status(p.status, 4 /* SPEC_ETIMEOUT */);
            }
            if (v != 0ull)
                m = race_merge(m, RaceState{__uint_as_float(static_cast<uint32_t>(v)),
                                            static_cast<int>(static_cast<uint32_t>(v >> 32) - 1u), -INFINITY});
        }
        m = warp_race_merge(m);
        if (lane == 0) s_best[0] = m;
    }
    __syncthreads();
    m = s_best[0];
    // The whole row again, by this block, from threshold t0 (over p_j when `bonus_of_p`).
    auto race_again = [&](bool res, float t0) {
        __syncthreads();
        if (threadIdx.x < NW) s_thr[threadIdx.x] = t0;
        __syncthreads();
        best = -INFINITY;
        thr = t0;
        best_idx = INT_MAX;
        lm_race_chunks(p, q, si, res, bg, bm_row, hs_t, hs_d, q.w_target, q.w_draft, 0, NW, wib, lane, s_thr, NW,
                       best, best_idx, thr);
        if (lane == 0) s_best[wib] = RaceState{best, best_idx, -INFINITY};
        __syncthreads();
        RaceState r = s_best[0];
        for (int k = 1; k < NW; ++k) r = race_merge(r, s_best[k]);
        return r;
    };
    // The starting threshold was above the winner (rare): tokens below it were never scored.
    // Race again from the best score found (a score some token has), or from nothing.
    if (!(m.best >= guess)) m = race_again(residual, m.idx == INT_MAX ? -INFINITY : m.best);
    // Every residual weight was zero (p <= q everywhere in fp32): draw from p_j.
    if (m.idx == INT_MAX) m = race_again(false, -INFINITY);
    if (threadIdx.x == 0) {
        p.out_tokens[static_cast<long long>(b) * (p.gamma + 1) + si.j] = m.idx;
        if (p.out_race) {
            p.out_race[2 * b] = m.best;
            p.out_race[2 * b + 1] = m.second;
        }
    }
}

}  // namespace specverify
