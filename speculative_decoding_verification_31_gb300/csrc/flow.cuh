// flow.cuh -- the sampling verify as one persistent (cooperative) launch in which each
// sequence's scan and race run as soon as its rows have been streamed, while the rows of later
// sequences are still being read (SPEC_FLAG_FUSED).
//
// The method is the same as the two-kernel path's ("How speculative decoding makes LLMs go
// brrr": pseudocode and module 3): per-row softmax statistics of p at T and q at T_d, the
// acceptance scan u_i < min(1, p_i(d_i) / q_i(d_i)) up to the first rejection j, then one draw
// from the residual max(0, p_j - q_j) (or from p_gamma) as an exponential race, with the same
// arithmetic in the same order, so the outputs are the same bits.  Only the schedule differs:
// one launch, no kernel boundary between the streaming pass and the races, and the races of
// the first sequences start while the last row items are still being read.
//
// Work:
//   row items   (b, r, piece) in sequence-major order, dealt round-robin to every warp (a
//               shared claim counter would throttle the stream: measured, its atomics cost
//               more than half the bandwidth): the streaming pass's item (partial softmax
//               statistics of one row piece, one packed 64-bit word), then one relaxed
//               increment of the sequence's item count.  Row items never wait.
//   race units  (b, u): tokens [u K, (u+1) K) of sequence b's raced row, claimed from a second
//               cursor once a warp finds no row item left, in spans of consecutive units that
//               shrink as the units run out (guided self-scheduling).  A span starting at unit
//               0 first waits (bounded) for the sequence's items, merges its rows, runs the
//               acceptance scan, writes the sequence's outputs and publishes the scan behind a
//               release flag; other spans wait (bounded) for that flag.  A span publishes its
//               winner as one packed word and takes one ticket per unit; the sequence's last
//               span merges the winners and writes the token.
// Every wait is for work of a warp that does not wait on it: row items are done by warps
// that never wait in them, and a scan by the warp holding unit 0, which waits only for row
// items (a claim that reaches into later sequences runs their unit-0 spans first).  Each wait
// gives up after kWaitLimitNs and records SPEC_ETIMEOUT.
//
// Measured on GB300 this schedule is slower than the two-kernel one at every size: the race
// and the streaming pass need the issue slots and registers of the same SMs (the race's
// registers leave 16 warps per SM for the stream, against 24 in row_stats), and a warp-level
// race unit cannot share its threshold the way a block does.
//
// The flow path's workspace (cursors, counts, flags, tickets, packed winners and the row
// partials in use, all meaning "nothing yet" when zero) is zeroed by prep_fill_kernel just
// before the flow kernel, which is its programmatic dependent where the device allows it.
#pragma once

#include "kernels.cuh"

namespace specverify {

#ifndef SPECVERIFY_FLOW_MINBLOCKS
#define SPECVERIFY_FLOW_MINBLOCKS 2
#endif
#ifndef SPECVERIFY_FLOW_LOADS
#define SPECVERIFY_FLOW_LOADS 16
#endif
#ifndef SPECVERIFY_FLOW_UNIT_CHUNKS
#define SPECVERIFY_FLOW_UNIT_CHUNKS 1
#endif
#ifndef SPECVERIFY_FLOW_CLAIM
#define SPECVERIFY_FLOW_CLAIM 8
#endif
constexpr int kFlowLoads = SPECVERIFY_FLOW_LOADS;  // 16-byte loads in flight per stream lane
constexpr int kFlowClaim = SPECVERIFY_FLOW_CLAIM;  // race units per claim, at most
// tokens of the raced row per race unit (small: the last sequences' races are the tail)
constexpr int kFlowUnitTokens = SPECVERIFY_FLOW_UNIT_CHUNKS * kRaceWarpTokens;

__device__ __forceinline__ void red_add_relaxed(int* p, int v) {
    asm volatile("red.relaxed.gpu.global.add.s32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_u64(unsigned long long* p, unsigned long long v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Exponential race over tokens [xa, xb) of one raced row by one warp.  The span is read in
// chunks of kRaceWarpTokens (the next chunk's vectors are loaded while the current one is
// scored); Philox blocks are computed kRaceChains at a time per lane; the threshold is seeded
// from each lane's largest logit (a fast lower bound of its score) and raised to the warp's
// best exact score after every group, and a token is scored exactly only if it passes the
// bound test (see kRaceBoundMargin2).  Each lane offers its tokens in increasing x, so the
// result is the same winner, bit for bit, as any other split of the row.  rt and rd hold
// tokens xoff, xoff + 1, ... of the row (a vocabulary shard; xoff a multiple of 8): random
// numbers and the winner's index are those of token x + xoff.
template <class ET>
__device__ __forceinline__ RaceState race_warp_span(const VerifyParams& p,
                                                   const typename ET::storage* rt,
                                                   const typename ET::storage* rd, bool residual,
                                                   uint32_t bg, uint32_t pos, int xa, int xb,
                                                   const SeqInfo& si, int lane, int xoff = 0) {
    constexpr int VPL = kRaceWarpTokens / (32 * ET::kVec);
    const RaceRowRng q = race_row_rng(p.rk, bg, pos);
    RaceState st{-INFINITY, INT_MAX, -INFINITY};
    auto word_at = [&](int x) {
        const uint4 blk = race_block_fast(q, p.rk, static_cast<uint32_t>(x + xoff) >> 2);
        return word_of(blk, static_cast<uint32_t>(x + xoff) & 3u);
    };
    auto offer_exact = [&](float xt, int x, uint32_t w) {
        const float xd = residual ? ET::load1(rd + x) : 0.0f;
        const float sc = race_exact_score(xt, xd, si, residual, w);
        if (sc > -INFINITY) race_offer(st, sc, x + xoff);
    };
    auto load_chunk = [&](int x0, uint4 (&dst)[VPL]) {
        const int x1 = min(xb, x0 + kRaceWarpTokens);
        if (residual) prefetch_l2(rd, x0, x1, lane);
        const bool ok = x0 < x1 && (reinterpret_cast<uintptr_t>(rt + x0) & 15u) == 0;
        const int nv = ok ? (x1 - x0) / ET::kVec : 0;
        const uint4* vt = reinterpret_cast<const uint4*>(rt + (ok ? x0 : 0));
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int v = lane + 32 * k;
            dst[k] = v < nv ? __ldg(vt + v) : make_uint4(ET::kNegInfWord, ET::kNegInfWord,
                                                         ET::kNegInfWord, ET::kNegInfWord);
        }
    };
    uint4 raw[VPL], raw_next[VPL];
    load_chunk(xa, raw);
    float thr = -INFINITY;
    bool first = true;
    for (int x0 = xa; x0 < xb; x0 += kRaceWarpTokens) {
        const int x1 = min(xb, x0 + kRaceWarpTokens);
        const bool vec_ok = (reinterpret_cast<uintptr_t>(rt + x0) & 15u) == 0;
        const int nvec = vec_ok ? (x1 - x0) / ET::kVec : 0;
        const bool more = x0 + kRaceWarpTokens < xb;
        if (more) load_chunk(x0 + kRaceWarpTokens, raw_next);
        if (first) {
            float seed = -INFINITY;
            if (vec_ok) {
                float vmax = -INFINITY;
                int xs = -1;
#pragma unroll
                for (int k = 0; k < VPL; ++k) {
                    float ft[ET::kVec];
                    ET::widen(raw[k], ft);
                    float m = ft[0];
#pragma unroll
                    for (int e = 1; e < ET::kVec; ++e) m = fmaxf(m, ft[e]);
                    if (m > vmax) {
                        vmax = m;
#pragma unroll
                        for (int e = ET::kVec - 1; e >= 0; --e)
                            if (ft[e] == m) xs = x0 + (lane + 32 * k) * ET::kVec + e;
                    }
                }
                if (xs >= 0) {
                    const float xd = residual ? ET::load1(rd + xs) : 0.0f;
                    seed = race_score_lower_bound(vmax, xd, si, residual, word_at(xs));
                }
            }
            thr = float_unorder(__reduce_max_sync(0xffffffffu, float_order(seed)));
            first = false;
        }
        if (vec_ok) {
            const float mpl = si.mp + si.l2sp;
            constexpr int BPV = ET::kVec / 4;  // Philox blocks per 16-byte vector
            constexpr int VG = kRaceChains / BPV;
            static_assert(VPL % VG == 0, "race vectors per lane must fill whole groups");
#pragma unroll
            for (int k0 = 0; k0 < VPL; k0 += VG) {
                const float C = (thr > -INFINITY) ? 32.0f + kRaceBoundMargin2 - thr * kLog2e - mpl
                                                  : INFINITY;
                uint4 blk[VG * BPV];
#pragma unroll
                for (int kk = 0; kk < VG; ++kk)
#pragma unroll
                    for (int gg = 0; gg < BPV; ++gg)
                        blk[kk * BPV + gg] = race_block_fast(
                            q, p.rk,
                            static_cast<uint32_t>(xoff + x0 + (lane + 32 * (k0 + kk)) * ET::kVec + 4 * gg) >> 2);
#pragma unroll
                for (int kk = 0; kk < VG; ++kk) {
                    const int v = lane + 32 * (k0 + kk);
                    if (v >= nvec) continue;
                    float ft[ET::kVec];
                    ET::widen(raw[k0 + kk], ft);
                    const int xv = x0 + v * ET::kVec;
                    uint32_t cand = vector_candidates<ET>(ft, blk + kk * BPV, si.cp, C);
                    while (cand) {  // rare: exact scores in increasing token order
                        const int e = __ffs(cand) - 1;
                        cand &= cand - 1;
                        offer_exact(ET::load1(rt + xv + e), xv + e, word_at(xv + e));
                    }
                }
                thr = fmaxf(thr, float_unorder(__reduce_max_sync(0xffffffffu, float_order(st.best))));
            }
            const int t0 = nvec * ET::kVec;
            if (lane < (x1 - x0) - t0)
                offer_exact(ET::load1(rt + x0 + t0 + lane), x0 + t0 + lane, word_at(x0 + t0 + lane));
        } else {
            for (int x = x0 + lane; x < x1; x += 32) offer_exact(ET::load1(rt + x), x, word_at(x));
        }
        if (more) {
#pragma unroll
            for (int k = 0; k < VPL; ++k) raw[k] = raw_next[k];
        }
    }
    return warp_race_merge(st);
}

// The scan of sequence b by the warp holding its race unit 0: wait (bounded) for the
// sequence's items, check the draft tokens, then 16 positions at a time merge their target and
// draft rows (one lane per row, fold_row_stats: the same bits as the two-kernel path) and
// decide them; write the sequence's outputs and publish the raced rows' statistics.  Returns
// 0 if a wait gave up.
template <class ET>
__device__ __noinline__ int flow_scan(const VerifyParams& p, int b, int lane, SeqInfo* out) {
    using S = typename ET::storage;
    const int g = p.gamma, R = 2 * g + 1, P = p.npieces;
    int ok = 1;
    if (lane == 0) {
        const int* cnt = p.flow.items + b;
        if (ld_relaxed(cnt) < R * P) {
            const unsigned long long t0 = global_time_ns();
            unsigned ns = 64;
            while (ld_relaxed(cnt) < R * P) {
                if (global_time_ns() - t0 > kWaitLimitNs) {
                    ok = 0;
                    set_status(p.status, 4 /* SPEC_ETIMEOUT */);
                    break;
                }
                __nanosleep(ns);
                if (ns < 1024) ns <<= 1;
            }
        }
    }
    if (!__shfl_sync(0xffffffffu, ok, 0)) return 0;
    const float cp = scale_of(seq_T(p, b)), cq = scale_of(seq_Td(p, b));
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    const long long tok0 = static_cast<long long>(b) * g;
    // any draft token outside [0, V) marks the whole sequence
    bool bad = false;
    for (int i = lane; i < g; i += 32) {
        const int d = p.tokens[tok0 + i];
        bad |= (d < 0 || d >= p.V);
    }
    bad = __any_sync(0xffffffffu, bad);
    const unsigned long long* parts =
        reinterpret_cast<const unsigned long long*>(p.stat_parts) + static_cast<long long>(b) * R * P;
    const bool diag = p.out_logZp || p.out_logZq || p.out_logp || p.out_logq || p.out_u;
    int j = g;
    float jmp = 0.0f, jlp = 0.0f, jmq = 0.0f, jlq = 0.0f;  // the raced rows' statistics
    // positions 16 at a time: lane l < 16 folds target row i0 + l, lane 16 + l draft row i0 + l
    const int half = lane >> 4, l = lane & 15;
    for (int i0 = 0; i0 <= g; i0 += 16) {
        const int i = i0 + l;
        const bool has = half == 0 ? (i <= g) : (i < g);
        const int r = half == 0 ? i : g + 1 + i;
        SoftmaxStat st{-FLT_MAX, 0.0f};
        if (has) st = fold_row_stats<true>(p, parts + static_cast<long long>(r) * P, P);
        const float l2s = log2f(st.s);
        if (has) {
            const float lz = (st.m + l2s) * kLn2;
            if (half == 0 && p.out_logZp) p.out_logZp[static_cast<long long>(b) * (g + 1) + i] = lz;
            if (half == 1 && p.out_logZq) p.out_logZq[tok0 + i] = lz;
        }
        const float dm = __shfl_sync(0xffffffffu, st.m, 16 + l);
        const float dl = __shfl_sync(0xffffffffu, l2s, 16 + l);
        // accept iff u < min(1, p/q); p(d) = 0 rejects, q(d) = 0 < p(d) accepts
        bool reject = false;
        if (half == 0 && i < g) {
            const long long k = tok0 + i;
            const float u = accept_uniform(p.key, bg, static_cast<uint32_t>(i));
            if (p.out_u) p.out_u[k] = u;
            if (bad) {
                if (p.out_logp) p.out_logp[k] = NAN;
                if (p.out_logq) p.out_logq[k] = NAN;
            } else {
                const int d = p.tokens[k];
                const float xt = ET::load1(static_cast<const S*>(p.target) +
                                           (static_cast<long long>(b) * (g + 1) + i) * p.V + d);
                const float xd = ET::load1(static_cast<const S*>(p.draft) + k * p.V + d);
                const float l2p = fmaf(xt, cp, -st.m) - l2s;
                const float l2q = fmaf(xd, cq, -dm) - dl;
                if (p.out_logp) p.out_logp[k] = l2p * kLn2;
                if (p.out_logq) p.out_logq[k] = l2q * kLn2;
                reject = !((l2p > -INFINITY) && (u < exp2f(l2p - l2q)));
            }
        }
        const unsigned rej = __ballot_sync(0xffffffffu, reject);
        if (!bad && j == g) {  // warp-uniform
            if (rej) {
                j = i0 + __ffs(rej) - 1;
                jmp = __shfl_sync(0xffffffffu, st.m, j - i0);
                jlp = __shfl_sync(0xffffffffu, l2s, j - i0);
                jmq = __shfl_sync(0xffffffffu, st.m, 16 + j - i0);
                jlq = __shfl_sync(0xffffffffu, l2s, 16 + j - i0);
            } else if (g - i0 < 16) {  // every draft accepted: the bonus row is in this chunk
                jmp = __shfl_sync(0xffffffffu, st.m, g - i0);
                jlp = __shfl_sync(0xffffffffu, l2s, g - i0);
            }
        }
        // rows past the first rejection decide nothing; diagnostics still cover every row
        if ((j < g || bad) && !diag) break;
    }
    if (bad) j = -1;
    if (lane == 0) {
        p.out_n[b] = j;
        if (j < 0) set_status(p.status, 3 /* SPEC_EBADTOKEN */);
    }
    int32_t* outt = p.out_tokens + static_cast<long long>(b) * (g + 1);
    for (int t = lane; t <= g; t += 32)
        if (t != j) outt[t] = (j >= 0 && t < j) ? p.tokens[tok0 + t] : -1;
    SeqInfo si;
    si.j = j;
    si.cp = cp;
    si.cq = cq;
    si.mp = jmp;
    si.l2sp = jlp;
    const bool residual = j >= 0 && j < g;
    si.mq = residual ? jmq : 0.0f;
    si.l2sq = residual ? jlq : 0.0f;
    si.pad = 0;
    if (lane == 0) {
        p.flow.seq[b] = si;
        __threadfence();
        if (!(p.debug_flags & kDebugNeverReady)) st_release(p.flow.ready + b, 1);
    }
    *out = si;
    return 1;
}

// Wait (bounded) for sequence b's published scan and read it.  Returns 0 if the wait gave up.
__device__ __forceinline__ int flow_wait_scan(const VerifyParams& p, int b, int lane, SeqInfo* out) {
    int ok = 0;
    if (lane == 0) {
        ok = ld_acquire(p.flow.ready + b);
        if (!ok) {
            const unsigned long long t0 = global_time_ns();
            unsigned ns = 64;
            while (!(ok = ld_acquire(p.flow.ready + b))) {
                if (global_time_ns() - t0 > kWaitLimitNs) break;
                __nanosleep(ns);
                if (ns < 1024) ns <<= 1;
            }
            if (!ok) set_status(p.status, 4 /* SPEC_ETIMEOUT */);
        }
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    __syncwarp();  // the other lanes' reads come after lane 0's acquire
    if (!ok) return 0;
    const int4 a = __ldcg(reinterpret_cast<const int4*>(p.flow.seq + b));
    const float4 q = __ldcg(reinterpret_cast<const float4*>(p.flow.seq + b) + 1);
    out->j = a.x;
    out->mp = __int_as_float(a.y);
    out->l2sp = __int_as_float(a.z);
    out->mq = __int_as_float(a.w);
    out->l2sq = q.x;
    out->cp = q.y;
    out->cq = q.z;
    out->pad = 0;
    return 1;
}

// Units [u0, u0 + n) of sequence b, raced by one warp as one span: the scan (when u0 = 0) or
// the wait for it, the race of tokens [u0 K, (u0 + n) K), the span's winner in slot u0 and
// "nothing" in the others, then n tickets; the sequence's last units merge every slot and
// write the token.
template <class ET>
__device__ __forceinline__ void flow_span(const VerifyParams& p, int b, int u0, int n, int lane) {
    using S = typename ET::storage;
    const int U = p.flow.units, g = p.gamma;
    SeqInfo si;
    int ok = (u0 == 0) ? flow_scan<ET>(p, b, lane, &si) : 1;
    if (ok && (u0 != 0 || (p.debug_flags & kDebugNeverReady))) ok = flow_wait_scan(p, b, lane, &si);
    const bool live = ok && si.j >= 0;
    const bool residual = live && si.j < g;
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    const S* rt = live ? static_cast<const S*>(p.target) + (static_cast<long long>(b) * (g + 1) + si.j) * p.V
                       : nullptr;
    const S* rd = residual ? static_cast<const S*>(p.draft) + (static_cast<long long>(b) * g + si.j) * p.V
                           : nullptr;
    RaceState st{-INFINITY, INT_MAX, -INFINITY};
    if (live)
        st = race_warp_span<ET>(p, rt, rd, residual, bg, static_cast<uint32_t>(si.j), u0 * kFlowUnitTokens,
                                min(p.V, (u0 + n) * kFlowUnitTokens), si, lane);
    const long long slot0 = static_cast<long long>(b) * U + u0;
    for (int k = lane; k < n; k += 32) {  // packed words are never zero
        p.flow.second[slot0 + k] = k == 0 ? st.second : -INFINITY;  // diagnostic only (never polled)
        st_relaxed_u64(p.flow.race + slot0 + k, k == 0 ? pack_race(st.best, st.idx) : pack_race(-INFINITY, INT_MAX));
    }
    __syncwarp();
    int t = 0;
    if (lane == 0) t = atomicAdd(p.flow.tickets + b, n);
    if (__shfl_sync(0xffffffffu, t, 0) + n != U) return;
    // the sequence's last units: every slot (each polled: arrivals carry no fence)
    RaceState m{-INFINITY, INT_MAX, -INFINITY};
    for (int k = lane; k < U; k += 32) {
        const unsigned long long v = poll_nonzero_u64(p, p.flow.race + static_cast<long long>(b) * U + k);
        if (v != 0ull) {
            const float sec = __ldcg(p.flow.second + static_cast<long long>(b) * U + k);
            m = race_merge(m, RaceState{__uint_as_float(static_cast<uint32_t>(v)),
                                        static_cast<int>(static_cast<uint32_t>(v >> 32) - 1u), sec});
        }
    }
    m = warp_race_merge(m);
    if (!live) return;
    if (m.idx == INT_MAX)  // every residual weight was zero (p <= q everywhere in fp32): draw from p_j
        m = race_piece<ET>(rt, nullptr, 0, p.V, si, false, p.rk, bg, static_cast<uint32_t>(si.j), lane);
    if (lane == 0) {
        p.out_tokens[static_cast<long long>(b) * (g + 1) + si.j] = m.idx;
        if (p.out_race) {
            p.out_race[2 * b] = m.best;
            p.out_race[2 * b + 1] = m.second;
        }
    }
}

template <class ET, int UNR>
__global__ void __launch_bounds__(256, SPECVERIFY_FLOW_MINBLOCKS) verify_flow_kernel(VerifyParams p) {
    const int lane = threadIdx.x & 31;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the flow region has been zeroed
    const long long RP = static_cast<long long>(2 * p.gamma + 1) * p.npieces;
    const long long total = static_cast<long long>(p.B) * RP;
    {  // every warp streams its row items (round-robin over the warps, in sequence-major
       // order: one shared claim counter throttles the stream), then races
        const long long nw = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
        for (long long g = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5; g < total;
             g += nw) {
            const int b = static_cast<int>(g / RP);
            const int within = static_cast<int>(g % RP);
            row_stats_item<ET, UNR, kFlowLoads>(p, b, within / p.npieces, within % p.npieces, lane);
            if (lane == 0) red_add_relaxed(p.flow.items + b, 1);
        }
    }
    // race units, claimed in spans that shrink as the units run out (guided self-scheduling:
    // about the remaining units over the warps, at most kFlowClaim)
    const int U = p.flow.units;
    const long long units = static_cast<long long>(p.B) * U;
    const long long nwarps = static_cast<long long>(gridDim.x) * (blockDim.x >> 5);
    while (true) {
        long long c = 0;
        int n = 0;
        if (lane == 0) {
            const long long left = units - static_cast<long long>(ld_relaxed_u64g(p.flow.cursors + 16));
            n = static_cast<int>(max(1LL, min(static_cast<long long>(kFlowClaim), left / nwarps)));
            c = static_cast<long long>(atomicAdd(p.flow.cursors + 16, static_cast<unsigned long long>(n)));
        }
        c = __shfl_sync(0xffffffffu, c, 0);
        n = __shfl_sync(0xffffffffu, n, 0);
        if (c >= units) break;
        // one span per sequence the claim touches; the later sequences' spans start at unit 0
        // (their scans wait for nothing but rows) and go first, so that no scan waits behind
        // the race of an earlier sequence's units
        const long long cend = min(c + n, units);
        const long long first_end = min(cend, (c / U + 1) * U);
        for (long long cc = first_end; cc < cend;) {
            const int nb = static_cast<int>(min(cend - cc, static_cast<long long>(U)));
            flow_span<ET>(p, static_cast<int>(cc / U), 0, nb, lane);
            cc += nb;
        }
        flow_span<ET>(p, static_cast<int>(c / U), static_cast<int>(c % U), static_cast<int>(first_end - c), lane);
    }
}

}  // namespace specverify
