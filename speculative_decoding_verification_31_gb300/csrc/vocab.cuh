// vocab.cuh -- the sampling verify with the vocabulary split over ranks (vocabulary-parallel
// logits, as a tensor-parallel LM head leaves them): rank w holds columns
// [x_w, x_w + V_w) of every target and draft row.
//
// Per call, on every rank:
//   vp_partials   per row, the (max, sum) softmax statistics of the rank's columns (the
//                 streaming pass over the shard, its pieces folded in order), and the logits
//                 at the draft tokens the rank owns (-inf where it does not);
//   (all-gather of the statistics, max all-reduce of the gathered logits)
//   vp_decide     merge every row's statistics in rank order, draw u_i, find the first
//                 rejection j ("How speculative decoding makes LLMs go brrr": pseudocode and
//                 module 3), write the accepted prefix and keep the raced rows' statistics;
//   vp_race       the exponential race over the rank's columns of the raced row, keyed by the
//                 global token index, so the union of the ranks' races is the one-GPU race;
//                 returns the packed winner (and, where the rank's residual weights are all
//                 zero, the winner of the race over p_j, the fallback for an empty residual);
//   (max all-reduce of the packed winners)
//   vp_finish     write the drawn token.
// The exchanged bytes are O(B gamma) against O(B gamma V) logits.  Decisions agree with the
// one-GPU verify except where the two merge orders round a near-tie differently.
#pragma once

#include "kernels.cuh"

namespace specverify {

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
    // (chunks start on multiples of four tokens; one off a 16-byte boundary is read with
    // narrower loads)
    auto load_chunk = [&](int x0, uint4 (&dst)[VPL]) {
        const int x1 = min(xb, x0 + kRaceWarpTokens);
        if (residual) prefetch_l2(rd, x0, x1, lane);
        const int nv = x0 < x1 ? (x1 - x0) / ET::kVec : 0;
        const typename ET::storage* base = rt + (x0 < x1 ? x0 : 0);
        const bool al = (reinterpret_cast<uintptr_t>(base) & 15u) == 0;
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int v = lane + 32 * k;
            dst[k] = v >= nv ? make_uint4(ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord)
                   : al ? __ldg(reinterpret_cast<const uint4*>(base) + v)
                        : ET::load_vec_unaligned(base + v * ET::kVec);
        }
    };
    uint4 raw[VPL], raw_next[VPL];
    load_chunk(xa, raw);
    float thr = -INFINITY;
    bool first = true;
    for (int x0 = xa; x0 < xb; x0 += kRaceWarpTokens) {
        const int x1 = min(xb, x0 + kRaceWarpTokens);
        const bool vec_ok = ((x0 + xoff) & 3) == 0;  // a vector's Philox blocks are whole
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
                // every vector's coarse test first, then (rarely) its tokens, scored exactly in
                // increasing token order
                bool coarse[VG];
                bool any = false;
#pragma unroll
                for (int kk = 0; kk < VG; ++kk) {
                    coarse[kk] = lane + 32 * (k0 + kk) < nvec &&
                                 vector_may_win<ET>(raw[k0 + kk], blk + kk * BPV, si.cp, C);
                    any |= coarse[kk];
                }
                if (any) {
#pragma unroll
                    for (int kk = 0; kk < VG; ++kk) {
                        if (!coarse[kk]) continue;
                        float ft[ET::kVec];
                        ET::widen(raw[k0 + kk], ft);
                        const int xv = x0 + (lane + 32 * (k0 + kk)) * ET::kVec;
                        uint32_t cand = token_candidates<ET>(ft, blk + kk * BPV, si.cp, C);
                        while (cand) {
                            const int e = __ffs(cand) - 1;
                            cand &= cand - 1;
                            offer_exact(ET::load1(rt + xv + e), xv + e, word_at(xv + e));
                        }
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

// Per-sequence state between vp_decide and vp_race / vp_finish (opaque to callers).
struct VpState {
    SeqInfo si;
};

// Signed 64-bit key of a race winner, ordered like (score, then lower index) under a signed
// max: the orderable image of the score in the high word, the complement of the index in the
// low word, the sign bit flipped so that signed order is unsigned order.  No winner: the
// smallest key.
__device__ __forceinline__ long long vp_key(float score, int idx) {
    if (idx == INT_MAX) return LLONG_MIN;
    const unsigned long long u = (static_cast<unsigned long long>(float_order(score)) << 32) |
                                 static_cast<uint32_t>(~static_cast<uint32_t>(idx));
    return static_cast<long long>(u ^ 0x8000000000000000ull);
}

__device__ __forceinline__ int vp_key_index(long long key) {
    return key == LLONG_MIN ? -1 : static_cast<int>(~static_cast<uint32_t>(static_cast<unsigned long long>(key)));
}

// One thread per row: fold the shard's piece partials (the streaming pass's output) into the
// row's (m, s), written as floats.
__global__ void __launch_bounds__(256) vp_fold_kernel(VerifyParams p, float2* out) {
    const int R = 2 * p.gamma + 1;
    const long long rows = static_cast<long long>(p.B) * R;
    for (long long r = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; r < rows;
         r += static_cast<long long>(gridDim.x) * blockDim.x) {
        const SoftmaxStat st = fold_row_stats(
            reinterpret_cast<const unsigned long long*>(p.stat_parts) + r * p.npieces, p.npieces);
        out[r] = make_float2(st.m, st.s);
    }
}

// One thread per (b, i): the target and draft logits at draft token d_i if this shard holds
// it, else -inf (a max over the ranks then gives the owner's values).
template <class ET>
__global__ void __launch_bounds__(256) vp_gather_kernel(VerifyParams p, int x_offset, float2* out) {
    using S = typename ET::storage;
    const long long n = static_cast<long long>(p.B) * p.gamma;
    for (long long k = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; k < n;
         k += static_cast<long long>(gridDim.x) * blockDim.x) {
        const long long b = k / p.gamma, i = k % p.gamma;
        const long long x = static_cast<long long>(p.tokens[k]) - x_offset;
        float2 v = make_float2(-INFINITY, -INFINITY);
        if (x >= 0 && x < p.V) {
            v.x = ET::load1(static_cast<const S*>(p.target) + (b * (p.gamma + 1) + i) * p.V + x);
            v.y = ET::load1(static_cast<const S*>(p.draft) + k * p.V + x);
        }
        out[k] = v;
    }
}

// One warp per sequence: merge each row's statistics over the W ranks in rank order, check
// the draft tokens against the whole vocabulary (p.V), decide the positions, write the
// accepted prefix and -1 padding, n_accepted, and the raced rows' statistics.
__global__ void __launch_bounds__(256) vp_decide_kernel(VerifyParams p, const float2* stats, int W,
                                                        const float2* gathered, VpState* state) {
    const int lane = threadIdx.x & 31;
    const int b = static_cast<int>((static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5);
    if (b >= p.B) return;
    const int g = p.gamma, R = 2 * g + 1;
    const float cp = scale_of(seq_T(p, b)), cq = scale_of(seq_Td(p, b));
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    const long long tok0 = static_cast<long long>(b) * g;
    auto row_stat = [&](int r, float& m, float& l2s) {
        SoftmaxStat st{-FLT_MAX, 0.0f};
        for (int w = 0; w < W; ++w) {
            const float2 v = stats[(static_cast<long long>(w) * p.B + b) * R + r];
            st = merge_stat(st, SoftmaxStat{v.x, v.y});
        }
        m = st.m;
        l2s = log2f(st.s);
    };
    bool bad = false;
    for (int i = lane; i < g; i += 32) {
        const int d = p.tokens[tok0 + i];
        bad |= (d < 0 || d >= p.V);
    }
    bad = __any_sync(0xffffffffu, bad);
    int j = g;
    for (int i0 = 0; i0 < g && !bad; i0 += 32) {
        const int i = i0 + lane;
        bool reject = false;
        if (i < g) {
            float mp, lp, mq, lq;
            row_stat(i, mp, lp);
            row_stat(g + 1 + i, mq, lq);
            const float2 x = gathered[tok0 + i];
            const float u = accept_uniform(p.key, bg, static_cast<uint32_t>(i));
            const float l2p = fmaf(x.x, cp, -mp) - lp;
            const float l2q = fmaf(x.y, cq, -mq) - lq;
            // accept iff u < min(1, p/q); p(d) = 0 rejects, q(d) = 0 < p(d) accepts
            reject = !((l2p > -INFINITY) && (u < exp2f(l2p - l2q)));
        }
        const unsigned rej = __ballot_sync(0xffffffffu, reject);
        if (rej) {
            j = i0 + __ffs(rej) - 1;
            break;
        }
    }
    if (bad) j = -1;
    int32_t* out = p.out_tokens + static_cast<long long>(b) * (g + 1);
    for (int t = lane; t <= g; t += 32)
        if (t != j) out[t] = (j >= 0 && t < j) ? p.tokens[tok0 + t] : -1;
    if (lane == 0) {
        p.out_n[b] = j;
        if (j < 0) set_status(p.status, 3 /* SPEC_EBADTOKEN */);
        SeqInfo si;
        si.j = j;
        si.cp = cp;
        si.cq = cq;
        si.mp = si.l2sp = si.mq = si.l2sq = 0.0f;
        if (j >= 0) row_stat(j, si.mp, si.l2sp);
        if (j >= 0 && j < g) row_stat(g + 1 + j, si.mq, si.l2sq);
        si.pad = 0;
        state[b].si = si;
    }
}

// One block per sequence: race the shard's columns of the raced row (global token index
// x_offset + x), 1024-token chunks over the block's warps.  A chunk whose residual weights are
// all zero also races p_j: if every rank's every chunk has none, those races together are the
// fallback race over p_j.  Writes the keys of the residual winner and of the fallback winner.
template <class ET>
__global__ void __launch_bounds__(256) vp_race_kernel(VerifyParams p, int x_offset, const VpState* state,
                                                      long long* out) {
    using S = typename ET::storage;
    __shared__ RaceState s_r[8], s_p[8];
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int b = blockIdx.x, g = p.gamma;
    const SeqInfo si = state[b].si;
    RaceState wr{-INFINITY, INT_MAX, -INFINITY}, wp{-INFINITY, INT_MAX, -INFINITY};
    if (si.j >= 0) {
        const bool residual = si.j < g;
        const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
        const S* rt = static_cast<const S*>(p.target) + (static_cast<long long>(b) * (g + 1) + si.j) * p.V;
        const S* rd = residual ? static_cast<const S*>(p.draft) + (static_cast<long long>(b) * g + si.j) * p.V
                               : nullptr;
        const int nchunks = (p.V + kRaceWarpTokens - 1) / kRaceWarpTokens;
        for (int c = wib; c < nchunks; c += 8) {
            const int xa = c * kRaceWarpTokens, xb = min(p.V, xa + kRaceWarpTokens);
            const RaceState r = race_warp_span<ET>(p, rt, rd, residual, bg, static_cast<uint32_t>(si.j),
                                                   xa, xb, si, lane, x_offset);
            wr = race_merge(wr, r);
            if (residual && r.idx == INT_MAX)
                wp = race_merge(wp, race_warp_span<ET>(p, rt, nullptr, false, bg, static_cast<uint32_t>(si.j),
                                                       xa, xb, si, lane, x_offset));
        }
    }
    if (lane == 0) {
        s_r[wib] = wr;
        s_p[wib] = wp;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        RaceState mr = s_r[0], mp = s_p[0];
        for (int k = 1; k < 8; ++k) {
            mr = race_merge(mr, s_r[k]);
            mp = race_merge(mp, s_p[k]);
        }
        out[2 * b] = vp_key(mr.best, mr.idx);
        out[2 * b + 1] = vp_key(mp.best, mp.idx);
    }
}

// One thread per sequence: the token from the reduced keys (the residual winner, else the
// fallback race over p_j).
__global__ void __launch_bounds__(256) vp_finish_kernel(int B, int gamma, const VpState* state,
                                                        const long long* keys, int32_t* out_tokens) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    const int j = state[b].si.j;
    if (j < 0) return;
    int y = vp_key_index(keys[2 * b]);
    if (y < 0) y = vp_key_index(keys[2 * b + 1]);
    out_tokens[static_cast<long long>(b) * (gamma + 1) + j] = y;
}

}  // namespace specverify
