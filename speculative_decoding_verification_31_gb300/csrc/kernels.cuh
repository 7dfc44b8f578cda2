// kernels.cuh -- the verify step's CUDA kernels (sm_103a).
//
// Sampling mode runs three kernels on the caller's stream:
//   row_stats   one pass over every target and draft logit: per (row, piece) partial
//               softmax statistics of p at T and q at T_d (max and sum of exponentials);
//   scan        one block per sequence: merge the partials into ln Z per row, gather
//               p_i(d_i) and q_i(d_i), draw u_i and find the first rejection j
//               ("How speculative decoding makes LLMs go brrr": pseudocode and module 3);
//   race        one pass over the one row each sequence still needs -- target and draft row
//               j for the residual max(0, p_j - q_j), or target row gamma for the bonus
//               token -- as an exponential race; the last warp to finish a sequence merges
//               the pieces and writes the token.
// Greedy mode runs row_argmax (first argmax per (row, piece)) and scan_greedy.
//
// Work is split into warp-sized items (one row piece each) taken round-robin by every warp
// of a grid sized to the GPU, so that no item ever waits for another.
#pragma once

#include <cfloat>
#include <climits>
#include <cstdint>

#include "device_common.cuh"
#include "philox.cuh"

namespace specverify {

// Per-sequence result of the scan, consumed by the race.
struct SeqInfo {
    int j;            // first rejected position (gamma: all accepted), -1: bad draft token
    float mp, l2sp;   // target row raced: scaled max and log2 of the sum
    float mq, l2sq;   // draft row j (residual only)
    float cp, cq;     // log2(e)/T_b, log2(e)/Td_b
};

struct RacePart {
    float best;
    int idx;
    float second;
    int pad;
};

struct VerifyParams {
    const void* target;         // [B, gamma+1, V]
    const void* draft;          // [B, gamma, V]
    const int32_t* tokens;      // [B, gamma]
    int B, gamma, V;
    int piece_len, npieces;     // elements per row piece, pieces per row
    float T, Td;                // scalar temperatures
    const float* T_seq;         // [B] or nullptr
    const float* Td_seq;        // [B] or nullptr
    PhiloxKey key;
    uint32_t seq_base;
    // workspace
    float2* stat_parts;         // [B][2*gamma+1][npieces] (m, s) or (value, index) in greedy
    SeqInfo* seq;               // [B]
    RacePart* race_parts;       // [B][npieces]
    int* tickets;               // [B] race arrival counters, zeroed by the scan
    int32_t* status;
    // outputs
    int32_t* out_tokens;        // [B, gamma+1]
    int32_t* out_n;             // [B]
    float* out_logp;
    float* out_logq;
    float* out_logZp;
    float* out_logZq;
    float* out_u;
    float* out_race;
};

__device__ __forceinline__ float seq_T(const VerifyParams& p, int b) {
    return p.T_seq ? p.T_seq[b] : p.T;
}
__device__ __forceinline__ float seq_Td(const VerifyParams& p, int b) {
    return p.Td_seq ? p.Td_seq[b] : p.Td;
}

// log2(e)/T, computed identically by every kernel that needs it.
__device__ __forceinline__ float scale_of(float T) { return kLog2e / T; }

// ----------------------------------------------------------------------------------------
// row_stats: partial (max, sum) of 2^(x*c - max) for one row piece per warp item.
// ----------------------------------------------------------------------------------------

__device__ __forceinline__ void stat_push1(SoftmaxStat& st, float x, float c) {
    const float mn = fmaxf(st.m, fmaxf(x * c, -FLT_MAX));
    st.s = st.s * ex2_fast(st.m - mn) + ex2_fast(fmaf(x, c, -mn));
    st.m = mn;
}

template <class ET, int U>
__device__ __forceinline__ SoftmaxStat stats_piece(const typename ET::storage* row, int x0, int x1,
                                                   float c, int lane) {
    SoftmaxStat st{-FLT_MAX, 0.0f};
    const RowSpan<ET> sp(row, x0, x1);
    if (lane < sp.head) stat_push1(st, ET::load1(sp.base + lane), c);
    const uint4* vp = sp.vec();
    for (int v0 = 0; v0 < sp.nvec; v0 += 32 * U) {
        uint4 raw[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int v = v0 + lane + 32 * k;
            raw[k] = v < sp.nvec ? ld_stream16(vp + v)
                                 : make_uint4(ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord,
                                              ET::kNegInfWord);
        }
        float f[U][ET::kVec];
#pragma unroll
        for (int k = 0; k < U; ++k) ET::widen(raw[k], f[k]);
        float bmax = f[0][0];
#pragma unroll
        for (int k = 0; k < U; ++k)
#pragma unroll
            for (int e = 0; e < ET::kVec; ++e) bmax = fmaxf(bmax, f[k][e]);
        const float mn = fmaxf(st.m, fmaxf(bmax * c, -FLT_MAX));
        float part[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            float t[ET::kVec];
#pragma unroll
            for (int e = 0; e < ET::kVec; ++e) t[e] = ex2_fast(fmaf(f[k][e], c, -mn));
#pragma unroll
            for (int w = ET::kVec / 2; w > 0; w >>= 1)
#pragma unroll
                for (int e = 0; e < w; ++e) t[e] += t[e + w];
            part[k] = t[0];
        }
#pragma unroll
        for (int w = U / 2; w > 0; w >>= 1)
#pragma unroll
            for (int k = 0; k < w; ++k) part[k] += part[k + w];
        st.s = st.s * ex2_fast(st.m - mn) + part[0];
        st.m = mn;
    }
    const int t0 = sp.head + sp.nvec * ET::kVec;
    if (lane < sp.tail) stat_push1(st, ET::load1(sp.base + t0 + lane), c);
    return warp_merge_stat(st);
}

template <class ET, int U>
__global__ void __launch_bounds__(256) row_stats_kernel(VerifyParams p) {
    using S = typename ET::storage;
    const int lane = threadIdx.x & 31;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int R = 2 * p.gamma + 1;
    const long long total = static_cast<long long>(p.B) * R * p.npieces;
    for (long long item = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         item < total; item += nwarps) {
        const int piece = static_cast<int>(item % p.npieces);
        const long long br = item / p.npieces;
        const int r = static_cast<int>(br % R);
        const int b = static_cast<int>(br / R);
        const S* row;
        float c;
        if (r <= p.gamma) {
            row = static_cast<const S*>(p.target) + (static_cast<long long>(b) * (p.gamma + 1) + r) * p.V;
            c = scale_of(seq_T(p, b));
        } else {
            row = static_cast<const S*>(p.draft) +
                  (static_cast<long long>(b) * p.gamma + (r - p.gamma - 1)) * p.V;
            c = scale_of(seq_Td(p, b));
        }
        const int x0 = piece * p.piece_len;
        const int x1 = min(p.V, x0 + p.piece_len);
        const SoftmaxStat st = stats_piece<ET, U>(row, x0, x1, c, lane);
        if (lane == 0) p.stat_parts[item] = make_float2(st.m, st.s);
    }
}

// ----------------------------------------------------------------------------------------
// row_argmax (greedy): first argmax of the raw logits per (target row, piece).
// ----------------------------------------------------------------------------------------

template <class ET, int U>
__device__ __forceinline__ ArgMax argmax_piece(const typename ET::storage* row, int x0, int x1,
                                               int lane) {
    ArgMax best{-INFINITY, INT_MAX};
    const RowSpan<ET> sp(row, x0, x1);
    if (lane < sp.head) {
        const ArgMax a{ET::load1(sp.base + lane), x0 + lane};
        if (argmax_better(a, best)) best = a;
    }
    const uint4* vp = sp.vec();
    const int xb = x0 + sp.head;
    for (int v0 = 0; v0 < sp.nvec; v0 += 32 * U) {
        uint4 raw[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int v = v0 + lane + 32 * k;
            raw[k] = v < sp.nvec ? ld_stream16(vp + v)
                                 : make_uint4(ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord,
                                              ET::kNegInfWord);
        }
        float f[U][ET::kVec];
#pragma unroll
        for (int k = 0; k < U; ++k) ET::widen(raw[k], f[k]);
        float bmax = f[0][0];
#pragma unroll
        for (int k = 0; k < U; ++k)
#pragma unroll
            for (int e = 0; e < ET::kVec; ++e) bmax = fmaxf(bmax, f[k][e]);
        if (bmax > best.v || best.i == INT_MAX) {
            // rare: locate the first element equal to the batch maximum (lowest index)
            int found = INT_MAX;
#pragma unroll
            for (int k = U - 1; k >= 0; --k) {
                const int v = v0 + lane + 32 * k;
#pragma unroll
                for (int e = ET::kVec - 1; e >= 0; --e)
                    if (v < sp.nvec && f[k][e] == bmax) found = xb + v * ET::kVec + e;
            }
            if (found != INT_MAX && (bmax > best.v || best.i == INT_MAX)) best = ArgMax{bmax, found};
        }
    }
    const int t0 = sp.head + sp.nvec * ET::kVec;
    if (lane < sp.tail) {
        const ArgMax a{ET::load1(sp.base + t0 + lane), x0 + t0 + lane};
        if (argmax_better(a, best)) best = a;
    }
    return warp_argmax(best);
}

template <class ET, int U>
__global__ void __launch_bounds__(256) row_argmax_kernel(VerifyParams p) {
    using S = typename ET::storage;
    const int lane = threadIdx.x & 31;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const int R = p.gamma + 1;
    const long long total = static_cast<long long>(p.B) * R * p.npieces;
    for (long long item = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         item < total; item += nwarps) {
        const int piece = static_cast<int>(item % p.npieces);
        const long long row_index = item / p.npieces;  // = b * (gamma+1) + i
        const S* row = static_cast<const S*>(p.target) + row_index * p.V;
        const int x0 = piece * p.piece_len;
        const int x1 = min(p.V, x0 + p.piece_len);
        const ArgMax a = argmax_piece<ET, U>(row, x0, x1, lane);
        if (lane == 0) p.stat_parts[item] = make_float2(a.v, __int_as_float(a.i));
    }
}

// ----------------------------------------------------------------------------------------
// scan: per sequence, ln Z of each row, p_i(d_i), q_i(d_i), u_i and the first rejection.
// ----------------------------------------------------------------------------------------

__device__ __forceinline__ void set_status(int32_t* status, int code) {
    atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

template <class ET>
__global__ void __launch_bounds__(256) scan_kernel(VerifyParams p) {
    using S = typename ET::storage;
    extern __shared__ float smem[];
    const int R = 2 * p.gamma + 1;
    float* sm_m = smem;        // [R] scaled max
    float* sm_l = smem + R;    // [R] log2 of the sum
    __shared__ int s_j, s_bad;
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) {
        s_j = p.gamma;
        s_bad = 0;
    }
    const float Tb = seq_T(p, b), Tdb = seq_Td(p, b);
    const float cp = scale_of(Tb), cq = scale_of(Tdb);
    for (int r = warp; r < R; r += nw) {
        SoftmaxStat st{-FLT_MAX, 0.0f};
        const float2* parts = p.stat_parts + (static_cast<long long>(b) * R + r) * p.npieces;
        for (int k = lane; k < p.npieces; k += 32) {
            const float2 q = parts[k];
            st = merge_stat(st, SoftmaxStat{q.x, q.y});
        }
        st = warp_merge_stat(st);
        if (lane == 0) {
            const float l2s = log2f(st.s);
            sm_m[r] = st.m;
            sm_l[r] = l2s;
            const float lz = (st.m + l2s) * kLn2;
            if (r <= p.gamma) {
                if (p.out_logZp) p.out_logZp[static_cast<long long>(b) * (p.gamma + 1) + r] = lz;
            } else if (p.out_logZq) {
                p.out_logZq[static_cast<long long>(b) * p.gamma + (r - p.gamma - 1)] = lz;
            }
        }
    }
    __syncthreads();
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    for (int i = threadIdx.x; i < p.gamma; i += blockDim.x) {
        const int d = p.tokens[static_cast<long long>(b) * p.gamma + i];
        const float u = accept_uniform(p.key, bg, static_cast<uint32_t>(i));
        const long long k = static_cast<long long>(b) * p.gamma + i;
        if (p.out_u) p.out_u[k] = u;
        if (d < 0 || d >= p.V) {
            s_bad = 1;
            if (p.out_logp) p.out_logp[k] = NAN;
            if (p.out_logq) p.out_logq[k] = NAN;
            continue;
        }
        const float xt = ET::load1(static_cast<const S*>(p.target) +
                                   (static_cast<long long>(b) * (p.gamma + 1) + i) * p.V + d);
        const float xd = ET::load1(static_cast<const S*>(p.draft) +
                                   (static_cast<long long>(b) * p.gamma + i) * p.V + d);
        const float l2p = fmaf(xt, cp, -sm_m[i]) - sm_l[i];
        const float l2q = fmaf(xd, cq, -sm_m[p.gamma + 1 + i]) - sm_l[p.gamma + 1 + i];
        if (p.out_logp) p.out_logp[k] = l2p * kLn2;
        if (p.out_logq) p.out_logq[k] = l2q * kLn2;
        // accept iff u < min(1, p/q); p(d) = 0 rejects, q(d) = 0 < p(d) accepts
        const bool accept = (l2p > -INFINITY) && (u < exp2f(l2p - l2q));
        if (!accept) atomicMin(&s_j, i);
    }
    __syncthreads();
    const int j = s_bad ? -1 : s_j;
    if (threadIdx.x == 0) {
        p.out_n[b] = j;
        SeqInfo si;
        si.j = j;
        si.cp = cp;
        si.cq = cq;
        const int rr = (j >= 0) ? j : 0;
        si.mp = sm_m[rr];
        si.l2sp = sm_l[rr];
        if (j >= 0 && j < p.gamma) {
            si.mq = sm_m[p.gamma + 1 + j];
            si.l2sq = sm_l[p.gamma + 1 + j];
        } else {
            si.mq = 0.0f;
            si.l2sq = 0.0f;
        }
        p.seq[b] = si;
        p.tickets[b] = 0;  // the race's per-sequence arrival counter starts from zero
        if (j < 0) set_status(p.status, 3 /* SPEC_EBADTOKEN */);
    }
    int32_t* out = p.out_tokens + static_cast<long long>(b) * (p.gamma + 1);
    for (int t = threadIdx.x; t <= p.gamma; t += blockDim.x)
        out[t] = (j >= 0 && t < j) ? p.tokens[static_cast<long long>(b) * p.gamma + t] : -1;
}

template <class ET>
__global__ void __launch_bounds__(256) scan_greedy_kernel(VerifyParams p) {
    extern __shared__ float smem[];
    int* sm_g = reinterpret_cast<int*>(smem);  // [gamma+1]
    __shared__ int s_j, s_bad;
    const int R = p.gamma + 1;
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    if (threadIdx.x == 0) {
        s_j = p.gamma;
        s_bad = 0;
    }
    for (int r = warp; r < R; r += nw) {
        ArgMax a{-INFINITY, INT_MAX};
        const float2* parts = p.stat_parts + (static_cast<long long>(b) * R + r) * p.npieces;
        for (int k = lane; k < p.npieces; k += 32) {
            const float2 q = parts[k];
            const ArgMax o{q.x, __float_as_int(q.y)};
            if (argmax_better(o, a)) a = o;
        }
        a = warp_argmax(a);
        if (lane == 0) sm_g[r] = a.i;
    }
    __syncthreads();
    for (int i = threadIdx.x; i < p.gamma; i += blockDim.x) {
        const int d = p.tokens[static_cast<long long>(b) * p.gamma + i];
        if (d < 0 || d >= p.V) {
            s_bad = 1;
            continue;
        }
        if (d != sm_g[i]) atomicMin(&s_j, i);
    }
    __syncthreads();
    const int j = s_bad ? -1 : s_j;
    if (threadIdx.x == 0) {
        p.out_n[b] = j;
        if (j < 0) set_status(p.status, 3 /* SPEC_EBADTOKEN */);
    }
    int32_t* out = p.out_tokens + static_cast<long long>(b) * (p.gamma + 1);
    for (int t = threadIdx.x; t <= p.gamma; t += blockDim.x) {
        int v = -1;
        if (j >= 0) {
            if (t < j) v = p.tokens[static_cast<long long>(b) * p.gamma + t];
            else if (t == j) v = sm_g[j];
        }
        out[t] = v;
    }
}

// ----------------------------------------------------------------------------------------
// race: exponential race over the residual row (or the bonus row) of each sequence.
// ----------------------------------------------------------------------------------------

struct RaceState {
    float best;
    int idx;
    float second;
};

// Offer token x (offered in increasing x by each lane): a strictly larger score wins, so
// an equal score keeps the lower x.
__device__ __forceinline__ void race_offer(RaceState& st, float score, int x) {
    if (score > st.best) {
        st.second = fmaxf(st.second, st.best);
        st.best = score;
        st.idx = x;
    } else {
        st.second = fmaxf(st.second, score);
    }
}

__device__ __forceinline__ RaceState race_merge(RaceState a, RaceState b) {
    const bool bw = b.best > a.best || (b.best == a.best && b.idx < a.idx);
    RaceState w = bw ? b : a, l = bw ? a : b;
    w.second = fmaxf(fmaxf(w.second, l.second), l.best);
    return w;
}

__device__ __forceinline__ RaceState warp_race_merge(RaceState s) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        RaceState o{__shfl_xor_sync(0xffffffffu, s.best, off), __shfl_xor_sync(0xffffffffu, s.idx, off),
                    __shfl_xor_sync(0xffffffffu, s.second, off)};
        s = race_merge(s, o);
    }
    return s;
}

// ln of the race weight of one token: ln p(x) for the bonus row, ln max(0, p - q) for the
// residual row (-inf when the weight is zero).  p and q are formed relative to each row's
// maximum, so the weights of likely tokens carry full fp32 precision.
__device__ __forceinline__ float race_log_weight(float xt, float xd, const SeqInfo& si, bool residual) {
    const float l2p = fmaf(xt, si.cp, -si.mp) - si.l2sp;
    if (!residual) return l2p > -INFINITY ? l2p * kLn2 : -INFINITY;
    const float l2q = fmaf(xd, si.cq, -si.mq) - si.l2sq;
    if (!(l2p > l2q)) return -INFINITY;
    // ln(p - q) = ln p + ln(1 - q/p) = ln p + ln(-expm1(ln q - ln p))
    return l2p * kLn2 + logf(-expm1f((l2q - l2p) * kLn2));
}

template <class ET>
__device__ __forceinline__ RaceState race_piece(const typename ET::storage* rt,
                                                const typename ET::storage* rd, int x0, int x1,
                                                const SeqInfo& si, bool residual, PhiloxKey key,
                                                uint32_t bg, uint32_t pos, int lane) {
    RaceState st{-INFINITY, INT_MAX, -INFINITY};
    const RowSpan<ET> sp(rt, x0, x1);
    // The vector path needs the residual's draft row to share the target row's alignment
    // and Philox blocks of four tokens to start on a vector boundary.
    const bool vec_ok =
        ((x0 + sp.head) & 3) == 0 &&
        (!residual || ((reinterpret_cast<uintptr_t>(rd + x0) & 15u) ==
                       (reinterpret_cast<uintptr_t>(rt + x0) & 15u)));
    auto scalar = [&](int x) {
        const float xt = ET::load1(rt + x);
        const float xd = residual ? ET::load1(rd + x) : 0.0f;
        const float lw = race_log_weight(xt, xd, si, residual);
        if (lw > -INFINITY) {
            const uint4 blk = race_block(key, bg, pos, static_cast<uint32_t>(x) >> 2);
            race_offer(st, lw - race_log_exponential(word_of(blk, static_cast<uint32_t>(x) & 3u)), x);
        }
    };
    if (!vec_ok) {
        for (int x = x0 + lane; x < x1; x += 32) scalar(x);  // (lane order is still increasing)
        return warp_race_merge(st);
    }
    if (lane < sp.head) scalar(x0 + lane);
    const int xb = x0 + sp.head;
    const uint4* vt = sp.vec();
    const uint4* vd = residual ? reinterpret_cast<const uint4*>(rd + xb) : nullptr;
    for (int v = lane; v < sp.nvec; v += 32) {
        float ft[ET::kVec], fd[ET::kVec];
        ET::widen(__ldg(vt + v), ft);
        if (residual) ET::widen(__ldg(vd + v), fd);
        const int xv = xb + v * ET::kVec;
#pragma unroll
        for (int g = 0; g < ET::kVec / 4; ++g) {
            float lw[4];
            bool any = false;
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                lw[e] = race_log_weight(ft[4 * g + e], residual ? fd[4 * g + e] : 0.0f, si, residual);
                any |= lw[e] > -INFINITY;
            }
            if (any) {
                const uint4 blk = race_block(key, bg, pos, static_cast<uint32_t>(xv + 4 * g) >> 2);
                const uint32_t w4[4] = {blk.x, blk.y, blk.z, blk.w};
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    if (lw[e] > -INFINITY)
                        race_offer(st, lw[e] - race_log_exponential(w4[e]), xv + 4 * g + e);
            }
        }
    }
    const int t0 = sp.head + sp.nvec * ET::kVec;
    if (lane < sp.tail) scalar(x0 + t0 + lane);
    return warp_race_merge(st);
}

template <class ET>
__global__ void __launch_bounds__(256) race_kernel(VerifyParams p) {
    using S = typename ET::storage;
    const int lane = threadIdx.x & 31;
    const long long nwarps = (static_cast<long long>(gridDim.x) * blockDim.x) >> 5;
    const long long total = static_cast<long long>(p.B) * p.npieces;
    for (long long item = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
         item < total; item += nwarps) {
        const int b = static_cast<int>(item / p.npieces);
        const int piece = static_cast<int>(item % p.npieces);
        const SeqInfo si = p.seq[b];
        if (si.j < 0) continue;  // bad draft token: nothing to draw
        const bool residual = si.j < p.gamma;
        const S* rt = static_cast<const S*>(p.target) + (static_cast<long long>(b) * (p.gamma + 1) + si.j) * p.V;
        const S* rd = residual ? static_cast<const S*>(p.draft) + (static_cast<long long>(b) * p.gamma + si.j) * p.V
                               : nullptr;
        const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
        const int x0 = piece * p.piece_len;
        const int x1 = min(p.V, x0 + p.piece_len);
        const RaceState st = race_piece<ET>(rt, rd, x0, x1, si, residual, p.key, bg,
                                            static_cast<uint32_t>(si.j), lane);
        if (lane == 0) {
            p.race_parts[item] = RacePart{st.best, st.idx, st.second, 0};
            __threadfence();
        }
        int ticket = 0;
        if (lane == 0) ticket = atomicAdd(p.tickets + b, 1);
        ticket = __shfl_sync(0xffffffffu, ticket, 0);
        if (ticket != p.npieces - 1) continue;
        // Last piece of this sequence: merge every piece's winner (read through L2).
        __threadfence();
        RaceState m{-INFINITY, INT_MAX, -INFINITY};
        for (int k = lane; k < p.npieces; k += 32) {
            const RacePart* rp = p.race_parts + static_cast<long long>(b) * p.npieces + k;
            const float4 raw = __ldcg(reinterpret_cast<const float4*>(rp));
            m = race_merge(m, RaceState{raw.x, __float_as_int(raw.y), raw.z});
        }
        m = warp_race_merge(m);
        if (m.idx == INT_MAX) {
            // Every residual weight was zero (p <= q everywhere in fp32): draw from p_j.
            m = race_piece<ET>(rt, nullptr, 0, p.V, si, false, p.key, bg,
                               static_cast<uint32_t>(si.j), lane);
        }
        if (lane == 0) {
            p.out_tokens[static_cast<long long>(b) * (p.gamma + 1) + si.j] = m.idx;
            if (p.out_race) {
                p.out_race[2 * b] = m.best;
                p.out_race[2 * b + 1] = m.second;
            }
        }
    }
}

}  // namespace specverify
