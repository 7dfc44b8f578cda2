// kernels.cuh -- the verify step's CUDA kernels (sm_103a).
//
// Sampling mode, default schedule: two kernels on the caller's stream.
//   row_stats   one pass over every target and draft logit: per (row, piece) partial
//               softmax statistics of p at T and q at T_d (max and sum of exponentials);
//   scan_race   G blocks per sequence: merge the partials into ln Z per row, gather
//               p_i(d_i) and q_i(d_i), draw u_i and find the first rejection j
//               ("How speculative decoding makes LLMs go brrr": pseudocode and module 3),
//               then race the one row each sequence still needs -- target and draft row j
//               for the residual max(0, p_j - q_j), or target row gamma for the bonus token
//               -- as an exponential race; the last block of a sequence merges the winners
//               and writes the token.
// Other schedules of the same computation: the early-exit kernel (below: reads rows only up
// to each sequence's first rejection), pair_stats (the streaming pass with per-position
// entropies and KL), and the token-tree kernels.
// Greedy mode runs row_argmax (first argmax per (row, piece)) and scan_greedy.
//
// Streaming work is split into warp-sized items (one row piece each); each SM's block takes a
// contiguous share and its warps claim the items one at a time (for_block_items), so that no
// item ever waits for another and the warps of an SM finish together.
#pragma once

#include <cfloat>
#include <climits>
#include <cstdint>

#include <cooperative_groups.h>

#include "device_common.cuh"
#include "philox.cuh"

namespace specverify {

// Per-sequence result of the scan, consumed by the race.
struct __align__(16) SeqInfo {
    int j;            // first rejected position (gamma: all accepted), -1: bad draft token
    float mp, l2sp;   // target row raced: scaled max and log2 of the sum
    float mq, l2sq;   // draft row j (residual only)
    float cp, cq;     // log2(e)/T_b, log2(e)/Td_b
    int pad;
};

struct RacePart {
    float best;
    int idx;
    float second;
    int pad;
};

// Element counts of the buffers a call's kernels index, for the index-checked build
// (SPECVERIFY_CHECKED): the caller's tensors and the workspace regions.
struct BufferCaps {
    long long target, draft, tokens, out_tokens;  // caller tensors
    long long stat;                               // stat_parts (float2)
    long long race;                               // race_parts (RacePart)
    long long row_stat, pos, rowarr, task, race_task, early_race;  // early-exit regions
};

struct VerifyParams {
    const void* target;         // [B, gamma+1, V]
    const void* draft;          // [B, gamma, V]
    const int32_t* tokens;      // [B, gamma]
    int B, gamma, V;
    int piece_len, npieces;     // elements per row piece, pieces per row (streaming pass)
    int rpieces;                // race pieces of kRaceBlockTokens per row (partial-slot sizing)
    int rgroups;                // scan-race blocks per sequence (each races rpieces / rgroups pieces)
    float T, Td;                // scalar temperatures
    const float* T_seq;         // [B] or nullptr
    const float* Td_seq;        // [B] or nullptr
    PhiloxKey key;
    PhiloxRoundKeys rk;         // round keys of `key`
    uint32_t seq_base;
    // workspace
    float2* stat_parts;         // [B][2*gamma+1][npieces] (m, s) or (value, index) in greedy
    SeqInfo* seq;               // [B]
    RacePart* race_parts;       // [B][rpieces]
    int* tickets;               // [B] race arrival counters, zeroed by the scan
    int32_t* status;
    float2* row_stat;           // [B][2*gamma+1] merged (scaled max, log2 sum) per row (early exit)
    uint32_t debug_flags;       // kDebug* test switches
    // early-exit path (verify_early_kernel): task queue and its counters
    int* task;                  // [task_cap] appended task descriptors (pre-filled kTaskEmpty)
    int task_cap;
    int n_init;                 // implicit initial tasks (position 0 rows, or bonus rows)
    int* task_tail;             // slots of `task` reserved so far
    unsigned long long* unit_cursor;  // units claimed so far
    int* row_arrivals;          // [B][R] pieces of each row finished
    int* pos_done;              // [B][gamma+1] completion events of each position
    int* enq_pos;               // [B] last position whose rows are queued, minus early_L0
    int early_L0;               // positions 0..early_L0 of every sequence are queued at the start
    int early_fill;             // positions in flight that keep the row warps busy
    int early_growth;           // extra positions queued ahead after an accepted position i: (i+1)*g/4
    int* race_done;             // [B] race units finished
    int* seq_decided;           // sequences whose first rejection (or bonus) is known
    int* seq_finished;          // sequences finished (token written)
    int* race_task;             // [B] race queue: sequence indices (pre-filled kTaskEmpty)
    int* race_tail;             // slots of race_task reserved so far
    unsigned long long* race_unit_cursor;  // race units claimed so far
    unsigned long long* early_race;  // [B][npieces] packed (score, index + 1) race winners
    void* mirror_target;        // early exit over host memory: device copies of the rows streamed,
    void* mirror_draft;         // laid out like the inputs (the race reads them there); or nullptr
    // outputs
    int32_t* out_tokens;        // [B, gamma+1]
    int32_t* out_n;             // [B]
    float* out_logp;
    float* out_logq;
    float* out_logZp;
    float* out_logZq;
    float* out_u;
    float* out_race;
    // per-position statistics (pair_stats / position_stats)
    float2* ext_parts;          // [B][2*gamma+1][npieces] entropy and cross terms per piece
    float* out_Hp;              // [B, gamma+1] entropy of p_i (nats), or nullptr
    float* out_Hq;              // [B, gamma]   entropy of q_i (nats), or nullptr
    float* out_KL;              // [B, gamma]   KL(p_i || q_i) (nats), or nullptr
    double* ctrl_centres;       // [B, 2] entropy class centres updated in place, or nullptr
    double ctrl_beta;
    // token-tree verify
    int32_t* out_nodes;         // [B, depth] accepted nodes, or nullptr
    struct TreeRace* tree_race; // [B] the node each sequence races
    BufferCaps caps;            // buffer sizes (checked by the index-checked build only)
};

// The index-checked build (compiled with SPECVERIFY_CHECKED): before an access through a
// computed index, sv_in_range(p, i, n) tests 0 <= i < n for the buffer's n elements; on
// failure it records SPEC_EINDEX (7) in the status word (the first error recorded stays) and
// the caller skips the access -- no trap, no assert, so the context stays usable.  In the
// normal build the test is the constant true and compiles away.
__device__ __forceinline__ bool sv_in_range(const VerifyParams& p, long long i, long long n) {
#ifdef SPECVERIFY_CHECKED
    if (i >= 0 && i < n) return true;
    atomicCAS(reinterpret_cast<int*>(p.status), 0, 7 /* SPEC_EINDEX */);
    return false;
#else
    (void)p; (void)i; (void)n;
    return true;
#endif
}

// Whether the elements [first, first + count) lie in a buffer of n elements (count >= 0).
__device__ __forceinline__ bool sv_span_in_range(const VerifyParams& p, long long first, long long count,
                                                 long long n) {
    return count <= 0 || (sv_in_range(p, first, n) && sv_in_range(p, first + count - 1, n));
}

// Race partial slots per sequence: at most one per block racing it.  A block of the
// scan-race grid takes at least one step of chunks, so a sequence meets at most
// ceil(V / kRaceBlockTokens) + 1 blocks; the tree and LM-head races use at most rpieces.
__host__ __device__ __forceinline__ int race_slots(int rpieces) { return rpieces + 1; }

// Row pieces of the streaming passes: between kMinPieceBytes and kMaxPieceBytes of logits
// (the early-exit path: kEarlyPieceBytes up to twice that, by the call's size).
#ifndef SPECVERIFY_PIECE_BYTES
#define SPECVERIFY_PIECE_BYTES 16384
#endif
constexpr int kPieceBytes = SPECVERIFY_PIECE_BYTES;  // default (no grid given)
constexpr int kMinPieceBytes = 8192;
constexpr int kMaxPieceBytes = 20480;  // larger pieces measured slower on the throughput workload
#ifndef SPECVERIFY_EARLY_PIECE_BYTES
#define SPECVERIFY_EARLY_PIECE_BYTES 8192
#endif
constexpr int kEarlyPieceBytes = SPECVERIFY_EARLY_PIECE_BYTES;
static_assert(kEarlyPieceBytes >= kMinPieceBytes, "the workspace holds rows of kMinPieceBytes pieces");

// Elements per piece for `rows` rows of V elements of es bytes streamed by `warps` warps.
// The pass takes about ceil(items / warps) item times (every warp takes about the same
// number of items), an item costing its piece plus a fixed overhead (the warp's reduction
// and partial store and the next item's first loads, about kItemOverheadBytes of
// streaming); the piece with the most useful bytes per unit of that time wins, the larger
// one on near-equal scores.  warps = 0: the default size.
constexpr float kItemOverheadBytes = 2048.0f;

inline int pick_piece_len(long long rows, int V, int es, long long warps) {
    int best_len = kPieceBytes / es;
    if (warps > 0) {
        const float fw = static_cast<float>(warps);
        const float work = static_cast<float>(rows) * static_cast<float>(V) * static_cast<float>(es);
        float best_eff = -1.0f;
        for (int bytes = kMaxPieceBytes; bytes >= kMinPieceBytes; bytes -= 1024) {
            const int l = bytes / es;
            const float items = static_cast<float>(rows) * static_cast<float>((V + l - 1) / l);
            const float eff = work / (ceilf(items / fw) * fw * (static_cast<float>(bytes) + kItemOverheadBytes));
            if (eff > best_eff + 0.005f) {
                best_eff = eff;
                best_len = l;
            }
        }
    }
    return best_len;
}

// (m, s) pairs travel as one naturally aligned 64-bit word, so a reader that polls the word
// sees both halves or neither and the writer needs no memory fence.  The early-exit path
// pre-fills them with kStatEmpty (two NaN halves; a real pair has s >= 1, or m = -FLT_MAX
// when every logit of the piece is -inf).
constexpr unsigned long long kStatEmpty = 0xFFFFFFFFFFFFFFFFull;

__device__ __forceinline__ void store_stat(float2* dst, float m, float s) {
    const unsigned long long v = (static_cast<unsigned long long>(__float_as_uint(s)) << 32) |
                                 __float_as_uint(m);
    *reinterpret_cast<unsigned long long*>(dst) = v;
}

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
    st.s = fmaf(st.s, ex2_fast(st.m - mn), ex2_fast(fmaf(x, c, -mn)));
    st.m = mn;
}

// Partial statistics of row[x0, x1) by one warp: 16-byte vectors L per lane in flight, taken
// U at a time (one running-max update per U vectors per lane).  The arithmetic depends on U
// only: any L (a multiple of U) gives the same bits; an all-padding batch changes nothing.
template <class ET, int U, int L = U, bool kMirror = false>
__device__ __forceinline__ SoftmaxStat stats_piece(const typename ET::storage* row, int x0, int x1,
                                                   float c, int lane,
                                                   typename ET::storage* mirror = nullptr) {
    static_assert(L % U == 0, "loads in flight must be whole batches");
    SoftmaxStat st{-FLT_MAX, 0.0f};
    const RowSpan<ET> sp(row, x0, x1);
    // kMirror: every element read is also written to the same place of the row `mirror`
    // (a device row with the same alignment as `row`)
    typename ET::storage* mb = kMirror ? mirror + x0 : nullptr;
    if (lane < sp.head) {
        if (kMirror) mb[lane] = sp.base[lane];
        stat_push1(st, ET::load1(sp.base + lane), c);
    }
    const uint4* vp = sp.vec();
    uint4* mv = kMirror ? reinterpret_cast<uint4*>(mb + sp.head) : nullptr;
    for (int v0 = 0; v0 < sp.nvec; v0 += 32 * L) {
        uint4 raw[L];
#pragma unroll
        for (int k = 0; k < L; ++k) {
            const int v = v0 + lane + 32 * k;
            raw[k] = v < sp.nvec ? ld_stream16(vp + v)
                                 : make_uint4(ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord,
                                              ET::kNegInfWord);
        }
        if (kMirror) {
#pragma unroll
            for (int k = 0; k < L; ++k) {
                const int v = v0 + lane + 32 * k;
                if (v < sp.nvec) mv[v] = raw[k];
            }
        }
#pragma unroll
        for (int h = 0; h < L / U; ++h) {
            float f[U][ET::kVec];
#pragma unroll
            for (int k = 0; k < U; ++k) ET::widen(raw[h * U + k], f[k]);
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
            st.s = fmaf(st.s, ex2_fast(st.m - mn), part[0]);
            st.m = mn;
        }
    }
    const int t0 = sp.head + sp.nvec * ET::kVec;
    if (lane < sp.tail) {
        if (kMirror) mb[t0 + lane] = sp.base[t0 + lane];
        stat_push1(st, ET::load1(sp.base + t0 + lane), c);
    }
    return warp_merge_stat(st);
}

// Row r of sequence b: target row r (r <= gamma, scale log2(e)/T_b) or draft row
// r - gamma - 1 (scale log2(e)/Td_b).  Writes the piece's partial statistics.
template <class ET, int U, int L = U>
__device__ __forceinline__ void row_stats_item(const VerifyParams& p, int b, int r, int piece,
                                               int lane) {
    using S = typename ET::storage;
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
    const int R = 2 * p.gamma + 1;
#ifdef SPECVERIFY_CHECKED
    {
        const bool tgt = r <= p.gamma;
        const long long off = tgt ? (static_cast<long long>(b) * (p.gamma + 1) + r) * p.V
                                  : (static_cast<long long>(b) * p.gamma + (r - p.gamma - 1)) * p.V;
        if (!(sv_span_in_range(p, off + x0, x1 - x0, tgt ? p.caps.target : p.caps.draft) &&
              sv_in_range(p, (static_cast<long long>(b) * R + r) * p.npieces + piece, p.caps.stat)))
            return;
    }
#endif
    const SoftmaxStat st = stats_piece<ET, U, L>(row, x0, x1, c, lane);
    if (lane == 0)  // one aligned 64-bit store: readers see both halves or neither
        store_stat(p.stat_parts + (static_cast<long long>(b) * R + r) * p.npieces + piece, st.m, st.s);
}

// The streaming passes (row_stats, pair_stats, row_argmax, tree_stats) run one block of
// kStreamThreads per SM.  Their items (one row piece per warp) are split into contiguous
// equal ranges, one per block, and the warps of a block claim the block's items one at a time
// from a shared counter, so the warps of an SM finish together.  (Dealt round-robin to the
// warps of three 256-thread blocks per SM, the same items ended over a 33 us window on the
// throughput workload: the blocks of one SM were not served alike, the last-placed block
// ending 16 us after the first.)
#ifndef SPECVERIFY_STREAM_THREADS
#define SPECVERIFY_STREAM_THREADS 768
#endif
#ifndef SPECVERIFY_STATS_MINBLOCKS
#define SPECVERIFY_STATS_MINBLOCKS 1
#endif
constexpr int kStreamThreads = SPECVERIFY_STREAM_THREADS;

// The streaming kernels are launched as programmatic dependents of whatever kernel precedes
// them on the stream: wait for it (and its memory) before the first access.
__device__ __forceinline__ void stream_pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Items [0, total) of a streaming pass, one item per warp at a time: with kClaim, this block's
// range, claimed by its warps from a shared counter (every thread of the block must call
// it); without, the item whose index is the global warp index (the launch shape of small
// calls, a warp for every item).
template <bool kClaim, class F>
__device__ __forceinline__ void for_block_items(long long total, F&& f) {
    if (!kClaim) {
        const long long item = (static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x) >> 5;
        if (item < total) f(item);
        return;
    }
    __shared__ int s_next;
    if (threadIdx.x == 0) s_next = 0;
    __syncthreads();
    const long long i0 = static_cast<long long>(blockIdx.x) * total / gridDim.x;
    const long long i1 = (static_cast<long long>(blockIdx.x) + 1) * total / gridDim.x;
    const int lane = threadIdx.x & 31;
    for (;;) {
        int k = 0;
        if (lane == 0) k = atomicAdd(&s_next, 1);
        const long long item = i0 + __shfl_sync(0xffffffffu, k, 0);
        if (item >= i1) break;
        f(item);
    }
}

// Also empties the race partials and arrival counters the scan-race kernel uses, and lets
// that kernel (launched as a programmatic dependent) start as soon as blocks retire.
template <class ET, int U, bool kClaim>
__global__ void __launch_bounds__(kStreamThreads, SPECVERIFY_STATS_MINBLOCKS) row_stats_kernel(VerifyParams p) {
    stream_pdl_wait();
    const int lane = threadIdx.x & 31;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (long long k = tid; k < static_cast<long long>(p.B) * race_slots(p.rpieces); k += nthreads)
        reinterpret_cast<uint4*>(p.race_parts)[k] = make_uint4(0u, 0u, 0u, 0u);
    for (long long k = tid; k < p.B; k += nthreads) p.tickets[k] = 0;
    const int R = 2 * p.gamma + 1;
    for_block_items<kClaim>(static_cast<long long>(p.B) * R * p.npieces, [&](long long item) {
        const int piece = static_cast<int>(item % p.npieces);
        const long long br = item / p.npieces;
        row_stats_item<ET, U>(p, static_cast<int>(br / R), static_cast<int>(br % R), piece, lane);
    });
    asm volatile("griddepcontrol.launch_dependents;");
}

// ----------------------------------------------------------------------------------------
// Per-position entropies and KL divergence, and the entropy class centres
// ("投机解码的第二本账" (SparseSpec-L), section 3.3: every draft token's entropy H_i; class
// centres of the entropies of accepted and rejected tokens kept as moving averages.  KL is
// the draft-target divergence quoted by "SubSpec: the target model's own low-bit shadow as
// the draft model").
//
// pair_stats replaces row_stats when these are asked for: one item is a piece of target
// row i together with the same piece of draft row i (target row gamma alone), so the same
// bytes are read once.  Besides each row's (max m, sum s) partial -- written exactly as
// row_stats writes it, so the scan and race read it unchanged -- a lane keeps, in base 2
// with t = x c - m,
//     A = sum 2^t t            (entropy: H = ln 2 (log2 s - A / s))
//     C = sum 2^tp tq          (p-weighted draft log-weights, relative to the draft max)
// so that KL(p || q) = ln 2 (A_p / s_p - log2 s_p - C / s_p + log2 s_q).  A change of a max
// from m to m' (delta = m - m') rescales A to 2^delta (A + s delta), and C to
// 2^delta_p (C + s_p delta_q).  A term whose weight 2^t is 0 contributes nothing (no 0 * inf).
// ----------------------------------------------------------------------------------------

struct PairStat {
    float mp, sp, ap, c;  // target row: max, sum, entropy term, cross term
    float mq, sq, aq;     // draft row
};

__device__ __forceinline__ void pair_rescale(float& m, float& s, float& a, float mn) {
    const float d = m - mn;  // <= 0
    const float f = ex2_fast(d);
    a = f * fmaf(s, d, a);
    s *= f;
    m = mn;
}

__device__ __forceinline__ PairStat pair_merge(PairStat x, PairStat y) {
    PairStat r;
    const float Mp = fmaxf(x.mp, y.mp), Mq = fmaxf(x.mq, y.mq);
    const float dxp = x.mp - Mp, dyp = y.mp - Mp, dxq = x.mq - Mq, dyq = y.mq - Mq;
    const float fxp = ex2_fast(dxp), fyp = ex2_fast(dyp), fxq = ex2_fast(dxq), fyq = ex2_fast(dyq);
    r.mp = Mp;
    r.mq = Mq;
    r.sp = x.sp * fxp + y.sp * fyp;
    r.ap = fxp * fmaf(x.sp, dxp, x.ap) + fyp * fmaf(y.sp, dyp, y.ap);
    r.c = fxp * fmaf(x.sp, dxq, x.c) + fyp * fmaf(y.sp, dyq, y.c);
    r.sq = x.sq * fxq + y.sq * fyq;
    r.aq = fxq * fmaf(x.sq, dxq, x.aq) + fyq * fmaf(y.sq, dyq, y.aq);
    return r;
}

__device__ __forceinline__ PairStat warp_pair_merge(PairStat v) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        PairStat o;
        o.mp = __shfl_xor_sync(0xffffffffu, v.mp, off);
        o.sp = __shfl_xor_sync(0xffffffffu, v.sp, off);
        o.ap = __shfl_xor_sync(0xffffffffu, v.ap, off);
        o.c = __shfl_xor_sync(0xffffffffu, v.c, off);
        o.mq = __shfl_xor_sync(0xffffffffu, v.mq, off);
        o.sq = __shfl_xor_sync(0xffffffffu, v.sq, off);
        o.aq = __shfl_xor_sync(0xffffffffu, v.aq, off);
        v = pair_merge(v, o);
    }
    return v;
}

// Exponents below this are clamped in the extra terms: a weight 2^t is then 0 and 0 times
// the clamp is 0, with no branch; a draft exponent at the clamp under a positive target
// weight (q(x) = 0 < p(x)) drives C below kKlInfinite, which position_stats reports as an
// infinite KL.  Exponents of real logits are far above both (|t| < 2^16 for |x c| < 2^15).
constexpr float kTermClamp = -1e30f;
constexpr float kKlInfinite = -1e20f;

// One element pair (target logit xp, draft logit xq; has_q: the position has a draft row).
__device__ __forceinline__ void pair_push(PairStat& st, float xp, float xq, float cp, float cq,
                                          bool has_q) {
    const float tp = fmaxf(fmaf(xp, cp, -st.mp), kTermClamp), ep = ex2_fast(tp);
    st.sp += ep;
    st.ap = fmaf(ep, tp, st.ap);
    if (has_q) {
        const float tq = fmaxf(fmaf(xq, cq, -st.mq), kTermClamp), eq = ex2_fast(tq);
        st.sq += eq;
        st.aq = fmaf(eq, tq, st.aq);
        st.c = fmaf(ep, tq, st.c);
    }
}

// Partial statistics of elements [x0, x1) of target row i and (has_q) draft row i, whose
// starts have the same alignment (both rows are V elements apart from their tensor's base,
// and both bases are 16-byte aligned).
template <class ET, int U>
__device__ __forceinline__ PairStat pair_piece(const typename ET::storage* rp,
                                               const typename ET::storage* rq, bool has_q,
                                               int x0, int x1, float cp, float cq, int lane) {
    PairStat st{-FLT_MAX, 0.0f, 0.0f, 0.0f, -FLT_MAX, 0.0f, 0.0f};
    const RowSpan<ET> sp(rp, x0, x1);
    const RowSpan<ET> sq(has_q ? rq : rp, x0, x1);
    const bool same = sp.head == sq.head;  // equal alignment: vectors pair up
    // raise the maxima to (mp, mq): C is shifted with the draft max, then rescaled with the
    // target weights
    auto raise = [&](float mp, float mq) {
        st.c = fmaf(st.sp, st.mq - mq, st.c);
        pair_rescale(st.mq, st.sq, st.aq, mq);
        const float d = st.mp - mp, f = ex2_fast(d);
        st.ap = f * fmaf(st.sp, d, st.ap);
        st.c *= f;
        st.sp *= f;
        st.mp = mp;
    };
    auto push_scalar = [&](int x) {
        const float xp = ET::load1(rp + x);
        const float xq = has_q ? ET::load1(rq + x) : -INFINITY;
        raise(fmaxf(st.mp, fmaxf(xp * cp, -FLT_MAX)), fmaxf(st.mq, fmaxf(xq * cq, -FLT_MAX)));
        pair_push(st, xp, xq, cp, cq, has_q);
    };
    if (!same) {  // unaligned pair (only when a caller's draft base breaks the rule): scalar
        for (int x = x0 + lane; x < x1; x += 32) push_scalar(x);
        return warp_pair_merge(st);
    }
    if (lane < sp.head) push_scalar(x0 + lane);
    const uint4* vp = sp.vec();
    const uint4* vq = sq.vec();
    for (int v0 = 0; v0 < sp.nvec; v0 += 32 * U) {
        uint4 rawp[U], rawq[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int v = v0 + lane + 32 * k;
            const uint4 ninf = make_uint4(ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord);
            rawp[k] = v < sp.nvec ? ld_stream16(vp + v) : ninf;
            rawq[k] = (has_q && v < sp.nvec) ? ld_stream16(vq + v) : ninf;
        }
        float bp = -INFINITY, bq = -INFINITY;
#pragma unroll
        for (int k = 0; k < U; ++k) {
            bp = fmaxf(bp, ET::vmax(rawp[k]));
            bq = fmaxf(bq, ET::vmax(rawq[k]));
        }
        raise(fmaxf(st.mp, fmaxf(bp * cp, -FLT_MAX)), fmaxf(st.mq, fmaxf(bq * cq, -FLT_MAX)));
#pragma unroll
        for (int k = 0; k < U; ++k) {
            float f[ET::kVec], g[ET::kVec];
            ET::widen(rawp[k], f);
            ET::widen(rawq[k], g);
#pragma unroll
            for (int e = 0; e < ET::kVec; ++e) pair_push(st, f[e], g[e], cp, cq, has_q);
        }
    }
    const int t0 = sp.head + sp.nvec * ET::kVec;
    if (lane < sp.tail) push_scalar(x0 + t0 + lane);
    return warp_pair_merge(st);
}

// pair_stats: row_stats with the extra terms (see above).  Item (b, i, piece), i <= gamma.
#ifndef SPECVERIFY_PAIR_MINBLOCKS
#define SPECVERIFY_PAIR_MINBLOCKS 1
#endif
template <class ET, int U, bool kClaim>
__global__ void __launch_bounds__(kStreamThreads, SPECVERIFY_PAIR_MINBLOCKS) pair_stats_kernel(VerifyParams p) {
    stream_pdl_wait();
    using S = typename ET::storage;
    const int lane = threadIdx.x & 31;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (long long k = tid; k < static_cast<long long>(p.B) * race_slots(p.rpieces); k += nthreads)
        reinterpret_cast<uint4*>(p.race_parts)[k] = make_uint4(0u, 0u, 0u, 0u);
    for (long long k = tid; k < p.B; k += nthreads) p.tickets[k] = 0;
    const int R = 2 * p.gamma + 1;
    for_block_items<kClaim>(static_cast<long long>(p.B) * (p.gamma + 1) * p.npieces, [&](long long item) {
        const int piece = static_cast<int>(item % p.npieces);
        const long long bi = item / p.npieces;
        const int b = static_cast<int>(bi / (p.gamma + 1)), i = static_cast<int>(bi % (p.gamma + 1));
        const bool has_q = i < p.gamma;
        const S* rp = static_cast<const S*>(p.target) + (static_cast<long long>(b) * (p.gamma + 1) + i) * p.V;
        const S* rq = has_q ? static_cast<const S*>(p.draft) + (static_cast<long long>(b) * p.gamma + i) * p.V
                            : rp;
        const int x0 = piece * p.piece_len;
        const PairStat st = pair_piece<ET, U>(rp, rq, has_q, x0, min(p.V, x0 + p.piece_len),
                                              scale_of(seq_T(p, b)), scale_of(seq_Td(p, b)), lane);
        if (lane == 0) {
            const long long kp = (static_cast<long long>(b) * R + i) * p.npieces + piece;
            store_stat(p.stat_parts + kp, st.mp, st.sp);
            p.ext_parts[kp] = make_float2(st.ap, st.c);
            if (has_q) {
                const long long kq = (static_cast<long long>(b) * R + p.gamma + 1 + i) * p.npieces + piece;
                store_stat(p.stat_parts + kq, st.mq, st.sq);
                p.ext_parts[kq] = make_float2(st.aq, 0.0f);
            }
        }
    });
    asm volatile("griddepcontrol.launch_dependents;");
}

// position_stats: one block per sequence merges the pieces of every position into H(p_i),
// H(q_i) and KL(p_i || q_i); then, given class centres, moves them with this verify's
// outcome (positions before the first rejection j update the accepted centre, position j
// the rejected one, in position order; c <- (1 - beta) c + beta H(q_i), in fp64 with every
// operation rounded on its own).  Runs after the scan, whose accepted counts it reads.
__global__ void __launch_bounds__(256) position_stats_kernel(VerifyParams p) {
    extern __shared__ float s_hq[];  // [gamma]
    // a programmatic dependent of the scan-race kernel (or of pair_stats): wait for it
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");  // (see scan_greedy_kernel)
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int b = blockIdx.x;
    const int R = 2 * p.gamma + 1;
    for (int i = wib; i <= p.gamma; i += 8) {
        const bool has_q = i < p.gamma;
        PairStat acc{-FLT_MAX, 0.0f, 0.0f, 0.0f, -FLT_MAX, 0.0f, 0.0f};
        const long long base_p = (static_cast<long long>(b) * R + i) * p.npieces;
        const long long base_q = (static_cast<long long>(b) * R + p.gamma + 1 + i) * p.npieces;
        for (int k = lane; k < p.npieces; k += 32) {
            const float2 sp = p.stat_parts[base_p + k], ep = p.ext_parts[base_p + k];
            PairStat x{sp.x, sp.y, ep.x, ep.y, -FLT_MAX, 0.0f, 0.0f};
            if (has_q) {
                const float2 sq = p.stat_parts[base_q + k], eq = p.ext_parts[base_q + k];
                x.mq = sq.x;
                x.sq = sq.y;
                x.aq = eq.x;
            }
            acc = pair_merge(acc, x);
        }
        acc = warp_pair_merge(acc);
        if (lane == 0) {
            const float l2p = log2f(acc.sp), l2q = log2f(acc.sq);
            const float hp = kLn2 * (l2p - acc.ap / acc.sp);
            if (p.out_Hp) p.out_Hp[static_cast<long long>(b) * (p.gamma + 1) + i] = hp;
            if (has_q) {
                const float hq = kLn2 * (l2q - acc.aq / acc.sq);
                const float cs = acc.c / acc.sp;
                const float kl = cs < kKlInfinite ? INFINITY
                                                  : kLn2 * (acc.ap / acc.sp - cs - l2p + l2q);
                if (p.out_Hq) p.out_Hq[static_cast<long long>(b) * p.gamma + i] = hq;
                if (p.out_KL) p.out_KL[static_cast<long long>(b) * p.gamma + i] = kl;
                s_hq[i] = hq;
            }
        }
    }
    __syncthreads();
    if (threadIdx.x == 0 && p.ctrl_centres) {
        const int j = p.out_n[b];
        if (j >= 0) {
            const double beta = p.ctrl_beta, keep = __dsub_rn(1.0, beta);
            for (int i = 0; i <= j && i < p.gamma; ++i) {
                double* c = p.ctrl_centres + 2 * static_cast<long long>(b) + (i < j ? 0 : 1);
                *c = __dadd_rn(__dmul_rn(keep, *c), __dmul_rn(beta, static_cast<double>(s_hq[i])));
            }
        }
    }
}

// ----------------------------------------------------------------------------------------
// Adaptive draft length ("投机解码的第二本账" (SparseSpec-L), section 3.3): each next draft
// token's acceptance probability p_i comes from its entropy's distances to the two class
// centres, p = d_rej / (d_acc + d_rej) (1/2 when both are 0), and the draft length is the
// candidate k maximising (1 + sum_{m=1..k} prod_{i<=m} p_i) / (k C_d + C_v), the earlier
// candidate on equal values.  One thread per sequence, fp64 with every operation rounded on
// its own, in the order of that definition.
// ----------------------------------------------------------------------------------------

constexpr int kMaxCandidates = 64;

struct AdaptiveKParams {
    const float* H;          // [B, K] next draft tokens' entropies
    const double* centres;   // [B, 2] (accepted, rejected)
    int B, K, n_cand;
    int cand[kMaxCandidates];
    double Cd, Cv;
    int32_t* out_k;          // [B]
    double* out_eff;         // [B] or nullptr
};

__device__ __forceinline__ double soft_accept(double H, double ca, double cr) {
    const double da = fabs(__dsub_rn(H, ca)), dr = fabs(__dsub_rn(H, cr));
    const double s = __dadd_rn(da, dr);
    return s == 0.0 ? 0.5 : __ddiv_rn(dr, s);
}

__global__ void adaptive_k_kernel(AdaptiveKParams a) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= a.B) return;
    const double ca = a.centres[2 * static_cast<long long>(b)];
    const double cr = a.centres[2 * static_cast<long long>(b) + 1];
    const float* h = a.H + static_cast<long long>(b) * a.K;
    int best_k = -1;
    double best = -INFINITY;
    for (int c = 0; c < a.n_cand; ++c) {
        const int k = a.cand[c];
        double prod = 1.0, expect = 0.0;
        for (int m = 0; m < k; ++m) {
            prod = __dmul_rn(prod, soft_accept(static_cast<double>(h[m]), ca, cr));
            expect = __dadd_rn(expect, prod);
        }
        const double eff = __ddiv_rn(__dadd_rn(1.0, expect),
                                     __dadd_rn(__dmul_rn(static_cast<double>(k), a.Cd), a.Cv));
        if (eff > best) {
            best = eff;
            best_k = k;
        }
    }
    a.out_k[b] = best_k;
    if (a.out_eff) a.out_eff[b] = best;
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

template <class ET, int U, bool kClaim>
__global__ void __launch_bounds__(kStreamThreads, 1) row_argmax_kernel(VerifyParams p) {
    stream_pdl_wait();
    using S = typename ET::storage;
    const int lane = threadIdx.x & 31;
    const int R = p.gamma + 1;
    for_block_items<kClaim>(static_cast<long long>(p.B) * R * p.npieces, [&](long long item) {
        const int piece = static_cast<int>(item % p.npieces);
        const long long row_index = item / p.npieces;  // = b * (gamma+1) + i
        const S* row = static_cast<const S*>(p.target) + row_index * p.V;
        const int x0 = piece * p.piece_len;
        const int x1 = min(p.V, x0 + p.piece_len);
#ifdef SPECVERIFY_CHECKED
        if (!(sv_span_in_range(p, row_index * p.V + x0, x1 - x0, p.caps.target) &&
              sv_in_range(p, item, p.caps.stat)))
            return;
#endif
        const ArgMax a = argmax_piece<ET, U>(row, x0, x1, lane);
        if (lane == 0) p.stat_parts[item] = make_float2(a.v, __int_as_float(a.i));
    });
    asm volatile("griddepcontrol.launch_dependents;");
}

// ----------------------------------------------------------------------------------------
// Bounded waits and the status word; scan_greedy: per sequence, the first position whose
// draft token is not the target row's argmax.
// ----------------------------------------------------------------------------------------

constexpr uint32_t kDebugNeverReady = 1u;  // early-exit race units never publish their winners (tests)
constexpr uint32_t kDebugRaceAgain = 2u;   // the LM-head race starts above any winner (tests)
constexpr unsigned long long kWaitLimitNs = 500000000ull;  // give up a wait after 0.5 s

__device__ __forceinline__ unsigned long long global_time_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void set_status(int32_t* status, int code) {
    atomicCAS(reinterpret_cast<int*>(status), 0, code);
}

template <class ET>
__global__ void __launch_bounds__(256) scan_greedy_kernel(VerifyParams p) {
    extern __shared__ float smem[];
    int* sm_g = reinterpret_cast<int*>(smem);  // [gamma+1]
    __shared__ int s_j, s_bad;
    const int R = p.gamma + 1;
    const int b = blockIdx.x;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
    // launched as a programmatic dependent of row_argmax: wait for its partials; a following
    // verify's streaming pass may be set up now (it waits for this grid)
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    if (threadIdx.x == 0) {
        s_j = p.gamma;
        s_bad = 0;
    }
    for (int r = warp; r < R; r += nw) {
        ArgMax a{-INFINITY, INT_MAX};
        const long long pbase = (static_cast<long long>(b) * R + r) * p.npieces;
        const float2* parts = p.stat_parts + pbase;
        if (!sv_span_in_range(p, pbase, p.npieces, p.caps.stat)) continue;
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
    if (!sv_span_in_range(p, static_cast<long long>(b) * (p.gamma + 1), p.gamma + 1, p.caps.out_tokens)) return;
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
// The generator as the verify kernels evaluate it, exposed for testing: form 0 runs the plain
// ten rounds (the acceptance uniforms' path), form 1 the race's evaluation of counter
// (c0, c1, c2, 1) with the per-row parts of rounds 1 and 2 precomputed (race_row_rng and
// race_block_fast, as every race calls them).
// ----------------------------------------------------------------------------------------

__global__ void __launch_bounds__(256) philox_probe_kernel(const uint4* ctr, const uint2* key, long long n,
                                                           int form, uint4* out) {
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const uint4 c = ctr[i];
        const PhiloxKey k{key[i].x, key[i].y};
        if (form == 0) {
            out[i] = philox4x32_10(c, k);
        } else {
            const PhiloxRoundKeys rk = philox_round_keys(k);
            out[i] = race_block_fast(race_row_rng(rk, c.z, c.y), rk, c.x);
        }
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

// Orderable integer image of a float (for a warp max with redux.sync).
__device__ __forceinline__ uint32_t float_order(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float float_unorder(uint32_t u) {
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}

__device__ __forceinline__ float lg2_fast(float x) {
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

// Exact fp32 race score ln w(x) - ln E_x of one token (-inf when its weight is zero).  Kept
// out of line: the filter below calls it for a handful of tokens per row.
__device__ __noinline__ float race_exact_score(float xt, float xd, SeqInfo si, bool residual,
                                               uint32_t w) {
    const float lw = race_log_weight(xt, xd, si, residual);
    return lw > -INFINITY ? lw - race_log_exponential(w) : -INFINITY;
}

// A token can win only if its score reaches the best exact score so far.  Its score is at
// most ln p(x) - ln U_x: the weight max(0, p - q) never exceeds p, and E = -log1p(-U) >= U.
// With U_x >= w 2^-32 the test  log2(w) <= log2 p(x) + 32 - best/ln2 + margin  is a
// necessary condition (w = 0 always passes), and costs one FFMA, one I2F and one lg2.approx.
// The margin (in log2 units) is far above the fp32 error of the exact score.
constexpr float kRaceBoundMargin2 = 1e-3f;

// A vector of tokens is first tested as a whole (vector_may_win), and its tokens one by one
// (token_candidates) only when that passes, which is rare.
constexpr float kVectorTestMargin = 1e-3f;

// The coarse test of one 16-byte vector `raw` (ET::kVec logits) whose Philox words are
// blk[0 .. kVec/4): false when no token of the vector can pass the bound, i.e. when its
// smallest word fails against its largest logit (a necessary condition, up to
// kVectorTestMargin, which covers lg2.approx not being exactly monotone).  Straight-line
// code, so that the tests of a group of vectors overlap; it fails for all but a few vectors
// in a thousand.
template <class ET>
__device__ __forceinline__ bool vector_may_win(const uint4& raw, const uint4* blk, float cp, float C) {
    constexpr int BPV = ET::kVec / 4;
    uint32_t wmin = 0xffffffffu;
#pragma unroll
    for (int gg = 0; gg < BPV; ++gg)
        wmin = min(wmin, min(min(blk[gg].x, blk[gg].y), min(blk[gg].z, blk[gg].w)));
    return lg2_fast(static_cast<float>(wmin)) - kVectorTestMargin <= fmaf(ET::vmax(raw), cp, C);
}

// The tokens of one vector (logits ft, Philox words blk) that pass the bound, as bits:
// token e passes iff lg2(w_e) <= ft[e] cp + C.
template <class ET>
__device__ __forceinline__ uint32_t token_candidates(const float (&ft)[ET::kVec], const uint4* blk, float cp,
                                                     float C) {
    constexpr int BPV = ET::kVec / 4;
    uint32_t cand = 0;
#pragma unroll
    for (int gg = 0; gg < BPV; ++gg) {
        const uint32_t w4[4] = {blk[gg].x, blk[gg].y, blk[gg].z, blk[gg].w};
#pragma unroll
        for (int e = 0; e < 4; ++e)
            cand |= (lg2_fast(static_cast<float>(w4[e])) <= fmaf(ft[4 * gg + e], cp, C)) ? (1u << (4 * gg + e)) : 0u;
    }
    return cand;
}

// Bring row[x0, x1) into L2, one prefetch per 128-byte line spread over the warp's lanes.
// The chunked races read the residual's draft row only at candidate tokens, one dependent
// load each; prefetched with the target vectors, those loads hit L2 (batched serving 59.4 ->
// 57.7 us; the early-exit path's 8 KB race units, which seed from a first pass over the
// piece, measured 1% slower with it and go without).
template <class S>
__device__ __forceinline__ void prefetch_l2(const S* row, int x0, int x1, int lane) {
    constexpr int kLine = 128 / static_cast<int>(sizeof(S));
    for (int x = x0 + lane * kLine; x < x1; x += 32 * kLine)
        asm volatile("prefetch.global.L2 [%0];" ::"l"(row + x));
}

// Race over tokens [x0, x1) of the raced row; every lane offers its tokens in increasing x.
// The residual's draft row is read only at candidate tokens.  kAligned: the vectors are the
// row span's 16-byte-aligned ones (sp as built); otherwise they start at x0 (sp.head = 0) and
// are read with narrower loads.
template <class ET, bool kAligned>
__device__ __forceinline__ RaceState race_piece_body(const typename ET::storage* rt,
                                                     const typename ET::storage* rd, int x0, int x1,
                                                     const RowSpan<ET>& sp, const SeqInfo& si,
                                                     bool residual, const PhiloxRoundKeys& rk,
                                                     uint32_t bg, uint32_t pos, int lane) {
    RaceState st{-INFINITY, INT_MAX, -INFINITY};
    const RaceRowRng q = race_row_rng(rk, bg, pos);
    auto word_at = [&](int x) {
        const uint4 blk = race_block_fast(q, rk, static_cast<uint32_t>(x) >> 2);
        return word_of(blk, static_cast<uint32_t>(x) & 3u);
    };
    auto offer_exact = [&](float xt, int x, uint32_t w) {
        const float xd = residual ? ET::load1(rd + x) : 0.0f;
        const float s = race_exact_score(xt, xd, si, residual, w);
        if (s > -INFINITY) race_offer(st, s, x);
    };
    if (lane < sp.head) offer_exact(ET::load1(sp.base + lane), x0 + lane, word_at(x0 + lane));
    const int xb = x0 + sp.head;
    const uint4* vt = reinterpret_cast<const uint4*>(sp.base + sp.head);
    auto vload = [&](int v) {
        if constexpr (kAligned) return __ldg(vt + v);
        else return ET::load_vec_unaligned(sp.base + v * ET::kVec);
    };
    // Seed the threshold: each lane finds its largest target logit (a cheap pass, no random
    // numbers) and scores that token exactly.  Any token's score is at most the final best,
    // and a lane's most likely token is usually close to it, so few tokens pass the filter.
    // Loads are issued kSeedBatch vectors at a time; the second pass finds the piece in L1.
    constexpr int kSeedBatch = 8;
    constexpr int kRaceBatch = 2;
    float seed = -INFINITY;
    {
        float vmax = -INFINITY;
        int xs = -1;
        for (int v0 = 0; v0 < sp.nvec; v0 += 32 * kSeedBatch) {
            uint4 raw[kSeedBatch];
#pragma unroll
            for (int k = 0; k < kSeedBatch; ++k) {
                const int v = v0 + lane + 32 * k;
                raw[k] = v < sp.nvec ? vload(v)
                                     : make_uint4(ET::kNegInfWord, ET::kNegInfWord,
                                                  ET::kNegInfWord, ET::kNegInfWord);
            }
#pragma unroll
            for (int k = 0; k < kSeedBatch; ++k) {
                float ft[ET::kVec];
                ET::widen(raw[k], ft);
                float m = ft[0];
#pragma unroll
                for (int e = 1; e < ET::kVec; ++e) m = fmaxf(m, ft[e]);
                if (m > vmax) {
                    vmax = m;
#pragma unroll
                    for (int e = ET::kVec - 1; e >= 0; --e)
                        if (ft[e] == m) xs = xb + (v0 + lane + 32 * k) * ET::kVec + e;
                }
            }
        }
        if (xs >= 0) {
            const float xd = residual ? ET::load1(rd + xs) : 0.0f;
            seed = race_exact_score(ET::load1(rt + xs), xd, si, residual, word_at(xs));
        }
    }
    float thr = float_unorder(__reduce_max_sync(0xffffffffu, float_order(fmaxf(seed, st.best))));
    const float mpl = si.mp + si.l2sp;
    for (int v0 = 0; v0 < sp.nvec; v0 += 32 * kRaceBatch) {
        // rhs(x) = log2 p(x) + 32 - thr/ln2 + margin, as one FFMA per token
        const float C = (thr > -INFINITY) ? 32.0f + kRaceBoundMargin2 - thr * kLog2e - mpl
                                          : INFINITY;
        uint4 raw[kRaceBatch];
#pragma unroll
        for (int k = 0; k < kRaceBatch; ++k) {
            const int v = v0 + lane + 32 * k;
            raw[k] = v < sp.nvec ? vload(v) : make_uint4(0u, 0u, 0u, 0u);
        }
        uint4 blk[kRaceBatch][ET::kVec / 4];
#pragma unroll
        for (int k = 0; k < kRaceBatch; ++k)
#pragma unroll
            for (int g = 0; g < ET::kVec / 4; ++g)
                blk[k][g] = race_block_fast(
                    q, rk, static_cast<uint32_t>(xb + (v0 + lane + 32 * k) * ET::kVec + 4 * g) >> 2);
        // each vector's coarse test, then (rarely) its tokens, scored exactly in increasing
        // token order
        bool coarse[kRaceBatch];
        bool any = false;
#pragma unroll
        for (int k = 0; k < kRaceBatch; ++k) {
            coarse[k] = v0 + lane + 32 * k < sp.nvec && vector_may_win<ET>(raw[k], blk[k], si.cp, C);
            any |= coarse[k];
        }
        if (any) {
#pragma unroll
            for (int k = 0; k < kRaceBatch; ++k) {
                if (!coarse[k]) continue;
                float ft[ET::kVec];
                ET::widen(raw[k], ft);
                uint32_t cand = token_candidates<ET>(ft, blk[k], si.cp, C);
                while (cand) {
                    const int e = __ffs(cand) - 1;
                    cand &= cand - 1;
                    const int x = xb + (v0 + lane + 32 * k) * ET::kVec + e;
                    offer_exact(ET::load1(rt + x), x, word_at(x));  // recomputed: no indexed registers
                }
            }
        }
        thr = fmaxf(thr, float_unorder(__reduce_max_sync(0xffffffffu, float_order(st.best))));
    }
    const int t0 = sp.head + sp.nvec * ET::kVec;
    if (lane < sp.tail) offer_exact(ET::load1(sp.base + t0 + lane), x0 + t0 + lane, word_at(x0 + t0 + lane));
    return warp_race_merge(st);
}

// The unaligned race over a piece, kept out of line so that the aligned one is compiled as
// if it were the only one.
template <class ET>
__device__ __noinline__ RaceState race_piece_unaligned(const typename ET::storage* rt,
                                                      const typename ET::storage* rd, int x0, int x1,
                                                      RowSpan<ET> sp, SeqInfo si, bool residual,
                                                      PhiloxRoundKeys rk, uint32_t bg, uint32_t pos,
                                                      int lane) {
    return race_piece_body<ET, false>(rt, rd, x0, x1, sp, si, residual, rk, bg, pos, lane);
}

// The race over [x0, x1): vectors of whole Philox blocks.  Where the row span's first 16-byte
// boundary does not fall on a multiple of four tokens (a row of an odd vocabulary), the
// vectors start at x0 instead (x0 is one) and are read with narrower loads.  kAligned: the
// caller knows rt + x0 is on a 16-byte boundary.
template <class ET, bool kAligned = false>
__device__ __forceinline__ RaceState race_piece(const typename ET::storage* rt,
                                                const typename ET::storage* rd, int x0, int x1,
                                                const SeqInfo& si, bool residual,
                                                const PhiloxRoundKeys& rk, uint32_t bg,
                                                uint32_t pos, int lane) {
    RowSpan<ET> sp(rt, x0, x1);
    if (kAligned || ((x0 + sp.head) & 3) == 0)
        return race_piece_body<ET, true>(rt, rd, x0, x1, sp, si, residual, rk, bg, pos, lane);
    if constexpr (kAligned) return RaceState{};  // (not reached)
    if ((x0 & 3) != 0) {  // (no caller starts a piece off a Philox block)
        const RaceRowRng q = race_row_rng(rk, bg, pos);
        RaceState st{-INFINITY, INT_MAX, -INFINITY};
        for (int x = x0 + lane; x < x1; x += 32) {
            const uint4 blk = race_block_fast(q, rk, static_cast<uint32_t>(x) >> 2);
            const float xd = residual ? ET::load1(rd + x) : 0.0f;
            const float sc = race_exact_score(ET::load1(rt + x), xd, si, residual, word_of(blk, static_cast<uint32_t>(x) & 3u));
            if (sc > -INFINITY) race_offer(st, sc, x);
        }
        return warp_race_merge(st);
    }
    sp.head = 0;
    sp.nvec = (x1 - x0) / ET::kVec;
    sp.tail = (x1 - x0) - sp.nvec * ET::kVec;
    return race_piece_unaligned<ET>(rt, rd, x0, x1, sp, si, residual, rk, bg, pos, lane);
}

// ----------------------------------------------------------------------------------------
// Race geometry: a warp scores kRaceWarpTokens tokens per step from registers (so each is
// read once), a block kRaceBlockTokens; thresholds are seeded from every lane's most likely
// token with a cheap lower bound of its score (no exact evaluation on the critical path).
// ----------------------------------------------------------------------------------------

constexpr int kRaceWarpTokens = 1024;
constexpr int kRaceBlockTokens = 8 * kRaceWarpTokens;
constexpr int kRaceBlockChunks = kRaceBlockTokens / kRaceWarpTokens;  // one chunk per warp
#ifndef SPECVERIFY_RACE_CHAINS
#define SPECVERIFY_RACE_CHAINS 8
#endif
constexpr int kRaceChains = SPECVERIFY_RACE_CHAINS;  // Philox blocks in flight per lane in the race
#ifndef SPECVERIFY_RACE_MINBLOCKS
#define SPECVERIFY_RACE_MINBLOCKS 2
#endif

// A lower bound of the exact score ln w(x) - ln E_x from fast approximations, or -inf.
// E = -log1p(-U) is formed as U (1 + U/2 + U^2/3) below U = 2^-8 (series, relative error
// below 2^-26) and as -ln(1 - U) from lg2.approx of the exact complement above it (relative
// error below 2^-15 there); ln w = ln p + ln(1 - q/p) from ex2/lg2.approx, given up (-inf)
// when 1 - q/p < 2^-10.  The result is reduced by a margin that covers these errors.
__device__ __forceinline__ float race_score_lower_bound(float xt, float xd, const SeqInfo& si,
                                                       bool residual, uint32_t w) {
    const float l2p = fmaf(xt, si.cp, -si.mp) - si.l2sp;
    if (!(l2p > -INFINITY)) return -INFINITY;
    float l2w = l2p;
    if (residual) {
        const float l2q = fmaf(xd, si.cq, -si.mq) - si.l2sq;
        const float one_minus = 1.0f - ex2_fast(l2q - l2p);
        if (!(one_minus > 0x1p-10f)) return -INFINITY;
        l2w += lg2_fast(one_minus);
    }
    float E;
    if (w < 0x01000000u) {
        const float U = (static_cast<float>(w) + 0.5f) * 0x1p-32f;
        E = U * fmaf(U, fmaf(U, 1.0f / 3.0f, 0.5f), 1.0f);
    } else {
        const float one_minus_U = (static_cast<float>(~w) + 0.5f) * 0x1p-32f;
        E = -lg2_fast(one_minus_U) * kLn2;
    }
    return (l2w - lg2_fast(E)) * kLn2 - 1e-3f;
}

// ----------------------------------------------------------------------------------------
// scan_race: G blocks per sequence b, block g racing pieces g, g + G, ... (kRaceBlockTokens
// tokens each) of the raced row, loading each next piece while computing the current one
// and sharing the warps' best scores as the next piece's threshold.  Every block of sequence
// b repeats the sequence's scan (row merges up to the first rejection, gathers, u_i) --
// cheap next to its share of the race -- so no separate scan launch sits between the
// streaming pass and the race; block 0 of the sequence writes the sequence's outputs.  The
// kernel is launched as a programmatic dependent of row_stats: before waiting for it, a
// block gathers p(d_i), q(d_i) inputs and draws its uniforms.  Race partials are single
// 64-bit words (score, index + 1), one per block, that the streaming pass emptied; the last
// block of a sequence (by a relaxed arrival count) polls them, so no fence is needed.
// ----------------------------------------------------------------------------------------

__device__ __forceinline__ unsigned long long pack_race(float best, int idx) {
    return (static_cast<unsigned long long>(static_cast<uint32_t>(idx) + 1u) << 32) |
           __float_as_uint(best);
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64g(const void* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// race_rows_block (below) for a raced row that starts on a 16-byte boundary (kAligned; so
// does every chunk, chunks being 1024 tokens) or not (a row of an odd vocabulary: the
// chunks' vectors are read with narrower loads -- still whole Philox blocks, chunks starting
// on multiples of four tokens).
template <class ET, int NW, class Sync, int CHAINS, bool kAligned>
__device__ __forceinline__ void race_rows_block_impl(const VerifyParams& p, int b,
                                                    const typename ET::storage* rt,
                                                    const typename ET::storage* rd, bool residual,
                                                    uint32_t pos, int32_t* out, int cb_begin,
                                                    int cb_end, int cb_step, int ch_limit, int slot,
                                                    int nslots,
                                                    const SeqInfo& si, float* s_thr,
                                                    RaceState* s_best, int& s_last, int wib, Sync sync) {
    using S = typename ET::storage;
    constexpr int VPL = kRaceWarpTokens / (32 * ET::kVec);
    const int lane = threadIdx.x & 31;
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    const RaceRowRng q = race_row_rng(p.rk, bg, pos);
    RaceState st{-INFINITY, INT_MAX, -INFINITY};
    auto word_at = [&](int x) {
        const uint4 blk = race_block_fast(q, p.rk, static_cast<uint32_t>(x) >> 2);
        return word_of(blk, static_cast<uint32_t>(x) & 3u);
    };
    auto offer_exact = [&](float xt, int x, uint32_t w) {
        const float xd = residual ? ET::load1(rd + x) : 0.0f;
        const float sc = race_exact_score(xt, xd, si, residual, w);
        if (sc > -INFINITY) race_offer(st, sc, x);
    };
    // Step k races chunks cb + w (warp w) of kRaceWarpTokens tokens, cb = cb_begin + k cb_step
    // < cb_end, chunks from ch_limit on excluded.  Vectors of the next step are loaded before
    // the current one is computed.
    auto chunk_x0 = [&](int cb) {
        const int ch = cb + wib;
        return ch < ch_limit ? ch * kRaceWarpTokens : p.V;
    };
    auto load_piece = [&](int cb, uint4 (&dst)[VPL]) {
        const int x0 = chunk_x0(cb);
        const int x1 = min(p.V, x0 + kRaceWarpTokens);
        if (residual) prefetch_l2(rd, x0, x1, lane);
        const int nv = x0 < x1 ? (x1 - x0) / ET::kVec : 0;
        const S* base = rt + (x0 < x1 ? x0 : 0);
#pragma unroll
        for (int k = 0; k < VPL; ++k) {
            const int v = lane + 32 * k;
            if constexpr (kAligned)
                dst[k] = v < nv ? __ldg(reinterpret_cast<const uint4*>(base) + v)
                                : make_uint4(ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord);
            else
                dst[k] = v < nv ? ET::load_vec_unaligned(base + v * ET::kVec)
                                : make_uint4(ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord, ET::kNegInfWord);
        }
    };
    uint4 raw[VPL], raw_next[VPL];
    load_piece(cb_begin, raw);
    float thr = -INFINITY;
    bool first = true;
    for (int cb = cb_begin; cb < cb_end; cb += cb_step) {
        const int x0 = chunk_x0(cb);
        const int x1 = min(p.V, x0 + kRaceWarpTokens);
        const bool vec_ok = x0 < x1 && (!kAligned || (reinterpret_cast<uintptr_t>(rt + x0) & 15u) == 0);
        const int nvec = vec_ok ? (x1 - x0) / ET::kVec : 0;
        if (cb + cb_step < cb_end) load_piece(cb + cb_step, raw_next);
        if (first) {
            // seed: each lane's largest logit, scored by a fast lower bound
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
            seed = float_unorder(__reduce_max_sync(0xffffffffu, float_order(seed)));
            if (lane == 0) s_thr[wib] = seed;
            sync();
            thr = s_thr[0];
#pragma unroll
            for (int k = 1; k < NW; ++k) thr = fmaxf(thr, s_thr[k]);
            first = false;
        }
        if (vec_ok) {
            const float mpl = si.mp + si.l2sp;
            // Philox blocks are computed CHAINS at a time (independent dependency chains, so
            // the rounds of one hide the latency of another), then tested
            constexpr int BPV = ET::kVec / 4;  // Philox blocks per 16-byte vector
            constexpr int VG = CHAINS / BPV;
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
                            q, p.rk, static_cast<uint32_t>(x0 + (lane + 32 * (k0 + kk)) * ET::kVec + 4 * gg) >> 2);
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
            if (lane < (x1 - x0) - t0) offer_exact(ET::load1(rt + x0 + t0 + lane), x0 + t0 + lane,
                                                   word_at(x0 + t0 + lane));
        } else {
            for (int x = x0 + lane; x < x1; x += 32) offer_exact(ET::load1(rt + x), x, word_at(x));
        }
        if (cb + cb_step < cb_end) {
            // every warp's best so far bounds the sequence's best from below: share them
            // through shared memory without a barrier (whatever value a slot holds, old or
            // new, is such a bound)
            volatile float* vt = s_thr;
            if (lane == 0) vt[wib] = thr;
            const float t = lane < NW ? vt[lane] : -INFINITY;
            thr = fmaxf(thr, float_unorder(__reduce_max_sync(0xffffffffu, float_order(t))));
#pragma unroll
            for (int k = 0; k < VPL; ++k) raw[k] = raw_next[k];
        }
    }
    st = warp_race_merge(st);
    if (lane == 0) s_best[wib] = st;
    sync();
    RacePart* parts = p.race_parts + static_cast<long long>(b) * race_slots(p.rpieces);
    if (wib == 0 && lane == 0) {
        RaceState m = s_best[0];
        for (int k = 1; k < NW; ++k) m = race_merge(m, s_best[k]);
        const long long ps = static_cast<long long>(b) * race_slots(p.rpieces) + slot;
        if (slot < race_slots(p.rpieces) && sv_in_range(p, ps, p.caps.race)) {
            parts[slot].second = m.second;  // diagnostic only
            *reinterpret_cast<unsigned long long*>(parts + slot) = pack_race(m.best, m.idx);
        }
        s_last = (atomicAdd(p.tickets + b, 1) == nslots - 1);
    }
    sync();
    if (!s_last || wib != 0) return;
    // last block of this sequence: merge every block's winner, waiting (bounded) for each
    RaceState m{-INFINITY, INT_MAX, -INFINITY};
    for (int k = lane; k < nslots; k += 32) {
        unsigned long long v = ld_relaxed_u64g(parts + k);
        if (v == 0ull) {
            const unsigned long long t0 = global_time_ns();
            while ((v = ld_relaxed_u64g(parts + k)) == 0ull) {
                if (global_time_ns() - t0 > kWaitLimitNs) break;
                __nanosleep(64);
            }
            if (v == 0ull) set_status(p.status, 4 /* SPEC_ETIMEOUT */);
        }
        if (v != 0ull) {
            const float sec = __ldcg(&parts[k].second);
            m = race_merge(m, RaceState{__uint_as_float(static_cast<uint32_t>(v)),
                                        static_cast<int>(static_cast<uint32_t>(v >> 32) - 1u), sec});
        }
    }
    m = warp_race_merge(m);
    if (m.idx == INT_MAX) {
        // Every residual weight was zero (p <= q everywhere in fp32): draw from p_j.
        m = race_piece<ET, kAligned>(rt, nullptr, 0, p.V, si, false, p.rk, bg, pos, lane);
    }
    if (lane == 0) {
        *out = m.idx;
        if (p.out_race) {
            p.out_race[2 * b] = m.best;
            p.out_race[2 * b + 1] = m.second;
        }
    }
}

// The rare unaligned case kept out of line, so that the aligned race is compiled as if it
// were the only one.
template <class ET, int NW, class Sync, int CHAINS>
__device__ __noinline__ void race_rows_block_unaligned(const VerifyParams& p, int b,
                                                       const typename ET::storage* rt,
                                                       const typename ET::storage* rd, bool residual,
                                                       uint32_t pos, int32_t* out, int cb_begin,
                                                       int cb_end, int cb_step, int ch_limit, int slot,
                                                       int nslots, SeqInfo si, float* s_thr,
                                                       RaceState* s_best, int* s_last, int wib, Sync sync) {
    race_rows_block_impl<ET, NW, Sync, CHAINS, false>(p, b, rt, rd, residual, pos, out, cb_begin, cb_end,
                                                      cb_step, ch_limit, slot, nslots, si, s_thr, s_best,
                                                      *s_last, wib, sync);
}

// The race of sequence b by one of the `nslots` groups of NW warps that share it (a block,
// or the racing warps of one), over target row rt (and, for a residual, draft row rd;
// statistics in si) with random-number row `pos`: race the chunks cb + w (warp w of the
// group, wib) for cb = cb_begin, cb_begin + cb_step, ... (< cb_end), chunks from ch_limit on
// excluded, publish the group's winner in partial slot `slot`, and if this is the sequence's
// last group to finish, merge the groups' winners and write the token to *out.  sync() is
// the group's barrier; CHAINS Philox blocks are computed at a time per lane.
// kRowsAligned: the caller knows every row starts on a 16-byte boundary (no out-of-line
// path compiled in).
template <class ET, int NW, class Sync, int CHAINS = kRaceChains, bool kRowsAligned = false>
__device__ __forceinline__ void race_rows_block(const VerifyParams& p, int b,
                                               const typename ET::storage* rt,
                                               const typename ET::storage* rd, bool residual,
                                               uint32_t pos, int32_t* out, int cb_begin,
                                               int cb_end, int cb_step, int ch_limit, int slot,
                                               int nslots,
                                               const SeqInfo& si, float* s_thr,
                                               RaceState* s_best, int& s_last, int wib, Sync sync) {
    if (kRowsAligned || (reinterpret_cast<uintptr_t>(rt) & 15u) == 0)
        race_rows_block_impl<ET, NW, Sync, CHAINS, true>(p, b, rt, rd, residual, pos, out, cb_begin, cb_end,
                                                         cb_step, ch_limit, slot, nslots, si, s_thr, s_best,
                                                         s_last, wib, sync);
    else if constexpr (!kRowsAligned)
        race_rows_block_unaligned<ET, NW, Sync, CHAINS>(p, b, rt, rd, residual, pos, out, cb_begin, cb_end,
                                                        cb_step, ch_limit, slot, nslots, si, s_thr, s_best,
                                                        &s_last, wib, sync);
}

// The chain's race: row j = si.j (the residual of position j < gamma, or the bonus row), by
// a group of NW warps (see race_rows_block).
template <class ET, int NW, class Sync, int CHAINS = kRaceChains, bool kRowsAligned = false>
__device__ __forceinline__ void race_sequence_block(const VerifyParams& p, int b, int cb_begin,
                                                   int cb_end, int cb_step, int ch_limit, int slot,
                                                   int nslots, const SeqInfo& si, float* s_thr,
                                                   RaceState* s_best, int& s_last, int wib, Sync sync) {
    using S = typename ET::storage;
    const int j = si.j;
    const bool residual = j < p.gamma;
    const S* rt = static_cast<const S*>(p.target) + (static_cast<long long>(b) * (p.gamma + 1) + j) * p.V;
    const S* rd = residual ? static_cast<const S*>(p.draft) + (static_cast<long long>(b) * p.gamma + j) * p.V
                           : nullptr;
    // (every block of the sequence takes the same branch: none arrives, none waits)
    if (!(sv_span_in_range(p, (static_cast<long long>(b) * (p.gamma + 1) + j) * p.V, p.V, p.caps.target) &&
          (!residual || sv_span_in_range(p, (static_cast<long long>(b) * p.gamma + j) * p.V, p.V, p.caps.draft)) &&
          sv_in_range(p, static_cast<long long>(b) * (p.gamma + 1) + j, p.caps.out_tokens)))
        return;
    race_rows_block<ET, NW, Sync, CHAINS, kRowsAligned>(p, b, rt, rd, residual, static_cast<uint32_t>(j),
                            p.out_tokens + static_cast<long long>(b) * (p.gamma + 1) + j, cb_begin,
                            cb_end, cb_step, ch_limit, slot, nslots, si, s_thr, s_best, s_last, wib,
                            sync);
}

// Eight partials (packed (m, s) words; past P: empty) merged as a balanced tree.
__device__ __forceinline__ SoftmaxStat fold8(const unsigned long long* v, int n) {
    SoftmaxStat t[8];
#pragma unroll
    for (int q = 0; q < 8; ++q)
        t[q] = q < n ? SoftmaxStat{__uint_as_float(static_cast<uint32_t>(v[q])),
                                   __uint_as_float(static_cast<uint32_t>(v[q] >> 32))}
                     : SoftmaxStat{-FLT_MAX, 0.0f};
    t[0] = merge_stat(t[0], t[1]);
    t[2] = merge_stat(t[2], t[3]);
    t[4] = merge_stat(t[4], t[5]);
    t[6] = merge_stat(t[6], t[7]);
    t[0] = merge_stat(t[0], t[2]);
    t[4] = merge_stat(t[4], t[6]);
    return merge_stat(t[0], t[4]);
}

// The merged statistics of one row from its P partials (packed (m, s) words, complete: they
// were written by an earlier kernel), by one thread in a fixed order: eight partials at a
// time merged as a balanced tree (pairs, pairs of pairs, root), the eight-partial results
// folded in piece order, so that every call merges a row's pieces into the same bits.
__device__ __forceinline__ SoftmaxStat fold_row_stats(const unsigned long long* parts, int P) {
    SoftmaxStat acc{-FLT_MAX, 0.0f};
    // sixteen loads in flight (two eight-partial groups), folded in the same order
    for (int k0 = 0; k0 < P; k0 += 16) {
        unsigned long long v[16];
#pragma unroll
        for (int q = 0; q < 16; ++q)
            v[q] = (k0 + q < P) ? __ldcg(parts + k0 + q) : 0ull;
        acc = merge_stat(acc, fold8(v, P - k0));
        if (k0 + 8 < P) acc = merge_stat(acc, fold8(v + 8, P - k0 - 8));
    }
    return acc;
}

// One sequence's scan by a group of nt threads (thread tid of them): the draft tokens and
// their logits, the acceptance uniforms, every row's merged statistics, the accept tests and
// the first rejection.  Split in two so that the inputs-only part can run before the
// statistics are complete: scan_prologue (positions i = tid < min(nt, kScanFast) gathered
// into shared memory), then, after the group's barrier, scan_sequence.
constexpr int kScanFast = 256;  // positions gathered ahead by the prologue, at most

struct ScanShared {
    int j, bad;
    int d[kScanFast];
    float xt[kScanFast], xd[kScanFast], u[kScanFast];
};

template <class ET>
__device__ __forceinline__ void scan_prologue(const VerifyParams& p, int b, int tid, ScanShared& sh) {
    using S = typename ET::storage;
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    const int i0 = tid;
    if (i0 < p.gamma && i0 < kScanFast) {
        const int d = p.tokens[static_cast<long long>(b) * p.gamma + i0];
        sh.d[i0] = d;
        sh.u[i0] = accept_uniform(p.key, bg, static_cast<uint32_t>(i0));
        float xt = 0.0f, xd = 0.0f;
        const long long kt = (static_cast<long long>(b) * (p.gamma + 1) + i0) * p.V + d;
        const long long kd = (static_cast<long long>(b) * p.gamma + i0) * p.V + d;
        if (d >= 0 && d < p.V && sv_in_range(p, kt, p.caps.target) && sv_in_range(p, kd, p.caps.draft)) {
            xt = ET::load1(static_cast<const S*>(p.target) + kt);
            xd = ET::load1(static_cast<const S*>(p.draft) + kd);
        }
        sh.xt[i0] = xt;
        sh.xd[i0] = xd;
    }
    if (tid == 0) {
        sh.j = p.gamma;
        sh.bad = 0;
    }
}

// The rest of the scan, after the prologue and a barrier: returns the first rejection j
// (gamma: all accepted; -1: a draft token outside [0, V)), with every row's scaled max and
// log2 sum in sm_m / sm_l.  The writer group also writes the sequence's outputs (n_accepted,
// the accepted prefix and the -1 padding; the drawn token is the race's) and diagnostics.
template <class ET, class Sync>
__device__ __forceinline__ int scan_sequence(const VerifyParams& p, int b, bool writer, int tid, int nt,
                                             ScanShared& sh, float* sm_m, float* sm_l, Sync sync) {
    using S = typename ET::storage;
    const int R = 2 * p.gamma + 1;
    const int nfast = min(nt, kScanFast);
    const float cp = scale_of(seq_T(p, b)), cq = scale_of(seq_Td(p, b));
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    // any draft token outside [0, V) marks the whole sequence
    for (int i = tid; i < p.gamma; i += nt) {
        const int d = (i < nfast) ? sh.d[i] : p.tokens[static_cast<long long>(b) * p.gamma + i];
        if (d < 0 || d >= p.V) sh.bad = 1;
    }
    auto decide = [&](int i) {  // one thread: the accept test at position i
        int d;
        float xt, xd, u;
        if (i < nfast) {
            d = sh.d[i]; xt = sh.xt[i]; xd = sh.xd[i]; u = sh.u[i];
        } else {
            d = p.tokens[static_cast<long long>(b) * p.gamma + i];
            u = accept_uniform(p.key, bg, static_cast<uint32_t>(i));
            const long long kt = (static_cast<long long>(b) * (p.gamma + 1) + i) * p.V + d;
            const long long kd = (static_cast<long long>(b) * p.gamma + i) * p.V + d;
            xt = sv_in_range(p, kt, p.caps.target) ? ET::load1(static_cast<const S*>(p.target) + kt) : 0.0f;
            xd = sv_in_range(p, kd, p.caps.draft) ? ET::load1(static_cast<const S*>(p.draft) + kd) : 0.0f;
        }
        const long long k = static_cast<long long>(b) * p.gamma + i;
        if (writer && p.out_u) p.out_u[k] = u;
        const float l2p = fmaf(xt, cp, -sm_m[i]) - sm_l[i];
        const float l2q = fmaf(xd, cq, -sm_m[p.gamma + 1 + i]) - sm_l[p.gamma + 1 + i];
        if (writer && p.out_logp) p.out_logp[k] = l2p * kLn2;
        if (writer && p.out_logq) p.out_logq[k] = l2q * kLn2;
        // accept iff u < min(1, p/q); p(d) = 0 rejects, q(d) = 0 < p(d) accepts
        if (!((l2p > -INFINITY) && (u < exp2f(l2p - l2q)))) atomicMin(&sh.j, i);
    };
    // every row's statistics, one thread per row (fold_row_stats: the order every schedule
    // uses); rows past the first rejection decide nothing but cost one L2 read per partial
    const unsigned long long* parts =
        reinterpret_cast<const unsigned long long*>(p.stat_parts) + static_cast<long long>(b) * R * p.npieces;
    for (int r = tid; r < R; r += nt) {
        const long long pbase = (static_cast<long long>(b) * R + r) * p.npieces;
        const SoftmaxStat st = sv_span_in_range(p, pbase, p.npieces, p.caps.stat)
            ? fold_row_stats(parts + static_cast<long long>(r) * p.npieces, p.npieces)
            : SoftmaxStat{-FLT_MAX, 1.0f};
        const float l2s = log2f(st.s);
        sm_m[r] = st.m;
        sm_l[r] = l2s;
        if (writer) {
            const float lz = (st.m + l2s) * kLn2;
            if (r <= p.gamma) {
                if (p.out_logZp) p.out_logZp[static_cast<long long>(b) * (p.gamma + 1) + r] = lz;
            } else if (p.out_logZq) {
                p.out_logZq[static_cast<long long>(b) * p.gamma + (r - p.gamma - 1)] = lz;
            }
        }
    }
    sync();
    if (sh.bad) {
        if (writer) {
            for (int i = tid; i < p.gamma; i += nt) {
                const long long k = static_cast<long long>(b) * p.gamma + i;
                if (p.out_u) p.out_u[k] = accept_uniform(p.key, bg, static_cast<uint32_t>(i));
                if (p.out_logp) p.out_logp[k] = NAN;
                if (p.out_logq) p.out_logq[k] = NAN;
            }
        }
    } else {
        for (int i = tid; i < p.gamma; i += nt) decide(i);
    }
    sync();
    const int j = sh.bad ? -1 : sh.j;
    if (writer) {
        if (tid == 0) {
            p.out_n[b] = j;
            if (j < 0) set_status(p.status, 3 /* SPEC_EBADTOKEN */);
        }
        int32_t* out = p.out_tokens + static_cast<long long>(b) * (p.gamma + 1);
        if (sv_span_in_range(p, static_cast<long long>(b) * (p.gamma + 1), p.gamma + 1, p.caps.out_tokens))
            for (int t = tid; t <= p.gamma; t += nt)
                if (t != j) out[t] = (j >= 0 && t < j) ? p.tokens[static_cast<long long>(b) * p.gamma + t] : -1;
    }
    return j;
}

// The statistics of sequence b's raced row j (target row j and, for a residual, draft row
// j) from the scan's shared row statistics.
__device__ __forceinline__ SeqInfo raced_row_info(const VerifyParams& p, int b, int j, const float* sm_m,
                                                  const float* sm_l) {
    SeqInfo si;
    si.j = j;
    si.cp = scale_of(seq_T(p, b));
    si.cq = scale_of(seq_Td(p, b));
    si.mp = sm_m[j];
    si.l2sp = sm_l[j];
    const bool residual = j < p.gamma;
    si.mq = residual ? sm_m[p.gamma + 1 + j] : 0.0f;
    si.l2sq = residual ? sm_l[p.gamma + 1 + j] : 0.0f;
    si.pad = 0;
    return si;
}

template <class ET>
__global__ void __launch_bounds__(256, SPECVERIFY_RACE_MINBLOCKS) scan_race_kernel(VerifyParams p) {
    extern __shared__ float smem[];  // [2R]: scaled max and log2 sum of every row
    __shared__ int s_last;
    __shared__ float s_thr[8];
    __shared__ RaceState s_best[8];
    __shared__ ScanShared sh;
    const int R = 2 * p.gamma + 1;
    float* sm_m = smem;
    float* sm_l = smem + R;
    auto sync = [] { __syncthreads(); };
    // This block's race chunks (kRaceWarpTokens tokens each), in one of two layouts:
    //   G = p.rgroups > 0: G blocks per sequence, block g racing steps g, g + G, ... of its
    //     sequence's row (a step: one chunk per warp); every block scans one sequence;
    //   G = 0: the T = B * CH chunks in sequence-major order split evenly, block k taking
    //     [k T / n, (k + 1) T / n) (at least one step each); a block whose range crosses a
    //     sequence boundary scans and races both sequences.
    const int CH = (p.V + kRaceWarpTokens - 1) / kRaceWarpTokens;
    const int G = p.rgroups;
    const long long T = static_cast<long long>(p.B) * CH;
    const long long nblk = gridDim.x;
    const long long q0 = G > 0 ? 0 : static_cast<long long>(blockIdx.x) * T / nblk;
    const long long q1 = G > 0 ? 1 : (static_cast<long long>(blockIdx.x) + 1) * T / nblk;
    auto block_of = [&](long long x) { return ((x + 1) * nblk - 1) / T; };  // block racing chunk x
    bool first = true;
    for (long long q = q0; q < q1;) {
        int b, cb_begin, cb_end, cb_step, ch_limit, slot, nslots;
        if (G > 0) {
            b = static_cast<int>(blockIdx.x / G);
            slot = static_cast<int>(blockIdx.x % G);
            nslots = G;
            cb_begin = slot * kRaceBlockChunks;
            cb_step = G * kRaceBlockChunks;
            cb_end = ch_limit = CH;
            q = q1;
        } else {
            b = static_cast<int>(q / CH);
            const int ch0 = static_cast<int>(q % CH);
            const int ch1 = static_cast<int>(min(static_cast<long long>(CH), ch0 + (q1 - q)));
            q += ch1 - ch0;
            const long long k_lo = block_of(static_cast<long long>(b) * CH);
            const long long k_hi = block_of(static_cast<long long>(b + 1) * CH - 1);
            slot = static_cast<int>(blockIdx.x - k_lo);
            nslots = static_cast<int>(k_hi - k_lo + 1);
            cb_begin = ch0;
            cb_end = ch_limit = ch1;
            cb_step = kRaceBlockChunks;
        }
        // inputs-only prologue: the first sequence's overlaps the streaming pass's tail
        scan_prologue<ET>(p, b, threadIdx.x, sh);
        if (first) {
            asm volatile("griddepcontrol.wait;" ::: "memory");
            // a following verify's streaming pass may be set up now: it waits for this grid
            asm volatile("griddepcontrol.launch_dependents;");
        }
        first = false;
        __syncthreads();  // sh.j and sh.bad are set before any thread reports a bad token
        const int j = scan_sequence<ET>(p, b, slot == 0, threadIdx.x, blockDim.x, sh, sm_m, sm_l, sync);
        if (j >= 0)
            race_sequence_block<ET, 8>(p, b, cb_begin, cb_end, cb_step, ch_limit, slot, nslots,
                                       raced_row_info(p, b, j, sm_m, sm_l), s_thr, s_best, s_last,
                                       static_cast<int>(threadIdx.x >> 5), sync);
        if (q < q1) __syncthreads();  // before the next sequence reuses shared memory
    }
}

// ----------------------------------------------------------------------------------------
// Static token-tree verification ("SubSpec: Speculate Deep and Accurate" (papernotes): the
// draft is a token tree whose candidate paths one target forward verifies; SubSpec keeps a
// static, deep and narrow tree).  The pages give no multi-branch rule; the one taken is
// multi-draft rejection sampling, lossless when the children of a node are independent
// draws from the node's draft distribution q_u: at node u try its children in node order
// against the running residual p' = max(0, p_u - c q_u) / N (c = 0, N = 1 at first):
// accept child v (token x) iff u_v < min(1, p'(x) / q_u(x)) and move to v; on a rejection
// set c <- c + N and N <- sum_x max(0, p_u(x) - c q_u(x)).  When every child is rejected the
// token is drawn from p' -- the race over max(0, p_u - c q_u), which is the chain's residual
// race with log2 c added to the draft row's log-normaliser -- and at a node without
// children the bonus token is drawn from p_u.  A chain-shaped tree is the chain verify.
//
// tree_stats   row statistics of the target row of every node and the draft row of every
//              internal node (the streaming pass of the chain, another row mapping);
// tree_walk    one block per sequence walks the tree from the root, merging the rows of
//              the nodes it visits; each rejection costs one block-wide pass over the node's
//              two rows for the next N;
// tree_race    the race of each sequence's last node, G blocks per sequence.
// ----------------------------------------------------------------------------------------

constexpr int kMaxTreeNodes = 512;

struct TreeShape {
    int N, M, D;                          // nodes, internal nodes (draft rows), depth
    int16_t drow[kMaxTreeNodes];          // draft row of node u (its rank among internal nodes), -1: leaf
    int16_t first_child[kMaxTreeNodes];   // -1: none
    int16_t next_sibling[kMaxTreeNodes];  // next child of the same parent in node order, -1: last
};

struct TreeRace {
    int node, k, residual, drow;  // node raced (-1: none), output slot, residual?, its draft row
};

// ----------------------------------------------------------------------------------------
// verify_small: the whole sampling verify of one sequence in one block, for calls whose
// sequences are so small that a second launch costs more than their work (every row's
// pieces read by the block's warps, and the raced row one race step long).  Warp w takes
// the sequence's row pieces w, w + 8, ... with the same pieces and arithmetic as row_stats,
// so the partials are the same bits; the block then scans and races the sequence exactly as
// scan_race does with one block per sequence.  The block empties its sequence's race slot
// and arrival count itself (row_stats does that on the two-kernel path).  Taken only when
// every row starts on a 16-byte boundary (V s a multiple of 16).
// ----------------------------------------------------------------------------------------
constexpr int kSmallSeqBytes = 64 * 1024;  // largest (2 gamma + 1) V s taken by verify_small

template <class ET, int U>
__global__ void __launch_bounds__(256, SPECVERIFY_RACE_MINBLOCKS) verify_small_kernel(VerifyParams p) {
    extern __shared__ float smem[];  // [2R]: scaled max and log2 sum of every row
    __shared__ int s_last;
    __shared__ float s_thr[8];
    __shared__ RaceState s_best[8];
    __shared__ ScanShared sh;
    const int R = 2 * p.gamma + 1;
    float* sm_m = smem;
    float* sm_l = smem + R;
    auto sync = [] { __syncthreads(); };
    const int lane = threadIdx.x & 31;
    const int warp = static_cast<int>(threadIdx.x >> 5);
    const int b = blockIdx.x;
    scan_prologue<ET>(p, b, threadIdx.x, sh);  // inputs only: overlaps the previous kernel
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const int ns = race_slots(p.rpieces);
    for (int k = threadIdx.x; k < ns; k += blockDim.x)
        if (sv_in_range(p, static_cast<long long>(b) * ns + k, p.caps.race))
            reinterpret_cast<uint4*>(p.race_parts + static_cast<long long>(b) * ns)[k] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) p.tickets[b] = 0;
    for (int item = warp; item < R * p.npieces; item += static_cast<int>(blockDim.x >> 5))
        row_stats_item<ET, U>(p, b, item / p.npieces, item % p.npieces, lane);
    __syncthreads();  // the partials (and sh, the emptied slots) are visible to the block
    const int j = scan_sequence<ET>(p, b, true, threadIdx.x, blockDim.x, sh, sm_m, sm_l, sync);
    const int CH = (p.V + kRaceWarpTokens - 1) / kRaceWarpTokens;
    if (j >= 0)
        race_sequence_block<ET, 8, decltype(sync), kRaceChains, true>(p, b, 0, CH, kRaceBlockChunks, CH, 0, 1,
                                   raced_row_info(p, b, j, sm_m, sm_l), s_thr, s_best, s_last, warp, sync);
}

template <class ET, int U, bool kClaim>
__global__ void __launch_bounds__(kStreamThreads, SPECVERIFY_STATS_MINBLOCKS) tree_stats_kernel(VerifyParams p, int N, int M) {
    stream_pdl_wait();
    using S = typename ET::storage;
    const int lane = threadIdx.x & 31;
    const long long nthreads = static_cast<long long>(gridDim.x) * blockDim.x;
    const long long tid = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x;
    for (long long k = tid; k < static_cast<long long>(p.B) * race_slots(p.rpieces); k += nthreads)
        reinterpret_cast<uint4*>(p.race_parts)[k] = make_uint4(0u, 0u, 0u, 0u);
    for (long long k = tid; k < p.B; k += nthreads) p.tickets[k] = 0;
    const int R = N + M;
    for_block_items<kClaim>(static_cast<long long>(p.B) * R * p.npieces, [&](long long item) {
        const int piece = static_cast<int>(item % p.npieces);
        const long long br = item / p.npieces;
        const int b = static_cast<int>(br / R), r = static_cast<int>(br % R);
        const S* row;
        float c;
        if (r < N) {
            row = static_cast<const S*>(p.target) + (static_cast<long long>(b) * N + r) * p.V;
            c = scale_of(seq_T(p, b));
        } else {
            row = static_cast<const S*>(p.draft) + (static_cast<long long>(b) * M + (r - N)) * p.V;
            c = scale_of(seq_Td(p, b));
        }
        const int x0 = piece * p.piece_len;
        const SoftmaxStat st = stats_piece<ET, U>(row, x0, min(p.V, x0 + p.piece_len), c, lane);
        if (lane == 0) store_stat(p.stat_parts + br * p.npieces + piece, st.m, st.s);
    });
    asm volatile("griddepcontrol.launch_dependents;");
}

constexpr int kTreeCluster = 8;  // CTAs per sequence in tree_walk (a portable cluster size)

// Cluster: sum over the row of max(0, p(x) - c q(x)), p(x) = 2^(xt cp - mp - l2sp) and
// q(x) = 2^(xd cq - mq - l2sq) (fp32; c > 0).  CTA r of the cluster sums elements
// r, r + kTreeCluster, ... (in 16-byte vectors when the two rows are aligned alike), the
// CTAs publish their sums in shared memory, and after a cluster barrier every CTA adds the
// kTreeCluster sums in rank order -- so every CTA gets the same value.
template <class ET>
__device__ float residual_mass_cluster(const typename ET::storage* rt, const typename ET::storage* rd,
                                       int V, float cp, float mp, float l2sp, float cq, float mq,
                                       float l2sq, float c, float* s_red, float* s_part) {
    namespace cg = cooperative_groups;
    cg::cluster_group cluster = cg::this_cluster();
    const int rank = static_cast<int>(cluster.block_rank());
    const float l2c = log2f(c);
    const float op = -mp - l2sp, oq = -mq - l2sq + l2c;
    float acc = 0.0f;
    auto term = [&](float xt, float xd) {
        const float p = ex2_fast(fmaf(xt, cp, op));
        const float cq_ = ex2_fast(fmaf(xd, cq, oq));
        return fmaxf(p - cq_, 0.0f);
    };
    const RowSpan<ET> st(rt, 0, V), sd(rd, 0, V);
    const int stride = blockDim.x * kTreeCluster;
    const int t = rank * blockDim.x + threadIdx.x;
    if (st.head == sd.head) {
        if (t < st.head) acc += term(ET::load1(rt + t), ET::load1(rd + t));
        const uint4* vt = st.vec();
        const uint4* vd = sd.vec();
        for (int v = t; v < st.nvec; v += stride) {
            float ft[ET::kVec], fd[ET::kVec];
            ET::widen(__ldg(vt + v), ft);
            ET::widen(__ldg(vd + v), fd);
#pragma unroll
            for (int e = 0; e < ET::kVec; ++e) acc += term(ft[e], fd[e]);
        }
        const int t0 = st.head + st.nvec * ET::kVec;
        if (t < st.tail) acc += term(ET::load1(rt + t0 + t), ET::load1(rd + t0 + t));
    } else {
        for (int x = t; x < V; x += stride) acc += term(ET::load1(rt + x), ET::load1(rd + x));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) s_red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        float sum = 0.0f;
        for (int k = 0; k < static_cast<int>(blockDim.x >> 5); ++k) sum += s_red[k];
        *s_part = sum;
    }
    cluster.sync();  // every CTA's sum is published
    float total = 0.0f;
    for (int r = 0; r < kTreeCluster; ++r) total += *cluster.map_shared_rank(s_part, r);
    cluster.sync();  // nobody overwrites a sum before every CTA has read it
    return total;
}

// One cluster of kTreeCluster CTAs per sequence: every CTA walks the tree with the same
// values (so they take the same decisions), and they share each residual pass; CTA 0
// writes the results.
template <class ET>
__global__ void __cluster_dims__(kTreeCluster, 1, 1) __launch_bounds__(256)
tree_walk_kernel(VerifyParams p, TreeShape t) {
    using S = typename ET::storage;
    namespace cg = cooperative_groups;
    __shared__ float s_m[2], s_l[2], s_red[8], s_part;
    __shared__ int s_bad, s_acc;
    const int lane = threadIdx.x & 31, wib = threadIdx.x >> 5;
    const int b = blockIdx.x / kTreeCluster;
    const bool leader = cg::this_cluster().block_rank() == 0;
    const int N = t.N, M = t.M, R = N + M;
    const float cp = scale_of(seq_T(p, b)), cq = scale_of(seq_Td(p, b));
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    const int32_t* tok = p.tokens + static_cast<long long>(b) * N;
    int32_t* out = p.out_tokens + static_cast<long long>(b) * (t.D + 1);
    int32_t* nodes = p.out_nodes ? p.out_nodes + static_cast<long long>(b) * t.D : nullptr;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    if (threadIdx.x == 0) s_bad = 0;
    if (leader) {
        for (int i = threadIdx.x; i <= t.D; i += blockDim.x) out[i] = -1;
        for (int i = threadIdx.x; nodes && i < t.D; i += blockDim.x) nodes[i] = -1;
    }
    __syncthreads();
    for (int n = 1 + threadIdx.x; n < N; n += blockDim.x)
        if (tok[n] < 0 || tok[n] >= p.V) s_bad = 1;
    __syncthreads();
    if (s_bad) {
        if (leader && threadIdx.x == 0) {
            p.out_n[b] = -1;
            p.tree_race[b] = TreeRace{-1, 0, 0, -1};
            set_status(p.status, 3 /* SPEC_EBADTOKEN */);
        }
        return;
    }
    auto merge_row = [&](int r, int slot) {  // one warp
        SoftmaxStat st{-FLT_MAX, 0.0f};
        const float2* parts = p.stat_parts + (static_cast<long long>(b) * R + r) * p.npieces;
        for (int k = lane; k < p.npieces; k += 32) {
            const float2 q = parts[k];
            st = merge_stat(st, SoftmaxStat{q.x, q.y});
        }
        st = warp_merge_stat(st);
        if (lane == 0) {
            s_m[slot] = st.m;
            s_l[slot] = log2f(st.s);
        }
    };
    int u = 0, k = 0;
    for (;;) {
        const int dr = t.drow[u];
        if (wib == 0) merge_row(u, 0);
        if (wib == 1 && dr >= 0) merge_row(N + dr, 1);
        __syncthreads();
        const float mp = s_m[0], l2sp = s_l[0];
        if (dr < 0) {  // no children: the bonus token from p_u
            if (leader && threadIdx.x == 0) {
                SeqInfo si{u, mp, l2sp, 0.0f, 0.0f, cp, cq, 0};
                p.seq[b] = si;
                p.tree_race[b] = TreeRace{u, k, 0, -1};
                p.out_n[b] = k;
            }
            return;
        }
        const float mq = s_m[1], l2sq = s_l[1];
        const S* rt = static_cast<const S*>(p.target) + (static_cast<long long>(b) * N + u) * p.V;
        const S* rd = static_cast<const S*>(p.draft) + (static_cast<long long>(b) * M + dr) * p.V;
        float c = 0.0f, mass = 1.0f;
        int accepted = -1;
        for (int v = t.first_child[u]; v >= 0; v = t.next_sibling[v]) {
            if (threadIdx.x == 0) {
                const int x = tok[v];
                const float l2p = fmaf(ET::load1(rt + x), cp, -mp) - l2sp;
                const float l2q = fmaf(ET::load1(rd + x), cq, -mq) - l2sq;
                float l2pp = l2p;  // log2 of the running residual p'(x)
                if (c > 0.0f) {
                    const float l2cq = l2q + log2f(c);
                    l2pp = (l2p > l2cq) ? l2p + log1pf(-exp2f(l2cq - l2p)) * kLog2e - log2f(mass)
                                        : -INFINITY;
                }
                const float uv = accept_uniform(p.key, bg, static_cast<uint32_t>(v - 1));
                // accept iff u < min(1, p'(x)/q(x)); p'(x) = 0 rejects, q(x) = 0 < p'(x) accepts
                s_acc = (l2pp > -INFINITY) && (uv < exp2f(l2pp - l2q));
            }
            __syncthreads();
            const int acc = s_acc;
            __syncthreads();
            if (acc) {
                accepted = v;
                break;
            }
            c += mass;
            mass = residual_mass_cluster<ET>(rt, rd, p.V, cp, mp, l2sp, cq, mq, l2sq, c, s_red, &s_part);
        }
        if (accepted >= 0) {
            if (leader && threadIdx.x == 0) {
                out[k] = tok[accepted];
                if (nodes) nodes[k] = accepted;
            }
            ++k;
            u = accepted;
            __syncthreads();
            continue;
        }
        // every child rejected: the race over max(0, p_u - c q_u)
        if (leader && threadIdx.x == 0) {
            SeqInfo si{u, mp, l2sp, mq, l2sq - log2f(c), cp, cq, 0};
            p.seq[b] = si;
            p.tree_race[b] = TreeRace{u, k, 1, dr};
            p.out_n[b] = k;
        }
        return;
    }
}

template <class ET>
__global__ void __launch_bounds__(256, SPECVERIFY_RACE_MINBLOCKS) tree_race_kernel(VerifyParams p, int N, int M, int D) {
    using S = typename ET::storage;
    __shared__ float s_thr[8];
    __shared__ RaceState s_best[8];
    __shared__ int s_last;
    const int G = p.rgroups;
    const int b = blockIdx.x / G, g = blockIdx.x % G;
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");  // (see scan_greedy_kernel)
    const TreeRace tr = p.tree_race[b];
    if (tr.node < 0) return;
    const SeqInfo si = p.seq[b];
    const S* rt = static_cast<const S*>(p.target) + (static_cast<long long>(b) * N + tr.node) * p.V;
    const S* rd = tr.residual ? static_cast<const S*>(p.draft) + (static_cast<long long>(b) * M + tr.drow) * p.V
                              : nullptr;
    race_rows_block<ET, 8>(p, b, rt, rd, tr.residual != 0, static_cast<uint32_t>(tr.node),
                           p.out_tokens + static_cast<long long>(b) * (D + 1) + tr.k, g * kRaceBlockChunks,
                           p.rpieces * kRaceBlockChunks, G * kRaceBlockChunks, INT_MAX, g, G, si, s_thr,
                           s_best, s_last, static_cast<int>(threadIdx.x >> 5), [] { __syncthreads(); });
}

__device__ __forceinline__ int ld_acquire(const int* p) {
    int v;
    asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ int ld_relaxed(const int* p) {
    int v;
    asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void st_release(int* p, int v) {
    asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const void* p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// Wait (bounded) until a pre-filled (m, s) word has been written; returns it.  On giving up
// it records SPEC_ETIMEOUT and returns an empty pair.
__device__ __forceinline__ float2 wait_stat(const VerifyParams& p, const float2* src) {
    unsigned long long v = ld_relaxed_u64(src);
    if (v == kStatEmpty) {
        const unsigned long long t0 = global_time_ns();
        while ((v = ld_relaxed_u64(src)) == kStatEmpty) {
            if (global_time_ns() - t0 > kWaitLimitNs) {
                set_status(p.status, 4 /* SPEC_ETIMEOUT */);
                return make_float2(-FLT_MAX, 0.0f);
            }
            __nanosleep(64);
        }
    }
    return make_float2(__uint_as_float(static_cast<uint32_t>(v)),
                       __uint_as_float(static_cast<uint32_t>(v >> 32)));
}

// ----------------------------------------------------------------------------------------
// verify_early: the early-exit sampling verify as one persistent (cooperative) launch that
// schedules its own work.  A sequence's rows are read one position at a time, and only up
// to its first rejection: the method discards the rest of the draft ("How speculative
// decoding makes LLMs go brrr": pseudocode, rejection step), so those rows never decide
// anything.
//
// Work comes from two queues of tasks, each task split into npieces units of piece_len
// logits:
//   row queue    (b, r): partial softmax statistics of row r of sequence b, one piece per
//                unit.  The first tasks (target and draft rows of position 0 of every
//                sequence, or the bonus rows when gamma = 0) are implicit; the rest are
//                appended as positions are accepted;
//   race queue   b: the exponential race over the raced row of b, one piece per unit,
//                appended when b is decided.
// Row warps (the first 8 - kEarlyRaceWarps of each block) claim row units in queue order
// from one counter; race warps claim race units from another, and row warps join them once
// every sequence is decided.  Keeping the races out of the row queue keeps the chain of a
// long-accepted draft (merge, decide, next position) from queueing behind race work.  The
// last unit of a row to finish merges the row; the second row of a position to be merged
// decides the position: on acceptance it appends the next position's two rows (or the bonus
// row after position gamma-1), on rejection -- or when the bonus row is merged -- it writes
// the sequence's outputs and appends its race.  The last race unit of a sequence merges the
// units' winners and writes the token.
//
// No unit ever waits on another claimed unit: a warp waits only for a queue slot that is
// not written yet, or for partial results whose writers have already counted their arrival
// (partials are pre-filled with empty markers and polled, so no fence is needed).  Each
// undecided sequence always has one task in the row queue, so a row slot a warp waits for
// is either written soon by the warp that reserved it, or lies past every queued row task,
// whose units are then all claimed by warps that do not wait; race warps hold no row work.
// Every wait gives up after kWaitLimitNs and records SPEC_ETIMEOUT.
// ----------------------------------------------------------------------------------------

constexpr int kTaskEmpty = -1;  // queue slot not written yet (the slots are pre-filled)

__device__ __forceinline__ void st_relaxed(int* p, int v) {
    asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Rows of position i: its target and draft rows, or the bonus row (target row gamma).
__device__ __forceinline__ int early_rows_of(const VerifyParams& p, int i) {
    return i < p.gamma ? 2 : 1;
}

// Events that complete position i: each of its rows merged and, after position 0, the
// acceptance of position i - 1.  Whoever brings the count to this decides the position.
__device__ __forceinline__ int early_events_of(const VerifyParams& p, int i) {
    return early_rows_of(p, i) + (i > 0 ? 1 : 0);
}

// Rows of positions 0..L (target row k, draft row k, ...; the bonus row last if L = gamma).
__device__ __forceinline__ int early_rows_upto(const VerifyParams& p, int L) {
    return L < p.gamma ? 2 * (L + 1) : 2 * p.gamma + 1;
}

// Row task descriptor b * R + r of initial slot q: positions 0..early_L0 of every sequence.
__device__ __forceinline__ int early_initial_task(const VerifyParams& p, int q) {
    const int R = 2 * p.gamma + 1;
    const int per = early_rows_upto(p, p.early_L0);
    const int b = q / per, m = q % per;
    const int k = m >> 1;
    return b * R + ((m & 1) ? p.gamma + 1 + k : k);
}

// Lane 0 waits (bounded) for queue slot `slot`; returns its value, or kTaskEmpty once
// *done reaches B (the slot will never be written) or the wait gave up.  Polls back off
// from 64 ns to 1 us, and look at *done (one word every waiting warp reads) every fourth
// time only.
__device__ __forceinline__ int early_wait_slot(const VerifyParams& p, const int* slot,
                                               const int* done) {
    int d = ld_acquire(slot);
    if (d != kTaskEmpty) return d;
    const unsigned long long t0 = global_time_ns();
    unsigned sleep_ns = 64;
    for (unsigned it = 0;; ++it) {
        if ((it & 3) == 3 && ld_relaxed(done) >= p.B) return kTaskEmpty;
        if (global_time_ns() - t0 > kWaitLimitNs) {
            set_status(p.status, 4 /* SPEC_ETIMEOUT */);
            return kTaskEmpty;
        }
        __nanosleep(sleep_ns);
        if (sleep_ns < 1024) sleep_ns *= 2;
        if ((d = ld_acquire(slot)) != kTaskEmpty) return d;
    }
}

// Lane 0: queue the rows of every position of sequence b up to `hi` not queued yet.
__device__ __forceinline__ void early_enqueue_upto(const VerifyParams& p, int b, int hi) {
    const int R = 2 * p.gamma + 1;
    const int old = atomicMax(p.enq_pos + b, hi - p.early_L0) + p.early_L0;
    if (hi <= old) return;
    const int n = early_rows_upto(p, hi) - early_rows_upto(p, old);
    int q = atomicAdd(p.task_tail, n);
    for (int k = old + 1; k <= hi; ++k) {
        if (sv_in_range(p, q, p.caps.task)) st_relaxed(p.task + q, b * R + k);
        ++q;
        if (k < p.gamma) {
            if (sv_in_range(p, q, p.caps.task)) st_relaxed(p.task + q, b * R + p.gamma + 1 + k);
            ++q;
        }
    }
}

// Warp: a finished sequence with a bad draft token (no race).
__device__ __forceinline__ void early_finish_bad(const VerifyParams& p, int b, int lane) {
    int32_t* out = p.out_tokens + static_cast<long long>(b) * (p.gamma + 1);
    for (int t = lane; t <= p.gamma; t += 32) out[t] = -1;
    if (lane == 0) {
        p.out_n[b] = -1;
        set_status(p.status, 3 /* SPEC_EBADTOKEN */);
        atomicAdd(p.seq_finished, 1);
        atomicAdd(p.seq_decided, 1);
    }
}

// Warp: sequence b is decided at j (first rejection, or gamma): outputs, then its race.
__device__ __forceinline__ void early_finish(const VerifyParams& p, int b, int j, float mp,
                                             float l2sp, float mq, float l2sq, int lane) {
    int32_t* out = p.out_tokens + static_cast<long long>(b) * (p.gamma + 1);
    const int32_t* tok = p.tokens + static_cast<long long>(b) * p.gamma;
    for (int t = lane; t <= p.gamma; t += 32)
        if (t != j) out[t] = t < j ? tok[t] : -1;
    if (lane == 0) {
        SeqInfo si;
        si.j = j;
        si.mp = mp;
        si.l2sp = l2sp;
        si.mq = mq;
        si.l2sq = l2sq;
        si.cp = scale_of(seq_T(p, b));
        si.cq = scale_of(seq_Td(p, b));
        si.pad = 0;
        p.seq[b] = si;
        p.out_n[b] = j;
        // the race reads seq[b] after acquiring this slot
        const int rs = atomicAdd(p.race_tail, 1);
        if (sv_in_range(p, rs, p.caps.race_task)) st_release(p.race_task + rs, b);
        atomicAdd(p.seq_decided, 1);
    }
}

// Count one event of an early-exit task (a row piece arrived, a row merged, a position
// accepted).  Over host memory with a mirror, the count also hands the mirror's contents to
// whoever acts on it: a fence before the increment (the writer's release) and one after (the
// reader's acquire), so the rows a sequence's race reads from the mirror were written before
// its race task was published.
__device__ __forceinline__ int early_event(const VerifyParams& p, int* addr) {
    if (!p.mirror_target) return atomicAdd(addr, 1);
    __threadfence();
    const int t = atomicAdd(addr, 1);
    __threadfence();
    return t;
}

// On acceptance at position i, queue (i+1)*g/4 extra positions ahead.  Throughput workload
// (16 KB units), us per call with g = 0 / 1 / 2 / 3 / 4: 152.4 / 152.4 / 145.7 / 149.0 / 162.3;
// the smaller workloads within 1 us of each other.  Rows in host memory read none ahead
// (g = 0): over the host link the rows read past a rejection cost as much as the others
// (1.80e6 rows/s end to end with g = 0, 1.53e6 with g = 2).
#ifndef SPECVERIFY_EARLY_GROWTH
#define SPECVERIFY_EARLY_GROWTH 2
#endif
constexpr int kEarlyGrowth = SPECVERIFY_EARLY_GROWTH;

// Warp: position i of sequence b is complete (its rows merged, the previous position
// accepted) -- decide it, and go on through the following positions while they are complete
// too.  On acceptance later positions are queued ahead of their decisions: a number that
// grows with the accepted prefix (so a long accepted draft needs few decide-and-queue round
// trips), and more when too few sequences are left undecided to keep the row warps busy.
// Rows read past a rejection are wasted; the growth bounds them by the rows the sequence
// needed.
template <class ET>
__device__ __forceinline__ void early_decide_from(const VerifyParams& p, int b, int i, int lane) {
    using S = typename ET::storage;
    const int R = 2 * p.gamma + 1;
    const int32_t* tok = p.tokens + static_cast<long long>(b) * p.gamma;
    const float2* rs = p.row_stat + static_cast<long long>(b) * R;
    if (i == 0) {  // any draft token outside [0, V) marks the whole sequence
        bool bad = false;
        for (int t = lane; t < p.gamma; t += 32) bad |= (tok[t] < 0 || tok[t] >= p.V);
        if (__any_sync(0xffffffffu, bad)) {
            early_finish_bad(p, b, lane);
            return;
        }
    }
    for (;;) {
        float2 sp = make_float2(0.0f, 0.0f), sq = make_float2(0.0f, 0.0f);
        int accept = 0;
        if (lane == 0) {
            sp = wait_stat(p, rs + i);
            if (i < p.gamma) {
                sq = wait_stat(p, rs + p.gamma + 1 + i);
                const int d = tok[i];
                const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
                const float u = accept_uniform(p.key, bg, static_cast<uint32_t>(i));
                const long long kt = (static_cast<long long>(b) * (p.gamma + 1) + i) * p.V + d;
                const long long kd = (static_cast<long long>(b) * p.gamma + i) * p.V + d;
                const float xt = sv_in_range(p, kt, p.caps.target) ? ET::load1(static_cast<const S*>(p.target) + kt) : 0.0f;
                const float xd = sv_in_range(p, kd, p.caps.draft) ? ET::load1(static_cast<const S*>(p.draft) + kd) : 0.0f;
                const float l2p = fmaf(xt, scale_of(seq_T(p, b)), -sp.x) - sp.y;
                const float l2q = fmaf(xd, scale_of(seq_Td(p, b)), -sq.x) - sq.y;
                // accept iff u < min(1, p/q); p(d) = 0 rejects, q(d) = 0 < p(d) accepts
                accept = (l2p > -INFINITY) && (u < exp2f(l2p - l2q));
            }
        }
        accept = __shfl_sync(0xffffffffu, accept, 0);
        if (!accept) {  // rejected at i, or i = gamma: the bonus row
            sp.x = __shfl_sync(0xffffffffu, sp.x, 0);
            sp.y = __shfl_sync(0xffffffffu, sp.y, 0);
            sq.x = __shfl_sync(0xffffffffu, sq.x, 0);
            sq.y = __shfl_sync(0xffffffffu, sq.y, 0);
            early_finish(p, b, i, sp.x, sp.y, i < p.gamma ? sq.x : 0.0f, i < p.gamma ? sq.y : 0.0f, lane);
            return;
        }
        int t = 0;
        if (lane == 0) {
            const int undecided = max(1, p.B - ld_relaxed(p.seq_decided));
            const int fill = (p.early_fill + undecided - 1) / undecided;
            const int grow = ((i + 1) * p.early_growth) >> 2;
            early_enqueue_upto(p, b, min(p.gamma, i + max(1, max(fill, 1 + grow))));
            t = early_event(p, p.pos_done + static_cast<long long>(b) * (p.gamma + 1) + i + 1);
        }
        t = __shfl_sync(0xffffffffu, t, 0);
        ++i;
        if (t != early_events_of(p, i) - 1) return;  // the last row of position i decides it
    }
}

// Warp: the last piece of row r of sequence b arrived -- merge the row; if that completes
// its position, decide.
template <class ET>
__device__ __forceinline__ void early_row_done(const VerifyParams& p, int b, int r, int lane) {
    const int R = 2 * p.gamma + 1;
    SoftmaxStat st{-FLT_MAX, 0.0f};
    const long long pbase = (static_cast<long long>(b) * R + r) * p.npieces;
    const float2* parts = p.stat_parts + pbase;
    if (!(sv_span_in_range(p, pbase, p.npieces, p.caps.stat) &&
          sv_span_in_range(p, static_cast<long long>(b) * R, R, p.caps.row_stat) &&
          sv_span_in_range(p, static_cast<long long>(b) * (p.gamma + 1), p.gamma + 1, p.caps.pos)))
        return;
    for (int k = lane; k < p.npieces; k += 32) {
        const float2 q = wait_stat(p, parts + k);
        st = merge_stat(st, SoftmaxStat{q.x, q.y});
    }
    st = warp_merge_stat(st);
    const int i = r <= p.gamma ? r : r - p.gamma - 1;
    int t = 0;
    if (lane == 0) {
        store_stat(p.row_stat + static_cast<long long>(b) * R + r, st.m, log2f(st.s));
        t = early_event(p, p.pos_done + static_cast<long long>(b) * (p.gamma + 1) + i);
    }
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t == early_events_of(p, i) - 1) early_decide_from<ET>(p, b, i, lane);
}

// Warp: one race unit (piece `piece` of the raced row of sequence b).
template <class ET>
__device__ __forceinline__ void early_race_unit(const VerifyParams& p, int b, int piece, int lane) {
    using S = typename ET::storage;
    SeqInfo si;
    {
        const int4 a = __ldcg(reinterpret_cast<const int4*>(p.seq + b));
        const float4 q = __ldcg(reinterpret_cast<const float4*>(p.seq + b) + 1);
        si.j = a.x;
        si.mp = __int_as_float(a.y);
        si.l2sp = __int_as_float(a.z);
        si.mq = __int_as_float(a.w);
        si.l2sq = q.x;
        si.cp = q.y;
        si.cq = q.z;
        si.pad = 0;
    }
    const int j = si.j;
    const bool residual = j < p.gamma;
    // the raced rows were streamed (and, over host memory, mirrored on the device) before
    // the sequence was decided
    const S* tb = static_cast<const S*>(p.mirror_target ? p.mirror_target : p.target);
    const S* db = static_cast<const S*>(p.mirror_target ? p.mirror_draft : p.draft);
    const S* rt = tb + (static_cast<long long>(b) * (p.gamma + 1) + j) * p.V;
    const S* rd = residual ? db + (static_cast<long long>(b) * p.gamma + j) * p.V : nullptr;
    const uint32_t bg = p.seq_base + static_cast<uint32_t>(b);
    const int x0 = piece * p.piece_len;
    const int x1 = min(p.V, x0 + p.piece_len);
    if (!(sv_span_in_range(p, (static_cast<long long>(b) * (p.gamma + 1) + j) * p.V, p.V, p.caps.target) &&
          (!residual || sv_span_in_range(p, (static_cast<long long>(b) * p.gamma + j) * p.V, p.V, p.caps.draft)) &&
          sv_span_in_range(p, static_cast<long long>(b) * p.npieces, p.npieces, p.caps.early_race) &&
          sv_in_range(p, static_cast<long long>(b) * (p.gamma + 1) + j, p.caps.out_tokens)))
        return;
    const RaceState st = race_piece<ET>(rt, rd, x0, x1, si, residual, p.rk, bg,
                                        static_cast<uint32_t>(j), lane);
    unsigned long long* parts = p.early_race + static_cast<long long>(b) * p.npieces;
    int t = 0;
    if (lane == 0) {
        // never zero: the index field is idx + 1.  (kDebugNeverReady, tests only: no unit
        // publishes its winner, so the last unit's bounded wait below runs out.)
        if (!(p.debug_flags & kDebugNeverReady)) parts[piece] = pack_race(st.best, st.idx);
        t = atomicAdd(p.race_done + b, 1);
    }
    t = __shfl_sync(0xffffffffu, t, 0);
    if (t != p.npieces - 1) return;
    // the sequence's last race unit: merge every unit's winner, waiting (bounded) for each
    RaceState m{-INFINITY, INT_MAX, -INFINITY};
    for (int k = lane; k < p.npieces; k += 32) {
        unsigned long long v = ld_relaxed_u64(parts + k);
        if (v == 0ull) {
            const unsigned long long t0 = global_time_ns();
            while ((v = ld_relaxed_u64(parts + k)) == 0ull) {
                if (global_time_ns() - t0 > kWaitLimitNs) break;
                __nanosleep(64);
            }
            if (v == 0ull) set_status(p.status, 4 /* SPEC_ETIMEOUT */);
        }
        if (v != 0ull)
            m = race_merge(m, RaceState{__uint_as_float(static_cast<uint32_t>(v)),
                                        static_cast<int>(static_cast<uint32_t>(v >> 32) - 1u),
                                        -INFINITY});
    }
    m = warp_race_merge(m);
    if (m.idx == INT_MAX) {
        // Every residual weight was zero (p <= q everywhere in fp32): draw from p_j.
        m = race_piece<ET>(rt, nullptr, 0, p.V, si, false, p.rk, bg, static_cast<uint32_t>(j), lane);
    }
    if (lane == 0) {
        p.out_tokens[static_cast<long long>(b) * (p.gamma + 1) + j] = m.idx;
        atomicAdd(p.seq_finished, 1);
    }
}

#ifndef SPECVERIFY_EARLY_MINBLOCKS
#define SPECVERIFY_EARLY_MINBLOCKS 2
#endif
#ifndef SPECVERIFY_EARLY_UNROLL
#define SPECVERIFY_EARLY_UNROLL 8
#endif
constexpr int kEarlyUnroll = SPECVERIFY_EARLY_UNROLL;

#ifndef SPECVERIFY_EARLY_RACE_WARPS
#define SPECVERIFY_EARLY_RACE_WARPS 2
#endif
constexpr int kEarlyRaceWarps = SPECVERIFY_EARLY_RACE_WARPS;  // of the 8 warps of a block

// Fill a[0, na) with fa and b[0, nb) with fb (8-byte words) before a launch that depends on
// them.  Launched as a programmatic dependent of the kernel before it, it waits for that one,
// then lets its own dependent be set up while it fills.
__global__ void __launch_bounds__(256) prep_fill_kernel(unsigned long long* a, long long na,
                                                        unsigned long long fa, unsigned long long* b,
                                                        long long nb, unsigned long long fb) {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;");
    const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
    for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < na + nb; i += stride) {
        if (i < na)
            a[i] = fa;
        else
            b[i - na] = fb;
    }
}

template <class ET, int U>
__global__ void __launch_bounds__(256, SPECVERIFY_EARLY_MINBLOCKS) verify_early_kernel(VerifyParams p) {
    using S = typename ET::storage;
    const int lane = threadIdx.x & 31;
    asm volatile("griddepcontrol.wait;" ::: "memory");  // the workspace fill (prep_fill_kernel)
    asm volatile("griddepcontrol.launch_dependents;");   // (see scan_greedy_kernel)
    const int R = 2 * p.gamma + 1;
    const int np = p.npieces;
    if ((threadIdx.x >> 5) < 8 - kEarlyRaceWarps) {
        // row units, until every sequence is decided
        const long long units_cap = static_cast<long long>(p.n_init + p.task_cap) * np;
        for (;;) {
            long long c = 0;
            if (lane == 0) c = static_cast<long long>(atomicAdd(p.unit_cursor, 1ull));
            c = __shfl_sync(0xffffffffu, c, 0);
            if (c >= units_cap) break;
            const int q = static_cast<int>(c / np);
            const int piece = static_cast<int>(c % np);
            int d;
            if (q < p.n_init) {
                d = early_initial_task(p, q);
            } else {
                d = 0;
                if (!sv_in_range(p, q - p.n_init, p.caps.task)) break;
                if (lane == 0) d = early_wait_slot(p, p.task + (q - p.n_init), p.seq_decided);
                d = __shfl_sync(0xffffffffu, d, 0);
                if (d == kTaskEmpty) break;
            }
            const int b = d / R, r = d % R;
#ifdef SPECVERIFY_CHECKED
            if (!(sv_in_range(p, static_cast<long long>(d) * np + piece, p.caps.stat) &&
                  sv_in_range(p, d, p.caps.rowarr) &&
                  sv_span_in_range(p, (r <= p.gamma ? static_cast<long long>(b) * (p.gamma + 1) + r
                                                     : static_cast<long long>(b) * p.gamma + (r - p.gamma - 1)) * p.V +
                                          static_cast<long long>(piece) * p.piece_len,
                                   min(p.V - piece * p.piece_len, p.piece_len),
                                   r <= p.gamma ? p.caps.target : p.caps.draft)))
                continue;
#endif
            const S* row;
            float cs;
            if (r <= p.gamma) {
                row = static_cast<const S*>(p.target) + (static_cast<long long>(b) * (p.gamma + 1) + r) * p.V;
                cs = scale_of(seq_T(p, b));
            } else {
                row = static_cast<const S*>(p.draft) +
                      (static_cast<long long>(b) * p.gamma + (r - p.gamma - 1)) * p.V;
                cs = scale_of(seq_Td(p, b));
            }
            const int x0 = piece * p.piece_len;
            SoftmaxStat st;
            if (p.mirror_target) {  // keep a device copy of the row for the race
                S* mrow = r <= p.gamma
                    ? static_cast<S*>(p.mirror_target) + (static_cast<long long>(b) * (p.gamma + 1) + r) * p.V
                    : static_cast<S*>(p.mirror_draft) + (static_cast<long long>(b) * p.gamma + (r - p.gamma - 1)) * p.V;
                st = stats_piece<ET, U, U, true>(row, x0, min(p.V, x0 + p.piece_len), cs, lane, mrow);
            } else {
                st = stats_piece<ET, U>(row, x0, min(p.V, x0 + p.piece_len), cs, lane);
            }
            int t = 0;
            if (lane == 0) {
                store_stat(p.stat_parts + static_cast<long long>(d) * np + piece, st.m, st.s);
                t = early_event(p, p.row_arrivals + d);
            }
            t = __shfl_sync(0xffffffffu, t, 0);
            if (t == np - 1) early_row_done<ET>(p, b, r, lane);
        }
    }
    // race units, until every sequence is finished
    const long long race_cap = static_cast<long long>(p.B) * np;
    for (;;) {
        long long c = 0;
        if (lane == 0) c = static_cast<long long>(atomicAdd(p.race_unit_cursor, 1ull));
        c = __shfl_sync(0xffffffffu, c, 0);
        if (c >= race_cap) break;
        int b = 0;
        if (!sv_in_range(p, c / np, p.caps.race_task)) break;
        if (lane == 0) b = early_wait_slot(p, p.race_task + c / np, p.seq_finished);
        b = __shfl_sync(0xffffffffu, b, 0);
        __syncwarp();  // the other lanes' reads of seq[b] follow lane 0's acquire
        if (b == kTaskEmpty) break;
        early_race_unit<ET>(p, b, static_cast<int>(c % np), lane);
    }
}

}  // namespace specverify
