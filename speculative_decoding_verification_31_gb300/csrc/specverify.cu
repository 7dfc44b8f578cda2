// specverify.cu -- host side of libspecverify: argument checks, workspace, launches.
//
// The C ABI is declared in include/specverify.h; the kernels are in kernels.cuh.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "kernels.cuh"
#include "vocab.cuh"
#include "lmhead.cuh"
#include "specverify.h"

using namespace specverify;

namespace {

constexpr int kMaxGamma = 2048;          // the scan keeps 2*gamma+1 row statistics in shared memory
constexpr int kThreads = 256;
#ifndef SPECVERIFY_UNROLL
#define SPECVERIFY_UNROLL 8
#endif
constexpr int kUnroll = SPECVERIFY_UNROLL;  // 16-byte loads in flight per lane in the streaming pass
constexpr int kMaxDevices = 64;

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

int elem_bytes(int dtype) { return dtype == SPEC_F32 ? 4 : 2; }

struct Layout {
    int piece_len, npieces;
    int rpieces;
    size_t stat_off, ext_off, seq_off, race_off, ticket_off;
    size_t tree_off;                    // token-tree verify: the node each sequence races
    int e_n_init, e_task_cap;           // early-exit path (verify_early_kernel)
    size_t e_rowstat_off, e_task_off, e_stat_off, e_zero_off, e_cursor_off, e_tail_off,
        e_finished_off, e_rowarr_off, e_pos_off, e_racedone_off, e_race_off, e_racetask_off,
        e_racecursor_off, e_racetail_off, e_decided_off, e_enq_off;
    size_t total;
};

// Pieces per row for the streaming pass (see pick_piece_len); stream_warps = 0 takes the
// default piece size (for sizing the workspace, which is allocated for the most pieces).
void choose_pieces(int B, int gamma, int V, int dtype, long long stream_warps, int* len, int* np) {
    const long long rows = static_cast<long long>(B) * (2 * gamma + 1);
    *len = pick_piece_len(rows, V, elem_bytes(dtype), stream_warps);
    *np = (V + *len - 1) / *len;
}

Layout layout_of(int B, int gamma, int V, int dtype, long long stream_warps = 0) {
    Layout L{};
    choose_pieces(B, gamma, V, dtype, stream_warps, &L.piece_len, &L.npieces);
    // the workspace always holds the most pieces any choice can give
    const int max_np = (V + kMinPieceBytes / elem_bytes(dtype) - 1) / (kMinPieceBytes / elem_bytes(dtype));
    // race pieces: one block of kRaceBlockTokens tokens each
    L.rpieces = (V + kRaceBlockTokens - 1) / kRaceBlockTokens;
    const size_t R = 2 * static_cast<size_t>(gamma) + 1;
    size_t off = 0;
    L.stat_off = off;
    off = align_up(off + static_cast<size_t>(B) * R * max_np * sizeof(float2), 256);
    L.ext_off = off;  // per-position statistics: entropy and cross terms per row piece
    off = align_up(off + static_cast<size_t>(B) * R * max_np * sizeof(float2) + 16, 256);
    L.seq_off = off;
    off = align_up(off + static_cast<size_t>(B) * sizeof(SeqInfo), 256);
    L.race_off = off;
    off = align_up(off + static_cast<size_t>(B) * race_slots(L.rpieces) * sizeof(RacePart), 256);
    L.ticket_off = off;
    off = align_up(off + static_cast<size_t>(B) * sizeof(int), 256);
    L.tree_off = off;
    off = align_up(off + static_cast<size_t>(B) * sizeof(TreeRace), 256);
    // early-exit region: a block filled with 0xFF before each call (merged rows, task queue,
    // then the row partials, last so that only the pieces in use need filling), then a
    // zeroed block (counters, then the race winners)
    L.e_n_init = gamma > 0 ? 2 * B : B;     // the fewest initial row tasks (launch_early may
    L.e_task_cap = B * (2 * gamma + 1) - L.e_n_init;  // queue more): the queue's capacity
    L.e_rowstat_off = off;
    off += static_cast<size_t>(B) * R * sizeof(float2);
    L.e_task_off = off;
    off += static_cast<size_t>(L.e_task_cap) * sizeof(int);
    L.e_racetask_off = off;
    off = align_up(off + static_cast<size_t>(B) * sizeof(int), 8);
    L.e_stat_off = off;
    off = align_up(off + static_cast<size_t>(B) * R * max_np * sizeof(float2), 256);
    L.e_zero_off = off;
    // each counter on its own 128-byte line: waiting warps poll two of them, and claims and
    // appends update the others
    L.e_cursor_off = off;
    off += 128;
    L.e_tail_off = off;
    off += 128;
    L.e_finished_off = off;
    off += 128;
    L.e_racecursor_off = off;
    off += 128;
    L.e_racetail_off = off;
    off += 128;
    L.e_decided_off = off;
    off += 128;
    L.e_rowarr_off = off;
    off += static_cast<size_t>(B) * R * sizeof(int);
    L.e_pos_off = off;
    off += static_cast<size_t>(B) * (gamma + 1) * sizeof(int);
    L.e_enq_off = off;
    off += static_cast<size_t>(B) * sizeof(int);
    L.e_racedone_off = off;
    off += static_cast<size_t>(B) * sizeof(int);
    off = align_up(off, 8);
    L.e_race_off = off;
    off = align_up(off + static_cast<size_t>(B) * max_np * sizeof(unsigned long long), 256);
    L.total = off;
    return L;
}

struct DeviceState {
    bool init = false;
    int sm_count = 0;
    int coop = 0;               // cooperative launch supported
    long long stream_warps[2] = {0, 0};  // warps of a full streaming grid, per dtype
    void* ws = nullptr;
    size_t ws_bytes = 0;
    void* mirror = nullptr;     // spec_verify_host: device copies of the rows it streams
    size_t mirror_bytes = 0;
    int32_t* status = nullptr;  // library status word (its own allocation)
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

int current_device(int* dev) {
    if (cudaGetDevice(dev) != cudaSuccess) return SPEC_ECUDA;
    if (*dev < 0 || *dev >= kMaxDevices) return SPEC_EINVAL;
    return SPEC_OK;
}

// Per-device state; allocates the status word on first use.  Caller holds g_mu.
int device_state(DeviceState** out) {
    int dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    DeviceState& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SPEC_ECUDA;
        if (cudaDeviceGetAttribute(&d.coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
            return SPEC_ECUDA;
        if (cudaMalloc(&d.status, sizeof(int32_t)) != cudaSuccess) return SPEC_ENOMEM;
        if (cudaMemset(d.status, 0, sizeof(int32_t)) != cudaSuccess) return SPEC_ECUDA;
        d.init = true;
    }
    *out = &d;
    return SPEC_OK;
}

// Grow the library workspace of this device to `bytes` (zero-filled).  Caller holds g_mu.
int ensure_workspace(DeviceState& d, size_t bytes) {
    if (d.ws_bytes >= bytes) return SPEC_OK;
    if (d.ws) {
        cudaDeviceSynchronize();
        cudaFree(d.ws);
        d.ws = nullptr;
        d.ws_bytes = 0;
    }
    if (cudaMalloc(&d.ws, bytes) != cudaSuccess) return SPEC_ENOMEM;
    if (cudaMemset(d.ws, 0, bytes) != cudaSuccess) return SPEC_ECUDA;
    d.ws_bytes = bytes;
    return SPEC_OK;
}

// Grow the host path's row mirror to `bytes`; false (and no mirror) if that fails.  Caller
// holds g_mu.
bool ensure_mirror(DeviceState& d, size_t bytes) {
    if (d.mirror_bytes >= bytes) return true;
    if (d.mirror) {
        cudaDeviceSynchronize();
        cudaFree(d.mirror);
        d.mirror = nullptr;
        d.mirror_bytes = 0;
    }
    if (cudaMalloc(&d.mirror, bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        d.mirror = nullptr;
        return false;
    }
    d.mirror_bytes = bytes;
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr uint32_t kKnownFlags = SPEC_DEBUG_NEVER_READY | SPEC_FLAG_EARLY_EXIT | SPEC_FLAG_FULL_READ;

bool good_temperature(float t) { return std::isfinite(t) && t > 0.0f; }

// Resident blocks per SM of `kernel` at `threads` threads and `smem` bytes of dynamic shared
// memory on the current device, or 0 if the query fails.  The answer cannot change within a
// process, and the query costs host microseconds on every call, so each (device, kernel,
// threads, smem) is queried once and kept.
struct OccupancyEntry {
    int dev, threads, value;
    const void* fn;
    size_t smem;
};
std::mutex g_occ_mu;
OccupancyEntry g_occ[64];
int g_occ_n = 0;

template <class K>
int blocks_per_sm(K kernel, int threads, size_t smem) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    const void* fn = reinterpret_cast<const void*>(kernel);
    std::lock_guard<std::mutex> lock(g_occ_mu);
    for (int i = 0; i < g_occ_n; ++i)
        if (g_occ[i].fn == fn && g_occ[i].dev == dev && g_occ[i].threads == threads && g_occ[i].smem == smem)
            return g_occ[i].value;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem) != cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    if (g_occ_n < 64) g_occ[g_occ_n++] = OccupancyEntry{dev, threads, per_sm, fn, smem};
    return per_sm;
}

// Launch of a streaming kernel: one block of kStreamThreads per SM (the claiming variant kc,
// whose warps share the block's items) when the items outnumber the warps of that grid;
// otherwise blocks of kThreads of the plain variant kp, one item per warp, so that a small
// call starts few threads and spreads its items over as many SMs as it can.  The launch is a
// programmatic dependent of the kernel before it on the stream (the kernel waits for that one
// to finish before touching memory), so its blocks are set up while the previous verify's
// last kernel drains.
template <class KC, class KP, class... A>
cudaError_t launch_stream(KC kc, KP kp, int sm_count, long long items, cudaStream_t s, A... args) {
    int per_sm = blocks_per_sm(kc, kStreamThreads, 0);
    if (per_sm < 1) per_sm = 1;
    const long long full = static_cast<long long>(sm_count) * per_sm;
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const bool claim = items >= full * (kStreamThreads / 32);
    const long long g = claim ? full : (items + (kThreads / 32) - 1) / (kThreads / 32);
    cfg.gridDim = dim3(static_cast<unsigned>(g < 1 ? 1 : g));
    cfg.blockDim = dim3(claim ? kStreamThreads : kThreads);
    cudaError_t e = claim ? cudaLaunchKernelEx(&cfg, kc, args...) : cudaLaunchKernelEx(&cfg, kp, args...);
    if (e != cudaSuccess) {  // a device without programmatic launches: a plain one
        cudaGetLastError();
        cfg.numAttrs = 0;
        e = claim ? cudaLaunchKernelEx(&cfg, kc, args...) : cudaLaunchKernelEx(&cfg, kp, args...);
    }
    return e;
}

// Warps of the streaming kernel's full grid.
long long stream_warps_of(int sm_count, int dtype) {
    int per_sm = dtype == SPEC_F32 ? blocks_per_sm(row_stats_kernel<F32Elem, kUnroll, true>, kStreamThreads, 0)
                                   : blocks_per_sm(row_stats_kernel<Bf16Elem, kUnroll, true>, kStreamThreads, 0);
    if (per_sm < 1) per_sm = 1;
    return static_cast<long long>(sm_count) * per_sm * (kStreamThreads / 32);
}

void record(const spec_verify_opts* o, int k, cudaStream_t s) {
    if (o && o->prof_events[k]) cudaEventRecord(static_cast<cudaEvent_t>(o->prof_events[k]), s);
}

// Element counts of the buffers the call's kernels index (checked by the index-checked
// build): the caller's tensors from the problem's sizes, the workspace regions from the
// layout.
void set_caps(VerifyParams& p, const Layout& L, int B, int gamma, int V) {
    const long long R = 2LL * gamma + 1;
    p.caps.target = static_cast<long long>(B) * (gamma + 1) * V;
    p.caps.draft = static_cast<long long>(B) * gamma * V;
    p.caps.tokens = static_cast<long long>(B) * gamma;
    p.caps.out_tokens = static_cast<long long>(B) * (gamma + 1);
    p.caps.stat = static_cast<long long>((L.ext_off - L.stat_off) / sizeof(float2));
    p.caps.race = static_cast<long long>((L.ticket_off - L.race_off) / sizeof(RacePart));
    p.caps.row_stat = B * R;
    p.caps.pos = static_cast<long long>(B) * (gamma + 1);
    p.caps.rowarr = B * R;
    p.caps.task = L.e_task_cap;
    p.caps.race_task = B;
    p.caps.early_race = static_cast<long long>((L.total - L.e_race_off) / sizeof(unsigned long long));
}

void bind_workspace(VerifyParams& p, const Layout& L, char* ws) {
    p.piece_len = L.piece_len;
    p.npieces = L.npieces;
    p.rpieces = L.rpieces;
    p.stat_parts = reinterpret_cast<float2*>(ws + L.stat_off);
    p.ext_parts = reinterpret_cast<float2*>(ws + L.ext_off);
    p.seq = reinterpret_cast<SeqInfo*>(ws + L.seq_off);
    p.race_parts = reinterpret_cast<RacePart*>(ws + L.race_off);
    p.tickets = reinterpret_cast<int*>(ws + L.ticket_off);
    p.tree_race = reinterpret_cast<TreeRace*>(ws + L.tree_off);
}

// Validated common set-up of a call: fills `p` with the workspace pointers.
int prepare(int B, int gamma, int V, int dtype, const spec_verify_opts* o, VerifyParams& p,
            DeviceState** dstate, char** ws_out = nullptr) {
    std::lock_guard<std::mutex> lock(g_mu);
    int rc = device_state(dstate);
    if (rc) return rc;
    long long& sw = (*dstate)->stream_warps[dtype == SPEC_F32 ? 0 : 1];
    if (sw == 0) sw = stream_warps_of((*dstate)->sm_count, dtype);
    const Layout L = layout_of(B, gamma, V, dtype, sw);
    char* ws;
    if (o && o->workspace) {
        if (o->workspace_bytes < L.total) return SPEC_ENOMEM;
        if (!aligned16(o->workspace)) return SPEC_EINVAL;
        ws = static_cast<char*>(o->workspace);
    } else {
        rc = ensure_workspace(**dstate, L.total);
        if (rc) return rc;
        ws = static_cast<char*>((*dstate)->ws);
    }
    bind_workspace(p, L, ws);
    set_caps(p, L, B, gamma, V);
    p.status = (o && o->d_status) ? o->d_status : (*dstate)->status;
    if (ws_out) *ws_out = ws;
    return SPEC_OK;
}

int check_common(const void* target, const int32_t* out_tokens, const int32_t* out_n, int B,
                 int gamma, int V, int dtype) {
    if (B < 0 || gamma < 0 || gamma > kMaxGamma || V < 1) return SPEC_EINVAL;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_EINVAL;
    if (static_cast<long long>(B) * (gamma + 1) * static_cast<long long>(V) >= (1LL << 40))
        return SPEC_EINVAL;
    if (B == 0) return SPEC_OK;
    if (!target || !out_tokens || !out_n) return SPEC_EINVAL;
    if (!aligned16(target)) return SPEC_EINVAL;
    return SPEC_OK;
}

// Launch with programmatic stream serialization when `pdl`: the kernel may start before the
// previous one on the stream ends, and waits for it with griddepcontrol.wait.
template <class K>
cudaError_t launch_pdl(K kernel, int grid, size_t smem, cudaStream_t s, bool pdl, const VerifyParams& p) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, p);
}

// Two-kernel sampling verify: the streaming pass, then the scan-race kernel as its
// programmatic dependent (its blocks start while the streaming pass drains).
#ifndef SPECVERIFY_PAIR_UNROLL
#define SPECVERIFY_PAIR_UNROLL 4
#endif
constexpr int kPairUnroll = SPECVERIFY_PAIR_UNROLL;  // 16-byte loads per row in flight per lane

// Whether a call asks for the per-position statistics (entropies, KL, class centres).
bool wants_position_stats(const VerifyParams& p) {
    return p.out_Hp || p.out_Hq || p.out_KL || p.ctrl_centres;
}

template <class ET>
int launch_sampling(VerifyParams& p, int sm_count, const spec_verify_opts* o, cudaStream_t s) {
    const int R = 2 * p.gamma + 1;
    const bool extra = wants_position_stats(p);
    record(o, 0, s);
    const long long seq_bytes = static_cast<long long>(R) * p.V * static_cast<long long>(sizeof(typename ET::storage));
    const bool rows_aligned = (static_cast<long long>(p.V) * static_cast<long long>(sizeof(typename ET::storage))) % 16 == 0;
    if (!extra && seq_bytes <= kSmallSeqBytes && p.V <= kRaceBlockTokens && rows_aligned) {
        // small sequences: one block each does the whole verify (one launch instead of two)
        if (launch_pdl(verify_small_kernel<ET, kUnroll>, p.B, 2 * R * sizeof(float), s, true, p) != cudaSuccess)
            return SPEC_ECUDA;
        record(o, 1, s);
        record(o, 2, s);
        return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
    }
    if (extra) {  // the same read of every logit, paired by position, with the extra terms
        // pieces chosen for this pass's items (position pairs, not rows) and grid
        int per_sm = blocks_per_sm(pair_stats_kernel<ET, kPairUnroll, true>, kStreamThreads, 0);
        if (per_sm < 1) per_sm = 1;
        p.piece_len = pick_piece_len(static_cast<long long>(p.B) * (p.gamma + 1), p.V,
                                     static_cast<int>(sizeof(typename ET::storage)),
                                     static_cast<long long>(sm_count) * per_sm * (kStreamThreads / 32));
        p.npieces = (p.V + p.piece_len - 1) / p.piece_len;
        const long long items = static_cast<long long>(p.B) * (p.gamma + 1) * p.npieces;
        if (launch_stream(pair_stats_kernel<ET, kPairUnroll, true>, pair_stats_kernel<ET, kPairUnroll, false>,
                      sm_count, items, s, p) != cudaSuccess)
            return SPEC_ECUDA;
    } else {
        const long long stat_items = static_cast<long long>(p.B) * R * p.npieces;
        if (launch_stream(row_stats_kernel<ET, kUnroll, true>, row_stats_kernel<ET, kUnroll, false>, sm_count,
                      stat_items, s, p) != cudaSuccess)
            return SPEC_ECUDA;
    }
    record(o, 1, s);
    // scan-race grid, one resident wave: G = wave / B blocks per sequence when that is at
    // least 2, or 1 when the sequences fill three quarters of the wave (every block scans one
    // sequence); else the race's B * CH chunks shared evenly over the wave, at least one
    // chunk per warp each (one block per sequence when the sequences alone fill the wave)
    long long grid;
    {
        int per_sm = blocks_per_sm(scan_race_kernel<ET>, kThreads, 2 * R * sizeof(float));
        if (per_sm < 1) per_sm = 1;
        const long long wave = static_cast<long long>(sm_count) * per_sm;
        const long long steps = static_cast<long long>(p.B) * ((p.V + kRaceWarpTokens - 1) / kRaceWarpTokens) /
                                kRaceBlockChunks;
        long long G = wave / p.B;
        if (G > p.rpieces) G = p.rpieces;
        // one block per sequence (G = 1) also when the sequences nearly fill the wave: shared
        // evenly, most blocks would straddle two sequences and scan both (throughput
        // workload, B = 256 on a 304-block wave: 57.9 -> 55.9 us)
        const bool whole = G == 1 && 4 * p.B >= 3 * wave;
        if (G >= 2 || whole) {
            p.rgroups = static_cast<int>(G);
            grid = p.B * G;
        } else {
            p.rgroups = 0;
            grid = p.B >= wave ? p.B : std::max<long long>(p.B, std::min(wave, steps));
        }
    }
    // (no PDL when an event is recorded between the kernels, so that each one is timed alone)
    if (launch_pdl(scan_race_kernel<ET>, static_cast<int>(grid), 2 * R * sizeof(float), s,
                   !(o && o->prof_events[1]), p) != cudaSuccess)
        return SPEC_ECUDA;
    record(o, 2, s);
    if (extra) {
        if (launch_pdl(position_stats_kernel, p.B, static_cast<size_t>(p.gamma) * sizeof(float), s,
                       !(o && o->prof_events[2]), p) != cudaSuccess)
            return SPEC_ECUDA;
        record(o, 3, s);
    }
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

// Early-exit sampling verify: fill the queue and the row partials with empty markers, zero
// the counters, then one cooperative launch (every block resident; the warps wait only for
// work that warps which never wait will publish).
template <class ET>
int launch_early(VerifyParams& p, int sm_count, const spec_verify_opts* o, cudaStream_t s,
                 const Layout& L, char* ws, bool host_rows) {
    auto kernel = verify_early_kernel<ET, kEarlyUnroll>;
    const int per_sm = blocks_per_sm(kernel, kThreads, 0);
    if (per_sm < 1) return SPEC_ECUDA;
    const int R = 2 * p.gamma + 1;
    const long long row_warps = static_cast<long long>(sm_count) * per_sm * (8 - kEarlyRaceWarps);
    // pieces: the largest of kEarlyPieceBytes x {2, 1.5, 1} that still gives every row warp
    // two units among the rows all sequences start with (larger units cost less per byte; a
    // few sequences need small ones to spread each row over many warps).  Measured per call:
    // throughput workload 167.5 / 155.0 / 152.1 us with 8 / 12 / 16 KB; single sequence
    // 32.6 / 37.0 / 40.2 us.  Rows in host memory keep kEarlyPieceBytes (over the host link
    // the throughput workload measured 1.80e6 rows/s with 8 KB, 1.72e6 with 16 KB).
    const long long rows0 = static_cast<long long>(p.B) * (p.gamma > 0 ? 2 : 1);
    const int es = static_cast<int>(sizeof(typename ET::storage));
    for (int k = host_rows ? 2 : 4; k >= 2; --k) {
        p.piece_len = (kEarlyPieceBytes * k / 2) / es;
        p.npieces = (p.V + p.piece_len - 1) / p.piece_len;
        if (rows0 * p.npieces >= 2 * row_warps) break;
    }
    p.stat_parts = reinterpret_cast<float2*>(ws + L.e_stat_off);
    p.row_stat = reinterpret_cast<float2*>(ws + L.e_rowstat_off);
    p.task = reinterpret_cast<int*>(ws + L.e_task_off);
    p.pos_done = reinterpret_cast<int*>(ws + L.e_pos_off);
    p.enq_pos = reinterpret_cast<int*>(ws + L.e_enq_off);
    // positions in flight that keep the row warps busy, and the positions every sequence
    // starts with (more than position 0 only when there are too few sequences for that)
    p.early_fill = static_cast<int>(std::max(1LL, row_warps / (2LL * p.npieces)));
    p.early_growth = host_rows ? 0 : kEarlyGrowth;
    p.early_L0 = std::min(p.gamma, std::max(0, (p.early_fill + p.B - 1) / p.B - 1));
    const int per_seq = p.early_L0 < p.gamma ? 2 * (p.early_L0 + 1) : 2 * p.gamma + 1;
    p.n_init = p.B * per_seq;
    p.task_cap = p.B * R - p.n_init;
    p.unit_cursor = reinterpret_cast<unsigned long long*>(ws + L.e_cursor_off);
    p.task_tail = reinterpret_cast<int*>(ws + L.e_tail_off);
    p.seq_finished = reinterpret_cast<int*>(ws + L.e_finished_off);
    p.seq_decided = reinterpret_cast<int*>(ws + L.e_decided_off);
    p.race_task = reinterpret_cast<int*>(ws + L.e_racetask_off);
    p.race_tail = reinterpret_cast<int*>(ws + L.e_racetail_off);
    p.race_unit_cursor = reinterpret_cast<unsigned long long*>(ws + L.e_racecursor_off);
    p.row_arrivals = reinterpret_cast<int*>(ws + L.e_rowarr_off);
    p.race_done = reinterpret_cast<int*>(ws + L.e_racedone_off);
    p.early_race = reinterpret_cast<unsigned long long*>(ws + L.e_race_off);
    const size_t rows = static_cast<size_t>(p.B) * R;
    // no more warps than the units queued at the start
    long long grid = static_cast<long long>(sm_count) * per_sm;
    const long long want = (static_cast<long long>(p.n_init) * p.npieces + (kThreads / 32) - 1) /
                           (kThreads / 32);
    if (want < grid) grid = want;
    // the row statistics and their partials start empty (every bit set), the counters, events
    // and race winners zero: one small kernel, the early-exit kernel its programmatic
    // dependent (it waits for the fill with griddepcontrol.wait)
    const size_t fill_bytes = (L.e_stat_off - L.e_rowstat_off) + rows * p.npieces * sizeof(float2);
    const size_t zero_bytes = (L.e_race_off - L.e_zero_off) +
                              static_cast<size_t>(p.B) * p.npieces * sizeof(unsigned long long);
    const long long n_fill = static_cast<long long>(fill_bytes / 8), n_zero = static_cast<long long>(zero_bytes / 8);
    long long prep_grid = (n_fill + n_zero + kThreads - 1) / kThreads;
    if (prep_grid > 2LL * sm_count) prep_grid = 2LL * sm_count;
    record(o, 0, s);
    cudaLaunchConfig_t cfg = {};
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeCooperative;
    attr[1].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.gridDim = dim3(static_cast<unsigned>(prep_grid < 1 ? 1 : prep_grid));
    cfg.blockDim = dim3(kThreads);
    cfg.numAttrs = 1;
    unsigned long long* fill = reinterpret_cast<unsigned long long*>(ws + L.e_rowstat_off);
    unsigned long long* zero = reinterpret_cast<unsigned long long*>(ws + L.e_zero_off);
    if (cudaLaunchKernelEx(&cfg, prep_fill_kernel, fill, n_fill, ~0ull, zero, n_zero, 0ull) != cudaSuccess) {
        (void)cudaGetLastError();  // no programmatic launches: a plain one
        cfg.numAttrs = 0;
        if (cudaLaunchKernelEx(&cfg, prep_fill_kernel, fill, n_fill, ~0ull, zero, n_zero, 0ull) != cudaSuccess)
            return SPEC_ECUDA;
    }
    cfg.gridDim = dim3(static_cast<unsigned>(grid));
    cfg.numAttrs = 2;
    if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess) {
        (void)cudaGetLastError();  // not accepted together: a plain cooperative launch
        cfg.attrs = attr + 1;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, kernel, p) != cudaSuccess) return SPEC_ECUDA;
    }
    record(o, 1, s);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

// Token-tree verify: the streaming pass, the walk (one cluster per sequence, a programmatic
// dependent), then the race (G blocks per sequence, another dependent).
template <class ET>
int launch_tree(VerifyParams& p, const TreeShape& t, int sm_count, const spec_verify_opts* o,
                cudaStream_t s) {
    const bool pdl = !(o && o->prof_events[1]);
    record(o, 0, s);
    const long long items = static_cast<long long>(p.B) * (t.N + t.M) * p.npieces;
    if (launch_stream(tree_stats_kernel<ET, kUnroll, true>, tree_stats_kernel<ET, kUnroll, false>, sm_count, items,
                  s, p, t.N, t.M) != cudaSuccess)
        return SPEC_ECUDA;
    record(o, 1, s);
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(p.B) * kTreeCluster);  // one cluster per sequence
        cfg.blockDim = dim3(kThreads);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, tree_walk_kernel<ET>, p, t) != cudaSuccess) return SPEC_ECUDA;
    }
    record(o, 2, s);
    int per_sm = blocks_per_sm(tree_race_kernel<ET>, kThreads, 0);
    if (per_sm < 1) per_sm = 1;
    long long G = static_cast<long long>(sm_count) * per_sm / p.B;
    if (G > p.rpieces) G = p.rpieces;
    if (G < 1) G = 1;
    p.rgroups = static_cast<int>(G);
    {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(static_cast<unsigned>(p.B * G));
        cfg.blockDim = dim3(kThreads);
        cfg.stream = s;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = pdl ? 1 : 0;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        if (cudaLaunchKernelEx(&cfg, tree_race_kernel<ET>, p, t.N, t.M, t.D) != cudaSuccess)
            return SPEC_ECUDA;
    }
    record(o, 3, s);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

template <class ET>
int launch_greedy(VerifyParams& p, int sm_count, const spec_verify_opts* o, cudaStream_t s) {
    const int R = p.gamma + 1;
    record(o, 0, s);
    const long long items = static_cast<long long>(p.B) * R * p.npieces;
    if (launch_stream(row_argmax_kernel<ET, kUnroll, true>, row_argmax_kernel<ET, kUnroll, false>, sm_count,
                  items, s, p) != cudaSuccess)
        return SPEC_ECUDA;
    record(o, 1, s);
    if (launch_pdl(scan_greedy_kernel<ET>, p.B, R * sizeof(int), s, !(o && o->prof_events[1]), p) != cudaSuccess)
        return SPEC_ECUDA;
    record(o, 2, s);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // namespace

extern "C" {

void spec_verify_opts_init(spec_verify_opts* opts) {
    if (!opts) return;
    std::memset(opts, 0, sizeof(*opts));
    opts->dtype = SPEC_BF16;
}

size_t spec_verify_workspace_bytes(int B, int gamma, int V, int dtype) {
    if (B < 0 || gamma < 0 || gamma > kMaxGamma || V < 1) return 0;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return 0;
    return layout_of(B, gamma, V, dtype).total;
}

}  // extern "C"

namespace {

// spec_verify_ex, and spec_verify_host's call of it (host_rows: the logits are in host memory;
// the early-exit kernel then mirrors the rows it streams on the device for the race).
int verify_ex_impl(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                   int B, int gamma, int V, float T, float T_d, uint64_t seed, int32_t* out_tokens,
                   int32_t* out_n_accepted, const spec_verify_opts* opts, void* stream, bool host_rows) {
    const int dtype = opts ? opts->dtype : SPEC_BF16;
    int rc = check_common(target_logits, out_tokens, out_n_accepted, B, gamma, V, dtype);
    if (rc || B == 0) return rc;
    if (gamma > 0 && (!draft_logits || !draft_tokens || !aligned16(draft_logits))) return SPEC_EINVAL;
    if (!(opts && opts->T_per_seq) && !good_temperature(T)) return SPEC_EINVAL;
    if (!(opts && opts->Td_per_seq) && !good_temperature(T_d)) return SPEC_EINVAL;
    VerifyParams p{};
    p.target = target_logits;
    p.draft = draft_logits;
    p.tokens = draft_tokens;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.T = T;
    p.Td = T_d;
    p.T_seq = opts ? opts->T_per_seq : nullptr;
    p.Td_seq = opts ? opts->Td_per_seq : nullptr;
    p.key = philox_key(seed);
    p.rk = philox_round_keys(p.key);
    p.seq_base = opts ? opts->seq_index_base : 0u;
    p.out_tokens = out_tokens;
    p.out_n = out_n_accepted;
    if (opts) {
        p.out_logp = opts->out_logp_draft;
        p.out_logq = opts->out_logq_draft;
        p.out_logZp = opts->out_logZ_p;
        p.out_logZq = opts->out_logZ_q;
        p.out_u = opts->out_u;
        p.out_race = opts->out_race;
        p.out_Hp = opts->out_H_p;
        p.out_Hq = opts->out_H_q;
        p.out_KL = opts->out_KL;
        p.ctrl_centres = opts->ctrl_centres;
        p.ctrl_beta = opts->ctrl_beta;
        if (p.ctrl_centres && !(p.ctrl_beta > 0.0 && p.ctrl_beta <= 1.0)) return SPEC_EINVAL;
    }
    if (opts && (opts->flags & ~kKnownFlags)) return SPEC_EINVAL;
    p.debug_flags = (opts && (opts->flags & SPEC_DEBUG_NEVER_READY)) ? kDebugNeverReady : 0u;
    DeviceState* d = nullptr;
    char* ws = nullptr;
    rc = prepare(B, gamma, V, dtype, opts, p, &d, &ws);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool diagnostics = p.out_logp || p.out_logq || p.out_logZp || p.out_logZq || p.out_u ||
                             p.out_race || wants_position_stats(p);
    const Layout L = layout_of(B, gamma, V, dtype, d->stream_warps[dtype == SPEC_F32 ? 0 : 1]);
    if (d->coop && opts && (opts->flags & SPEC_FLAG_EARLY_EXIT) && !diagnostics) {
        if (host_rows) {  // a device copy of every row the kernel streams, for the race
            const size_t es = static_cast<size_t>(elem_bytes(dtype));
            const size_t tb = align_up(static_cast<size_t>(B) * (gamma + 1) * V * es, 256);
            const size_t db = static_cast<size_t>(B) * gamma * V * es;
            std::lock_guard<std::mutex> lock(g_mu);
            if (ensure_mirror(*d, tb + db)) {
                p.mirror_target = d->mirror;
                p.mirror_draft = static_cast<char*>(d->mirror) + tb;
            }
        }
        return dtype == SPEC_F32 ? launch_early<F32Elem>(p, d->sm_count, opts, s, L, ws, host_rows)
                                 : launch_early<Bf16Elem>(p, d->sm_count, opts, s, L, ws, host_rows);
    }
    return dtype == SPEC_F32 ? launch_sampling<F32Elem>(p, d->sm_count, opts, s)
                             : launch_sampling<Bf16Elem>(p, d->sm_count, opts, s);
}

}  // namespace

extern "C" {

int spec_verify_ex(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                   int B, int gamma, int V, float T, float T_d, uint64_t seed, int32_t* out_tokens,
                   int32_t* out_n_accepted, const spec_verify_opts* opts, void* stream) {
    return verify_ex_impl(target_logits, draft_logits, draft_tokens, B, gamma, V, T, T_d, seed,
                          out_tokens, out_n_accepted, opts, stream, false);
}

int spec_verify(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                int B, int gamma, int V, float T, float T_d, uint64_t seed, int32_t* out_tokens,
                int32_t* out_n_accepted, void* stream) {
    return spec_verify_ex(target_logits, draft_logits, draft_tokens, B, gamma, V, T, T_d, seed,
                          out_tokens, out_n_accepted, nullptr, stream);
}

int spec_verify_greedy_ex(const void* target_logits, const int32_t* draft_tokens, int B, int gamma,
                          int V, int32_t* out_tokens, int32_t* out_n_accepted,
                          const spec_verify_opts* opts, void* stream) {
    const int dtype = opts ? opts->dtype : SPEC_BF16;
    int rc = check_common(target_logits, out_tokens, out_n_accepted, B, gamma, V, dtype);
    if (rc || B == 0) return rc;
    if (gamma > 0 && !draft_tokens) return SPEC_EINVAL;
    VerifyParams p{};
    p.target = target_logits;
    p.tokens = draft_tokens;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.out_tokens = out_tokens;
    p.out_n = out_n_accepted;
    DeviceState* d = nullptr;
    rc = prepare(B, gamma, V, dtype, opts, p, &d);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == SPEC_F32 ? launch_greedy<F32Elem>(p, d->sm_count, opts, s)
                             : launch_greedy<Bf16Elem>(p, d->sm_count, opts, s);
}

int spec_verify_greedy(const void* target_logits, const int32_t* draft_tokens, int B, int gamma,
                       int V, int32_t* out_tokens, int32_t* out_n_accepted, void* stream) {
    return spec_verify_greedy_ex(target_logits, draft_tokens, B, gamma, V, out_tokens,
                                 out_n_accepted, nullptr, stream);
}

int spec_philox4x32_10(const uint32_t* counters, const uint32_t* keys, int64_t n, int form,
                       uint32_t* out, void* stream) {
    if (n < 0 || (form != 0 && form != 1)) return SPEC_EINVAL;
    if (n == 0) return SPEC_OK;
    if (!counters || !keys || !out || !aligned16(counters) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(keys) & 7u) != 0)
        return SPEC_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long blocks = std::min<long long>((n + kThreads - 1) / kThreads, 1LL << 20);
    philox_probe_kernel<<<static_cast<unsigned>(blocks), kThreads, 0, s>>>(
        reinterpret_cast<const uint4*>(counters), reinterpret_cast<const uint2*>(keys), n, form,
        reinterpret_cast<uint4*>(out));
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int spec_verify_check(void* stream, int32_t* d_status) {
    int32_t* st = d_status;
    if (!st) {
        std::lock_guard<std::mutex> lock(g_mu);
        DeviceState* d = nullptr;
        int rc = device_state(&d);
        if (rc) return rc;
        st = d->status;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int32_t h = 0;
    if (cudaMemcpyAsync(&h, st, sizeof(h), cudaMemcpyDeviceToHost, s) != cudaSuccess) return SPEC_ECUDA;
    if (cudaMemsetAsync(st, 0, sizeof(int32_t), s) != cudaSuccess) return SPEC_ECUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return SPEC_ECUDA;
    return h;
}

}  // extern "C"

namespace {

// The device address of a buffer the GPU can reach: device memory as it is, mapped pinned
// host memory (cudaHostAlloc / cudaHostRegister) through its device alias.  Anything else
// (pageable host memory) is refused.
template <class P>
int device_alias(P* ptr, P** out) {
    *out = ptr;
    if (!ptr) return SPEC_OK;
    cudaPointerAttributes a{};
    if (cudaPointerGetAttributes(&a, ptr) != cudaSuccess) {
        cudaGetLastError();  // clear the sticky-free error of an unknown pointer
        return SPEC_EINVAL;
    }
    if (a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged) return SPEC_OK;
    if (a.type == cudaMemoryTypeHost && a.devicePointer) {
        *out = static_cast<P*>(a.devicePointer);
        return SPEC_OK;
    }
    return SPEC_EINVAL;
}

}  // namespace

extern "C" {

int spec_verify_host(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                     int B, int gamma, int V, float T, float T_d, uint64_t seed, int32_t* out_tokens,
                     int32_t* out_n_accepted, const spec_verify_opts* opts, void* stream) {
    if (B == 0) return check_common(target_logits, out_tokens, out_n_accepted, B, gamma, V,
                                    opts ? opts->dtype : SPEC_BF16);
    const void *t = nullptr, *d = nullptr;
    const int32_t* tok = nullptr;
    int32_t *ot = nullptr, *on = nullptr;
    if (device_alias(target_logits, &t) || device_alias(draft_logits, &d) ||
        device_alias(draft_tokens, &tok) || device_alias(out_tokens, &ot) ||
        device_alias(out_n_accepted, &on))
        return SPEC_EINVAL;
    spec_verify_opts o;
    if (opts) o = *opts;
    else spec_verify_opts_init(&o);
    if (device_alias(o.T_per_seq, &o.T_per_seq) || device_alias(o.Td_per_seq, &o.Td_per_seq))
        return SPEC_EINVAL;
    if (!(o.flags & SPEC_FLAG_FULL_READ)) o.flags |= SPEC_FLAG_EARLY_EXIT;
    return verify_ex_impl(t, d, tok, B, gamma, V, T, T_d, seed, ot, on, &o, stream, true);
}

int spec_verify_tree(const void* target_logits, const void* draft_logits, const int32_t* draft_tokens,
                     const int32_t* parent, int B, int N, int V, float T, float T_d, uint64_t seed,
                     int32_t* out_tokens, int32_t* out_nodes, int32_t* out_n_accepted,
                     const spec_verify_opts* opts, void* stream) {
    const int dtype = opts ? opts->dtype : SPEC_BF16;
    if (N < 1 || N > kMaxTreeNodes || !parent) return SPEC_EINVAL;
    if (parent[0] != -1) return SPEC_EINVAL;
    TreeShape t{};
    t.N = N;
    int depth[kMaxTreeNodes] = {0};
    int nchild[kMaxTreeNodes] = {0};
    int last_child[kMaxTreeNodes];
    for (int n = 0; n < N; ++n) {
        t.first_child[n] = -1;
        t.next_sibling[n] = -1;
        last_child[n] = -1;
    }
    for (int n = 1; n < N; ++n) {
        const int u = parent[n];
        if (u < 0 || u >= n) return SPEC_EINVAL;
        depth[n] = depth[u] + 1;
        t.D = std::max(t.D, depth[n]);
        if (last_child[u] < 0) t.first_child[u] = static_cast<int16_t>(n);
        else t.next_sibling[last_child[u]] = static_cast<int16_t>(n);
        last_child[u] = n;
        ++nchild[u];
    }
    for (int n = 0; n < N; ++n) t.drow[n] = static_cast<int16_t>(nchild[n] > 0 ? t.M++ : -1);
    const int R = N + t.M;
    const int gamma_eq = R / 2;  // the workspace holds 2 * gamma_eq + 1 >= R rows per sequence
    int rc = check_common(target_logits, out_tokens, out_n_accepted, B, gamma_eq, V, dtype);
    if (rc || B == 0) return rc;
    if (static_cast<long long>(B) * N * static_cast<long long>(V) >= (1LL << 40)) return SPEC_EINVAL;
    if (t.M > 0 && (!draft_logits || !aligned16(draft_logits))) return SPEC_EINVAL;
    if (N > 1 && !draft_tokens) return SPEC_EINVAL;
    if (!(opts && opts->T_per_seq) && !good_temperature(T)) return SPEC_EINVAL;
    if (!(opts && opts->Td_per_seq) && !good_temperature(T_d)) return SPEC_EINVAL;
    VerifyParams p{};
    p.target = target_logits;
    p.draft = draft_logits;
    p.tokens = draft_tokens;
    p.B = B;
    p.gamma = gamma_eq;
    p.V = V;
    p.T = T;
    p.Td = T_d;
    p.T_seq = opts ? opts->T_per_seq : nullptr;
    p.Td_seq = opts ? opts->Td_per_seq : nullptr;
    p.key = philox_key(seed);
    p.rk = philox_round_keys(p.key);
    p.seq_base = opts ? opts->seq_index_base : 0u;
    p.out_tokens = out_tokens;
    p.out_n = out_n_accepted;
    p.out_nodes = out_nodes;
    DeviceState* d = nullptr;
    rc = prepare(B, gamma_eq, V, dtype, opts, p, &d);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return dtype == SPEC_F32 ? launch_tree<F32Elem>(p, t, d->sm_count, opts, s)
                             : launch_tree<Bf16Elem>(p, t, d->sm_count, opts, s);
}

}  // extern "C"

namespace {

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    });
    return fn;
}

// 2-D bf16 tensor map of a row-major [rows, cols] matrix, box of box_rows x 64 elements
// (128 bytes: one 128-byte swizzle row).
int bf16_tensor_map(CUtensorMap* map, const void* base, int rows, int cols, int box_rows) {
    auto enc = tensor_map_encoder();
    if (!enc) return SPEC_ECUDA;
    const cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    const cuuint64_t strides[1] = {static_cast<cuuint64_t>(cols) * 2};
    const cuuint32_t box[2] = {static_cast<cuuint32_t>(kGemmBK), static_cast<cuuint32_t>(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
                           box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                           CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? SPEC_OK : SPEC_EINVAL;
}

int lmhead_check(const void* H, const void* W, int rows, int V, int d) {
    if (rows < 0 || V < 1 || d < kGemmBK || d % kGemmBK != 0) return SPEC_EINVAL;
    if (static_cast<long long>(rows) * V >= (1LL << 40)) return SPEC_EINVAL;
    if (rows == 0) return SPEC_OK;
    if (!H || !W || !aligned16(H) || !aligned16(W)) return SPEC_EINVAL;
    return SPEC_OK;
}

// Grid of the LM-head kernel: one grid row per row tile (of both parts), the vocabulary
// tiles split into chunks so that the CTAs fill the GPU about once (one CTA per SM: each
// holds 512 TMEM columns and 193 KB of shared memory).  The CTAs of one chunk sweep the same
// head tiles in step, so each head is read from HBM about once.
void lmhead_grid(int rows0, int rows1, int V, int sm_count, LmHeadParams& lp, dim3& grid) {
    const int m0 = (rows0 + kGemmBM - 1) / kGemmBM, m1 = (rows1 + kGemmBM - 1) / kGemmBM;
    const int n_tiles = (V + kGemmBN - 1) / kGemmBN;
    long long want = sm_count / std::max(1, m0 + m1);  // chunks per row tile
    if (want < 1) want = 1;
    if (want > n_tiles) want = n_tiles;
    lp.tiles_per_cta = static_cast<int>((n_tiles + want - 1) / want);
    lp.nchunks = (n_tiles + lp.tiles_per_cta - 1) / lp.tiles_per_cta;
    lp.m_tiles0 = m0;
    grid = dim3(static_cast<unsigned>(lp.nchunks), static_cast<unsigned>(m0 + m1));
}

// Launch part 0 = (H0, W0) and, if lp.part[1].rows > 0, part 1 = (H1, W1) in one grid.
template <bool kLogits>
int launch_lmhead(const void* H0, const void* W0, const void* H1, const void* W1, LmHeadParams& lp,
                  int sm_count, cudaStream_t s) {
    CUtensorMap mh0, mw0, mh1, mw1;
    int rc = bf16_tensor_map(&mh0, H0, lp.part[0].rows, lp.d, kGemmBM);
    if (rc) return rc;
    rc = bf16_tensor_map(&mw0, W0, lp.V, lp.d, kGemmBN);
    if (rc) return rc;
    if (lp.part[1].rows > 0) {
        rc = bf16_tensor_map(&mh1, H1, lp.part[1].rows, lp.d, kGemmBM);
        if (rc) return rc;
        rc = bf16_tensor_map(&mw1, W1, lp.V, lp.d, kGemmBN);
        if (rc) return rc;
    } else {
        mh1 = mh0;
        mw1 = mw0;
    }
    dim3 grid;
    lmhead_grid(lp.part[0].rows, lp.part[1].rows, lp.V, sm_count, lp, grid);
    auto kernel = lmhead_kernel<kLogits>;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGemmSmem) != cudaSuccess)
        return SPEC_ECUDA;
    kernel<<<grid, kGemmThreads, kGemmSmem, s>>>(mh0, mw0, mh1, mw1, lp);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

// The merge kernel's view of one part.
LmHeadParams part_view(const LmHeadParams& lp, int k) {
    LmHeadParams v = lp;
    v.rows = lp.part[k].rows;
    v.T_row = lp.part[k].T_row;
    v.token_row = lp.part[k].token_row;
    v.stat_parts = lp.part[k].stat_parts;
    v.token_logit = lp.part[k].token_logit;
    return v;
}

}  // namespace

extern "C" {

int spec_lmhead_logits(const void* hidden, const void* weight, int rows, int V, int d,
                       float* out_logits, void* stream) {
    int rc = lmhead_check(hidden, weight, rows, V, d);
    if (rc || rows == 0) return rc;
    if (!out_logits) return SPEC_EINVAL;
    DeviceState* dev = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        rc = device_state(&dev);
        if (rc) return rc;
    }
    LmHeadParams lp{};
    lp.V = V;
    lp.d = d;
    lp.part[0].rows = rows;
    lp.part[0].logits = out_logits;
    lp.status = dev->status;
    return launch_lmhead<true>(hidden, weight, nullptr, nullptr, lp, dev->sm_count,
                               static_cast<cudaStream_t>(stream));
}

}  // extern "C"

namespace {

// Merge each row's chunk partials: ln Z = (m + log2 s) ln 2 and, when a token is given,
// ln p(token) = x_token / T - ln Z.  One warp per row.
__global__ void __launch_bounds__(256) lmhead_merge_kernel(LmHeadParams p, float* out_logZ,
                                                           float* out_logp_token) {
    const int lane = threadIdx.x & 31;
    const int row = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (row >= p.rows) return;
    SoftmaxStat st{-FLT_MAX, 0.0f};
    for (int k = lane; k < p.nchunks; k += 32) {
        const float2 q = p.stat_parts[static_cast<long long>(row) * p.nchunks + k];
        st = merge_stat(st, SoftmaxStat{q.x, q.y});
    }
    st = warp_merge_stat(st);
    if (lane == 0) {
        const float lz = (st.m + log2f(st.s)) * kLn2;
        if (out_logZ) out_logZ[row] = lz;
        if (out_logp_token) {
            const int tok = p.token_row ? p.token_row[row] : -1;
            out_logp_token[row] = (tok >= 0 && tok < p.V) ? p.token_logit[row] / p.T_row[row] - lz : NAN;
        }
    }
}

}  // namespace

extern "C" {

int spec_lmhead_row_stats(const void* hidden, const void* weight, int rows, int V, int d,
                          const float* T_row, const int32_t* token_row, float* out_logZ,
                          float* out_logp_token, void* stream) {
    int rc = lmhead_check(hidden, weight, rows, V, d);
    if (rc || rows == 0) return rc;
    if (!T_row || (!out_logZ && !out_logp_token)) return SPEC_EINVAL;
    if (out_logp_token && !token_row) return SPEC_EINVAL;
    DeviceState* dev = nullptr;
    char* ws = nullptr;
    LmHeadParams lp{};
    lp.V = V;
    lp.d = d;
    lp.part[0].rows = rows;
    dim3 grid;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        rc = device_state(&dev);
        if (rc) return rc;
        lmhead_grid(rows, 0, V, dev->sm_count, lp, grid);
        // workspace: [rows][nchunks] partials, then [rows] token logits
        const size_t need = align_up(static_cast<size_t>(rows) * lp.nchunks * sizeof(float2), 256) +
                            align_up(static_cast<size_t>(rows) * sizeof(float), 256);
        rc = ensure_workspace(*dev, need);
        if (rc) return rc;
        ws = static_cast<char*>(dev->ws);
    }
    lp.part[0].T_row = T_row;
    lp.part[0].token_row = token_row;
    lp.part[0].stat_parts = reinterpret_cast<float2*>(ws);
    lp.part[0].token_logit = reinterpret_cast<float*>(
        ws + align_up(static_cast<size_t>(rows) * lp.nchunks * sizeof(float2), 256));
    lp.status = dev->status;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    rc = launch_lmhead<false>(hidden, weight, nullptr, nullptr, lp, dev->sm_count, s);
    if (rc) return rc;
    lmhead_merge_kernel<<<(rows * 32 + 255) / 256, 256, 0, s>>>(part_view(lp, 0), out_logZ, out_logp_token);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int spec_verify_lmhead(const void* h_target, const void* w_target, const void* h_draft,
                       const void* w_draft, const int32_t* draft_tokens, int B, int gamma, int V,
                       int d, float T, float T_d, uint64_t seed, int32_t* out_tokens,
                       int32_t* out_n_accepted, const spec_verify_opts* opts, void* stream) {
    if (B < 0 || gamma < 0 || gamma > kMaxGamma) return SPEC_EINVAL;
    if (d > kLmMaxD) return SPEC_EINVAL;
    int rc = lmhead_check(h_target, w_target, B * (gamma + 1), V, d);
    if (rc) return rc;
    if (B == 0) return SPEC_OK;
    if (!out_tokens || !out_n_accepted) return SPEC_EINVAL;
    if (gamma > 0) {
        rc = lmhead_check(h_draft, w_draft, B * gamma, V, d);
        if (rc) return rc;
        if (!draft_tokens) return SPEC_EINVAL;
    }
    if (!(opts && opts->T_per_seq) && !good_temperature(T)) return SPEC_EINVAL;
    if (!(opts && opts->Td_per_seq) && !good_temperature(T_d)) return SPEC_EINVAL;
    const int rows_t = B * (gamma + 1), rows_d = B * gamma;
    DeviceState* dev = nullptr;
    LmHeadParams ps{};  // statistics: part 0 the target rows, part 1 the draft rows
    ps.V = V;
    ps.d = d;
    ps.part[0].rows = rows_t;
    ps.part[1].rows = rows_d;
    dim3 grid_s;
    const int rpieces = (V + kRaceBlockTokens - 1) / kRaceBlockTokens;
    // workspace carve-up
    size_t off = 0;
    auto take = [&](size_t bytes) { const size_t o = off; off = align_up(off + bytes, 256); return o; };
    char* ws = nullptr;
    size_t o_Tt, o_tokt, o_partt, o_xt, o_Zt, o_pt, o_Td, o_tokd, o_partd, o_xd, o_Zd, o_qd, o_bm, o_seq,
        o_race, o_tick;
    const int nbm = lm_block_stride(V);
    {
        std::lock_guard<std::mutex> lock(g_mu);
        rc = device_state(&dev);
        if (rc) return rc;
        lmhead_grid(rows_t, rows_d, V, dev->sm_count, ps, grid_s);
        o_Tt = take(rows_t * sizeof(float));
        o_tokt = take(rows_t * sizeof(int32_t));
        o_partt = take(static_cast<size_t>(rows_t) * ps.nchunks * sizeof(float2));
        o_xt = take(rows_t * sizeof(float));
        o_Zt = take(rows_t * sizeof(float));
        o_pt = take(rows_t * sizeof(float));
        o_Td = take(rows_d * sizeof(float) + 4);
        o_tokd = take(rows_d * sizeof(int32_t) + 4);
        o_partd = take(static_cast<size_t>(rows_d) * ps.nchunks * sizeof(float2) + 8);
        o_xd = take(rows_d * sizeof(float) + 4);
        o_Zd = take(rows_d * sizeof(float) + 4);
        o_qd = take(rows_d * sizeof(float) + 4);
        o_bm = take(static_cast<size_t>(rows_t) * nbm * sizeof(uint16_t));  // target rows' block maxima
        o_seq = take(static_cast<size_t>(B) * sizeof(SeqInfo));
        o_race = take(static_cast<size_t>(B) * race_slots(rpieces) * sizeof(RacePart));
        o_tick = take(static_cast<size_t>(B) * sizeof(int));
        rc = ensure_workspace(*dev, off);
        if (rc) return rc;
        ws = static_cast<char*>(dev->ws);
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    LmVerifyParams q{};
    q.B = B;
    q.gamma = gamma;
    q.V = V;
    q.d = d;
    q.h_target = static_cast<const uint16_t*>(h_target);
    q.h_draft = static_cast<const uint16_t*>(h_draft);
    q.tokens = draft_tokens;
    q.logZ_t = reinterpret_cast<float*>(ws + o_Zt);
    q.logp_t = reinterpret_cast<float*>(ws + o_pt);
    q.logZ_d = reinterpret_cast<float*>(ws + o_Zd);
    q.logq_d = reinterpret_cast<float*>(ws + o_qd);
    q.seq = reinterpret_cast<SeqInfo*>(ws + o_seq);
    q.T = T;
    q.Td = T_d;
    q.T_seq = opts ? opts->T_per_seq : nullptr;
    q.Td_seq = opts ? opts->Td_per_seq : nullptr;
    q.key = philox_key(seed);
    q.seq_base = opts ? opts->seq_index_base : 0u;
    q.out_tokens = out_tokens;
    q.out_n = out_n_accepted;
    q.status = (opts && opts->d_status) ? opts->d_status : dev->status;
    record(opts, 0, s);
    {
        const long long n = rows_t;
        lmhead_rows_kernel<<<static_cast<unsigned>((n + 255) / 256), 256, 0, s>>>(
            q, reinterpret_cast<float*>(ws + o_Tt), reinterpret_cast<int32_t*>(ws + o_tokt),
            reinterpret_cast<float*>(ws + o_Td), reinterpret_cast<int32_t*>(ws + o_tokd));
    }
    if (cudaMemsetAsync(ws + o_race, 0, static_cast<size_t>(B) * race_slots(rpieces) * sizeof(RacePart), s) != cudaSuccess ||
        cudaMemsetAsync(ws + o_tick, 0, static_cast<size_t>(B) * sizeof(int), s) != cudaSuccess)
        return SPEC_ECUDA;
    // row statistics of the target rows (T_b) and the draft rows (Td_b), with the draft
    // tokens and the target rows' block maxima, in one launch
    ps.part[0].block_max = reinterpret_cast<uint16_t*>(ws + o_bm);
    ps.part[0].T_row = reinterpret_cast<float*>(ws + o_Tt);
    ps.part[0].token_row = reinterpret_cast<int32_t*>(ws + o_tokt);
    ps.part[0].stat_parts = reinterpret_cast<float2*>(ws + o_partt);
    ps.part[0].token_logit = reinterpret_cast<float*>(ws + o_xt);
    ps.part[1].T_row = reinterpret_cast<float*>(ws + o_Td);
    ps.part[1].token_row = reinterpret_cast<int32_t*>(ws + o_tokd);
    ps.part[1].stat_parts = reinterpret_cast<float2*>(ws + o_partd);
    ps.part[1].token_logit = reinterpret_cast<float*>(ws + o_xd);
    ps.status = q.status;
    rc = launch_lmhead<false>(h_target, w_target, h_draft, w_draft, ps, dev->sm_count, s);
    if (rc) return rc;
    lmhead_merge_kernel<<<(rows_t * 32 + 255) / 256, 256, 0, s>>>(part_view(ps, 0), reinterpret_cast<float*>(ws + o_Zt),
                                                                 reinterpret_cast<float*>(ws + o_pt));
    if (rows_d)
        lmhead_merge_kernel<<<(rows_d * 32 + 255) / 256, 256, 0, s>>>(part_view(ps, 1), reinterpret_cast<float*>(ws + o_Zd),
                                                                     reinterpret_cast<float*>(ws + o_qd));
    record(opts, 1, s);
    lmhead_scan_kernel<<<(B * 32 + 255) / 256, 256, 0, s>>>(q);
    record(opts, 2, s);
    VerifyParams p{};
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.key = q.key;
    p.rk = philox_round_keys(q.key);
    p.seq_base = q.seq_base;
    p.seq = q.seq;
    p.rpieces = rpieces;
    p.race_parts = reinterpret_cast<RacePart*>(ws + o_race);
    p.tickets = reinterpret_cast<int*>(ws + o_tick);
    p.status = q.status;
    p.out_tokens = out_tokens;
    p.out_n = out_n_accepted;
    p.caps.out_tokens = static_cast<long long>(B) * (gamma + 1);
    p.caps.race = static_cast<long long>(B) * race_slots(rpieces);
    p.debug_flags = (opts && (opts->flags & SPEC_DEBUG_RACE_AGAIN)) ? kDebugRaceAgain : 0u;
    LmRaceParams lq{};
    lq.h_target = static_cast<const uint16_t*>(h_target);
    lq.h_draft = static_cast<const uint16_t*>(h_draft);
    lq.w_target = static_cast<const uint16_t*>(w_target);
    lq.w_draft = static_cast<const uint16_t*>(gamma > 0 ? w_draft : w_target);
    lq.block_max = reinterpret_cast<const uint16_t*>(ws + o_bm);
    lq.logp_t = q.logp_t;
    lq.logq_d = q.logq_d;
    lq.d = d;
    lq.nbm = nbm;
    const size_t race_smem = static_cast<size_t>(d) * 4;  // the two raced hidden states, bf16
    if (race_smem > 48 * 1024 &&
        cudaFuncSetAttribute(lmhead_race_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(race_smem)) != cudaSuccess)
        return SPEC_ECUDA;
    int per_sm = blocks_per_sm(lmhead_race_kernel, kThreads, race_smem);
    if (per_sm < 1) per_sm = 1;
    long long G = static_cast<long long>(dev->sm_count) * per_sm / B;
    if (G > rpieces) G = rpieces;
    if (G < 1) G = 1;
    p.rgroups = static_cast<int>(G);
    lmhead_race_kernel<<<static_cast<unsigned>(B * G), kThreads, race_smem, s>>>(p, lq);
    record(opts, 3, s);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int spec_adaptive_k(const float* H_next, int B, int K, const double* centres,
                    const int32_t* candidates, int n_cand, double C_d, double C_v,
                    int32_t* out_k, double* out_eff, void* stream) {
    if (B < 0 || K < 1 || n_cand < 1 || n_cand > kMaxCandidates || !candidates) return SPEC_EINVAL;
    if (!std::isfinite(C_d) || !std::isfinite(C_v)) return SPEC_EINVAL;
    AdaptiveKParams a{};
    for (int c = 0; c < n_cand; ++c) {
        if (candidates[c] < 1 || candidates[c] > K) return SPEC_EINVAL;
        if (!(static_cast<double>(candidates[c]) * C_d + C_v > 0.0)) return SPEC_EINVAL;
        a.cand[c] = candidates[c];
    }
    if (B == 0) return SPEC_OK;
    if (!H_next || !centres || !out_k) return SPEC_EINVAL;
    a.H = H_next;
    a.centres = centres;
    a.B = B;
    a.K = K;
    a.n_cand = n_cand;
    a.Cd = C_d;
    a.Cv = C_v;
    a.out_k = out_k;
    a.out_eff = out_eff;
    adaptive_k_kernel<<<(B + 127) / 128, 128, 0, static_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int spec_row_entropy(const void* logits, int rows, int V, float T, int dtype, float* out_H,
                     void* stream) {
    int rc = check_common(logits, reinterpret_cast<const int32_t*>(out_H),
                          reinterpret_cast<const int32_t*>(out_H), rows, 0, V, dtype);
    if (rc || rows == 0) return rc;
    if (!good_temperature(T)) return SPEC_EINVAL;
    VerifyParams p{};
    p.target = logits;
    p.B = rows;
    p.gamma = 0;
    p.V = V;
    p.T = T;
    p.Td = T;
    p.out_Hp = out_H;
    DeviceState* d = nullptr;
    rc = prepare(rows, 0, V, dtype, nullptr, p, &d);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const long long items = static_cast<long long>(rows) * p.npieces;
    const cudaError_t e = dtype == SPEC_F32
        ? launch_stream(pair_stats_kernel<F32Elem, kPairUnroll, true>, pair_stats_kernel<F32Elem, kPairUnroll, false>,
                        d->sm_count, items, s, p)
        : launch_stream(pair_stats_kernel<Bf16Elem, kPairUnroll, true>, pair_stats_kernel<Bf16Elem, kPairUnroll, false>,
                        d->sm_count, items, s, p);
    if (e != cudaSuccess) return SPEC_ECUDA;
    position_stats_kernel<<<rows, kThreads, 0, s>>>(p);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

const char* spec_verify_strerror(int status) {
    switch (status) {
        case SPEC_OK: return "success";
        case SPEC_EINVAL: return "invalid argument";
        case SPEC_ECUDA: return "CUDA runtime error";
        case SPEC_EBADTOKEN: return "draft token outside [0, V)";
        case SPEC_ETIMEOUT: return "bounded device wait timed out";
        case SPEC_ENOMEM: return "workspace allocation failed or caller workspace too small";
        case SPEC_ESCRATCH: return "problem needs more scratch than the static no-alloc buffer";
        case SPEC_EINDEX: return "index outside its buffer (index-checked build): access skipped";
        default: return "unknown status";
    }
}

}  // extern "C"

// ------------------------------------------------------------------------------------------
// Vocabulary-parallel verify (vocab.cuh): each rank's steps around two small collectives that
// the caller runs (an all-gather of the row statistics and the gathered logits' max, then a
// max of the race keys).
// ------------------------------------------------------------------------------------------

namespace {

// The parameters shared by the vocabulary-parallel steps; V is the shard's width (or, for
// vp_decide, the whole vocabulary).
void vp_params(VerifyParams& p, const void* target, const void* draft, const int32_t* tokens, int B,
               int gamma, int V, float T, float T_d, uint64_t seed, const spec_verify_opts* o) {
    p.target = target;
    p.draft = draft;
    p.tokens = tokens;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.T = T;
    p.Td = T_d;
    p.T_seq = o ? o->T_per_seq : nullptr;
    p.Td_seq = o ? o->Td_per_seq : nullptr;
    p.key = philox_key(seed);
    p.rk = philox_round_keys(p.key);
    p.seq_base = o ? o->seq_index_base : 0u;
}

int vp_shape_ok(int B, int gamma, int V, int x_offset, int dtype) {
    if (B < 0 || gamma < 0 || gamma > kMaxGamma || V < 1 || x_offset < 0 || (x_offset & 7)) return SPEC_EINVAL;
    if (dtype != SPEC_F32 && dtype != SPEC_BF16) return SPEC_EINVAL;
    if (static_cast<long long>(B) * (gamma + 1) * static_cast<long long>(V) >= (1LL << 40)) return SPEC_EINVAL;
    return SPEC_OK;
}

int vp_temps_ok(float T, float T_d, const spec_verify_opts* o) {
    if (!(o && o->T_per_seq) && !good_temperature(T)) return SPEC_EINVAL;
    if (!(o && o->Td_per_seq) && !good_temperature(T_d)) return SPEC_EINVAL;
    return SPEC_OK;
}

int status_word(const spec_verify_opts* o, int32_t** st) {
    if (o && o->d_status) {
        *st = o->d_status;
        return SPEC_OK;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceState* d = nullptr;
    const int rc = device_state(&d);
    if (rc) return rc;
    *st = d->status;
    return SPEC_OK;
}

template <class ET>
int launch_vp_partials(VerifyParams& p, int sm_count, int x_offset, float2* stats, float2* gathered,
                       cudaStream_t s) {
    const int R = 2 * p.gamma + 1;
    const long long items = static_cast<long long>(p.B) * R * p.npieces;
    if (launch_stream(row_stats_kernel<ET, kUnroll, true>, row_stats_kernel<ET, kUnroll, false>, sm_count, items, s,
                  p) != cudaSuccess)
        return SPEC_ECUDA;
    const long long rows = static_cast<long long>(p.B) * R;
    vp_fold_kernel<<<static_cast<unsigned>(std::min<long long>((rows + kThreads - 1) / kThreads, 4LL * sm_count)),
                     kThreads, 0, s>>>(p, stats);
    const long long n = static_cast<long long>(p.B) * p.gamma;
    if (n > 0)
        vp_gather_kernel<ET><<<static_cast<unsigned>(std::min<long long>((n + kThreads - 1) / kThreads, 4LL * sm_count)),
                               kThreads, 0, s>>>(p, x_offset, gathered);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // namespace

extern "C" {

size_t spec_vp_state_bytes(int B) { return B > 0 ? static_cast<size_t>(B) * sizeof(VpState) : 0; }

int spec_vp_partials(const void* target_shard, const void* draft_shard, const int32_t* draft_tokens,
                     int B, int gamma, int V_shard, int x_offset, float T, float T_d, float* out_stats,
                     float* out_gathered, const spec_verify_opts* opts, void* stream) {
    const int dtype = opts ? opts->dtype : SPEC_BF16;
    int rc = vp_shape_ok(B, gamma, V_shard, x_offset, dtype);
    if (rc || B == 0) return rc;
    if (!target_shard || !aligned16(target_shard) || !out_stats) return SPEC_EINVAL;
    if (gamma > 0 && (!draft_shard || !aligned16(draft_shard) || !draft_tokens || !out_gathered))
        return SPEC_EINVAL;
    if ((rc = vp_temps_ok(T, T_d, opts))) return rc;
    VerifyParams p{};
    vp_params(p, target_shard, draft_shard, draft_tokens, B, gamma, V_shard, T, T_d, 0, opts);
    DeviceState* d = nullptr;
    rc = prepare(B, gamma, V_shard, dtype, opts, p, &d);
    if (rc) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    float2* st = reinterpret_cast<float2*>(out_stats);
    float2* ga = reinterpret_cast<float2*>(out_gathered);
    return dtype == SPEC_F32 ? launch_vp_partials<F32Elem>(p, d->sm_count, x_offset, st, ga, s)
                             : launch_vp_partials<Bf16Elem>(p, d->sm_count, x_offset, st, ga, s);
}

int spec_vp_decide(const float* stats_all, int world, const float* gathered, const int32_t* draft_tokens,
                   int B, int gamma, int V, float T, float T_d, uint64_t seed, int32_t* out_tokens,
                   int32_t* out_n_accepted, void* state, const spec_verify_opts* opts, void* stream) {
    const int dtype = opts ? opts->dtype : SPEC_BF16;
    int rc = vp_shape_ok(B, gamma, V, 0, dtype);
    if (rc || B == 0) return rc;
    if (world < 1 || !stats_all || !out_tokens || !out_n_accepted || !state) return SPEC_EINVAL;
    if (gamma > 0 && (!gathered || !draft_tokens)) return SPEC_EINVAL;
    if ((rc = vp_temps_ok(T, T_d, opts))) return rc;
    VerifyParams p{};
    vp_params(p, nullptr, nullptr, draft_tokens, B, gamma, V, T, T_d, seed, opts);
    p.out_tokens = out_tokens;
    p.out_n = out_n_accepted;
    if ((rc = status_word(opts, &p.status))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    vp_decide_kernel<<<static_cast<unsigned>((static_cast<long long>(B) * 32 + kThreads - 1) / kThreads), kThreads, 0,
                       s>>>(p, reinterpret_cast<const float2*>(stats_all), world,
                            reinterpret_cast<const float2*>(gathered), static_cast<VpState*>(state));
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int spec_vp_race(const void* target_shard, const void* draft_shard, int B, int gamma, int V_shard,
                 int x_offset, uint64_t seed, const void* state, int64_t* out_keys,
                 const spec_verify_opts* opts, void* stream) {
    const int dtype = opts ? opts->dtype : SPEC_BF16;
    int rc = vp_shape_ok(B, gamma, V_shard, x_offset, dtype);
    if (rc || B == 0) return rc;
    if (!target_shard || !aligned16(target_shard) || !state || !out_keys) return SPEC_EINVAL;
    if (gamma > 0 && (!draft_shard || !aligned16(draft_shard))) return SPEC_EINVAL;
    VerifyParams p{};
    vp_params(p, target_shard, draft_shard, nullptr, B, gamma, V_shard, 1.0f, 1.0f, seed, opts);
    if ((rc = status_word(opts, &p.status))) return rc;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    auto* keys = reinterpret_cast<long long*>(out_keys);
    const auto* vs = static_cast<const VpState*>(state);
    if (dtype == SPEC_F32)
        vp_race_kernel<F32Elem><<<static_cast<unsigned>(B), kThreads, 0, s>>>(p, x_offset, vs, keys);
    else
        vp_race_kernel<Bf16Elem><<<static_cast<unsigned>(B), kThreads, 0, s>>>(p, x_offset, vs, keys);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

int spec_vp_finish(const int64_t* keys, const void* state, int B, int gamma, int32_t* out_tokens,
                   void* stream) {
    if (B < 0 || gamma < 0 || gamma > kMaxGamma) return SPEC_EINVAL;
    if (B == 0) return SPEC_OK;
    if (!keys || !state || !out_tokens) return SPEC_EINVAL;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    vp_finish_kernel<<<static_cast<unsigned>((B + kThreads - 1) / kThreads), kThreads, 0, s>>>(
        B, gamma, static_cast<const VpState*>(state), reinterpret_cast<const long long*>(keys), out_tokens);
    return cudaGetLastError() == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // extern "C"

// ------------------------------------------------------------------------------------------
// spec_verify_noalloc: the sampling verify with its scratch in a file-scope device array, for
// callers that cannot let the library allocate device memory.
// ------------------------------------------------------------------------------------------

static __device__ __align__(256) unsigned char g_noalloc_scratch[SPEC_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr size_t kNoallocStatusOff = SPEC_NOALLOC_SCRATCH_BYTES - 256;  // last 256 bytes

struct NoallocDevice {
    bool ready = false;
    char* scratch = nullptr;  // device address of g_noalloc_scratch on this device
    int sm_count = 0;
    int coop = 0;             // cooperative launch supported
    long long stream_warps[2] = {0, 0};
};

std::mutex g_noalloc_mu;
NoallocDevice g_noalloc[kMaxDevices];

// Once per device, with that device current: the array's device address (host code cannot
// use the symbol itself, which names a host-side stand-in) and the SM count.
int noalloc_device(NoallocDevice** out) {
    int dev;
    int rc = current_device(&dev);
    if (rc) return rc;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    NoallocDevice& d = g_noalloc[dev];
    if (!d.ready) {
        void* ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
            return SPEC_ECUDA;
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return SPEC_ECUDA;
        if (cudaDeviceGetAttribute(&d.coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess)
            return SPEC_ECUDA;
        d.scratch = static_cast<char*>(ptr);
        d.stream_warps[0] = stream_warps_of(d.sm_count, SPEC_F32);
        d.stream_warps[1] = stream_warps_of(d.sm_count, SPEC_BF16);
        d.ready = true;
    }
    *out = &d;
    return SPEC_OK;
}

}  // namespace

extern "C" int spec_verify_noalloc(const void* target_logits, const void* draft_logits,
                                   const int32_t* draft_tokens, int B, int gamma, int V, float T,
                                   float T_d, uint64_t seed, int32_t* out_tokens,
                                   int32_t* out_n_accepted, const spec_verify_opts* opts,
                                   void* stream) {
    const int dtype = opts ? opts->dtype : SPEC_BF16;
    int rc = check_common(target_logits, out_tokens, out_n_accepted, B, gamma, V, dtype);
    if (rc || B == 0) return rc;
    if (opts && opts->workspace) return SPEC_EINVAL;
    if (opts && (opts->flags & ~kKnownFlags)) return SPEC_EINVAL;
    if (gamma > 0 && (!draft_logits || !draft_tokens || !aligned16(draft_logits))) return SPEC_EINVAL;
    if (!(opts && opts->T_per_seq) && !good_temperature(T)) return SPEC_EINVAL;
    if (!(opts && opts->Td_per_seq) && !good_temperature(T_d)) return SPEC_EINVAL;
    if (layout_of(B, gamma, V, dtype).total > kNoallocStatusOff) return SPEC_ESCRATCH;
    NoallocDevice* nd = nullptr;
    rc = noalloc_device(&nd);
    if (rc) return rc;
    const Layout L = layout_of(B, gamma, V, dtype, nd->stream_warps[dtype == SPEC_F32 ? 0 : 1]);
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    VerifyParams p{};
    p.target = target_logits;
    p.draft = draft_logits;
    p.tokens = draft_tokens;
    p.B = B;
    p.gamma = gamma;
    p.V = V;
    p.T = T;
    p.Td = T_d;
    p.T_seq = opts ? opts->T_per_seq : nullptr;
    p.Td_seq = opts ? opts->Td_per_seq : nullptr;
    p.key = philox_key(seed);
    p.rk = philox_round_keys(p.key);
    p.seq_base = opts ? opts->seq_index_base : 0u;
    p.out_tokens = out_tokens;
    p.out_n = out_n_accepted;
    if (opts) {
        p.out_logp = opts->out_logp_draft;
        p.out_logq = opts->out_logq_draft;
        p.out_logZp = opts->out_logZ_p;
        p.out_logZq = opts->out_logZ_q;
        p.out_u = opts->out_u;
        p.out_race = opts->out_race;
    }
    char* ws = nd->scratch;
    bind_workspace(p, L, ws);
    set_caps(p, L, B, gamma, V);
    if (opts && opts->d_status) {
        p.status = opts->d_status;
    } else {
        p.status = reinterpret_cast<int32_t*>(ws + kNoallocStatusOff);
        if (cudaMemsetAsync(p.status, 0, sizeof(int32_t), s) != cudaSuccess) return SPEC_ECUDA;
    }
    return dtype == SPEC_F32 ? launch_sampling<F32Elem>(p, nd->sm_count, opts, s)
                             : launch_sampling<Bf16Elem>(p, nd->sm_count, opts, s);
}
