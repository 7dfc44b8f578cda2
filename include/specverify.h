/*
 * specverify.h -- C ABI of libspecverify, the speculative-decoding verify step on
 * NVIDIA GB300 (sm_103a).
 *
 * One speculative cycle drafts gamma tokens d_0..d_{gamma-1} with a draft distribution q,
 * runs the target once over gamma + 1 positions to get p, and then verifies: position i is
 * accepted while a fresh uniform u_i < min(1, p_i(d_i) / q_i(d_i)); at the first rejection j
 * one token is drawn from norm(max(0, p_j - q_j)) and the rest of the draft is dropped; if
 * every draft token survives one bonus token is drawn from p_gamma.  Each cycle therefore
 * emits between 1 and gamma + 1 tokens and the emitted tokens follow p exactly.
 * ("How speculative decoding makes LLMs go brrr": the pseudocode of one speculative cycle,
 * module 3 on rejection sampling and losslessness, module 4 on tau in [1, gamma + 1].)
 * p is the softmax of the target logits at temperature T; q is the softmax of the draft
 * logits at the draft temperature T_d, which may be sharper than T ("SubSpec: the target
 * model's own low-bit shadow as the draft model", section 2.2 and section 3.4, Table 5).
 * The greedy (T = 0) mode accepts a draft token when it equals the target's argmax
 * (SubSpec's Tables 1-2 run at T = 0).
 *
 * Random numbers (both u_i and the draws) come from Philox4x32-10 (Salmon et al., SC'11)
 * keyed by (lo32(seed), hi32(seed)); b below is the global sequence index
 * (opts->seq_index_base + local index):
 *   u_i          counter (0, i, b, 0), word 0 w:          u = (w >> 8) * 2^-24
 *   draw at row r counter (x >> 2, r, b, 1), word (x & 3) w: E_x = -log1p(-(w + 0.5) * 2^-32)
 * A draw from weights w(x) is the exponential race argmax_x w(x) / E_x (lowest x on equal
 * scores), so no prefix sum over the vocabulary decides the token.  The same
 * (inputs, seed, seq_index_base) always give the same tokens.
 *
 * Conventions for every entry point:
 *   - Every pointer argument is device memory owned by the caller; the library never frees
 *     it.  Logit base pointers must be 16-byte aligned; V need not be a multiple of 8.
 *   - Layouts are row-major and contiguous: target [B, gamma+1, V], draft [B, gamma, V],
 *     draft_tokens [B, gamma] int32, out_tokens [B, gamma+1] int32, out_n_accepted [B].
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy default stream)
 *     and return once the work is enqueued.  The return value reports argument and launch
 *     errors only; errors found on the device (a draft token outside [0, V)) are recorded in
 *     a device status word read by spec_verify_check().
 *   - B == 0 is an empty batch: nothing is launched and SPEC_OK is returned.
 *   - gamma == 0 is plain sampling from row 0 (sampling) or its argmax (greedy).
 *   - Output tokens are padded with -1 after the last emitted token.  out_n_accepted[b] is
 *     the number j of accepted draft tokens (0..gamma); the cycle emitted j + 1 tokens.
 *     A sequence holding a draft token outside [0, V) gets n_accepted = -1 and all -1
 *     tokens, and the status word records SPEC_EBADTOKEN.
 *   - The plain entry points use a workspace the library allocates per device on first use
 *     (and grows when a larger problem arrives); calls that use it must not run
 *     concurrently on one device.  The _ex entry points can take a caller workspace.
 *   - Kernels and stream order: each call's first kernel is launched with programmatic
 *     stream serialization and waits (griddepcontrol.wait) for the kernel before it on the
 *     stream before touching memory, so inputs written by that kernel are read; each call's
 *     last kernel lets a following kernel that was itself launched with programmatic stream
 *     serialization be scheduled early.  Such a kernel must wait for its prerequisite grid
 *     (griddepcontrol.wait / cudaGridDependencySynchronize) before it reads this call's
 *     outputs, as programmatic launches require; ordinary launches, copies and events see
 *     the call complete as usual.
 */
#ifndef SPECVERIFY_H
#define SPECVERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes. */
typedef enum {
    SPEC_OK = 0,
    SPEC_EINVAL = 1,     /* bad argument (size, NULL pointer, alignment, temperature) */
    SPEC_ECUDA = 2,      /* a CUDA runtime call or launch failed */
    SPEC_EBADTOKEN = 3,  /* (device) a draft token outside [0, V) */
    SPEC_ETIMEOUT = 4,   /* (device) a bounded wait gave up */
    SPEC_ENOMEM = 5,     /* workspace allocation failed or caller workspace too small */
    SPEC_ESCRATCH = 6,   /* problem needs more scratch than spec_verify_noalloc's static
                            buffer (SPEC_NOALLOC_SCRATCH_BYTES) holds */
    SPEC_EINDEX = 7      /* (device, index-checked build only) a computed index fell outside
                            its buffer; the access was skipped and the outputs are invalid */
} spec_status;

/* The index-checked build.  libspecverify_checked.so is the same library compiled with
 * SPECVERIFY_CHECKED: in the sampling (default and early-exit) and greedy kernels every
 * computed index into the logits, the draft tokens, the outputs, the workspace's partial
 * statistics, race partials and queues is tested against its buffer's size before the
 * access; an index outside it records SPEC_EINDEX in the status word and skips the access
 * (no trap and no assert: waits that then go unanswered end after their bounded time).  It
 * stands in for a memory checker on this GPU; it is slower and meant for tests. */

/* Element type of the logits. */
typedef enum { SPEC_F32 = 0, SPEC_BF16 = 1 } spec_dtype;

/* Options of the _ex entry points.  Zero-initialise (spec_verify_opts_init) and set what is
 * needed; every pointer may be NULL. */
typedef struct {
    int32_t dtype;              /* spec_dtype of both logit tensors */
    uint32_t seq_index_base;    /* global index of sequence 0 in the random-number counters */
    const float *T_per_seq;     /* [B] device: target temperature of each sequence (NULL: T) */
    const float *Td_per_seq;    /* [B] device: draft temperature of each sequence (NULL: T_d) */
    void *workspace;            /* device scratch of workspace_bytes (NULL: library's own);
                                   no initial contents are needed.  Calls sharing one
                                   workspace must not overlap on the device. */
    size_t workspace_bytes;
    int32_t *d_status;          /* device int32 status word (NULL: the library's own, which
                                   spec_verify_check(stream, NULL) reads on the current
                                   device) */
    /* Diagnostic outputs (device, NULL = not written), all fp32: */
    float *out_logp_draft;      /* [B, gamma]   ln p_i(d_i) */
    float *out_logq_draft;      /* [B, gamma]   ln q_i(d_i) */
    float *out_logZ_p;          /* [B, gamma+1] ln sum_x exp(L_t[b,i,x] / T_b) */
    float *out_logZ_q;          /* [B, gamma]   ln sum_x exp(L_d[b,i,x] / Td_b) */
    float *out_u;               /* [B, gamma]   acceptance uniforms */
    float *out_race;            /* [B, 2]       winning race score ln(w(y)/E_y), and the
                                                runner-up score (approximate: the best of
                                                the tokens scored exactly, which can vary
                                                from call to call) */
    void *prof_events[4];       /* optional cudaEvent_t: recorded before the first kernel and
                                   after each kernel of the call (sampling: two kernels, three
                                   with per-position statistics, one with SPEC_FLAG_EARLY_EXIT;
                                   greedy: two) */
    uint32_t flags;             /* SPEC_FLAG_* / SPEC_DEBUG_* bits; 0 in normal use; any other
                                   bit is SPEC_EINVAL */
    /* Per-position statistics ("投机解码的第二本账" (SparseSpec-L), section 3.3: every draft
     * token's entropy feeds two class centres, accepted and rejected, kept as moving
     * averages; "SubSpec: the target model's own low-bit shadow as the draft model" quotes
     * the draft-target KL divergence).  Device, NULL = not computed; all in nats.  Asking
     * for any of them reads every logit in one pass paired by position (target row i with
     * draft row i) and runs the full read whatever the flags say. */
    float *out_H_p;             /* [B, gamma+1] entropy of p_i = softmax(L_t[b,i] / T_b) */
    float *out_H_q;             /* [B, gamma]   entropy of q_i = softmax(L_d[b,i] / Td_b) */
    float *out_KL;              /* [B, gamma]   KL(p_i || q_i) (+inf where q = 0 < p) */
    double *ctrl_centres;       /* [B, 2] device (accepted, rejected) class centres of draft
                                   entropies, updated in place after the verify: positions
                                   before the first rejection j move the accepted centre,
                                   position j (if j < gamma) the rejected one, in position
                                   order, c <- (1 - beta) c + beta H(q_i); positions after j
                                   and sequences with a bad draft token leave them alone */
    double ctrl_beta;           /* the moving averages' rate, 0 < beta <= 1 (else SPEC_EINVAL
                                   when ctrl_centres is set) */
} spec_verify_opts;

/* flags bits (bit 0 is unused). */
#define SPEC_DEBUG_NEVER_READY 2u /* tests only, with SPEC_FLAG_EARLY_EXIT: no race unit
                                     publishes its winner, so each sequence's last race unit
                                     waits for them until its bounded wait (0.5 s) gives up,
                                     records SPEC_ETIMEOUT and draws from p_j instead (the
                                     outputs are then invalid).  Exercises the bounded waits
                                     without faulting or hanging the device. */
#define SPEC_FLAG_EARLY_EXIT 4u   /* sampling, spec_verify_ex only: read each sequence's rows one
                                     position at a time and stop after its first rejection (the
                                     rows the method discards); one persistent cooperative
                                     kernel schedules the rows, decisions and races.  Same
                                     outputs under the same rules as the full read; fewer bytes
                                     when drafts are rejected early.  Ignored (the full read
                                     runs) when any diagnostic output is requested, since those
                                     cover every row, or when the device has no cooperative
                                     launch. */

#define SPEC_FLAG_FULL_READ 8u    /* spec_verify_host only: read every row (the default there
                                     is SPEC_FLAG_EARLY_EXIT) */
#define SPEC_DEBUG_RACE_AGAIN 16u /* tests only, spec_verify_lmhead: the race starts from a score
                                     above any winner, so every sequence is raced a second time
                                     from nothing; the outputs must not change. */

/* Zero every field and set dtype = SPEC_BF16. */
void spec_verify_opts_init(spec_verify_opts *opts);

/*
 * Sampling-mode verify on bf16 logits with scalar temperatures T > 0 and T_d > 0
 * ("How speculative decoding makes LLMs go brrr", pseudocode and module 3).
 * target_logits [B, gamma+1, V] bf16, draft_logits [B, gamma, V] bf16,
 * draft_tokens [B, gamma] int32; writes out_tokens [B, gamma+1] and out_n_accepted [B].
 * Returns SPEC_EINVAL for B < 0, gamma < 0, V < 1, a non-finite or non-positive
 * temperature, a NULL pointer (other than draft_logits / draft_tokens when gamma == 0) or a
 * misaligned logit pointer; SPEC_ECUDA / SPEC_ENOMEM on runtime failures.
 */
int spec_verify(const void *target_logits, const void *draft_logits,
                const int32_t *draft_tokens, int B, int gamma, int V, float T, float T_d,
                uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted, void *stream);

/*
 * Greedy (T = 0) verify on bf16 target logits: g_i = the first argmax of row i of the raw
 * target logits; draft token i is accepted while d_i == g_i; the cycle emits
 * d_0..d_{j-1}, g_j.  The draft logits are not needed.
 * (SubSpec's report runs its main tables at T = 0; the argmax-match rule is the plain
 * reading of greedy verification.)
 */
int spec_verify_greedy(const void *target_logits, const int32_t *draft_tokens, int B, int gamma,
                       int V, int32_t *out_tokens, int32_t *out_n_accepted, void *stream);

/* Full form of spec_verify: element type, per-sequence temperatures, caller workspace,
 * status word, global sequence index and diagnostic outputs through `opts` (NULL = the
 * defaults of spec_verify). */
int spec_verify_ex(const void *target_logits, const void *draft_logits,
                   const int32_t *draft_tokens, int B, int gamma, int V, float T, float T_d,
                   uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted,
                   const spec_verify_opts *opts, void *stream);

/* Full form of spec_verify_greedy (uses opts->dtype, workspace, d_status, prof_events). */
int spec_verify_greedy_ex(const void *target_logits, const int32_t *draft_tokens, int B,
                          int gamma, int V, int32_t *out_tokens, int32_t *out_n_accepted,
                          const spec_verify_opts *opts, void *stream);

/* Bytes of caller workspace the _ex entry points need for this problem (either mode).
 * Returns 0 for invalid sizes. */
size_t spec_verify_workspace_bytes(int B, int gamma, int V, int dtype);

/* Synchronise `stream`, read the device status word (NULL = the library's own status word
 * of the current device), reset it to SPEC_OK and return what it held (or SPEC_ECUDA). */
int spec_verify_check(void *stream, int32_t *d_status);

/*
 * Diagnostic: Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 * 1, 2, 3", SC'11, section 4) exactly as the verify kernels evaluate it, for testing the
 * device generator word for word.  counters [n, 4] and out [n, 4] uint32 (16-byte aligned),
 * keys [n, 2] uint32 (8-byte aligned), all device memory: out[i] = Philox4x32-10 of counter
 * i under key (keys[i][0], keys[i][1]).  form 0: the plain ten rounds (the acceptance
 * uniforms' path); form 1: the race's evaluation, which takes counter word 3 as 1 and
 * precomputes the per-row parts of rounds 1 and 2.  Asynchronous on `stream`; SPEC_EINVAL
 * for n < 0, another form, NULL or misaligned pointers.
 */
int spec_philox4x32_10(const uint32_t *counters, const uint32_t *keys, int64_t n, int form,
                       uint32_t *out, void *stream);

/* Static English text of a status code. */
const char *spec_verify_strerror(int status);

/*
 * Allocation-free form of spec_verify_ex.  The pages have no counterpart: this entry point
 * exists for callers that cannot let a library call cudaMalloc -- an inference server that
 * reserves nearly all device memory for its own pool up front, or a latency-critical caller
 * that may not block on the device synchronisation cudaMalloc/cudaFree can imply.  (The
 * other entry points allocate the library's status word, and the plain ones its workspace,
 * on first use.)
 *
 * The scratch (per-row partial statistics, per-sequence scan results, race partials and
 * arrival counters, and a status word) lives in one file-scope device array of
 * SPEC_NOALLOC_SCRATCH_BYTES, which every GPU that loads the library holds until the process
 * exits.  The caller still passes the inputs and outputs, exactly as for spec_verify_ex;
 * opts->workspace must be NULL.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress, with that device current); make that first call before any
 * stream capture.  Calls share the one array and it keeps the last call's contents: calls
 * that overlap on the GPU (other streams, other threads) race and give wrong results, so
 * serialise them.  Nothing in the array needs to start at zero: every call writes what it
 * reads.  Device-side errors go to opts->d_status when given; otherwise to a word inside the
 * array that this call clears first and that spec_verify_check cannot read: a caller who
 * needs to see SPEC_EBADTOKEN must pass opts->d_status (a bad draft token also shows as
 * n_accepted = -1).  This entry point runs the default two-kernel schedule only, whose one
 * wait (the last race block of a sequence polling the others' winners, bounded) follows
 * blocks that have already counted their arrival.  No cudaMalloc, cudaFree or allocating
 * library routine is called.
 * SPEC_FLAG_EARLY_EXIT, SPEC_DEBUG_NEVER_READY and the per-position statistics (out_H_p,
 * out_H_q, out_KL, ctrl_centres) are ignored here; other flag bits are SPEC_EINVAL.
 * Returns SPEC_ESCRATCH, without launching anything, when spec_verify_workspace_bytes() of
 * the problem exceeds SPEC_NOALLOC_SCRATCH_BYTES - 256; otherwise as spec_verify_ex.
 */
#define SPEC_NOALLOC_SCRATCH_BYTES (8u << 20) /* 8 MiB: B=256, gamma=12, V=152064 bf16 needs
                                                 6.1 MB */
int spec_verify_noalloc(const void *target_logits, const void *draft_logits,
                        const int32_t *draft_tokens, int B, int gamma, int V, float T, float T_d,
                        uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted,
                        const spec_verify_opts *opts, void *stream);

/*
 * Sampling verify on buffers in host memory.  Every pointer (logits, draft tokens,
 * outputs, and the per-sequence temperatures of opts) may be device memory or pinned host
 * memory mapped into the device address space (cudaHostAlloc, cudaHostRegister -- on this
 * GPU's coherent host link the kernels read and write it in place); pageable host memory
 * is refused with SPEC_EINVAL.  Reading logits over the host link is the bottleneck, so
 * this entry point verifies with SPEC_FLAG_EARLY_EXIT (only the rows up to each sequence's
 * first rejection cross the link) unless opts->flags has SPEC_FLAG_FULL_READ or a
 * diagnostic output is requested.  With early exit the rows it streams are also copied
 * into a library-owned device buffer the size of the logits (allocated on first use, grown
 * as needed), from which each sequence's race then reads its raced rows instead of crossing
 * the link a second time; if that allocation fails the race reads host memory.  Outputs land
 * in host memory when the stream's work completes: synchronise the stream before reading
 * them.  Otherwise as spec_verify_ex.
 */
int spec_verify_host(const void *target_logits, const void *draft_logits,
                     const int32_t *draft_tokens, int B, int gamma, int V, float T, float T_d,
                     uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted,
                     const spec_verify_opts *opts, void *stream);

/*
 * Static token-tree verify ("SubSpec: Speculate Deep and Accurate" (papernotes): a draft
 * token tree whose candidate paths one target forward verifies; SubSpec's tree is static,
 * deep and narrow).  The pages give no multi-branch rule; the one implemented is
 * multi-draft rejection sampling, lossless when the children of a node are independent
 * draws from that node's draft distribution: at node u its children are tried in node
 * order against the running residual p' = max(0, p_u - c q_u) / N (c = 0, N = 1 first;
 * after a rejection c <- c + N, N <- sum_x max(0, p_u(x) - c q_u(x))): child v with token x
 * is accepted iff u_v < min(1, p'(x) / q_u(x)), and the walk moves to v.  When every child
 * is rejected the token is drawn from p' (an exponential race); at a node without children
 * the bonus token is drawn from p_u.  A chain-shaped tree (parent[n] = n - 1) gives exactly
 * spec_verify_ex's tokens.
 * Random numbers: child v's uniform is counter (0, v - 1, b, 0) word 0; the race at node u
 * uses counters (x >> 2, u, b, 1) (b = seq_index_base + sequence).
 *   target_logits [B, N, V]: p at every node n (node 0 the root: the distribution after the
 *                 prefix; node n: after the path to n);
 *   draft_logits  [B, M, V]: q at every internal node (a node with children), row m = the
 *                 node's rank among internal nodes in node order (NULL when M = 0);
 *   draft_tokens  [B, N] int32: the token of node n >= 1 (column 0 unused);
 *   parent        [N] HOST int32: parent[0] = -1, 0 <= parent[n] < n; N <= 512;
 *   out_tokens    [B, D+1] int32 (D = the tree's depth): the accepted path's tokens, then
 *                 the drawn token, -1 padded; out_nodes [B, D] (device, NULL: skipped): the
 *                 accepted nodes, -1 padded; out_n_accepted [B]: accepted count (-1: a
 *                 draft token outside [0, V), which also sets SPEC_EBADTOKEN).
 * opts: dtype, per-sequence temperatures, seq_index_base, workspace, d_status and
 * prof_events (before the first kernel and after each of the three) are honoured; the
 * diagnostic and per-position outputs and the flags are not.  SPEC_EINVAL for a bad tree or
 * sizes, NULL or misaligned pointers, bad temperatures.
 */
int spec_verify_tree(const void *target_logits, const void *draft_logits,
                     const int32_t *draft_tokens, const int32_t *parent, int B, int N, int V,
                     float T, float T_d, uint64_t seed, int32_t *out_tokens, int32_t *out_nodes,
                     int32_t *out_n_accepted, const spec_verify_opts *opts, void *stream);

/*
 * The LM head on the tensor cores (tcgen05): logits L = H W^T with hidden states H
 * [rows, d] and head weights W [V, d], both bf16 row-major in device memory (16-byte
 * aligned), d a multiple of 64, accumulated in fp32.  spec_lmhead_logits writes L
 * [rows, V] fp32.  spec_lmhead_row_stats never writes L: its epilogue folds each tile into
 * the row's online softmax statistics at temperature T_row[row] (device [rows]) and keeps
 * the logit at token_row[row] (device [rows], -1: none; NULL when out_logp_token is NULL),
 * then writes out_logZ [rows] = ln sum_x exp(L[row, x] / T) and out_logp_token [rows] =
 * L[row, token] / T - ln Z (NaN without a token); either output may be NULL, not both.
 * These are the row statistics of the verify step ("How speculative decoding makes LLMs go
 * brrr", module 2: p_i = softmax of the target's logits at position i) computed from the
 * model's last hidden states, so the B (gamma+1) x V logits are never written and read
 * back.  spec_lmhead_row_stats uses the library's own workspace.  SPEC_EINVAL for bad sizes,
 * NULL or misaligned pointers; SPEC_ECUDA if the tensor-map encoder is unavailable.
 */
int spec_lmhead_logits(const void *hidden, const void *weight, int rows, int V, int d,
                       float *out_logits, void *stream);
int spec_lmhead_row_stats(const void *hidden, const void *weight, int rows, int V, int d,
                          const float *T_row, const int32_t *token_row, float *out_logZ,
                          float *out_logp_token, void *stream);

/*
 * The sampling verify step from the models' last hidden states ("How speculative decoding
 * makes LLMs go brrr", module 2: the gamma+1 target distributions of one forward pass, here
 * from the hidden states through the LM head): h_target [B, gamma+1, d]
 * with the target LM head w_target [V, d], and h_draft [B, gamma, d] with the draft LM head
 * w_draft [V, d] (may be w_target), all bf16 row-major device memory, d a multiple of 64 and
 * at most 32768.  The target and draft row statistics come from spec_lmhead_row_stats'
 * kernel (one pass over each head on the tensor cores; the B (2 gamma + 1) x V logits are
 * never written), which also keeps the largest logit of every 8-token block of the target
 * rows; each sequence's race then draws every token's random number, drops the tokens whose
 * block maximum cannot reach the best score found so far, and computes the logits h . w_x
 * of the rest (a few dozen per sequence) by dot products in fp32.  Outputs, decisions and
 * random numbers are those of spec_verify_ex run on the logits H W^T.  opts: per-sequence
 * temperatures, seq_index_base, d_status and prof_events (before the first kernel, after
 * the statistics, after the scan, after the race) are honoured; the library's own
 * workspace is used (B (gamma + 1) ceil(V / 8) bf16 block maxima plus a few words
 * per row).  Of opts->flags only SPEC_DEBUG_RACE_AGAIN is read.  SPEC_EINVAL for bad sizes,
 * NULL or misaligned pointers.
 */
int spec_verify_lmhead(const void *h_target, const void *w_target, const void *h_draft,
                       const void *w_draft, const int32_t *draft_tokens, int B, int gamma, int V,
                       int d, float T, float T_d, uint64_t seed, int32_t *out_tokens,
                       int32_t *out_n_accepted, const spec_verify_opts *opts, void *stream);

/*
 * Entropy of softmax(L / T) of each of `rows` contiguous rows of V logits (dtype
 * spec_dtype), in nats, into out_H [rows] (device) -- e.g. the next draft tokens' entropies
 * for spec_adaptive_k.  Uses the library's own workspace.  SPEC_EINVAL for bad sizes, a
 * non-positive or non-finite T, NULL or misaligned pointers.
 */
int spec_row_entropy(const void *logits, int rows, int V, float T, int dtype, float *out_H,
                     void *stream);

/*
 * Adaptive draft length ("投机解码的第二本账" (SparseSpec-L), section 3.3).  For each of B
 * sequences, the acceptance probability of its next draft tokens i = 1..K comes from their
 * entropies H_next [B, K] (device, fp32) and the sequence's class centres [B, 2] (device,
 * fp64: accepted, rejected): p_i = d_rej / (d_acc + d_rej) with d = |H_i - centre| (1/2 when
 * both distances are 0).  The chosen length is the candidate k maximising
 *     (1 + sum_{m=1..k} prod_{i=1..m} p_i) / (k C_d + C_v),
 * the earlier candidate on equal values; candidates (host array, 1..64 values, each in
 * 1..K) are the caller's, as are the draft and verify costs C_d and C_v.  Writes out_k [B]
 * (device int32) and, if not NULL, the best value into out_eff [B] (device fp64).  Computed
 * in fp64, each operation rounded on its own, in the order of the formula.  SPEC_EINVAL for
 * bad sizes, candidates outside 1..K, non-finite costs or a non-positive k C_d + C_v.
 */
int spec_adaptive_k(const float *H_next, int B, int K, const double *centres,
                    const int32_t *candidates, int n_cand, double C_d, double C_v,
                    int32_t *out_k, double *out_eff, void *stream);

/*
 * Vocabulary-parallel sampling verify ("How speculative decoding makes LLMs go brrr":
 * pseudocode and module 3, with the logits split by vocabulary column over W ranks, as a
 * tensor-parallel LM head leaves them).  Rank w holds target_shard [B, gamma+1, V_w] and
 * draft_shard [B, gamma, V_w]: columns [x_w, x_w + V_w) of every row, x_w a multiple of 8.
 * One verify is, on every rank, in this order on one stream:
 *   1. spec_vp_partials   -> stats [B, 2 gamma + 1, 2] (fp32 scaled max and sum of each row's
 *                            columns, base 2) and gathered [B, gamma, 2] (the target and draft
 *                            logits at each draft token the rank holds, -inf where it does not);
 *   2. the caller all-gathers stats into stats_all [W, B, 2 gamma + 1, 2] (rank order) and
 *      max-reduces gathered over the ranks;
 *   3. spec_vp_decide     -> out_tokens (accepted prefix, -1 padding; the drawn token's slot
 *                            is written in step 6), out_n_accepted, and state;
 *   4. spec_vp_race       -> keys [B, 2] int64: the rank's race winners (the residual race,
 *                            and the race over p_j where the rank's residual weights are all
 *                            zero), each as a key whose signed maximum is the winner;
 *   5. the caller max-reduces keys over the ranks;
 *   6. spec_vp_finish     -> the drawn token into out_tokens[b, j].
 * Random numbers are keyed by the global token index, so the result is the one-GPU verify's,
 * except that the two merge orders may round a near-tie (|u - p/q| or the top two race
 * scores within the tolerances of spec_verify) the other way.  All pointers are device
 * memory owned by the caller; state holds spec_vp_state_bytes(B) bytes (opaque), written by
 * step 3 and read by steps 4 and 6.  opts (may be NULL) supplies dtype, T_per_seq,
 * Td_per_seq, seq_index_base and d_status as in spec_verify_ex; step 1 uses the library
 * workspace (or opts->workspace, of spec_verify_workspace_bytes(B, gamma, V_w, dtype)).
 * Draft tokens outside [0, V) are reported by step 3 as in spec_verify (n_accepted = -1,
 * SPEC_EBADTOKEN in the status word).  SPEC_EINVAL for bad sizes, NULL or misaligned
 * pointers, an x_offset that is not a multiple of 8, bad temperatures.
 */
size_t spec_vp_state_bytes(int B);
int spec_vp_partials(const void *target_shard, const void *draft_shard, const int32_t *draft_tokens,
                     int B, int gamma, int V_shard, int x_offset, float T, float T_d,
                     float *out_stats, float *out_gathered, const spec_verify_opts *opts,
                     void *stream);
int spec_vp_decide(const float *stats_all, int world, const float *gathered,
                   const int32_t *draft_tokens, int B, int gamma, int V, float T, float T_d,
                   uint64_t seed, int32_t *out_tokens, int32_t *out_n_accepted, void *state,
                   const spec_verify_opts *opts, void *stream);
int spec_vp_race(const void *target_shard, const void *draft_shard, int B, int gamma, int V_shard,
                 int x_offset, uint64_t seed, const void *state, int64_t *out_keys,
                 const spec_verify_opts *opts, void *stream);
int spec_vp_finish(const int64_t *keys, const void *state, int B, int gamma, int32_t *out_tokens,
                   void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SPECVERIFY_H */
