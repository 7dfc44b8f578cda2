/*
 * specverify_oracle.c -- plain CPU oracle of the speculative-decoding verify step.
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT.  This is the slow, single-threaded,
 * fp64 restatement of what the CUDA library computes.  Only the tests, the smoke check
 * and the CPU-baseline leg of the benchmark load it.  It includes nothing from the CUDA
 * path and the CUDA path includes nothing from it; the two meet only through the
 * seeded input generators and the published definitions below.
 *
 * What it follows (web pages, cited by title and section):
 *   [GO-BRRR]  "How speculative decoding makes LLMs go brrr": the pseudocode of one
 *              speculative cycle (accept with a fresh uniform while it is below
 *              min(1, p/q); on the first rejection resample from the residual and drop
 *              the suffix; if every draft survives take one bonus token from row gamma),
 *              module 3 "rejection sampling and losslessness" (acceptance ratio, the
 *              residual norm(max(0, p - q)), the min(p, q) / max(0, p - q) mass split),
 *              module 4 (tau in [1, gamma + 1]).
 *   [SUBSPEC]  "SubSpec: the target model's own low-bit shadow as the draft model",
 *              section 2.2 and section 3.4 / Table 5 (the draft distribution is sharpened
 *              at its own temperature T_d), Tables 1-2 (greedy T = 0 runs).
 *   Philox4x32-10: Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as
 *              1, 2, 3", SC'11, section 4 (the Philox S-box: two 32x32->64 multiplies
 *              per round, Weyl-sequence key schedule, ten rounds).
 *
 * Readings where the pages are silent (each also listed in the design notes):
 *   - temperature: p = softmax(L / T), q = softmax(L_d / T_d); greedy is its own mode;
 *   - the accept test is strict, u < min(1, p/q); u has 24 random bits;
 *   - p(d) = 0 rejects; q(d) = 0 with p(d) > 0 accepts;
 *   - "sample from norm(max(0, p - q))" is an exponential race
 *     argmax_x r(x) / E_x over x with r(x) > 0, E_x ~ Exp(1) from Philox (the race is
 *     scale-free, so the normalisation needs no sum); if every r(x) is 0 the race runs
 *     over p instead; equal scores go to the lowest x;
 *   - the bonus token is the same race over p at row gamma;
 *   - greedy: g_i = first argmax of the raw target logits of row i; accept while d_i == g_i.
 *
 * Precision: every floating-point quantity is computed in fp64 (inputs are widened
 * exactly: bf16 -> fp32 -> fp64).  A decision that turns floating point into an integer
 * (the accept test, the race argmax) is taken on the fp32 rounding of the fp64 value,
 * the precision the GPU path decides in; the fp64 margins are reported so that the
 * caller can flag near-ties.
 *
 * Random-number contract (Philox4x32-10, key = (lo32(seed), hi32(seed)), b = global
 * sequence index):
 *   acceptance uniform of position i:  counter (0, i, b, 0), word 0 w;
 *                                      u = (w >> 8) * 2^-24          (exact in fp32)
 *   race exponential of token x at row pos: counter (x >> 2, pos, b, 1), word (x & 3) w;
 *                                      U = (w + 0.5) * 2^-32, E = -log1p(-U)
 *
 * Build: gcc -O2 -std=c11 -ffp-contract=off -fPIC -shared -o liboracle.so specverify_oracle.c -lm
 * (-ffp-contract=off keeps the arithmetic identical on x86-64 and aarch64).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTATION
#define ORACLE_MUTATION 0 /* tests build deliberately broken copies to show the pins bite */
#endif

/* ------------------------------------------------------------------------------------ */
/* Philox4x32-10 (SC'11, section 4).                                                     */
/* ------------------------------------------------------------------------------------ */

/* The two round multipliers and the two Weyl key increments chosen in the paper. */
#define PHILOX_M0 0xD2511F53u
#define PHILOX_M1 0xCD9E8D57u
#define PHILOX_W0 0x9E3779B9u /* golden ratio */
#define PHILOX_W1 0xBB67AE85u /* sqrt(3) - 1 */

static void mul_hilo32(uint32_t a, uint32_t b, uint32_t *hi, uint32_t *lo) {
    uint64_t p = (uint64_t)a * (uint64_t)b;
    *hi = (uint32_t)(p >> 32);
    *lo = (uint32_t)p;
}

void oracle_philox4x32_10(const uint32_t ctr_in[4], const uint32_t key_in[2], uint32_t out[4]) {
    uint32_t c0 = ctr_in[0], c1 = ctr_in[1], c2 = ctr_in[2], c3 = ctr_in[3];
    uint32_t k0 = key_in[0], k1 = key_in[1];
    for (int round = 0; round < 10; ++round) {
        if (round > 0) { /* key schedule: bump between rounds */
            k0 += PHILOX_W0;
            k1 += PHILOX_W1;
        }
        uint32_t hi0, lo0, hi1, lo1;
        mul_hilo32(PHILOX_M0, c0, &hi0, &lo0);
        mul_hilo32(PHILOX_M1, c2, &hi1, &lo1);
        uint32_t n0 = hi1 ^ c1 ^ k0;
        uint32_t n1 = lo1;
        uint32_t n2 = hi0 ^ c3 ^ k1;
        uint32_t n3 = lo0;
        c0 = n0; c1 = n1; c2 = n2; c3 = n3;
    }
    out[0] = c0; out[1] = c1; out[2] = c2; out[3] = c3;
}

static uint32_t philox_word(uint64_t seed, uint32_t c0, uint32_t c1, uint32_t c2, uint32_t c3,
                            int word) {
    uint32_t ctr[4] = {c0, c1, c2, c3};
    uint32_t key[2] = {(uint32_t)(seed & 0xffffffffu), (uint32_t)(seed >> 32)};
    uint32_t out[4];
    oracle_philox4x32_10(ctr, key, out);
    return out[word];
}

/* Acceptance uniform of (sequence b, draft position i): 24 random bits, exact in fp32. */
double oracle_accept_uniform(uint64_t seed, uint32_t b, uint32_t i) {
    uint32_t w = philox_word(seed, 0u, i, b, 0u, 0);
    return (double)(w >> 8) * (1.0 / 16777216.0);
}

/* Exp(1) variate of token x in the race at row `pos` of sequence b. */
double oracle_race_exponential(uint64_t seed, uint32_t b, uint32_t pos, uint32_t x) {
    uint32_t w = philox_word(seed, x >> 2, pos, b, 1u, (int)(x & 3u));
    double U = ((double)w + 0.5) * (1.0 / 4294967296.0);
    return -log1p(-U);
}

/* Bulk forms of the three functions above (for the statistical pins). */
void oracle_philox_bulk(const uint32_t *ctr, const uint32_t *key, int64_t n, uint32_t *out) {
    for (int64_t k = 0; k < n; ++k) oracle_philox4x32_10(ctr + 4 * k, key + 2 * k, out + 4 * k);
}

void oracle_accept_uniforms(uint64_t seed, uint32_t b_base, int B, int gamma, double *out) {
    for (int b = 0; b < B; ++b)
        for (int i = 0; i < gamma; ++i)
            out[(int64_t)b * gamma + i] = oracle_accept_uniform(seed, b_base + (uint32_t)b, (uint32_t)i);
}

void oracle_race_exponentials(uint64_t seed, uint32_t b, uint32_t pos, uint32_t x0, int64_t n,
                              double *out) {
    for (int64_t k = 0; k < n; ++k) out[k] = oracle_race_exponential(seed, b, pos, x0 + (uint32_t)k);
}

/* ------------------------------------------------------------------------------------ */
/* Input widening and per-row softmax statistics.                                        */
/* ------------------------------------------------------------------------------------ */

enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

static double widen(int dtype, const void *base, int64_t idx) {
    if (dtype == ORACLE_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

/* log of the softmax normaliser of one row at temperature temp:
 *   log Z = log sum_x exp(L[x] / temp), computed as M + log sum exp(L/temp - M). */
static double row_log_normaliser(int dtype, const void *base, int64_t row_off, int V, double temp) {
    double M = -INFINITY;
    for (int x = 0; x < V; ++x) {
        double l = widen(dtype, base, row_off + x) / temp;
        if (l > M) M = l;
    }
    if (M == -INFINITY) return -INFINITY;
    double S = 0.0;
    for (int x = 0; x < V; ++x) S += exp(widen(dtype, base, row_off + x) / temp - M);
    return M + log(S);
}

/* Public helper: log Z for each of `rows` contiguous rows (used by the p, q pins). */
void oracle_row_log_normalisers(int dtype, const void *base, int rows, int V,
                                const double *temp_per_row, double *out) {
    for (int r = 0; r < rows; ++r)
        out[r] = row_log_normaliser(dtype, base, (int64_t)r * V, V, temp_per_row[r]);
}

/* Public helper: per-row acceptance mass sum_x min(p(x), q(x)) [GO-BRRR module 3: the
 * mass that accepted draft tokens cover].  Used to calibrate the synthetic workloads. */
void oracle_row_overlap(int dtype, const void *target, const void *draft, int rows, int V,
                        const double *T_per_row, const double *Td_per_row, double *out) {
    for (int r = 0; r < rows; ++r) {
        int64_t off = (int64_t)r * V;
        double zp = row_log_normaliser(dtype, target, off, V, T_per_row[r]);
        double zq = row_log_normaliser(dtype, draft, off, V, Td_per_row[r]);
        double acc = 0.0;
        for (int x = 0; x < V; ++x) {
            double p = exp(widen(dtype, target, off + x) / T_per_row[r] - zp);
            double q = exp(widen(dtype, draft, off + x) / Td_per_row[r] - zq);
            acc += p < q ? p : q;
        }
        out[r] = acc;
    }
}

/* ------------------------------------------------------------------------------------ */
/* The exponential race: argmax_x w(x) / E_x in log form, log w(x) - log E_x.            */
/* ------------------------------------------------------------------------------------ */

typedef struct {
    int winner;          /* argmax on fp32-rounded scores, lowest x on equal scores; -1 if none */
    double best, second; /* fp64 top-two scores (for near-tie flags); -inf when absent */
} race_result;

/* Offer token x (offered in increasing x) with fp64 score.  The winner changes only on a
 * strictly larger fp32 score, so equal fp32 scores keep the lower x.  `second` tracks the
 * largest fp64 score of every other candidate; it can exceed `best` by less than one fp32
 * ulp when the fp32 decision kept an earlier equal score, which the near-tie flag catches. */
static void race_offer(race_result *r, int x, double score) {
    if (r->winner >= 0 && !((float)score > (float)r->best)) {
        if (score > r->second) r->second = score;
        return;
    }
    if (r->winner >= 0 && r->best > r->second) r->second = r->best;
    r->best = score;
    r->winner = x;
}

/* Race for the residual row (q_row != NULL) or the bonus / fallback row (q_row == NULL).
 *   residual weight r(x) = max(0, p(x) - q(x))                 [GO-BRRR module 3]
 *   log r(x) = log p(x) + log(1 - q(x)/p(x)) = lp + log(-expm1(lq - lp)), p > q.  */
static race_result run_race(int dtype, const void *target, int64_t t_off, double T, double logZp,
                            const void *draft, int64_t d_off, double Td, double logZq, int V,
                            uint64_t seed, uint32_t bg, uint32_t pos, int residual) {
    race_result r = {-1, -INFINITY, -INFINITY};
    for (int x = 0; x < V; ++x) {
        double lp = widen(dtype, target, t_off + x) / T - logZp;
        double lw;
        if (residual) {
            double lq = widen(dtype, draft, d_off + x) / Td - logZq;
#if ORACLE_MUTATION == 1 /* planted: residual max(0, q - p) instead of max(0, p - q) */
            { double t = lp; lp = lq; lq = t; }
#endif
#if ORACLE_MUTATION == 5 /* planted: residual ignores q entirely (samples p) */
            lq = -INFINITY;
#endif
            if (!(lp > lq)) continue; /* r(x) = 0: excluded */
            lw = (lq == -INFINITY) ? lp : lp + log(-expm1(lq - lp));
        } else {
            if (lp == -INFINITY) continue;
            lw = lp;
        }
        double E = oracle_race_exponential(seed, bg, pos, (uint32_t)x);
        race_offer(&r, x, lw - log(E));
    }
    return r;
}

/* ------------------------------------------------------------------------------------ */
/* Sampling-mode verify.                                                                 */
/* ------------------------------------------------------------------------------------ */

/* Output flags per sequence. */
#define ORACLE_FLAG_ACCEPT_NEAR_TIE 1 /* some tested position had |u - p/q| < 1e-5 */
#define ORACLE_FLAG_RACE_NEAR_TIE 2   /* top-two race scores within 1e-6 (relative) */
#define ORACLE_FLAG_BAD_TOKEN 4       /* a draft token outside [0, V) */
#define ORACLE_FLAG_RESIDUAL_EMPTY 8  /* every r(x) was 0: the race fell back to p */

/*
 * target [B, gamma+1, V], draft [B, gamma, V] (dtype ORACLE_F32 or ORACLE_BF16),
 * tokens [B, gamma], T/Td per sequence [B], b_base = global index of sequence 0.
 * Outputs (NULL = skip): out_tokens [B, gamma+1] (-1 padded), out_n [B] (-1 = bad token),
 * out_logp/out_logq/out_u/out_a [B, gamma] (ln p(d_i), ln q(d_i), u_i, p/q at every
 * position, tested or not), out_logZp [B, gamma+1], out_logZq [B, gamma],
 * out_race [B, 3] (best score, second score, row raced), out_flags [B].
 * Returns 0, or -1 on bad arguments.
 */
int oracle_verify(int dtype, const void *target, const void *draft, const int32_t *tokens, int B,
                  int gamma, int V, const double *T, const double *Td, uint64_t seed,
                  uint32_t b_base, int32_t *out_tokens, int32_t *out_n, double *out_logp,
                  double *out_logq, double *out_u, double *out_a, double *out_logZp,
                  double *out_logZq, double *out_race, int32_t *out_flags) {
    if (B < 0 || gamma < 0 || V < 1 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16)) return -1;
    double *lzp = (double *)malloc(sizeof(double) * (size_t)(gamma + 1));
    double *lzq = (double *)malloc(sizeof(double) * (size_t)(gamma + 1));
    if (!lzp || !lzq) { free(lzp); free(lzq); return -1; }

    for (int b = 0; b < B; ++b) {
        const uint32_t bg = b_base + (uint32_t)b;
        const double Tb = T[b], Tdb = Td[b];
        int32_t flags = 0;
        /* row statistics: target rows 0..gamma at T, draft rows 0..gamma-1 at T_d */
        for (int i = 0; i <= gamma; ++i) {
            lzp[i] = row_log_normaliser(dtype, target, ((int64_t)b * (gamma + 1) + i) * V, V, Tb);
            if (out_logZp) out_logZp[(int64_t)b * (gamma + 1) + i] = lzp[i];
        }
        for (int i = 0; i < gamma; ++i) {
#if ORACLE_MUTATION == 2 /* planted: draft normalised at T instead of T_d */
            lzq[i] = row_log_normaliser(dtype, draft, ((int64_t)b * gamma + i) * V, V, Tb);
#else
            lzq[i] = row_log_normaliser(dtype, draft, ((int64_t)b * gamma + i) * V, V, Tdb);
#endif
            if (out_logZq) out_logZq[(int64_t)b * gamma + i] = lzq[i];
        }
        int bad = 0;
        for (int i = 0; i < gamma; ++i) {
            int32_t d = tokens[(int64_t)b * gamma + i];
            if (d < 0 || d >= V) bad = 1;
        }
        /* per-position p(d_i), q(d_i), u_i, a_i */
        int j = gamma;
        for (int i = 0; i < gamma; ++i) {
            int32_t d = tokens[(int64_t)b * gamma + i];
            double lp = NAN, lq = NAN, a = NAN;
            double u = oracle_accept_uniform(seed, bg, (uint32_t)i);
            if (!bad) {
                lp = widen(dtype, target, ((int64_t)b * (gamma + 1) + i) * V + d) / Tb - lzp[i];
#if ORACLE_MUTATION == 2
                lq = widen(dtype, draft, ((int64_t)b * gamma + i) * V + d) / Tb - lzq[i];
#else
                lq = widen(dtype, draft, ((int64_t)b * gamma + i) * V + d) / Tdb - lzq[i];
#endif
                /* a = p/q in the log domain so that underflow never gives 0/0 */
                if (lp == -INFINITY) a = 0.0;
                else if (lq == -INFINITY) a = INFINITY;
                else a = exp(lp - lq);
            }
            const int64_t k = (int64_t)b * gamma + i;
            if (out_logp) out_logp[k] = lp;
            if (out_logq) out_logq[k] = lq;
            if (out_u) out_u[k] = u;
            if (out_a) out_a[k] = a;
            if (!bad && j == gamma) { /* still in the accepted prefix: this position is tested */
                if (fabs(u - a) < 1e-5) flags |= ORACLE_FLAG_ACCEPT_NEAR_TIE;
#if ORACLE_MUTATION == 3 /* planted: non-strict comparison and ratio inverted */
                int accept = (float)u <= (float)(1.0 / a);
#else
                int accept = (float)u < (float)a; /* [GO-BRRR pseudocode / module 3] */
#endif
                if (!accept) j = i;
            }
        }
        int32_t *tok = out_tokens ? out_tokens + (int64_t)b * (gamma + 1) : NULL;
        if (bad) {
            flags |= ORACLE_FLAG_BAD_TOKEN;
            if (tok) for (int i = 0; i <= gamma; ++i) tok[i] = -1;
            if (out_n) out_n[b] = -1;
            if (out_race) { out_race[3 * b] = NAN; out_race[3 * b + 1] = NAN; out_race[3 * b + 2] = -1; }
            if (out_flags) out_flags[b] = flags;
            continue;
        }
        race_result rr;
        int race_row;
        if (j < gamma) {
            /* first rejection at j: resample from norm(max(0, p_j - q_j)), drop the suffix */
            race_row = j;
            rr = run_race(dtype, target, ((int64_t)b * (gamma + 1) + j) * V, Tb, lzp[j], draft,
                          ((int64_t)b * gamma + j) * V,
#if ORACLE_MUTATION == 2
                          Tb,
#else
                          Tdb,
#endif
                          lzq[j], V, seed, bg, (uint32_t)j, 1);
            if (rr.winner < 0) { /* every r(x) == 0: fall back to p_j */
                flags |= ORACLE_FLAG_RESIDUAL_EMPTY;
                rr = run_race(dtype, target, ((int64_t)b * (gamma + 1) + j) * V, Tb, lzp[j], NULL, 0,
                              1.0, 0.0, V, seed, bg, (uint32_t)j, 0);
            }
        } else {
            /* every draft accepted: one bonus token from row gamma */
#if ORACLE_MUTATION == 4 /* planted: bonus drawn from row gamma-1 */
            race_row = gamma > 0 ? gamma - 1 : 0;
#else
            race_row = gamma;
#endif
            rr = run_race(dtype, target, ((int64_t)b * (gamma + 1) + race_row) * V, Tb,
                          lzp[race_row], NULL, 0, 1.0, 0.0, V, seed, bg, (uint32_t)gamma, 0);
        }
        if (rr.second > -INFINITY && rr.best - rr.second < 1e-6) flags |= ORACLE_FLAG_RACE_NEAR_TIE;
        if (tok) {
            for (int i = 0; i < j; ++i) tok[i] = tokens[(int64_t)b * gamma + i];
            tok[j] = rr.winner;
            for (int i = j + 1; i <= gamma; ++i) tok[i] = -1;
        }
        if (out_n) out_n[b] = j;
        if (out_race) {
            out_race[3 * b] = rr.best;
            out_race[3 * b + 1] = rr.second;
            out_race[3 * b + 2] = (double)race_row;
        }
        if (out_flags) out_flags[b] = flags;
    }
    free(lzp);
    free(lzq);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Greedy (T = 0) verify [SUBSPEC Tables 1-2 run greedily; rule: argmax match].          */
/* ------------------------------------------------------------------------------------ */

int oracle_verify_greedy(int dtype, const void *target, const int32_t *tokens, int B, int gamma,
                         int V, int32_t *out_tokens, int32_t *out_n, int32_t *out_argmax) {
    if (B < 0 || gamma < 0 || V < 1 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16)) return -1;
    int32_t *g = (int32_t *)malloc(sizeof(int32_t) * (size_t)(gamma + 1));
    if (!g) return -1;
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i <= gamma; ++i) {
            const int64_t off = ((int64_t)b * (gamma + 1) + i) * V;
            int best = 0;
            double bv = widen(dtype, target, off);
            for (int x = 1; x < V; ++x) {
                double v = widen(dtype, target, off + x);
                if (v > bv) { bv = v; best = x; } /* strict: ties keep the lowest index */
            }
            g[i] = best;
            if (out_argmax) out_argmax[(int64_t)b * (gamma + 1) + i] = best;
        }
        int bad = 0;
        for (int i = 0; i < gamma; ++i) {
            int32_t d = tokens[(int64_t)b * gamma + i];
            if (d < 0 || d >= V) bad = 1;
        }
        int32_t *tok = out_tokens ? out_tokens + (int64_t)b * (gamma + 1) : NULL;
        if (bad) {
            if (tok) for (int i = 0; i <= gamma; ++i) tok[i] = -1;
            if (out_n) out_n[b] = -1;
            continue;
        }
        int j = gamma;
        for (int i = 0; i < gamma; ++i)
            if (tokens[(int64_t)b * gamma + i] != g[i]) { j = i; break; }
        if (tok) {
            for (int i = 0; i < j; ++i) tok[i] = tokens[(int64_t)b * gamma + i];
            tok[j] = g[j];
            for (int i = j + 1; i <= gamma; ++i) tok[i] = -1;
        }
        if (out_n) out_n[b] = j;
    }
    free(g);
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Per-position draft statistics and the adaptive draft length.                          */
/*                                                                                       */
/* [SPARSESPEC] "投机解码的第二本账" (SparseSpec-L), section 3.3: every draft token        */
/* records the entropy H_i of its distribution; after verification the entropies of     */
/* accepted and of rejected tokens feed two class centres kept as exponential moving    */
/* averages; a new draft token is classified softly by its distances to the two centres, */
/* giving an acceptance probability p_i; the draft length is the k of a candidate set    */
/* that maximises (1 + sum_{m=1..k} prod_{i=1..m} p_i) / (k C_d + C_v).                  */
/* [SUBSPEC] "SubSpec: the target model's own low-bit shadow as the draft model" quotes   */
/* the draft-target KL divergence as its alignment measure; KL(p_i || q_i) per position   */
/* is reported beside the entropies.                                                     */
/*                                                                                       */
/* Readings where the page is silent (each also listed in the design notes):            */
/*   - H_i is the entropy of the draft distribution q_i = softmax(L_d / T_d), the one    */
/*     the draft token was drawn from, in nats;                                          */
/*   - after a verify with first rejection j, positions i < j update the accepted centre */
/*     and position j (if j < gamma) the rejected centre, in position order; positions   */
/*     after j were never tested and leave the centres alone; c <- (1 - beta) c +       */
/*     beta H_i with beta given by the caller;                                           */
/*   - soft classification: p = d_rej / (d_acc + d_rej) with d = |H - centre| (1/2 when  */
/*     both distances are 0);                                                            */
/*   - the candidate set, C_d and C_v are the caller's; equal efficiencies keep the      */
/*     earlier candidate.                                                                */
/* ------------------------------------------------------------------------------------ */

/* Entropy of softmax(L / temp) of one row, in nats: -sum_x p(x) log p(x) (0 log 0 = 0). */
static double row_entropy(int dtype, const void *base, int64_t off, int V, double temp) {
    const double lz = row_log_normaliser(dtype, base, off, V, temp);
    double h = 0.0;
    for (int x = 0; x < V; ++x) {
        const double l = widen(dtype, base, off + x) / temp - lz;
        const double p = exp(l);
#if ORACLE_MUTATION == 9 /* planted: the entropy sums p log p with the wrong sign */
        if (p > 0.0) h += p * l;
#else
        if (p > 0.0) h -= p * l;
#endif
    }
    return h;
}

/* KL(p || q) of one position: sum_x p(x) (log p(x) - log q(x)); terms with p(x) = 0 are 0,
 * and q(x) = 0 < p(x) makes it +inf. */
static double row_kl(int dtype, const void *target, const void *draft, int64_t off, int V,
                     double T, double Td) {
    const double zp = row_log_normaliser(dtype, target, off, V, T);
    const double zq = row_log_normaliser(dtype, draft, off, V, Td);
    double kl = 0.0;
    for (int x = 0; x < V; ++x) {
        const double lp = widen(dtype, target, off + x) / T - zp;
        const double p = exp(lp);
        if (p == 0.0) continue;
        const double lq = widen(dtype, draft, off + x) / Td - zq;
        kl += p * (lp - lq);
    }
    return kl;
}

/* H(p_i) for i <= gamma, H(q_i) and KL(p_i || q_i) for i < gamma, every sequence (NULL
 * outputs are skipped).  T, Td: per sequence. */
void oracle_position_stats(int dtype, const void *target, const void *draft, int B, int gamma,
                           int V, const double *T, const double *Td, double *out_Hp,
                           double *out_Hq, double *out_KL) {
    for (int b = 0; b < B; ++b) {
        for (int i = 0; i <= gamma; ++i) {
            const int64_t toff = ((int64_t)b * (gamma + 1) + i) * V;
            if (out_Hp) out_Hp[(int64_t)b * (gamma + 1) + i] = row_entropy(dtype, target, toff, V, T[b]);
            if (i == gamma) continue;
            const int64_t doff = ((int64_t)b * gamma + i) * V;
            if (out_Hq) out_Hq[(int64_t)b * gamma + i] = row_entropy(dtype, draft, doff, V, Td[b]);
            if (out_KL) {
                /* target row i and draft row i have different offsets: KL over the pair */
                const double zp = row_log_normaliser(dtype, target, toff, V, T[b]);
                const double zq = row_log_normaliser(dtype, draft, doff, V, Td[b]);
                double kl = 0.0;
                for (int x = 0; x < V; ++x) {
                    const double lp = widen(dtype, target, toff + x) / T[b] - zp;
                    const double p = exp(lp);
                    if (p == 0.0) continue;
                    kl += p * (lp - (widen(dtype, draft, doff + x) / Td[b] - zq));
                }
                out_KL[(int64_t)b * gamma + i] = kl;
            }
        }
    }
}

/* Rows laid out alike (row r of `target` and of `draft`): KL per row (for the pins). */
void oracle_row_kl(int dtype, const void *target, const void *draft, int rows, int V,
                   double T, double Td, double *out) {
    for (int r = 0; r < rows; ++r) out[r] = row_kl(dtype, target, draft, (int64_t)r * V, V, T, Td);
}

/* Entropy of each of `rows` contiguous rows at temperature temp. */
void oracle_row_entropies(int dtype, const void *base, int rows, int V, double temp, double *out) {
    for (int r = 0; r < rows; ++r) out[r] = row_entropy(dtype, base, (int64_t)r * V, V, temp);
}

/* Class centres after a verify: centres[b] = {accepted, rejected}, Hq[b][i] the draft
 * entropies, n[b] the accepted count (gamma: all accepted; -1: bad draft, no update). */
void oracle_entropy_centres_update(int B, int gamma, const double *Hq, const int32_t *n,
                                   double beta, double *centres) {
    for (int b = 0; b < B; ++b) {
        const int j = n[b];
        if (j < 0) continue;
        for (int i = 0; i <= j && i < gamma; ++i) {
#if ORACLE_MUTATION == 6 /* planted: the accepted and rejected centres swapped */
            double *c = centres + 2 * (int64_t)b + (i < j ? 1 : 0);
#else
            double *c = centres + 2 * (int64_t)b + (i < j ? 0 : 1);
#endif
            *c = (1.0 - beta) * *c + beta * Hq[(int64_t)b * gamma + i];
        }
    }
}

/* Acceptance probability of a draft token of entropy H. */
double oracle_soft_accept(double H, double c_acc, double c_rej) {
    const double da = fabs(H - c_acc), dr = fabs(H - c_rej);
    if (da + dr == 0.0) return 0.5;
#if ORACLE_MUTATION == 7 /* planted: soft classification inverted */
    return da / (da + dr);
#else
    return dr / (da + dr);
#endif
}

/* k* per sequence from the entropies H[b][0..K-1] of its next K draft tokens: candidates
 * cand[0..n_cand-1] (each in 1..K); out_eff[b] = the best efficiency (NULL: skipped). */
int oracle_adaptive_k(int B, int K, const double *H, const double *centres,
                      const int32_t *cand, int n_cand, double Cd, double Cv, int32_t *out_k,
                      double *out_eff) {
    for (int c = 0; c < n_cand; ++c)
        if (cand[c] < 1 || cand[c] > K) return -1;
    for (int b = 0; b < B; ++b) {
        int best_k = -1;
        double best = -INFINITY;
        for (int c = 0; c < n_cand; ++c) {
            const int k = cand[c];
            double prod = 1.0, expect = 0.0;
            for (int m = 0; m < k; ++m) {
#if ORACLE_MUTATION == 8 /* planted: expected yield sums p_i instead of prefix products */
                prod = oracle_soft_accept(H[(int64_t)b * K + m], centres[2 * (int64_t)b],
                                          centres[2 * (int64_t)b + 1]);
#else
                prod *= oracle_soft_accept(H[(int64_t)b * K + m], centres[2 * (int64_t)b],
                                           centres[2 * (int64_t)b + 1]);
#endif
                expect += prod;
            }
            const double eff = (1.0 + expect) / ((double)k * Cd + Cv);
            if (eff > best) {
                best = eff;
                best_k = k;
            }
        }
        out_k[b] = best_k;
        if (out_eff) out_eff[b] = best;
    }
    return 0;
}

/* ------------------------------------------------------------------------------------ */
/* Static token-tree verification.                                                       */
/*                                                                                       */
/* [SUBSPEC] "SubSpec: Speculate Deep and Accurate" (papernotes), on SpecInfer: the draft */
/* is a token tree whose candidate paths one target forward verifies in parallel; SubSpec */
/* keeps a static tree, deep and narrow (k = 6, depth 48).  The pages do not give the     */
/* multi-branch acceptance rule.  Reading taken (SpecInfer's multi-draft speculative      */
/* sampling, which is lossless when the children of a node are independent draws from    */
/* that node's draft distribution q_u):                                                  */
/*   at node u, with target distribution p_u, try its children v (in node order) with    */
/*   the running residual p' = max(0, p_u - c q_u) / N (c = 0, N = 1 at first):          */
/*   accept child v, token x, iff u_v < min(1, p'(x) / q_u(x)); on acceptance move to v; */
/*   on rejection set c <- c + N, N <- sum_x max(0, p_u(x) - c q_u(x)) (the next         */
/*   residual, norm(max(0, p' - q_u)) written in closed form) and try the next child.    */
/*   If every child is rejected, draw from p' (the race over max(0, p_u - c q_u)); at a   */
/*   node without children (an accepted leaf, or a root with none), draw the bonus token  */
/*   from p_u.  A chain-shaped tree is exactly the chain verify above.                  */
/* Random numbers: child v's uniform is counter (0, v - 1, b, 0) word 0 (a chain's node  */
/* v is its draft position v - 1); the race at node u uses counters (x >> 2, u, b, 1).    */
/* ------------------------------------------------------------------------------------ */

/* Race over max(0, p - c q) (c > 0), or over p (c == 0). */
static race_result run_race_scaled(int dtype, const void *target, int64_t t_off, double T,
                                   double logZp, const void *draft, int64_t d_off, double Td,
                                   double logZq, double c, int V, uint64_t seed, uint32_t bg,
                                   uint32_t pos) {
    race_result r = {-1, -INFINITY, -INFINITY};
    const double logc = c > 0.0 ? log(c) : 0.0;
    for (int x = 0; x < V; ++x) {
        const double lp = widen(dtype, target, t_off + x) / T - logZp;
        double lw;
        if (c > 0.0) {
            const double lq = widen(dtype, draft, d_off + x) / Td - logZq + logc; /* log(c q) */
            if (!(lp > lq)) continue;
            lw = (lq == -INFINITY) ? lp : lp + log(-expm1(lq - lp));
        } else {
            if (lp == -INFINITY) continue;
            lw = lp;
        }
        race_offer(&r, x, lw - log(oracle_race_exponential(seed, bg, pos, (uint32_t)x)));
    }
    return r;
}

/*
 * target [B, N, V]: p at every node (node 0 the root); draft [B, M, V]: q at every internal
 * node (draft row m = the node's rank among the nodes with children); tokens [B, N]: the
 * token of node n >= 1 (column 0 unused); parent [N]: parent[0] = -1, 0 <= parent[n] < n.
 * Outputs (NULL = skip): out_tokens [B, D+1] (accepted path tokens then the drawn token,
 * -1 padded; D = the tree's depth), out_nodes [B, D] (accepted nodes, -1 padded), out_n [B]
 * (accepted count, -1 = bad token), out_flags [B].  Returns 0, or -1 on bad arguments.
 */
int oracle_verify_tree(int dtype, const void *target, const void *draft, const int32_t *tokens,
                       const int32_t *parent, int B, int N, int V, const double *T,
                       const double *Td, uint64_t seed, uint32_t b_base, int32_t *out_tokens,
                       int32_t *out_nodes, int32_t *out_n, int32_t *out_flags) {
    if (B < 0 || N < 1 || V < 1 || (dtype != ORACLE_F32 && dtype != ORACLE_BF16)) return -1;
    if (parent[0] != -1) return -1;
    for (int n = 1; n < N; ++n)
        if (parent[n] < 0 || parent[n] >= n) return -1;
    int *depth = (int *)calloc((size_t)N, sizeof(int));
    int *nchild = (int *)calloc((size_t)N, sizeof(int));
    int *drow = (int *)malloc(sizeof(int) * (size_t)N);
    if (!depth || !nchild || !drow) { free(depth); free(nchild); free(drow); return -1; }
    int D = 0, M = 0;
    for (int n = 1; n < N; ++n) {
        depth[n] = depth[parent[n]] + 1;
        if (depth[n] > D) D = depth[n];
        nchild[parent[n]]++;
    }
    for (int n = 0; n < N; ++n) drow[n] = nchild[n] > 0 ? M++ : -1;
    for (int b = 0; b < B; ++b) {
        const uint32_t bg = b_base + (uint32_t)b;
        const double Tb = T[b], Tdb = Td[b];
        int32_t flags = 0;
        int32_t *tok = out_tokens ? out_tokens + (int64_t)b * (D + 1) : NULL;
        int32_t *nodes = out_nodes ? out_nodes + (int64_t)b * D : NULL;
        if (tok) for (int i = 0; i <= D; ++i) tok[i] = -1;
        if (nodes) for (int i = 0; i < D; ++i) nodes[i] = -1;
        int bad = 0;
        for (int n = 1; n < N; ++n) {
            const int32_t d = tokens[(int64_t)b * N + n];
            if (d < 0 || d >= V) bad = 1;
        }
        if (bad) {
            if (out_n) out_n[b] = -1;
            if (out_flags) out_flags[b] = ORACLE_FLAG_BAD_TOKEN;
            continue;
        }
        int u = 0, k = 0;
        race_result rr;
        for (;;) {
            const int64_t t_off = ((int64_t)b * N + u) * V;
            const double lzp = row_log_normaliser(dtype, target, t_off, V, Tb);
            if (nchild[u] == 0) { /* bonus token from p_u */
                rr = run_race_scaled(dtype, target, t_off, Tb, lzp, NULL, 0, 1.0, 0.0, 0.0, V,
                                     seed, bg, (uint32_t)u);
                break;
            }
            const int64_t d_off = ((int64_t)b * M + drow[u]) * V;
            const double lzq = row_log_normaliser(dtype, draft, d_off, V, Tdb);
            double c = 0.0, Nc = 1.0;
            int accepted = -1;
            for (int v = u + 1; v < N; ++v) {
                if (parent[v] != u) continue;
                const int32_t x = tokens[(int64_t)b * N + v];
                const double lp = widen(dtype, target, t_off + x) / Tb - lzp;
                const double lq = widen(dtype, draft, d_off + x) / Tdb - lzq;
                /* p'(x) = max(0, p(x) - c q(x)) / N, in the log domain */
                double lpp;
                if (c == 0.0) lpp = lp;
                else {
                    const double lcq = lq + log(c);
#if ORACLE_MUTATION == 11 /* planted: the running residual is not renormalised */
                    lpp = (lp > lcq) ? ((lcq == -INFINITY) ? lp : lp + log(-expm1(lcq - lp)))
                                     : -INFINITY;
#else
                    lpp = (lp > lcq) ? ((lcq == -INFINITY) ? lp : lp + log(-expm1(lcq - lp))) - log(Nc)
                                     : -INFINITY;
#endif
                }
                double a;
                if (lpp == -INFINITY) a = 0.0;
                else if (lq == -INFINITY) a = INFINITY;
                else a = exp(lpp - lq);
                const double uv = oracle_accept_uniform(seed, bg, (uint32_t)(v - 1));
                if (fabs(uv - a) < 1e-5) flags |= ORACLE_FLAG_ACCEPT_NEAR_TIE;
                if ((float)uv < (float)a) { accepted = v; break; }
#if ORACLE_MUTATION == 10 /* planted: the residual coefficient stops at 1 */
                c = 1.0;
#else
                c += Nc;
#endif
                double s = 0.0;
                for (int y = 0; y < V; ++y) {
                    const double p = exp(widen(dtype, target, t_off + y) / Tb - lzp);
                    const double q = exp(widen(dtype, draft, d_off + y) / Tdb - lzq);
                    if (p > c * q) s += p - c * q;
                }
                Nc = s;
            }
            if (accepted >= 0) {
                if (tok) tok[k] = tokens[(int64_t)b * N + accepted];
                if (nodes) nodes[k] = accepted;
                ++k;
                u = accepted;
                continue;
            }
            rr = run_race_scaled(dtype, target, t_off, Tb, lzp, draft, d_off, Tdb, lzq, c, V,
                                 seed, bg, (uint32_t)u);
            if (rr.winner < 0) { /* every residual weight was 0: fall back to p_u */
                flags |= ORACLE_FLAG_RESIDUAL_EMPTY;
                rr = run_race_scaled(dtype, target, t_off, Tb, lzp, NULL, 0, 1.0, 0.0, 0.0, V,
                                     seed, bg, (uint32_t)u);
            }
            break;
        }
        if (rr.second > -INFINITY && rr.best - rr.second < 1e-6) flags |= ORACLE_FLAG_RACE_NEAR_TIE;
        if (tok) tok[k] = rr.winner;
        if (out_n) out_n[b] = k;
        if (out_flags) out_flags[b] = flags;
    }
    free(depth);
    free(nchild);
    free(drow);
    return 0;
}
