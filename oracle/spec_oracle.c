/*
 * spec_oracle.c -- plain fp64 CPU oracle of the batched speculative-decoding
 * verify/commit step and of the confidence-scheduled verify-length pre-pass.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the independent checker for the CUDA
 * library: only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline /
 * reference arm load it.  It shares no code, header, table or helper with the
 * CUDA path (speculative_decoding_verification_15_gb300/csrc), and the product
 * path never calls it.
 *
 * Sources (page title -- section):
 *  [ALX]  "From draft-then-verify to DSpark" (alexine.rip) -- "How speculative
 *         decoding works": accept x with probability min(1, p(x)/q(x)); on
 *         rejection resample from normalise(max(0, p - q)); lossless.
 *  [PPR]  "Accelerating Large-Model Inference ..." (princepride.github.io) --
 *         Sec. 1 "Producing Multiple Tokens in a Single Forward Pass" (propose /
 *         verify / commit table: accept the longest prefix, resample at the first
 *         disagreement) and its worked examples.
 *  [VBK]  "DSpark paper review" (vllmbangkok.com) -- Sec. 4.2.1 (prefix survival
 *         c_1 x ... x c_k, non-increasing) and Sec. 4.2.2 (hardware-aware prefix
 *         scheduler: rank all draft tokens by survival, add one at a time, look up
 *         the startup step-time table; production variant searches the whole
 *         table instead of stopping at the first drop).
 *  [MTL]  "Bringing DSpark to vLLM Metal" (mhdimo.github.io) -- "Correctness is
 *         the feature": greedy path compares the target's argmax with the draft;
 *         "Making the draft cheaper": top-K Markov drafting (the correction only
 *         on the candidates picked from the base logits).
 *  [PPR2] "Accelerating Large-Model Inference ..." -- the drafting-engine table
 *         (layer 2, Markov head: a low-rank bias applied left to right, the bias at
 *         position k+1 set by the token chosen at position k).
 *  [SC11] Salmon, Moraes, Dror, Shaw, "Parallel random numbers: as easy as 1, 2,
 *         3", SC'11 -- Philox4x32-10.
 *
 * Readings where the pages are silent are stated at each function.  Everything
 * is fp64 with the host libm (exp, log); no blocking, fusion or reordering
 * beyond what the definitions state.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_BF16 0
#define OR_F32 1

/* per-request status codes (same meaning as the library's out_status) */
#define ST_OK 0
#define ST_BAD_TOKEN 1
#define ST_BAD_K 2
#define ST_BAD_T 3
#define ST_NONFINITE 4 /* a row that is read holds NaN or +inf, or is all -inf */

/* near-tie flag bits */
#define FL_THRESH 1     /* |u - P/Q| < 1e-5 * P/Q at a scanned position            */
#define FL_GUMBEL 2     /* top-2 Gumbel scores closer than 1e-5 * max(1,|top|)      */
#define FL_DEGENERATE 4 /* residual max(0, p - q) has empty support                 */
#define FL_ILLCOND 8    /* residual top-2 gap within the log(p-q) conditioning band */

#define REL_TIE 1e-5

/* ------------------------------------------------------------------------- */
/* Philox4x32-10 [SC11]: 10 rounds of the 4x32 S-box with multipliers         */
/* M0, M1 and the Weyl key schedule W0, W1.                                   */
/* ------------------------------------------------------------------------- */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
    const uint64_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    const uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
    uint32_t k0 = key[0], k1 = key[1];
    int round;
    for (round = 0; round < 10; ++round) {
        uint64_t prod0 = M0 * (uint64_t)x0;
        uint64_t prod1 = M1 * (uint64_t)x2;
        uint32_t y0 = (uint32_t)(prod1 >> 32) ^ x1 ^ k0;
        uint32_t y1 = (uint32_t)prod1;
        uint32_t y2 = (uint32_t)(prod0 >> 32) ^ x3 ^ k1;
        uint32_t y3 = (uint32_t)prod0;
        x0 = y0; x1 = y1; x2 = y2; x3 = y3;
        k0 += W0;
        k1 += W1;
    }
    out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

/*
 * Random word for vocabulary entry v of draw `purpose` at logit row `row` of
 * request b.  Reading (the pages define no RNG): key = (seed lo, seed hi);
 * counter = (v >> 2, b, (row << 4) | purpose, step lo); word v & 3.
 * Purposes: 0 = acceptance uniform (v = 0), 1 = residual Gumbel noise at the
 * first rejected row, 2 = bonus Gumbel noise at row k_b.
 */
uint32_t oracle_rand_word(uint64_t seed, uint64_t step, int b, int row, int purpose, int v) {
    uint32_t ctr[4], key[2], out[4];
    key[0] = (uint32_t)(seed & 0xffffffffu);
    key[1] = (uint32_t)(seed >> 32);
    ctr[0] = (uint32_t)v >> 2;
    ctr[1] = (uint32_t)b;
    ctr[2] = ((uint32_t)row << 4) | (uint32_t)purpose;
    ctr[3] = (uint32_t)(step & 0xffffffffu);
    oracle_philox4x32_10(ctr, key, out);
    return out[(uint32_t)v & 3u];
}

/* Uniform in (0,1): (2 * (w >> 9) + 1) * 2^-24, exact in fp32 and fp64. */
double oracle_u01(uint32_t w) { return (double)(2u * (w >> 9) + 1u) * (1.0 / 16777216.0); }

/* Gumbel(0,1) noise: g = -log(-log u). */
double oracle_gumbel(uint32_t w) { return -log(-log(oracle_u01(w))); }

/* ------------------------------------------------------------------------- */
/* Decoding and the temperature softmax                                      */
/* ------------------------------------------------------------------------- */
static double decode(const void *base, int dtype, int64_t idx) {
    if (dtype == OR_BF16) {
        uint16_t h = ((const uint16_t *)base)[idx];
        uint32_t bits = (uint32_t)h << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    }
    return (double)((const float *)base)[idx];
}

/* Max over a row with NaN propagation: NaN if any element is NaN. */
static double row_max_nan(const double *x, int V) {
    double m = -INFINITY;
    int v;
    for (v = 0; v < V; ++v) {
        if (isnan(x[v])) return NAN;
        if (x[v] > m) m = x[v];
    }
    return m;
}

/*
 * log p_v for p = softmax(x / T) over the full vocabulary [ALX] (p and q are the
 * target's and the draft's next-token distributions).  Reading: both target and
 * draft logits are divided by the request's temperature T > 0 before the
 * softmax; the max is subtracted for stability (it cancels exactly).
 */
void oracle_row_logprobs(const double *x, int V, double T, double *logp) {
    double m = -INFINITY, s = 0.0, ls;
    int v;
    for (v = 0; v < V; ++v) {
        double z = x[v] / T;
        if (z > m) m = z;
    }
    for (v = 0; v < V; ++v) s += exp(x[v] / T - m);
    ls = log(s);
    for (v = 0; v < V; ++v) logp[v] = x[v] / T - m - ls;
}

/* ------------------------------------------------------------------------- */
/* The acceptance rule and the residual [ALX]                                 */
/* ------------------------------------------------------------------------- */

/* Acceptance probability of a draft token with target probability P and draft
 * probability Q: min(1, P/Q).  Q = 0 (the draft could not have proposed it):
 * reading -- accept iff P > 0. */
double oracle_accept_prob(double P, double Q) {
    if (Q > 0.0) return P / Q < 1.0 ? P / Q : 1.0;
    return P > 0.0 ? 1.0 : 0.0;
}

/* Unnormalised residual weights r_v = max(0, p_v - q_v). */
void oracle_residual_weights(const double *p, const double *q, int V, double *r) {
    int v;
    for (v = 0; v < V; ++v) r[v] = p[v] > q[v] ? p[v] - q[v] : 0.0;
}

/*
 * Gumbel-max draw over log-weights lw (entries of -inf excluded): returns
 * argmax_v (lw_v + g_v), lowest v on exact ties, or -1 if every entry is -inf.
 * g_v comes from oracle_rand_word(seed, step, b, row, purpose, v).
 * *gap receives the difference between the two best scores (+inf if < 2);
 * *top the best score; *second_v the runner-up's index (-1 if none).
 */
static int gumbel_argmax(const double *lw, int V, uint64_t seed, uint64_t step, int b, int row,
                         int purpose, double *gap, double *top, int *second_v) {
    double best = -INFINITY, second = -INFINITY;
    int bi = -1, si = -1, v;
    for (v = 0; v < V; ++v) {
        double s;
        if (lw[v] == -INFINITY) continue;
        s = lw[v] + oracle_gumbel(oracle_rand_word(seed, step, b, row, purpose, v));
        if (s > best) {
            second = best; si = bi;
            best = s; bi = v;
        } else if (s > second) {
            second = s; si = v;
        }
    }
    *gap = (si >= 0) ? best - second : INFINITY;
    *top = best;
    *second_v = si;
    return bi;
}

/* Exposed for the Gumbel-max pin: draw from weights w (w_v = 0 excluded). */
int oracle_gumbel_sample(const double *w, int V, uint64_t seed, uint64_t step, int b, int row, int purpose) {
    double *lw = (double *)malloc(sizeof(double) * (size_t)(V > 0 ? V : 1));
    double gap, top;
    int sv, v, r;
    for (v = 0; v < V; ++v) lw[v] = w[v] > 0.0 ? log(w[v]) : -INFINITY;
    r = gumbel_argmax(lw, V, seed, step, b, row, purpose, &gap, &top, &sv);
    free(lw);
    return r;
}

/* Greedy argmax over raw values, lowest index on ties [MTL]. */
static int argmax_lowest(const double *x, int V) {
    int bi = 0, v;
    for (v = 1; v < V; ++v)
        if (x[v] > x[bi]) bi = v;
    return bi;
}

/* ------------------------------------------------------------------------- */
/* Per-request verify                                                         */
/* ------------------------------------------------------------------------- */
typedef struct {
    const void *target, *draft;
    int dtype, B, Kmax, V;
    int64_t ld_row;
    const int32_t *draft_tokens, *num_draft;
    const float *temperature; /* NULL: greedy for every request */
    uint64_t seed, step;
    int32_t *out_tokens, *out_accepted, *out_status, *out_flags;
    int32_t *out_flag_pos; /* first scanned position with a threshold near-tie, -1 if none */
    double *out_p, *out_q, *out_gap;
    /* early exit: read the rows position by position and stop at the first
     * rejection [PPR, ALX]; only rows read are checked for non-finite values and
     * p/q stay -1 past the first rejected position */
    int early_exit;
} verify_args;

static void load_row(const void *base, int dtype, int64_t row, int64_t ld_row, int V, double *dst) {
    int v;
    for (v = 0; v < V; ++v) dst[v] = decode(base, dtype, row * ld_row + v);
}

/* A request with a non-zero status emits nothing: accepted 0, tokens and p/q -1. */
static void fail_request(const verify_args *a, int b, int status) {
    int i;
    for (i = 0; i <= a->Kmax; ++i) a->out_tokens[(int64_t)b * (a->Kmax + 1) + i] = -1;
    for (i = 0; i < a->Kmax; ++i) {
        if (a->out_p) a->out_p[(int64_t)b * a->Kmax + i] = -1.0;
        if (a->out_q) a->out_q[(int64_t)b * a->Kmax + i] = -1.0;
    }
    a->out_status[b] = status;
    a->out_accepted[b] = 0;
    if (a->out_flags) a->out_flags[b] = 0;
    if (a->out_flag_pos) a->out_flag_pos[b] = -1;
    if (a->out_gap) a->out_gap[b] = INFINITY;
}

static void verify_one(const verify_args *a, int b, double *xt, double *xd, double *lpt, double *lpd,
                       double *tmp) {
    const int K1 = a->Kmax + 1, V = a->V;
    int32_t *tok = a->out_tokens + (int64_t)b * K1;
    const int32_t *x = a->draft_tokens + (int64_t)b * a->Kmax;
    int kb = a->num_draft ? a->num_draft[b] : a->Kmax;
    int i, v, status = ST_OK, greedy, A = 0, flags = 0, flag_pos = -1;
    double T = 0.0;
    double min_gap = INFINITY;

    for (i = 0; i < K1; ++i) tok[i] = -1;
    for (i = 0; i < a->Kmax; ++i) {
        if (a->out_p) a->out_p[(int64_t)b * a->Kmax + i] = -1.0;
        if (a->out_q) a->out_q[(int64_t)b * a->Kmax + i] = -1.0;
    }

    /* status checks, in this order: k_b, temperature, tokens, non-finite rows */
    if (kb < 0 || kb > a->Kmax) status = ST_BAD_K;
    if (!status && a->temperature) {
        T = (double)a->temperature[b];
        if (!(T >= 0.0) || isinf(T)) status = ST_BAD_T;
    }
    greedy = (a->temperature == NULL) || (T == 0.0);
    if (!status)
        for (i = 0; i < kb; ++i)
            if (x[i] < 0 || x[i] >= V) status = ST_BAD_TOKEN;
    if (!status && !a->early_exit) {
        /* rows of the draft positions: target 0..k_b-1, draft 0..k_b-1 (sampling only).
         * Reading: the target row k_b is checked only when it is read, i.e. when every
         * draft is accepted and the bonus (or greedy) token comes from it. */
        for (i = 0; i < kb && !status; ++i) {
            load_row(a->target, a->dtype, (int64_t)b * K1 + i, a->ld_row, V, xt);
            if (!isfinite(row_max_nan(xt, V))) status = ST_NONFINITE;
        }
        for (i = 0; i < kb && !greedy && !status; ++i) {
            load_row(a->draft, a->dtype, (int64_t)b * a->Kmax + i, a->ld_row, V, xd);
            if (!isfinite(row_max_nan(xd, V))) status = ST_NONFINITE;
        }
    }
    a->out_status[b] = status;
    if (a->out_flag_pos) a->out_flag_pos[b] = -1;
    if (status) {
        a->out_accepted[b] = 0;
        if (a->out_flags) a->out_flags[b] = 0;
        if (a->out_gap) a->out_gap[b] = INFINITY;
        return;
    }

    if (greedy) {
        /* greedy: y_i = argmax of the raw target row; accept while y_i == x_i [MTL] */
        int y = 0;
        for (i = 0; i <= kb; ++i) {
            load_row(a->target, a->dtype, (int64_t)b * K1 + i, a->ld_row, V, xt);
            if ((i == kb || a->early_exit) && !isfinite(row_max_nan(xt, V))) {
                fail_request(a, b, ST_NONFINITE);
                return;
            }
            y = argmax_lowest(xt, V);
            if (i == kb || y != x[i]) break;
            tok[i] = x[i];
            ++A;
        }
        tok[A] = y;
        a->out_accepted[b] = A;
        if (a->out_flags) a->out_flags[b] = 0;
        if (a->out_gap) a->out_gap[b] = INFINITY;
        return;
    }

    /* sampling: P_i = p_i(x_i), Q_i = q_i(x_i) for every draft position */
    {
        int rejected = 0;
        for (i = 0; i < kb; ++i) {
            double P, Q, u, ratio;
            load_row(a->target, a->dtype, (int64_t)b * K1 + i, a->ld_row, V, xt);
            load_row(a->draft, a->dtype, (int64_t)b * a->Kmax + i, a->ld_row, V, xd);
            if (a->early_exit && (!isfinite(row_max_nan(xt, V)) || !isfinite(row_max_nan(xd, V)))) {
                fail_request(a, b, ST_NONFINITE);
                return;
            }
            oracle_row_logprobs(xt, V, T, lpt);
            oracle_row_logprobs(xd, V, T, lpd);
            P = exp(lpt[x[i]]);
            Q = exp(lpd[x[i]]);
            if (a->out_p) a->out_p[(int64_t)b * a->Kmax + i] = P;
            if (a->out_q) a->out_q[(int64_t)b * a->Kmax + i] = Q;
            if (rejected) continue;
            /* accept with probability min(1, P/Q): u < P/Q with u uniform in (0,1) [ALX] */
            u = oracle_u01(oracle_rand_word(a->seed, a->step, b, i, 0, 0));
            if (Q > 0.0) {
                ratio = P / Q;
                if (fabs(u - ratio) < REL_TIE * ratio) {
                    flags |= FL_THRESH;
                    if (flag_pos < 0) flag_pos = i;
                }
                if (u < ratio) { tok[i] = x[i]; ++A; continue; }
            } else if (P > 0.0) {
                tok[i] = x[i]; ++A; continue;
            }
            rejected = 1; /* first rejection: position A == i [PPR] */
            if (a->early_exit) break;
        }
    }

    if (A < kb) {
        /* correction at j = A: Gumbel-max over log max(0, p_j - q_j) [ALX] */
        const int j = A;
        double gap, top;
        int tk, sv;
        load_row(a->target, a->dtype, (int64_t)b * K1 + j, a->ld_row, V, xt);
        load_row(a->draft, a->dtype, (int64_t)b * a->Kmax + j, a->ld_row, V, xd);
        oracle_row_logprobs(xt, V, T, lpt);
        oracle_row_logprobs(xd, V, T, lpd);
        for (v = 0; v < V; ++v) { lpt[v] = exp(lpt[v]); lpd[v] = exp(lpd[v]); }
        oracle_residual_weights(lpt, lpd, V, tmp);
        for (v = 0; v < V; ++v) tmp[v] = tmp[v] > 0.0 ? log(tmp[v]) : -INFINITY;
        tk = gumbel_argmax(tmp, V, a->seed, a->step, b, j, 1, &gap, &top, &sv);
        if (tk >= 0) {
            double tol = REL_TIE * (fabs(top) > 1.0 ? fabs(top) : 1.0);
            if (gap < tol) flags |= FL_GUMBEL;
            /* conditioning of log(p - q) = log p + log(1 - q/p): an fp32 error e in
             * log(q/p) moves the score by ~ e * q / (p - q); widen the band by that
             * factor for the two contenders */
            if (sv >= 0) {
                double k1 = lpd[tk] / (lpt[tk] - lpd[tk]);
                double k2 = lpd[sv] / (lpt[sv] - lpd[sv]);
                if (gap < tol * (k1 + k2)) flags |= FL_ILLCOND;
            }
            min_gap = gap;
        } else {
            /* reading: empty support (p <= q everywhere, only possible by rounding):
             * draw from the target row j with the same purpose-1 noise */
            flags |= FL_DEGENERATE;
            oracle_row_logprobs(xt, V, T, lpt);
            tk = gumbel_argmax(lpt, V, a->seed, a->step, b, j, 1, &gap, &top, &sv);
            min_gap = gap;
        }
        tok[j] = tk;
    } else {
        /* bonus: every draft accepted; sample from the target's row k_b */
        double gap, top;
        int tk, sv;
        load_row(a->target, a->dtype, (int64_t)b * K1 + kb, a->ld_row, V, xt);
        if (!isfinite(row_max_nan(xt, V))) {
            fail_request(a, b, ST_NONFINITE);
            return;
        }
        oracle_row_logprobs(xt, V, T, lpt);
        tk = gumbel_argmax(lpt, V, a->seed, a->step, b, kb, 2, &gap, &top, &sv);
        if (gap < REL_TIE * (fabs(top) > 1.0 ? fabs(top) : 1.0)) flags |= FL_GUMBEL;
        min_gap = gap;
        tok[kb] = tk;
    }
    a->out_accepted[b] = A;
    if (a->out_flags) a->out_flags[b] = flags;
    if (a->out_flag_pos) a->out_flag_pos[b] = flag_pos;
    if (a->out_gap) a->out_gap[b] = min_gap;
}

static int run_verify(const verify_args *a, int nthreads) {
    int b;
    if (a->B <= 0) return 0;
    (void)nthreads;
#ifdef _OPENMP
#pragma omp parallel num_threads(nthreads > 0 ? nthreads : 1)
#endif
    {
        double *buf = (double *)malloc(sizeof(double) * (size_t)a->V * 5);
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (b = 0; b < a->B; ++b)
            verify_one(a, b, buf, buf + a->V, buf + 2 * (size_t)a->V, buf + 3 * (size_t)a->V,
                       buf + 4 * (size_t)a->V);
        free(buf);
    }
    return 0;
}

/*
 * Sampling verify for a batch.  Layout as the library's: target row (b,i) at
 * (b*(Kmax+1)+i)*ld_row, draft row (b,i) at (b*Kmax+i)*ld_row, V contiguous.
 * temperature[b] == 0 marks a greedy request (reading).  out_tokens [B,Kmax+1]
 * (-1 = unused), out_accepted [B], out_p/out_q [B,Kmax] (-1 where not computed),
 * out_status [B], out_flags [B] (near-tie bits), out_flag_pos [B] (the first
 * scanned position with a threshold near-tie, -1 if none; may be NULL), out_gap [B]
 * (top-2 gap of the Gumbel draw, +inf if none).  nthreads: OpenMP threads over
 * requests.
 */
static int verify_sample_args(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                              int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                              const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                              int32_t *out_accepted, double *out_p, double *out_q, int32_t *out_status,
                              int32_t *out_flags, int32_t *out_flag_pos, double *out_gap, int nthreads,
                              int early_exit) {
    verify_args a;
    memset(&a, 0, sizeof a);
    a.early_exit = early_exit;
    a.target = target; a.draft = draft; a.dtype = dtype; a.B = B; a.Kmax = Kmax; a.V = V;
    a.ld_row = ld_row; a.draft_tokens = draft_tokens; a.num_draft = num_draft;
    a.temperature = temperature; a.seed = seed; a.step = step;
    a.out_tokens = out_tokens; a.out_accepted = out_accepted; a.out_status = out_status;
    a.out_flags = out_flags; a.out_flag_pos = out_flag_pos; a.out_p = out_p; a.out_q = out_q;
    a.out_gap = out_gap;
    return run_verify(&a, nthreads);
}

int oracle_verify_sample(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                         int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                         const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                         int32_t *out_accepted, double *out_p, double *out_q, int32_t *out_status,
                         int32_t *out_flags, int32_t *out_flag_pos, double *out_gap, int nthreads) {
    return verify_sample_args(target, draft, dtype, B, Kmax, V, ld_row, draft_tokens, num_draft, temperature,
                              seed, step, out_tokens, out_accepted, out_p, out_q, out_status, out_flags,
                              out_flag_pos, out_gap, nthreads, 0);
}

/* The same with early exit: rows are read in position order and reading stops at
 * the first rejected position, so a non-finite row after it is never seen (status
 * 0) and p/q are -1 after it.  Tokens and accepted counts equal the full scan's
 * whenever every row read is finite. */
int oracle_verify_sample_early_exit(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                                    int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                                    const float *temperature, uint64_t seed, uint64_t step,
                                    int32_t *out_tokens, int32_t *out_accepted, double *out_p, double *out_q,
                                    int32_t *out_status, int32_t *out_flags, int32_t *out_flag_pos,
                                    double *out_gap, int nthreads) {
    return verify_sample_args(target, draft, dtype, B, Kmax, V, ld_row, draft_tokens, num_draft, temperature,
                              seed, step, out_tokens, out_accepted, out_p, out_q, out_status, out_flags,
                              out_flag_pos, out_gap, nthreads, 1);
}

/* Greedy verify for a batch (draft logits are never read). */
static int verify_greedy_args(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                              const int32_t *draft_tokens, const int32_t *num_draft, int32_t *out_tokens,
                              int32_t *out_accepted, int32_t *out_status, int nthreads, int early_exit) {
    verify_args a;
    memset(&a, 0, sizeof a);
    a.target = target; a.dtype = dtype; a.B = B; a.Kmax = Kmax; a.V = V; a.ld_row = ld_row;
    a.draft_tokens = draft_tokens; a.num_draft = num_draft;
    a.out_tokens = out_tokens; a.out_accepted = out_accepted; a.out_status = out_status;
    a.early_exit = early_exit;
    return run_verify(&a, nthreads);
}

int oracle_verify_greedy(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                         const int32_t *draft_tokens, const int32_t *num_draft, int32_t *out_tokens,
                         int32_t *out_accepted, int32_t *out_status, int nthreads) {
    return verify_greedy_args(target, dtype, B, Kmax, V, ld_row, draft_tokens, num_draft, out_tokens,
                              out_accepted, out_status, nthreads, 0);
}

/* Greedy verify with early exit: target rows in position order up to the first
 * mismatch (or row k_b); only those are checked for non-finite values. */
int oracle_verify_greedy_early_exit(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                                    const int32_t *draft_tokens, const int32_t *num_draft, int32_t *out_tokens,
                                    int32_t *out_accepted, int32_t *out_status, int nthreads) {
    return verify_greedy_args(target, dtype, B, Kmax, V, ld_row, draft_tokens, num_draft, out_tokens,
                              out_accepted, out_status, nthreads, 1);
}

/* ------------------------------------------------------------------------- */
/* Confidence-scheduled verify length [VBK Sec. 4.2.1, 4.2.2]                 */
/* ------------------------------------------------------------------------- */
typedef struct {
    double s;
    int b, i;
} cand_t;

static int cand_cmp(const void *pa, const void *pb) {
    const cand_t *x = (const cand_t *)pa, *y = (const cand_t *)pb;
    if (x->s > y->s) return -1;
    if (x->s < y->s) return 1;
    if (x->b != y->b) return x->b < y->b ? -1 : 1;
    return x->i < y->i ? -1 : (x->i > y->i);
}

/*
 * Survival S_{b,i} = c_{b,0} * ... * c_{b,i} (fp64, left to right) [VBK 4.2.1];
 * E_b(L) = sum_{i<L} S_{b,i} is the expected number of accepted drafts when L
 * are verified.  Every request keeps m_b = min(min_len, maxlen_b) slots; the
 * other slots (b,i), m_b <= i < maxlen_b, are ranked by S descending (ties: b
 * then i ascending) and added one at a time [VBK 4.2.2].  For every total
 * n = n0 .. min(budget, n0 + #candidates, n_table - 1) the expected throughput
 * F(n) = (B + sum_b E_b) / tau[n] is evaluated (B: the one target token every
 * request emits) and the best n over the whole table is kept, ties to the
 * smallest n (full search, [VBK 4.2.2] production variant).
 * Readings: n counts draft slots; confidences are clamped to [0,1] (NaN -> 0);
 * maxlen_b = clamp(max_len[b], 0, Kmax) (NULL: Kmax); tau[n] <= 0 or
 * non-finite makes n unusable.
 * out_len [B]; out_info[3] = {n*, B + sum E, F(n*)}; *out_flags: 1 = the best
 * two F values within 1e-9 relative, 2 = survival tie (1e-12) across the cut.
 * Returns 0, or 1 for invalid arguments.
 */
int oracle_schedule_verify_len(const float *conf, const int32_t *max_len, int B, int Kmax,
                               const float *step_time_us, int n_table, int budget, int min_len,
                               int32_t *out_len, double *out_info, int32_t *out_flags) {
    double *S = (double *)malloc(sizeof(double) * (size_t)(B > 0 ? B : 1) * (size_t)(Kmax > 0 ? Kmax : 1));
    int *mand = (int *)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1));
    int *mlen = (int *)malloc(sizeof(int) * (size_t)(B > 0 ? B : 1));
    cand_t *cand = (cand_t *)malloc(sizeof(cand_t) * ((size_t)(B > 0 ? B : 1) * (size_t)(Kmax > 0 ? Kmax : 1)));
    int b, i, nc = 0, n0 = 0, nhi, n, nbest, take, flags = 0;
    double E0 = 0.0, E, Fbest = -INFINITY, Fsecond = -INFINITY;

    if (B < 0 || Kmax < 0 || min_len < 0 || n_table < 1 || budget < 0 ||
        (int64_t)budget < (int64_t)B * min_len || (int64_t)n_table - 1 < (int64_t)B * min_len) {
        free(S); free(mand); free(mlen); free(cand);
        return 1;
    }
    for (b = 0; b < B; ++b) {
        double surv = 1.0;
        int ml = max_len ? max_len[b] : Kmax;
        if (ml < 0) ml = 0;
        if (ml > Kmax) ml = Kmax;
        mlen[b] = ml;
        mand[b] = min_len < ml ? min_len : ml;
        for (i = 0; i < Kmax; ++i) {
            double c = (double)conf[(int64_t)b * Kmax + i];
            if (isnan(c) || c < 0.0) c = 0.0;
            if (c > 1.0) c = 1.0;
            surv = surv * c;
            S[(int64_t)b * Kmax + i] = surv;
        }
        n0 += mand[b];
        for (i = 0; i < mand[b]; ++i) E0 += S[(int64_t)b * Kmax + i];
        for (i = mand[b]; i < ml; ++i) {
            cand[nc].s = S[(int64_t)b * Kmax + i];
            cand[nc].b = b;
            cand[nc].i = i;
            ++nc;
        }
    }
    qsort(cand, (size_t)nc, sizeof(cand_t), cand_cmp);

    nhi = n0 + nc;
    if (budget < nhi) nhi = budget;
    if (n_table - 1 < nhi) nhi = n_table - 1;
    nbest = n0;
    E = E0;
    for (n = n0; n <= nhi; ++n) {
        double tau, F;
        if (n > n0) E += cand[n - n0 - 1].s;
        tau = (double)step_time_us[n];
        F = (tau > 0.0 && isfinite(tau)) ? ((double)B + E) / tau : -INFINITY;
        if (F > Fbest) {
            Fsecond = Fbest;
            Fbest = F;
            nbest = n;
        } else if (F > Fsecond) {
            Fsecond = F;
        }
    }
    if (isfinite(Fbest) && isfinite(Fsecond) && Fbest - Fsecond < 1e-9 * Fbest) flags |= 1;

    take = nbest - n0;
    if (take < 0) take = 0;
    for (b = 0; b < B; ++b) out_len[b] = mand[b];
    for (i = 0; i < take; ++i) out_len[cand[i].b] += 1;
    if (take > 0 && take < nc && fabs(cand[take - 1].s - cand[take].s) < 1e-12) flags |= 2;

    E = E0;
    for (i = 0; i < take; ++i) E += cand[i].s;
    if (out_info) {
        out_info[0] = (double)nbest;
        out_info[1] = (double)B + E;
        out_info[2] = (nbest >= 0 && nbest < n_table && step_time_us[nbest] > 0.0f)
                          ? ((double)B + E) / (double)step_time_us[nbest]
                          : 0.0;
    }
    if (out_flags) *out_flags = flags;
    free(S); free(mand); free(mlen); free(cand);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Scheduler variants [PPR prefix scheduler; VBK 4.2.2, 3]                    */
/* ------------------------------------------------------------------------- */
/*
 * Static threshold truncation [PPR "Prefix scheduler": scan left to right and
 * truncate at the first position whose confidence falls below the threshold;
 * VBK Sec. 3: cut draft tokens whose confidence is below a fixed cutoff].
 * L_b = the first i < maxlen_b with c_{b,i} < threshold (NaN counts as below),
 * else maxlen_b; maxlen_b = clamp(max_len[b], 0, Kmax) (NULL: Kmax).  Reading:
 * the score compared is the per-position confidence, as both passages state.
 */
int oracle_schedule_threshold(const float *conf, const int32_t *max_len, int B, int Kmax, float threshold,
                              int32_t *out_len) {
    int b, i;
    if (B < 0 || Kmax < 0 || isnan(threshold)) return 1;
    for (b = 0; b < B; ++b) {
        int ml = max_len ? max_len[b] : Kmax, L;
        if (ml < 0) ml = 0;
        if (ml > Kmax) ml = Kmax;
        L = ml;
        for (i = 0; i < ml; ++i) {
            const double c = (double)conf[(int64_t)b * Kmax + i];
            if (!(c >= (double)threshold)) { /* below, or NaN */
                L = i;
                break;
            }
        }
        out_len[b] = L;
    }
    return 0;
}

/*
 * Two-step-stale batch sizing [VBK 4.2.2, production: the engine prepares the
 * next batch while the GPU is busy, so the batch size comes from the scores of
 * two steps earlier and the tokens are chosen with the latest scores].
 * n* = the total that oracle_schedule_verify_len picks from conf_stale (same
 * table, budget, min_len and max_len); then every request keeps its mandatory
 * m_b slots and the n* - sum m_b remaining slots go to the candidates ranked by
 * the survival of conf (latest), as in the plain scheduler.
 * out_info[3] = {n*, B + sum E under conf, (B + sum E) / tau[n*]};
 * *out_flags: bit 1 from the stale search, bit 2 a survival tie across the cut
 * of the latest ranking.
 */
int oracle_schedule_verify_len_stale(const float *conf_stale, const float *conf, const int32_t *max_len, int B,
                                     int Kmax, const float *step_time_us, int n_table, int budget, int min_len,
                                     int32_t *out_len, double *out_info, int32_t *out_flags) {
    double info[3];
    int32_t flags_stale = 0, flags_now = 0, nstar, b, rc;
    int32_t *len_now = (int32_t *)malloc(sizeof(int32_t) * (size_t)(B > 0 ? B : 1));
    rc = oracle_schedule_verify_len(conf_stale, max_len, B, Kmax, step_time_us, n_table, budget, min_len,
                                    out_len, info, &flags_stale);
    if (rc) {
        free(len_now);
        return rc;
    }
    nstar = (int32_t)info[0];
    /* the latest scores under a table on which n* is the only usable total: the
     * plain scheduler then grants exactly the n* - sum m_b best candidates */
    {
        /* (the table must also reach B * min_len, which argument checking requires) */
        const int top = nstar > B * min_len ? nstar : B * min_len;
        float *tau1 = (float *)malloc(sizeof(float) * (size_t)(top + 1));
        int n;
        for (n = 0; n <= top; ++n) tau1[n] = n == nstar ? 1.0f : -1.0f;
        rc = oracle_schedule_verify_len(conf, max_len, B, Kmax, tau1, top + 1, top, min_len, len_now, info,
                                        &flags_now);
        free(tau1);
    }
    if (rc || (int32_t)info[0] != nstar) {
        free(len_now);
        return 1;
    }
    for (b = 0; b < B; ++b) out_len[b] = len_now[b];
    if (out_info) {
        out_info[0] = (double)nstar;
        out_info[1] = info[1];
        out_info[2] = (step_time_us[nstar] > 0.0f) ? info[1] / (double)step_time_us[nstar] : 0.0;
    }
    if (out_flags) *out_flags = (flags_stale & 1) | (flags_now & 2);
    free(len_now);
    return 0;
}

/* ------------------------------------------------------------------------- */
/* Markov-head drafting [PPR2], [VBK] Sec. 4.1, [MTL]                         */
/* ------------------------------------------------------------------------- */
/*
 * Near-tie band of a draw.  An fp32 implementation forms bias_v as a sum of r
 * products and adds it to the base logit; the products of the stored factors are
 * exact (bf16 x bf16) or carry one rounding (fp32), and a tensor-core style sum
 * aligns and truncates its terms, so |error| <= r * 2^-22 * S_v with
 * S_v = sum_j |emb[prev, j] * proj[v, j]| covers any summation order and rounding
 * mode; adding the base costs |z_v| 2^-24.  The draw then scales by 1 / T (two
 * roundings), adds the fp32 Gumbel noise (a few ulp of |g|, bounded by 8 ulp here)
 * and rounds the sum (|score| 2^-24).  Position k is flagged when the best entry and
 * some other entry are closer than the sum of their two bounds: only there can an
 * fp32 score order differ from the exact one (an exact tie, gap 0, counts too).
 */
static double markov_score_bound(double S, double z, double T, double g, double score, int rank) {
    const double u = 1.0 / 16777216.0;
    const double ez = (double)rank * 4.0 * u * S + fabs(z) * u;
    if (T == 0.0) return ez;
    return ez / T + fabs(z / T) * 2.0 * u + fabs(g) * 8.0 * u + fabs(score) * u;
}

/*
 * Semi-autoregressive drafting of one block.  For request b and positions
 * k = 0 .. K-1, left to right:
 *   prev = anchor[b] (k = 0) or x_{k-1};
 *   bias_v = sum_j emb[prev, j] * proj[v, j]   (rank-r factors, both [V, r]);
 *   z_v = U[b, k, v] + bias_v for v in the candidate set, -inf elsewhere;
 *   candidates: every v (topk = 0), or the topk entries with the largest base
 *   logit U[b, k, v], lower v first among equal values [MTL];
 *   x_k = argmax_v z_v (T_b = 0, lowest v on ties), else the Gumbel-max draw
 *   argmax_v z_v / T_b + g_v with g_v from purpose 3 at row k.
 * Readings (the pages name the bias "low-rank" and its input "the token chosen at
 * the previous position", and give the default rank 256, not the factorisation):
 * the bias row of token prev is the product of prev's row of an embedding factor
 * with a projection factor; the temperature of the draw is the request's
 * temperature; the draw uses the library's counter-based noise with its own
 * purpose.  Status: 1 anchor outside [0, V), 3 bad temperature, 4 a corrected row
 * with NaN or +inf among the candidates or no finite candidate; a request with a
 * non-zero status has every token -1.
 * out_logits [B, K, V] (may be NULL): the corrected logits z (the draft
 * distribution the verify step needs is softmax(z / T)).  out_tie [B]: the first
 * position where the best score and another lie within the sum of their fp32 error
 * bounds (markov_score_bound; K if none): the draws from there on are not decided
 * by fp64 alone.
 */
typedef struct {
    double val;
    int v;
} mcand_t;

static int mcand_desc(const void *pa, const void *pb) {
    const mcand_t *a = (const mcand_t *)pa, *b = (const mcand_t *)pb;
    if (a->val > b->val) return -1;
    if (a->val < b->val) return 1;
    return a->v < b->v ? -1 : (a->v > b->v);
}

int oracle_markov_draft(const void *base, int dtype, int B, int K, int V, int64_t ld_row, const int32_t *anchor,
                        const void *emb, const void *proj, int rank, const float *temperature, uint64_t seed,
                        uint64_t step, int topk, int32_t *out_tokens, double *out_logits, int32_t *out_status,
                        int32_t *out_tie, int nthreads) {
    int b;
    if (B < 0 || K < 0 || V <= 0 || rank <= 0 || ld_row < V || topk < 0 || !anchor || !emb || !proj ||
        !out_tokens || !out_status || !out_tie)
        return 1;
    (void)nthreads;
#pragma omp parallel for schedule(dynamic, 1) num_threads(nthreads > 0 ? nthreads : 1)
    for (b = 0; b < B; ++b) {
        double *u = (double *)malloc(sizeof(double) * (size_t)V);
        double *z = (double *)malloc(sizeof(double) * (size_t)V);
        double *h = (double *)malloc(sizeof(double) * (size_t)rank);
        double *sabs = (double *)malloc(sizeof(double) * (size_t)V);  /* S_v of markov_score_bound */
        double *scv = (double *)malloc(sizeof(double) * (size_t)V);   /* score of every entry */
        double *gv = (double *)malloc(sizeof(double) * (size_t)V);    /* its noise (0 when greedy) */
        mcand_t *cs = (mcand_t *)malloc(sizeof(mcand_t) * (size_t)V);
        const double T = temperature ? (double)temperature[b] : 0.0;
        int st = ST_OK, k, v, j, prev = anchor[b], tie = K;
        if (prev < 0 || prev >= V) st = ST_BAD_TOKEN;
        if (st == ST_OK && (!(T >= 0.0) || isinf(T))) st = ST_BAD_T;
        for (k = 0; k < K && st == ST_OK; ++k) {
            const int ncand = (topk == 0 || topk > V) ? V : topk;
            double best = -INFINITY, second = -INFINITY;
            int bi = -1, bad = 0;
            load_row(base, dtype, (int64_t)b * K + k, ld_row, V, u);
            for (j = 0; j < rank; ++j) h[j] = decode(emb, dtype, (int64_t)prev * rank + j);
            for (v = 0; v < V; ++v) z[v] = -INFINITY;
            if (ncand == V) {
                for (v = 0; v < V; ++v) cs[v].v = v;
            } else {
                for (v = 0; v < V; ++v) {
                    cs[v].val = isnan(u[v]) ? INFINITY : u[v]; /* a NaN is a candidate: it must be seen */
                    cs[v].v = v;
                }
                qsort(cs, (size_t)V, sizeof(mcand_t), mcand_desc);
            }
            for (v = 0; v < V; ++v) sabs[v] = 0.0;
            for (v = 0; v < ncand; ++v) {
                const int c = cs[v].v;
                double bias = 0.0, sa = 0.0;
                for (j = 0; j < rank; ++j) {
                    const double t = h[j] * decode(proj, dtype, (int64_t)c * rank + j);
                    bias += t;
                    sa += fabs(t);
                }
                z[c] = u[c] + bias;
                sabs[c] = sa;
            }
            if (out_logits)
                for (v = 0; v < V; ++v) out_logits[((int64_t)b * K + k) * V + v] = z[v];
            for (v = 0; v < V; ++v) {
                double sc;
                scv[v] = -INFINITY;
                gv[v] = 0.0;
                if (isnan(z[v]) || z[v] == INFINITY) bad = 1;
                if (!(z[v] > -INFINITY)) continue;
                if (T != 0.0) gv[v] = oracle_gumbel(oracle_rand_word(seed, step, b, k, 3, v));
                sc = (T == 0.0) ? z[v] : z[v] / T + gv[v];
                scv[v] = sc;
                if (sc > best) {
                    second = best;
                    best = sc;
                    bi = v;
                } else if (sc > second) {
                    second = sc;
                }
            }
            (void)second;
            if (bad || bi < 0) {
                st = ST_NONFINITE;
                break;
            }
            if (tie == K) {
                const double eb = markov_score_bound(sabs[bi], z[bi], T, gv[bi], best, rank);
                for (v = 0; v < V && tie == K; ++v)
                    if (v != bi && scv[v] > -INFINITY &&
                        best - scv[v] <= eb + markov_score_bound(sabs[v], z[v], T, gv[v], scv[v], rank))
                        tie = k;
            }
            out_tokens[(int64_t)b * K + k] = bi;
            prev = bi;
        }
        if (st != ST_OK)
            for (k = 0; k < K; ++k) out_tokens[(int64_t)b * K + k] = -1;
        out_status[b] = st;
        out_tie[b] = st == ST_OK ? tie : K;
        free(u);
        free(z);
        free(h);
        free(sabs);
        free(scv);
        free(gv);
        free(cs);
    }
    return 0;
}
