/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) speculative-decoding verify/commit
 * library (libspecverify.so).
 *
 * What it computes (page title -- section):
 *  - "From draft-then-verify to DSpark" (alexine.rip) -- "How speculative decoding
 *    works": each draft token x is accepted with probability min(1, p(x)/q(x)),
 *    p the target's and q the draft's next-token distribution; at the first
 *    rejection a token is drawn from normalise(max(0, p - q)); the emitted tokens
 *    are distributed exactly as the target's.
 *  - "Accelerating Large-Model Inference ... DSpark Speculative Decoding"
 *    (princepride.github.io) -- Sec. 1, propose/verify/commit table: the target
 *    scores all draft positions in one pass; the longest accepted prefix is kept
 *    and one more token is emitted (a correction at the first rejection, or a
 *    bonus token from the target's row after the last draft).
 *  - "Bringing DSpark to vLLM Metal" (mhdimo.github.io) -- greedy path: compare the
 *    target's argmax with each draft token.  The target's logits cover the K draft
 *    positions plus the one after them (K+1 rows), where the bonus token comes from.
 *  - "DSpark paper review" (vllmbangkok.com) -- Sec. 4.2.1 prefix survival
 *    c_1 x ... x c_k; Sec. 4.2.2 hardware-aware prefix scheduler over a step-time
 *    table profiled at startup, searching the whole table; Sec. 5.3 ragged batches
 *    where each request verifies its own number of drafts.
 *
 * Conventions for every entry point:
 *  - Array pointers are DEVICE pointers owned by the caller; the library keeps no
 *    reference after the call returns and allocates no device memory per call.
 *    Logit pointers must lie on the current device (or in managed memory), else
 *    SPEC_EINVAL.  Scratch space is the caller's workspace (size from the
 *    *_workspace_size query).
 *  - Calls are asynchronous on `cuda_stream` (a cudaStream_t; NULL = the legacy
 *    default stream) and never synchronise the host.
 *  - Logits are row-major with V contiguous and a row stride of ld_row elements
 *    (ld_row >= V).  Target row (b, i), i = 0..Kmax, starts at element
 *    (b*(Kmax+1) + i) * ld_row; draft row (b, i), i = 0..Kmax-1, at
 *    (b*Kmax + i) * ld_row.  Requests verify k_b = num_draft[b] <= Kmax drafts;
 *    target rows i > k_b and draft rows i >= k_b are never read.  Logit pointers
 *    must be aligned to their element size; rows need no further alignment.
 *  - Host-checkable argument errors return SPEC_EINVAL / SPEC_EWORKSPACE /
 *    SPEC_EUNSUPPORTED before anything is launched; a failed launch returns
 *    SPEC_ECUDA.  Data-dependent errors are reported per request in out_status.
 *  - Emitted tokens: out_tokens[b, 0 .. out_accepted[b]] (accepted drafts, then
 *    the correction or bonus token); unused slots are -1.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Return codes. */
typedef enum {
    SPEC_OK = 0,
    SPEC_EINVAL = 1,        /* bad argument (null pointer, size out of range) */
    SPEC_ECUDA = 2,         /* a CUDA runtime call or launch failed           */
    SPEC_EUNSUPPORTED = 3,  /* valid but outside what this library supports   */
    SPEC_EWORKSPACE = 4,    /* workspace pointer null or too small            */
    SPEC_ESCRATCH = 5       /* sizes need more than the fixed scratch of
                               spec_verify_sample_noalloc                    */
} spec_err;

/* Logit element types. */
typedef enum { SPEC_BF16 = 0, SPEC_F32 = 1 } spec_dtype;

/* Per-request status codes written to out_status (checked in this order). */
#define SPEC_STATUS_OK 0
#define SPEC_STATUS_BAD_TOKEN 1        /* a draft token x_i (i < k_b) is outside [0, V)          */
#define SPEC_STATUS_BAD_K 2            /* num_draft[b] outside [0, Kmax]                          */
#define SPEC_STATUS_BAD_TEMPERATURE 3  /* temperature[b] < 0, NaN or infinite                     */
#define SPEC_STATUS_NONFINITE 4        /* a row that was read holds NaN or +inf, or is all -inf   */
#define SPEC_STATUS_INTERNAL 5         /* a bounded internal wait gave up, or the workspace was not
                                          zeroed before its first use; results are not valid   */
/* Rows read: target and draft rows 0..k_b-1 (target only for greedy requests); the
 * target row k_b only when every draft is accepted (it holds the bonus token).
 * A request with a non-zero status has out_accepted[b] = 0, every token -1 and
 * out_p / out_q -1. */

/* Limits of this library. */
#define SPEC_MAX_BATCH 8192        /* B                                   */
#define SPEC_MAX_DRAFTS 255        /* Kmax                                */
#define SPEC_MAX_SCHED_ITEMS 8192  /* B * Kmax for the scheduler          */
#define SPEC_MARKOV_MAX_RANK 512   /* rank r of the Markov head's factors (a multiple of 4) */
#define SPEC_MARKOV_MAX_TOPK 1024  /* candidates a position of top-K Markov drafting corrects */

/*
 * Bytes of device workspace that spec_verify_greedy / spec_verify_sample (and their
 * _flat forms) need for (B, Kmax, V, dtype).  Returns 0 for invalid sizes.  The
 * workspace holds the main pass's chunk-ticket counter (always at its start), one
 * 16-byte statistic and 16 two-byte seed pointers per chunk of every row the main
 * pass reads (rows of at most 64 KB chunks), and per request a 128-byte line for the
 * commit pieces' counter and shared bound, and the commit pieces' results:
 *   256 + align256(4 (B + 1)) + align256(128 B) + align256(16 B R cpr)
 *       + align256(32 B R cpr) + align256(16 B P),
 * with R = 2 Kmax main-pass rows a request (sampling), cpr = the chunks a row
 * (ceil(V / floor(65504 / elsize)) for elsize 2 or 4, then ceil(V / ce) with
 * ce = ceil(V / cpr) rounded up to a multiple of 8) and P = ceil(ceil(V / 1024) / 8)
 * commit pieces a request.
 * ZERO-FILL the workspace once before its first use (cudaMemset(ws, 0, bytes)):
 * the ticket counter must start at 0.  Every call leaves it ready for the next
 * call, so one workspace serves any number of calls made in stream order; calls
 * that may overlap need one workspace each.  A call on a workspace that was not
 * zeroed reports status 5 for the requests it could not verify, and leaves the
 * workspace ready for the next call.  Calls with B at or above the device's SM
 * count run one persistent kernel, preceded in stream order by a memset of the
 * counters and request lines: for them any workspace contents serve.
 */
size_t spec_verify_workspace_size(int B, int Kmax, int V, int dtype);

/*
 * Greedy verify ("Bringing DSpark to vLLM Metal" -- greedy serving path; the
 * propose/verify/commit table of "Accelerating Large-Model Inference", Sec. 1).
 * For each request b and i = 0..k_b, y_i = argmax_v target[b, i, v] over the raw
 * logits, lowest v on ties.  A = first i < k_b with y_i != x_i, else k_b.
 * Emits x_0 .. x_{A-1}, then y_A.  Draft logits are not an input.
 *
 *  target        [B, Kmax+1, ld_row] logits of type dtype
 *  draft_tokens  [B, Kmax] int32 draft tokens x_i
 *  num_draft     [B] int32 k_b, or NULL for k_b = Kmax
 *  out_tokens    [B, Kmax+1] int32; out_accepted [B] int32 (= A); out_status [B]
 *  ws, ws_bytes  workspace of at least spec_verify_workspace_size(B, Kmax, V, dtype)
 * B = 0 is a no-op.  Kmax = 0 verifies nothing and emits y_0.
 */
int spec_verify_greedy(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                       const int32_t *draft_tokens, const int32_t *num_draft, int32_t *out_tokens,
                       int32_t *out_accepted, int32_t *out_status, void *ws, size_t ws_bytes,
                       void *cuda_stream);

/*
 * Sampling verify by rejection sampling ("From draft-then-verify to DSpark" --
 * "How speculative decoding works").  For request b with temperature T_b > 0:
 *   p_i = softmax(target[b, i, :] / T_b), q_i = softmax(draft[b, i, :] / T_b) over
 *   all V entries (numerically stable, fp32 with per-segment maxima);
 *   draft i is accepted iff u_i * q_i(x_i) < p_i(x_i), u_i uniform in (0, 1)
 *   (probability min(1, p/q)); scanning stops at the first rejection j;
 *   correction at j: argmax_v over {p_j(v) > q_j(v)} of log(p_j(v) - q_j(v)) + g_v
 *   (Gumbel-max draw from normalise(max(0, p_j - q_j))), lowest v on ties;
 *   bonus when all k_b are accepted: argmax_v log p_{k_b}(v) + g_v from the
 *   target's row k_b.
 * temperature[b] == 0 makes request b greedy (as spec_verify_greedy).
 * Random numbers: Philox4x32-10 (Salmon et al., SC'11) with key (seed lo, seed hi)
 * and counter (v >> 2, b, (row << 4) | purpose, step lo), word v & 3; purpose 0 =
 * acceptance uniform (v = 0), 1 = correction noise at row j, 2 = bonus noise at
 * row k_b.  A word w maps to u = (2 (w >> 9) + 1) 2^-24 and g = -log(-log u).
 * Outputs p_i(x_i) / q_i(x_i) for i < k_b go to out_p / out_q (may be NULL; -1
 * where not computed).  out_tokens, out_accepted, out_status as for greedy.
 * If p_j <= q_j everywhere (only possible by rounding), the correction is drawn
 * from p_j with the same noise.
 */
int spec_verify_sample(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                       int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                       const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                       int32_t *out_accepted, float *out_p, float *out_q, int32_t *out_status, void *ws,
                       size_t ws_bytes, void *cuda_stream);

/*
 * Flattened ragged layout ("DSpark paper review", Sec. 4, production results: to
 * verify a different number of tokens per request in one batch, the engine
 * flattens every token and tracks each one's request).  The same computation as
 * spec_verify_greedy / spec_verify_sample, with no padding rows.  Request b's k_b
 * draft positions are cu_draft[b] .. cu_draft[b+1] - 1 (k_b = cu_draft[b+1] -
 * cu_draft[b]), and:
 *  draft row i       at row cu_draft[b] + i of draft (ld_row elements a row);
 *  target row i      at row cu_draft[b] + b + i of target, i = 0 .. k_b (k_b + 1 rows);
 *  draft token x_i   draft_tokens[cu_draft[b] + i];
 *  out_tokens        k_b + 1 slots from cu_draft[b] + b (accepted drafts, then the
 *                    correction or bonus token, then -1);
 *  out_p / out_q     k_b entries from cu_draft[b];
 *  out_accepted, out_status  [B] as before.
 * Kmax is the caller's bound on every k_b: it sizes the workspace
 * (spec_verify_workspace_size(B, Kmax, V, dtype)), and a request with k_b outside
 * [0, Kmax] reports status 2.  cu_draft need not start at 0.  The arrays must hold
 * the rows and slots the offsets name; the library cannot check their sizes.
 */
int spec_verify_greedy_flat(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                            const int32_t *cu_draft, const int32_t *draft_tokens, int32_t *out_tokens,
                            int32_t *out_accepted, int32_t *out_status, void *ws, size_t ws_bytes,
                            void *cuda_stream);
int spec_verify_sample_flat(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                            int64_t ld_row, const int32_t *cu_draft, const int32_t *draft_tokens,
                            const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                            int32_t *out_accepted, float *out_p, float *out_q, int32_t *out_status, void *ws,
                            size_t ws_bytes, void *cuda_stream);

/*
 * Early-exit verify ("Accelerating Large-Model Inference ... DSpark", Sec. 1: only
 * the longest accepted prefix and one more token are committed, so no row after
 * the first rejected position is needed; "From draft-then-verify to DSpark": the
 * rejection test at each position in turn).  Same arguments, layout and results
 * as spec_verify_sample / spec_verify_greedy (padded layout), except that:
 *  - the rows are read in position order and reading stops at the first rejection
 *    (sampling) or mismatch (greedy); target row k_b only when every draft passes;
 *  - status 4 (non-finite) covers only the rows read, so a request whose bad row
 *    lies after its first rejection reports status 0;
 *  - out_p / out_q hold p_i(x_i), q_i(x_i) up to and including the first rejected
 *    position and -1 after it.
 * Tokens and accepted counts equal spec_verify_sample's whenever every row read
 * is finite.  One kernel, one cluster of CTAs per request walking its positions;
 * no workspace.
 */
int spec_verify_sample_early_exit(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                                  int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                                  const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                                  int32_t *out_accepted, float *out_p, float *out_q, int32_t *out_status,
                                  void *cuda_stream);
int spec_verify_greedy_early_exit(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                                  const int32_t *draft_tokens, const int32_t *num_draft, int32_t *out_tokens,
                                  int32_t *out_accepted, int32_t *out_status, void *cuda_stream);

/*
 * Markov-head drafting of one block ("Accelerating Large-Model Inference ...
 * DSpark", drafting-engine table, layer 2: the backbone's logits are corrected left
 * to right by a low-rank bias set by the token chosen at the previous position;
 * "DSpark paper review" Sec. 4.1: the head runs once per position, default rank
 * 256).  For request b and positions k = 0 .. K-1 in order:
 *   prev = anchor[b] (k = 0) or x_{k-1};
 *   z_v  = base[b, k, v] + sum_j emb[prev, j] * proj[v, j];
 *   x_k  = argmax_v z_v (temperature NULL or T_b = 0; lowest v on ties), else the
 *          Gumbel-max draw argmax_v z_v / T_b + g_v with noise purpose 3 at row k.
 * z is computed in fp32 (the products of the stored factors are exact).
 *
 *  base         [B, K, ld_row] backbone logits of type dtype
 *  anchor       [B] int32: the token before the block
 *  emb, proj    [V, rank] row-major factors of type dtype (row prev of emb, row v of
 *               proj); rank a multiple of 4, at most SPEC_MARKOV_MAX_RANK
 *  temperature  [B] float, or NULL for greedy drafting
 *  out_tokens   [B, K] int32 draft tokens
 *  out_logits   [B, K, V] float corrected logits z (the draft distribution that
 *               verify needs is softmax(z / T)); rows of a failed request are
 *               unspecified
 *  out_status   [B]: 0, 1 (anchor outside [0, V)), 3 (bad temperature) or 4 (a
 *               corrected row with NaN or +inf, or all -inf); a failed request has
 *               every token -1
 * All pointers are device pointers owned by the caller.  2 K kernel launches on
 * the stream, no host synchronisation, no workspace.  Host-checkable errors return
 * before any launch.
 */
int spec_markov_draft(const void *base, int dtype, int B, int K, int V, int64_t ld_row, const int32_t *anchor,
                      const void *emb, const void *proj, int rank, const float *temperature, uint64_t seed,
                      uint64_t step, int32_t *out_tokens, float *out_logits, int32_t *out_status,
                      void *cuda_stream);

/*
 * Top-K Markov-head drafting ("Bringing DSpark to vLLM Metal" -- "Making the draft
 * cheaper": only the top-K candidate rows of each position are corrected).  As
 * spec_markov_draft, with the candidate set of row (b, k) restricted to the
 * n = min(topk, V) entries with the largest backbone logit base[b, k, v] (a NaN
 * counts as +inf; lower v first among equal values):
 *   z_v = base[b, k, v] + sum_j emb[prev, j] * proj[v, j] for the candidates, -inf
 *         for the others;
 *   x_k = argmax over the candidates of z_v (greedy) or z_v / T_b + g_v (noise
 *         purpose 3 at row k, as spec_markov_draft).
 *  topk          1 .. SPEC_MARKOV_MAX_TOPK
 *  out_logits    [B, K, V] float (z, -inf outside the candidates), or NULL
 *  ws, ws_bytes  device workspace of at least spec_markov_topk_workspace_size
 *                (B, K, V, topk) bytes, 16-byte aligned: the candidate lists
 *                (B K n int32); nothing persists between calls
 * Statuses and failed requests as spec_markov_draft (status 4 when a candidate's z
 * is NaN or +inf, or no candidate is finite).  Two kernel launches (the selection
 * of every row, then the walk over the positions), no host synchronisation.
 */
size_t spec_markov_topk_workspace_size(int B, int K, int V, int topk);
int spec_markov_draft_topk(const void *base, int dtype, int B, int K, int V, int64_t ld_row,
                           const int32_t *anchor, const void *emb, const void *proj, int rank,
                           const float *temperature, uint64_t seed, uint64_t step, int topk,
                           int32_t *out_tokens, float *out_logits, int32_t *out_status, void *ws,
                           size_t ws_bytes, void *cuda_stream);

/*
 * spec_verify_sample without a workspace argument.  The method on the pages has no
 * counterpart to this entry point: it exists for callers that cannot hand over
 * device memory per call.  Examples are a C host program with no device allocator
 * of its own, and a serving loop that sized its caches to fill the GPU at start-up
 * and must not call cudaMalloc / cudaFree while decoding, since those calls can
 * synchronise the whole device and stall the pipelined steps around them.
 *
 * Scratch is one array of SPEC_STATIC_SCRATCH_BYTES bytes that the library holds in
 * its own module's device memory (one copy per device).  This entry point calls no
 * allocating routine.  Arguments, outputs and results are those of
 * spec_verify_sample, and the two agree on the same inputs.
 *  - Set-up: the first call on each device looks the array's address up with that
 *    device current (and sets the kernels' shared-memory limits, as the
 *    workspace entry points do).  Make that first call before any stream capture.
 *  - Limit: sizes whose spec_verify_workspace_size(B, Kmax, V, dtype) exceeds
 *    SPEC_STATIC_SCRATCH_BYTES return SPEC_ESCRATCH before anything is launched.
 *    The scratch grows with B * Kmax * (chunks a row) (see the formula at
 *    spec_verify_workspace_size): at V = 151936, Kmax = 7 fits B up to 1104 for
 *    bf16 logits (5 chunks a row) and B up to 586 for fp32 (10 chunks a row).
 *  - Zeroing: the array is zero when the module loads, and every call leaves the
 *    part that must start at zero (the chunk-ticket counter) at zero.
 *  - Races: every call on a device uses the same array, so two calls that can
 *    overlap (different streams, or host threads without ordering between them)
 *    corrupt each other's results.  Order the calls on one stream.
 */
#define SPEC_STATIC_SCRATCH_BYTES ((size_t)4 << 20)
int spec_verify_sample_noalloc(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                               int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                               const float *temperature, uint64_t seed, uint64_t step,
                               int32_t *out_tokens, int32_t *out_accepted, float *out_p, float *out_q,
                               int32_t *out_status, void *cuda_stream);

/*
 * Confidence-scheduled verify lengths ("DSpark paper review", Sec. 4.2.1 and
 * 4.2.2).  Survival S_{b,i} = c_{b,0} * ... * c_{b,i} in fp64 (confidences clamped
 * to [0, 1], NaN as 0); E_b(L) = sum_{i<L} S_{b,i} is the expected accepted length.
 * Every request keeps m_b = min(min_len, maxlen_b) slots, maxlen_b =
 * clamp(max_len[b], 0, Kmax) (max_len NULL: Kmax).  The remaining slots of all
 * requests are ranked by survival (ties: lower b, then lower i) and granted one at
 * a time; for every total n from sum m_b to min(budget, n_table - 1, all slots)
 * the expected throughput F(n) = (B + sum_b E_b) / step_time_us[n] is evaluated
 * and the largest is kept (ties: smallest n) -- a search of the whole table, not
 * a stop at the first drop.  Entries step_time_us[n] <= 0 make n unusable.
 *
 *  conf          [B, Kmax] float32 per-token confidences c_{b,i}
 *  max_len       [B] int32 or NULL
 *  step_time_us  [n_table] float32 step time with n verified draft slots
 *  out_len       [B] int32 verify length L_b (feed it to num_draft)
 *  out_info      [3] double {n*, B + sum E, F(n*)} or NULL
 * Errors: SPEC_EINVAL if budget < B*min_len or n_table - 1 < B*min_len;
 * SPEC_EUNSUPPORTED if B*Kmax > SPEC_MAX_SCHED_ITEMS.  Uses no workspace.
 */
int spec_schedule_verify_len(const float *conf, const int32_t *max_len, int B, int Kmax,
                             const float *step_time_us, int n_table, int budget, int min_len,
                             int32_t *out_len, double *out_info, void *cuda_stream);

/*
 * Two-step-stale batch sizing ("DSpark paper review", Sec. 4.2.2, production
 * variant).  The engine prepares the next batch while the GPU is still busy, so
 * the total number of verified slots n* comes from the scores of two steps
 * earlier (conf_stale), chosen exactly as spec_schedule_verify_len chooses it.
 * The n* slots then go to the requests by the latest scores (conf): every
 * request keeps its m_b mandatory slots and the rest are the best survivals of
 * conf (ties: lower b, then lower i).
 *  conf_stale, conf  [B, Kmax] float32; the other arguments as for
 *                    spec_schedule_verify_len
 *  out_info          [3] double {n*, B + sum E under conf, that / step_time_us[n*]}
 */
int spec_schedule_verify_len_stale(const float *conf_stale, const float *conf, const int32_t *max_len, int B,
                                   int Kmax, const float *step_time_us, int n_table, int budget, int min_len,
                                   int32_t *out_len, double *out_info, void *cuda_stream);

/*
 * Static threshold truncation ("Accelerating Large-Model Inference ... DSpark",
 * prefix scheduler: scan left to right and truncate at the first score below the
 * threshold; "DSpark paper review", Sec. 3: a fixed confidence cutoff).
 * out_len[b] = the first i < maxlen_b with conf[b, i] < threshold (NaN counts as
 * below), else maxlen_b = clamp(max_len[b], 0, Kmax) (max_len NULL: Kmax).
 * SPEC_EINVAL for a NaN threshold.  Uses no workspace.
 */
int spec_schedule_threshold(const float *conf, const int32_t *max_len, int B, int Kmax, float threshold,
                            int32_t *out_len, void *cuda_stream);

/* Short text for a return code. */
const char *spec_error_string(int err);

/* The CUDA error (cudaError_t value) behind the last SPEC_ECUDA on this thread. */
int spec_last_cuda_error(void);

/*
 * Kernel timing for measurement.  While enabled, every verify call records CUDA
 * events on its stream around each kernel it launches; spec_profile_read waits for
 * the last call's events and writes up to n durations in milliseconds, in launch
 * order (the main pass over the draft positions' rows, then the commit pass that
 * combines them, runs the acceptance scan and draws the extra token; greedy and
 * sampling calls launch the same two; the early-exit calls launch one), returning
 * how many were written (negative spec_err on failure).
 */
int spec_profile_enable(int on);
int spec_profile_read(float *ms, int n);

#ifdef __cplusplus
}
#endif

#endif /* SPEC_VERIFY_H */
