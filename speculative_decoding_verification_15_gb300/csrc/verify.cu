// verify.cu -- batched speculative-decoding verify/commit on sm_103a.
//
// What is computed (page title -- section):
//  * "From draft-then-verify to DSpark" -- "How speculative decoding works": accept
//    draft x with probability min(1, p(x)/q(x)); at the first rejection draw from
//    normalise(max(0, p - q)); the output distribution equals the target's.
//  * "Accelerating Large-Model Inference ... DSpark Speculative Decoding", Sec. 1:
//    one target pass scores every draft position; the longest accepted prefix is
//    committed plus one token (correction, or bonus from the row after the drafts).
//  * "Bringing DSpark to vLLM Metal" -- greedy path: target argmax vs draft token.
//
// Kernels per call (fixed grids, no host synchronisation, so a call can be captured
// in a CUDA graph):
//  rows_kernel    one streaming pass over every needed logit row, split into equal
//                 contiguous per-warp ranges of the flattened rows.  Per segment:
//                 softmax statistics (max and sum of 2^(x*log2e/T - max')) for the
//                 target and draft rows of the draft positions, the Gumbel-max bonus
//                 draw on the target row after the last draft, or the raw argmax of
//                 greedy requests.  This is the HBM-bound kernel.
//  accept_kernel  one warp per request: combines the segments, sets the status,
//                 computes p(x_i) and q(x_i), runs the acceptance scan, emits the
//                 accepted drafts and the bonus / greedy token, and queues a
//                 correction job at the first rejection.
//  resid_kernel   second streaming pass, over the target row of each queued job:
//                 Gumbel-max over log(max(0, p - q)); draft values are gathered only
//                 at the few entries that can still win.
//  final_kernel   one warp per job: combines the residual segments into the token.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "spec_common.cuh"
#include "spec_verify.h"

using namespace specv;

namespace {

constexpr int kThreads = 256;
constexpr int kWarpsPerBlock = kThreads / 32;
constexpr int kBlocksPerSM = 4;
constexpr int kBatch = 4;  // vectors each lane loads before reducing them

struct ResJob {
    int b, j;
    float invT, Ct, Cd;
    int pad[3];
};

// =================================================================== segments
template <class Vec>
__device__ __forceinline__ void load_batch(Vec (&d)[kBatch], const void *row, int64_t b0, int64_t vend) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int u = 0; u < kBatch; ++u) {
        const int64_t vi = b0 + lane + 32 * u;
        d[u] = vi < vend ? Vec::load(row, vi) : Vec::neg_inf();
    }
}

template <class Vec>
__device__ __forceinline__ float batch_max(const Vec (&d)[kBatch]) {
    float tm = d[0].vmax();
#pragma unroll
    for (int u = 1; u < kBatch; ++u) tm = max_nan_f32(tm, d[u].vmax());
    return tm;
}

// first (lowest-index) element of this lane's batch equal to x, or -1
template <class Vec>
__device__ __forceinline__ int batch_find(const Vec (&d)[kBatch], int64_t b0, float x) {
    const int lane = threadIdx.x & 31;
    int found = -1;
#pragma unroll
    for (int u = 0; u < kBatch; ++u)
#pragma unroll
        for (int e = 0; e < Vec::VE; ++e)
            if (found < 0 && d[u].get(e) == x) found = (int)((b0 + lane + 32 * u) * Vec::VE + e);
    return found;
}

// Softmax statistics of a row segment: m = max x (NaN-propagating), and
// s = sum_v 2^(x_v c - fl(m c)) with c = log2(e) / T.
template <class Vec>
__device__ Part seg_stats(const void *row, int64_t vb, int64_t vend, float c) {
    float m = kNegInf, mc = 0.f, s = 0.f;
    for (int64_t b0 = vb; b0 < vend; b0 += 32 * kBatch) {
        Vec d[kBatch];
        load_batch(d, row, b0, vend);
        const float tm = batch_max(d);
        if (!(tm <= m)) {  // new maximum, or NaN
            const float mcn = tm * c;
            s = (m == kNegInf) ? 0.f : s * ex2_approx(mc - mcn);
            m = tm;
            mc = mcn;
        }
        const float ms = (m == kNegInf) ? 0.f : mc;
        float acc = 0.f;
#pragma unroll
        for (int u = 0; u < kBatch; ++u) {
            float t = 0.f;
#pragma unroll
            for (int e = 0; e < Vec::VE; ++e) t += ex2_approx(fmaf(d[u].get(e), c, -ms));
            acc += t;
        }
        s += acc;
    }
    const float M = warp_max_nan(m);
    const float MC = M * c;
    const float sc = (m == kNegInf || s == 0.f) ? 0.f : s * ex2_approx(mc - MC);
    Part p;
    p.m = M;
    p.s = (float)warp_sum_d((double)sc);
    p.best = 0.f;
    p.idx = -1;
    return p;
}

// Raw argmax of a row segment, lowest index on ties; m = NaN if any NaN.
template <class Vec>
__device__ Part seg_argmax(const void *row, int64_t vb, int64_t vend) {
    float m = kNegInf;
    int idx = -1;
    bool nan_seen = false;
    for (int64_t b0 = vb; b0 < vend; b0 += 32 * kBatch) {
        Vec d[kBatch];
        load_batch(d, row, b0, vend);
        const float tm = batch_max(d);
        if (tm != tm) {
            nan_seen = true;
        } else if (tm > m) {
            idx = batch_find(d, b0, tm);
            m = tm;
        }
    }
    const bool any_nan = __any_sync(0xffffffffu, nan_seen);
    warp_argmax(m, idx);
    Part p;
    p.m = any_nan ? __int_as_float(0x7fc00000) : m;
    p.s = 0.f;
    p.best = 0.f;
    p.idx = idx;
    return p;
}

// Gumbel-max over z_v + g_v, z = x / T, on the target row after the last draft.
// The argmax is exact: an entry is skipped only when it provably cannot reach the
// best score this warp has already seen, either because z + 17 < best (no 32-bit
// word gives more than 16.64 of noise) or because 1 - u > 1.001 exp(z - best)
// (then -log u >= 1 - u makes g < best - z).
template <class Vec>
__device__ Part seg_bonus(const void *row, int64_t vb, int64_t vend, float invT, uint64_t seed,
                          uint32_t step, uint32_t b, uint32_t rowid) {
    float m = kNegInf, best = kNegInf, thr = kNegInf;
    int bidx = -1;
    bool seeded = false;
    for (int64_t b0 = vb; b0 < vend; b0 += 32 * kBatch) {
        Vec d[kBatch];
        load_batch(d, row, b0, vend);
        const float tm = batch_max(d);
        m = max_nan_f32(m, tm);
        if (!seeded) {  // seed the bound with each lane's largest entry
            seeded = true;
            if (tm == tm && tm > kNegInf) {
                const int v = batch_find(d, b0, tm);
                const uint4 r4 = rand_group(seed, step, b, rowid, PURPOSE_BONUS, (uint32_t)v >> 2);
                best = tm * invT + gumbel_of_word(word_of(r4, v & 3));
                bidx = v;
            }
            thr = warp_max(best);
        }
        if (tm * invT + kGumbelMax >= thr) {
            const int lane = threadIdx.x & 31;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t vi = b0 + lane + 32 * u;
                if (vi >= vend) continue;
#pragma unroll
                for (int g = 0; g < (Vec::VE + 3) / 4; ++g) {
                    if (!(d[u].gmax(g) * invT + kGumbelMax >= thr)) continue;
                    const int64_t v0 = vi * Vec::VE + 4 * g;
                    const uint4 r4 = rand_group(seed, step, b, rowid, PURPOSE_BONUS, (uint32_t)(v0 >> 2));
#pragma unroll
                    for (int k = 0; k < (Vec::VE < 4 ? Vec::VE : 4); ++k) {
                        const int v = (int)(v0 + k);
                        const float z = d[u].get(4 * g + k) * invT;
                        const uint32_t w = word_of(r4, v & 3);
                        const float lim = ex2_approx((z - thr) * kLog2e) * 1.001f;
                        if (one_minus_u01(w) <= lim) {
                            const float sc = z + gumbel_of_word(w);
                            if (better(sc, v, best, bidx)) { best = sc; bidx = v; }
                        }
                    }
                }
            }
        }
        thr = warp_max(best);
    }
    m = warp_max_nan(m);
    warp_argmax(best, bidx);
    Part p;
    p.m = m;
    p.s = 0.f;
    p.best = best;
    p.idx = bidx;
    return p;
}

// Correction draw at the first rejected row j: argmax over {v : p_v > q_v} of
// log(p_v - q_v) + g_v, with log p_v = x_v / T - Ct and log q_v = y_v / T - Cd.
// Same exact pruning as seg_bonus, using log(p - q) <= log p; the draft row is read
// only at the entries that survive it.
template <class Vec>
__device__ Part seg_residual(const void *trow, const void *drow, int dtype, int64_t vb, int64_t vend,
                             float invT, float Ct, float Cd, uint64_t seed, uint32_t step, uint32_t b,
                             uint32_t rowid) {
    float best = kNegInf, thr = kNegInf;
    int bidx = -1;
    bool seeded = false;
    for (int64_t b0 = vb; b0 < vend; b0 += 32 * kBatch) {
        Vec d[kBatch];
        load_batch(d, trow, b0, vend);
        const float tm = batch_max(d);
        if (!seeded) {
            seeded = true;
            if (tm > kNegInf) {
                const int v = batch_find(d, b0, tm);
                const float lp = fmaf(tm, invT, -Ct);
                const float lq = fmaf(load_logit(drow, dtype, v), invT, -Cd);
                if (lq < lp) {
                    const uint4 r4 = rand_group(seed, step, b, rowid, PURPOSE_RESIDUAL, (uint32_t)v >> 2);
                    best = lp + logf(-expm1f(lq - lp)) + gumbel_of_word(word_of(r4, v & 3));
                    bidx = v;
                }
            }
            thr = warp_max(best);
        }
        if (fmaf(tm, invT, -Ct) + kGumbelMax >= thr) {
            const int lane = threadIdx.x & 31;
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int64_t vi = b0 + lane + 32 * u;
                if (vi >= vend) continue;
#pragma unroll
                for (int g = 0; g < (Vec::VE + 3) / 4; ++g) {
                    if (!(fmaf(d[u].gmax(g), invT, -Ct) + kGumbelMax >= thr)) continue;
                    const int64_t v0 = vi * Vec::VE + 4 * g;
                    const uint4 r4 = rand_group(seed, step, b, rowid, PURPOSE_RESIDUAL, (uint32_t)(v0 >> 2));
#pragma unroll
                    for (int k = 0; k < (Vec::VE < 4 ? Vec::VE : 4); ++k) {
                        const int v = (int)(v0 + k);
                        const float lp = fmaf(d[u].get(4 * g + k), invT, -Ct);
                        const uint32_t w = word_of(r4, v & 3);
                        const float lim = ex2_approx((lp - thr) * kLog2e) * 1.001f;
                        if (one_minus_u01(w) <= lim) {
                            const float lq = fmaf(load_logit(drow, dtype, v), invT, -Cd);
                            if (lq < lp) {
                                const float sc = lp + logf(-expm1f(lq - lp)) + gumbel_of_word(w);
                                if (better(sc, v, best, bidx)) { best = sc; bidx = v; }
                            }
                        }
                    }
                }
            }
        }
        thr = warp_max(best);
    }
    warp_argmax(best, bidx);
    Part p;
    p.m = 0.f;
    p.s = 0.f;
    p.best = best;
    p.idx = bidx;
    return p;
}

// =================================================================== rows_kernel
struct RowsParams {
    const void *target;
    const void *draft;
    int64_t ld_row;
    int B, Kmax, V;
    const int32_t *num_draft;
    const float *temperature;  // NULL: every request greedy
    uint64_t seed;
    uint32_t step;
    int *row_start;  // [B+1], written by block 0 for accept_kernel
    Part *parts;     // [warps * nseg]
    int nseg;
    int *job_count;  // reset by block 0
};

__device__ __forceinline__ int request_rows(const int32_t *num_draft, const float *temperature, int Kmax,
                                            int b) {
    const int kb = num_draft ? num_draft[b] : Kmax;
    if (kb < 0 || kb > Kmax) return 0;
    if (temperature) {
        const float T = temperature[b];
        if (!(T >= 0.f) || isinf(T)) return 0;
        return T == 0.f ? kb + 1 : 2 * kb + 1;
    }
    return kb + 1;
}

// s[b] = number of needed rows of requests 0..b-1 (s[B] = total), in shared memory.
// Row order inside a request: sampling [target 0..k-1 | target k | draft 0..k-1],
// greedy [target 0..k].
__device__ void scan_request_rows(int *s, int B, const int32_t *num_draft, const float *temperature,
                                  int Kmax) {
    __shared__ int warp_tot[kWarpsPerBlock];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int per = (B + kThreads - 1) / kThreads;
    const int lo = min(tid * per, B), hi = min(lo + per, B);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += request_rows(num_draft, temperature, Kmax, i);
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    int wbase = 0;
    for (int k = 0; k < wid; ++k) wbase += warp_tot[k];
    int run = wbase + incl - local;
    for (int i = lo; i < hi; ++i) {
        s[i] = run;
        run += request_rows(num_draft, temperature, Kmax, i);
    }
    if (tid == kThreads - 1) s[B] = wbase + incl;
    __syncthreads();
}

__device__ __forceinline__ int find_request(const int *rs, int B, int r) {
    int lo = 0, hi = B - 1;
    while (lo < hi) {  // largest b with rs[b] <= r
        const int mid = (lo + hi + 1) >> 1;
        if (rs[mid] <= r) lo = mid; else hi = mid - 1;
    }
    return lo;
}

template <class Vec>
__global__ void __launch_bounds__(kThreads, kBlocksPerSM) rows_kernel(RowsParams p) {
    extern __shared__ int s_rs[];
    scan_request_rows(s_rs, p.B, p.num_draft, p.temperature, p.Kmax);
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i <= p.B; i += kThreads) p.row_start[i] = s_rs[i];
        if (threadIdx.x == 0) *p.job_count = 0;
    }
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerBlock;
    const int64_t w = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int64_t V = p.V;
    const int64_t total = (int64_t)s_rs[p.B] * V;
    const int64_t range = warp_range(total, nwarps, Vec::VE);
    const int64_t f1 = min(w * range + range, total);
    const int64_t esz = Vec::ESIZE;
    int seg = 0;
    for (int64_t f = w * range; f < f1; ++seg) {
        const int r = (int)(f / V);
        const int64_t rowbase = (int64_t)r * V;
        const int64_t v1 = min(f1 - rowbase, V);
        const int64_t vb = (f - rowbase) / Vec::VE, ve = v1 / Vec::VE;
        const int b = find_request(s_rs, p.B, r);
        const int local = r - s_rs[b];
        const int kb = p.num_draft ? p.num_draft[b] : p.Kmax;
        const float T = p.temperature ? p.temperature[b] : 0.f;
        const char *tb = (const char *)p.target + (int64_t)b * (p.Kmax + 1) * p.ld_row * esz;
        Part part;
        if (T == 0.f) {
            part = seg_argmax<Vec>(tb + local * p.ld_row * esz, vb, ve);
        } else if (local < kb) {
            part = seg_stats<Vec>(tb + local * p.ld_row * esz, vb, ve, __fdiv_rn(kLog2e, T));
        } else if (local == kb) {
            part = seg_bonus<Vec>(tb + (int64_t)kb * p.ld_row * esz, vb, ve, __fdiv_rn(1.f, T), p.seed,
                                  p.step, (uint32_t)b, (uint32_t)kb);
        } else {
            const char *drow = (const char *)p.draft +
                               ((int64_t)b * p.Kmax + (local - kb - 1)) * p.ld_row * esz;
            part = seg_stats<Vec>(drow, vb, ve, __fdiv_rn(kLog2e, T));
        }
        if (lane == 0 && seg < p.nseg) p.parts[w * p.nseg + seg] = part;
        f = rowbase + v1;
    }
}

// =================================================================== combine helpers
// Warps whose ranges intersect flat row r, and the slot of row r in warp w.
struct Split {
    int64_t range;
    int64_t V;
    int nseg;
    __device__ __forceinline__ int64_t w_lo(int r) const { return ((int64_t)r * V) / range; }
    __device__ __forceinline__ int64_t w_hi(int r) const { return ((int64_t)r * V + V - 1) / range; }
    __device__ __forceinline__ int64_t slot(int64_t w, int r) const {
        return w * nseg + (r - (w * range) / V);
    }
};

__device__ float combine_max(const Part *parts, const Split &sp, int r) {
    const int lane = threadIdx.x & 31;
    float m = kNegInf;
    for (int64_t w = sp.w_lo(r) + lane; w <= sp.w_hi(r); w += 32) m = max_nan_f32(m, parts[sp.slot(w, r)].m);
    return warp_max_nan(m);
}

// Row statistics: M (raw max), MC = fl(M c), l2S = log2 sum_v 2^(x_v c - MC).
__device__ void combine_stats(const Part *parts, const Split &sp, int r, float c, float &M, float &MC,
                              float &l2S) {
    const int lane = threadIdx.x & 31;
    M = combine_max(parts, sp, r);
    MC = M * c;
    double s = 0.0;
    for (int64_t w = sp.w_lo(r) + lane; w <= sp.w_hi(r); w += 32) {
        const Part q = parts[sp.slot(w, r)];
        if (q.m != kNegInf && q.s != 0.f) s += (double)q.s * (double)exp2f(q.m * c - MC);
    }
    s = warp_sum_d(s);
    l2S = (float)log2(s);
}

__device__ void combine_argmax(const Part *parts, const Split &sp, int r, bool use_best, float &score,
                               int &idx) {
    const int lane = threadIdx.x & 31;
    score = kNegInf;
    idx = -1;
    for (int64_t w = sp.w_lo(r) + lane; w <= sp.w_hi(r); w += 32) {
        const Part q = parts[sp.slot(w, r)];
        const float s = use_best ? q.best : q.m;
        if (better(s, q.idx, score, idx)) { score = s; idx = q.idx; }
    }
    warp_argmax(score, idx);
}

// =================================================================== accept_kernel
struct AcceptParams {
    const void *target;
    const void *draft;
    int dtype;
    int64_t ld_row;
    int B, Kmax, V;
    const int32_t *draft_tokens;
    const int32_t *num_draft;
    const float *temperature;  // NULL: greedy
    uint64_t seed;
    uint32_t step;
    const int *row_start;
    const Part *parts;
    int nseg;
    int64_t nwarps;  // warps of rows_kernel
    int ve;          // vector width rows_kernel used
    int32_t *out_tokens;
    int32_t *out_accepted;
    float *out_p;
    float *out_q;
    int32_t *out_status;
    ResJob *jobs;
    int *job_list;
    int *job_count;
};

__global__ void __launch_bounds__(kThreads) accept_kernel(AcceptParams p) {
    const int lane = threadIdx.x & 31;
    const int b = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    if (b >= p.B) return;
    const int K1 = p.Kmax + 1;
    int32_t *tok = p.out_tokens + (int64_t)b * K1;
    for (int i = lane; i < K1; i += 32) tok[i] = -1;
    if (p.out_p)
        for (int i = lane; i < p.Kmax; i += 32) p.out_p[(int64_t)b * p.Kmax + i] = -1.f;
    if (p.out_q)
        for (int i = lane; i < p.Kmax; i += 32) p.out_q[(int64_t)b * p.Kmax + i] = -1.f;

    // statuses, in order: k_b, temperature, tokens, non-finite rows
    const int kb = p.num_draft ? p.num_draft[b] : p.Kmax;
    int status = SPEC_STATUS_OK;
    float T = 0.f;
    if (kb < 0 || kb > p.Kmax) status = SPEC_STATUS_BAD_K;
    if (status == SPEC_STATUS_OK && p.temperature) {
        T = p.temperature[b];
        if (!(T >= 0.f) || isinf(T)) status = SPEC_STATUS_BAD_TEMPERATURE;
    }
    const bool greedy = (T == 0.f);
    const int32_t *x = p.draft_tokens + (int64_t)b * p.Kmax;
    if (status == SPEC_STATUS_OK) {
        bool bad = false;
        for (int i = lane; i < kb; i += 32) bad |= (x[i] < 0 || x[i] >= p.V);
        if (__any_sync(0xffffffffu, bad)) status = SPEC_STATUS_BAD_TOKEN;
    }
    Split sp;
    sp.range = warp_range((int64_t)p.row_start[p.B] * p.V, p.nwarps, p.ve);
    sp.V = p.V;
    sp.nseg = p.nseg;
    const int r0 = p.row_start[b];
    if (status == SPEC_STATUS_OK) {
        const int nrows = greedy ? kb + 1 : 2 * kb + 1;
        bool nonfinite = false;
        for (int rr = 0; rr < nrows; ++rr) {
            const float M = combine_max(p.parts, sp, r0 + rr);
            nonfinite |= !(fabsf(M) < __int_as_float(0x7f800000));
        }
        if (nonfinite) status = SPEC_STATUS_NONFINITE;
    }
    if (status != SPEC_STATUS_OK) {
        if (lane == 0) {
            p.out_status[b] = status;
            p.out_accepted[b] = 0;
        }
        return;
    }

    int A = 0;
    if (greedy) {
        int y = -1;
        for (int i = 0; i <= kb; ++i) {
            float m;
            combine_argmax(p.parts, sp, r0 + i, false, m, y);
            if (i == kb || y != x[i]) break;
            ++A;
        }
        if (lane == 0) {
            for (int i = 0; i < A; ++i) tok[i] = x[i];
            tok[A] = y;
        }
    } else {
        const float c = __fdiv_rn(kLog2e, T);
        const int64_t esz = p.dtype == SPEC_BF16 ? 2 : 4;
        bool rejected = false;
        float rej_Ct = 0.f, rej_Cd = 0.f;
        for (int i = 0; i < kb; ++i) {
            float Mt, MCt, l2St, Md, MCd, l2Sd;
            combine_stats(p.parts, sp, r0 + i, c, Mt, MCt, l2St);
            combine_stats(p.parts, sp, r0 + kb + 1 + i, c, Md, MCd, l2Sd);
            const int64_t trow = ((int64_t)b * K1 + i) * p.ld_row;
            const int64_t drow = ((int64_t)b * p.Kmax + i) * p.ld_row;
            const float xt = load_logit(p.target, p.dtype, trow + x[i]);
            const float xd = load_logit(p.draft, p.dtype, drow + x[i]);
            const float l2p = fmaf(xt, c, -MCt) - l2St;  // log2 p_i(x_i)
            const float l2q = fmaf(xd, c, -MCd) - l2Sd;  // log2 q_i(x_i)
            (void)esz;
            if (lane == 0) {
                if (p.out_p) p.out_p[(int64_t)b * p.Kmax + i] = exp2f(l2p);
                if (p.out_q) p.out_q[(int64_t)b * p.Kmax + i] = exp2f(l2q);
            }
            if (rejected) continue;
            // accept iff u q < p, i.e. log2 u < log2 p - log2 q (Q = 0 < P accepts; P = 0 rejects)
            const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)i, PURPOSE_ACCEPT, 0u);
            const float u = u01(r4.x);
            if (log2f(u) < l2p - l2q) {
                ++A;
            } else {
                rejected = true;
                // natural-log offsets: log p_v = x_v / T - Ct, log q_v = y_v / T - Cd
                rej_Ct = (float)(((double)MCt + (double)l2St) * 0.6931471805599453);
                rej_Cd = (float)(((double)MCd + (double)l2Sd) * 0.6931471805599453);
            }
        }
        if (lane == 0) {
            for (int i = 0; i < A; ++i) tok[i] = x[i];
        }
        if (A == kb) {
            float best;
            int idx;
            combine_argmax(p.parts, sp, r0 + kb, true, best, idx);
            if (lane == 0) tok[kb] = idx;
        } else if (lane == 0) {
            ResJob job;
            job.b = b;
            job.j = A;
            job.invT = __fdiv_rn(1.f, T);
            job.Ct = rej_Ct;
            job.Cd = rej_Cd;
            job.pad[0] = job.pad[1] = job.pad[2] = 0;
            p.jobs[b] = job;
            const int pos = atomicAdd(p.job_count, 1);
            p.job_list[pos] = b;
        }
    }
    if (lane == 0) {
        p.out_status[b] = SPEC_STATUS_OK;
        p.out_accepted[b] = A;
    }
}

// =================================================================== residual
struct ResidParams {
    const void *target;
    const void *draft;
    int dtype;
    int64_t ld_row;
    int Kmax, V;
    uint64_t seed;
    uint32_t step;
    const ResJob *jobs;
    const int *job_list;
    const int *job_count;
    Part *parts;
    int nseg;
};

template <class Vec>
__global__ void __launch_bounds__(kThreads, kBlocksPerSM) resid_kernel(ResidParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * kWarpsPerBlock;
    const int64_t w = (int64_t)blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int64_t V = p.V;
    const int64_t total = (int64_t)(*p.job_count) * V;
    const int64_t range = warp_range(total, nwarps, Vec::VE);
    const int64_t f1 = min(w * range + range, total);
    const int64_t esz = Vec::ESIZE;
    int seg = 0;
    for (int64_t f = w * range; f < f1; ++seg) {
        const int r = (int)(f / V);
        const int64_t rowbase = (int64_t)r * V;
        const int64_t v1 = min(f1 - rowbase, V);
        const int64_t vb = (f - rowbase) / Vec::VE, ve = v1 / Vec::VE;
        const ResJob job = p.jobs[p.job_list[r]];
        const char *trow = (const char *)p.target + ((int64_t)job.b * (p.Kmax + 1) + job.j) * p.ld_row * esz;
        const char *drow = (const char *)p.draft + ((int64_t)job.b * p.Kmax + job.j) * p.ld_row * esz;
        const Part part = seg_residual<Vec>(trow, drow, p.dtype, vb, ve, job.invT, job.Ct, job.Cd, p.seed,
                                            p.step, (uint32_t)job.b, (uint32_t)job.j);
        if (lane == 0 && seg < p.nseg) p.parts[w * p.nseg + seg] = part;
        f = rowbase + v1;
    }
}

struct FinalParams {
    const void *target;
    int dtype;
    int64_t ld_row;
    int B, Kmax, V;
    uint64_t seed;
    uint32_t step;
    const ResJob *jobs;
    const int *job_list;
    const int *job_count;
    const Part *parts;
    int nseg;
    int64_t nwarps;  // warps of resid_kernel
    int ve;
    int32_t *out_tokens;
};

__global__ void __launch_bounds__(kThreads) final_kernel(FinalParams p) {
    const int lane = threadIdx.x & 31;
    const int jb = blockIdx.x * kWarpsPerBlock + (threadIdx.x >> 5);
    const int njobs = *p.job_count;
    if (jb >= njobs) return;
    Split sp;
    sp.range = warp_range((int64_t)njobs * p.V, p.nwarps, p.ve);
    sp.V = p.V;
    sp.nseg = p.nseg;
    float best;
    int idx;
    combine_argmax(p.parts, sp, jb, true, best, idx);
    const ResJob job = p.jobs[p.job_list[jb]];
    if (idx < 0) {
        // p <= q everywhere (only by rounding): draw from p_j with the same noise
        const int64_t trow = ((int64_t)job.b * (p.Kmax + 1) + job.j) * p.ld_row;
        best = kNegInf;
        for (int v = lane; v < p.V; v += 32) {
            const float lp = fmaf(load_logit(p.target, p.dtype, trow + v), job.invT, -job.Ct);
            if (!(lp > kNegInf)) continue;
            const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)job.b, (uint32_t)job.j, PURPOSE_RESIDUAL,
                                        (uint32_t)v >> 2);
            const float sc = lp + gumbel_of_word(word_of(r4, v & 3));
            if (better(sc, v, best, idx)) { best = sc; idx = v; }
        }
        warp_argmax(best, idx);
    }
    if (lane == 0) p.out_tokens[(int64_t)job.b * (p.Kmax + 1) + job.j] = idx;
}

// =================================================================== host side
thread_local int t_last_cuda_error = 0;

struct DeviceInfo {
    int sms = 0;
};

std::mutex g_mu;
DeviceInfo g_dev[64];

int device_sms(int *out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    if (dev < 0 || dev >= 64) return SPEC_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_dev[dev].sms == 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
        g_dev[dev].sms = sms;
    }
    *out = g_dev[dev].sms;
    return SPEC_OK;
}

// profiling: events around each kernel of the last call
constexpr int kMaxProfKernels = 4;
bool g_prof = false;
int g_prof_dev = -1;
int g_prof_n = 0;
cudaEvent_t g_prof_ev[2 * kMaxProfKernels];

int prof_prepare() {
    if (!g_prof) return SPEC_OK;
    int dev = 0;
    cudaGetDevice(&dev);
    if (g_prof_dev != dev) {
        if (g_prof_dev >= 0) {
            int cur = dev;
            cudaSetDevice(g_prof_dev);
            for (auto &e : g_prof_ev) cudaEventDestroy(e);
            cudaSetDevice(cur);
        }
        for (auto &e : g_prof_ev) {
            cudaError_t err = cudaEventCreate(&e);
            if (err != cudaSuccess) { t_last_cuda_error = (int)err; return SPEC_ECUDA; }
        }
        g_prof_dev = dev;
    }
    g_prof_n = 0;
    return SPEC_OK;
}

struct ProfScope {
    cudaStream_t s;
    int k;
    ProfScope(cudaStream_t st) : s(st), k(-1) {
        if (g_prof && g_prof_n < kMaxProfKernels) {
            k = g_prof_n++;
            cudaEventRecord(g_prof_ev[2 * k], s);
        }
    }
    ~ProfScope() {
        if (k >= 0) cudaEventRecord(g_prof_ev[2 * k + 1], s);
    }
};

struct Layout {
    size_t off_row_start, off_parts, off_jobs, off_job_list, off_job_count, off_rparts, total;
    int nseg_rows, nseg_res;
    int64_t nwarps;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

// rows_per_request: 2*Kmax+1 (sampling) or Kmax+1 (greedy); ve: vector width used
Layout make_layout(int B, int Kmax, int V, int sms, int rows_per_request, int ve) {
    Layout L;
    L.nwarps = (int64_t)sms * kBlocksPerSM * kWarpsPerBlock;
    const int64_t tot_rows = (int64_t)B * rows_per_request * V;
    L.nseg_rows = segs_per_warp(warp_range(tot_rows, L.nwarps, ve), V);
    L.nseg_res = segs_per_warp(warp_range((int64_t)B * V, L.nwarps, ve), V);
    size_t o = 0;
    L.off_row_start = o;
    o = align256(o + sizeof(int) * (size_t)(B + 1));
    L.off_parts = o;
    o = align256(o + sizeof(Part) * (size_t)L.nwarps * (size_t)L.nseg_rows);
    L.off_jobs = o;
    o = align256(o + sizeof(ResJob) * (size_t)B);
    L.off_job_list = o;
    o = align256(o + sizeof(int) * (size_t)B);
    L.off_job_count = o;
    o = align256(o + sizeof(int));
    L.off_rparts = o;
    o = align256(o + sizeof(Part) * (size_t)L.nwarps * (size_t)L.nseg_res);
    L.total = o;
    return L;
}

bool vector_ok(const void *a, const void *b, int64_t ld_row, int V, int dtype) {
    const int esz = dtype == SPEC_BF16 ? 2 : 4;
    const int ve = 16 / esz;
    if (((uintptr_t)a & 15) != 0) return false;
    if (b && ((uintptr_t)b & 15) != 0) return false;
    if (((ld_row * esz) & 15) != 0) return false;
    return V % ve == 0;
}

int check_launch() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    return SPEC_OK;
}

template <class Vec>
int launch_all(const RowsParams &rp, AcceptParams ap, ResidParams qp, FinalParams fp, int sms, bool sample,
               cudaStream_t st) {
    const int grid = sms * kBlocksPerSM;
    const size_t smem = sizeof(int) * (size_t)(rp.B + 1);
    {
        ProfScope ps(st);
        rows_kernel<Vec><<<grid, kThreads, smem, st>>>(rp);
    }
    int rc = check_launch();
    if (rc) return rc;
    const int ablocks = (rp.B + kWarpsPerBlock - 1) / kWarpsPerBlock;
    {
        ProfScope ps(st);
        accept_kernel<<<ablocks, kThreads, 0, st>>>(ap);
    }
    rc = check_launch();
    if (rc || !sample) return rc;
    {
        ProfScope ps(st);
        resid_kernel<Vec><<<grid, kThreads, 0, st>>>(qp);
    }
    rc = check_launch();
    if (rc) return rc;
    {
        ProfScope ps(st);
        final_kernel<<<ablocks, kThreads, 0, st>>>(fp);
    }
    return check_launch();
}

int verify_impl(const void *target, const void *draft, int dtype, int B, int Kmax, int V, int64_t ld_row,
                const int32_t *draft_tokens, const int32_t *num_draft, const float *temperature,
                uint64_t seed, uint64_t step, int32_t *out_tokens, int32_t *out_accepted, float *out_p,
                float *out_q, int32_t *out_status, void *ws, size_t ws_bytes, void *cuda_stream,
                bool sample) {
    if (B < 0 || Kmax < 0 || V <= 0 || ld_row < V) return SPEC_EINVAL;
    if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_EINVAL;
    if (B == 0) return SPEC_OK;
    if (B > SPEC_MAX_BATCH || Kmax > SPEC_MAX_DRAFTS) return SPEC_EUNSUPPORTED;
    if (!target || !out_tokens || !out_accepted || !out_status) return SPEC_EINVAL;
    if (Kmax > 0 && !draft_tokens) return SPEC_EINVAL;
    if (sample && (!temperature || (Kmax > 0 && !draft))) return SPEC_EINVAL;
    if ((int64_t)B * (2 * Kmax + 1) * (int64_t)V > ((int64_t)1 << 50)) return SPEC_EUNSUPPORTED;
    int sms = 0;
    int rc = device_sms(&sms);
    if (rc) return rc;
    const bool vec = vector_ok(target, sample ? draft : nullptr, ld_row, V, dtype);
    const int ve = vec ? (dtype == SPEC_BF16 ? 8 : 4) : 1;
    const Layout L = make_layout(B, Kmax, V, sms, sample ? 2 * Kmax + 1 : Kmax + 1, ve);
    if (!ws) return SPEC_EWORKSPACE;
    if (ws_bytes < L.total) return SPEC_EWORKSPACE;
    rc = prof_prepare();
    if (rc) return rc;

    char *w = (char *)ws;
    RowsParams rp;
    rp.target = target;
    rp.draft = draft;
    rp.ld_row = ld_row;
    rp.B = B;
    rp.Kmax = Kmax;
    rp.V = V;
    rp.num_draft = num_draft;
    rp.temperature = sample ? temperature : nullptr;
    rp.seed = seed;
    rp.step = (uint32_t)step;
    rp.row_start = (int *)(w + L.off_row_start);
    rp.parts = (Part *)(w + L.off_parts);
    rp.nseg = L.nseg_rows;
    rp.job_count = (int *)(w + L.off_job_count);

    AcceptParams ap;
    ap.target = target;
    ap.draft = draft;
    ap.dtype = dtype;
    ap.ld_row = ld_row;
    ap.B = B;
    ap.Kmax = Kmax;
    ap.V = V;
    ap.draft_tokens = draft_tokens;
    ap.num_draft = num_draft;
    ap.temperature = rp.temperature;
    ap.seed = seed;
    ap.step = (uint32_t)step;
    ap.row_start = rp.row_start;
    ap.parts = rp.parts;
    ap.nseg = L.nseg_rows;
    ap.nwarps = L.nwarps;
    ap.ve = ve;
    ap.out_tokens = out_tokens;
    ap.out_accepted = out_accepted;
    ap.out_p = sample ? out_p : nullptr;
    ap.out_q = sample ? out_q : nullptr;
    ap.out_status = out_status;
    ap.jobs = (ResJob *)(w + L.off_jobs);
    ap.job_list = (int *)(w + L.off_job_list);
    ap.job_count = rp.job_count;

    ResidParams qp;
    qp.target = target;
    qp.draft = draft;
    qp.dtype = dtype;
    qp.ld_row = ld_row;
    qp.Kmax = Kmax;
    qp.V = V;
    qp.seed = seed;
    qp.step = (uint32_t)step;
    qp.jobs = ap.jobs;
    qp.job_list = ap.job_list;
    qp.job_count = rp.job_count;
    qp.parts = (Part *)(w + L.off_rparts);
    qp.nseg = L.nseg_res;

    FinalParams fp;
    fp.target = target;
    fp.dtype = dtype;
    fp.ld_row = ld_row;
    fp.B = B;
    fp.Kmax = Kmax;
    fp.V = V;
    fp.seed = seed;
    fp.step = (uint32_t)step;
    fp.jobs = ap.jobs;
    fp.job_list = ap.job_list;
    fp.job_count = rp.job_count;
    fp.parts = qp.parts;
    fp.nseg = L.nseg_res;
    fp.nwarps = L.nwarps;
    fp.ve = ve;
    fp.out_tokens = out_tokens;

    cudaStream_t st = (cudaStream_t)cuda_stream;
    if (dtype == SPEC_BF16)
        return vec ? launch_all<VecBF16>(rp, ap, qp, fp, sms, sample, st)
                   : launch_all<ScalarBF16>(rp, ap, qp, fp, sms, sample, st);
    return vec ? launch_all<VecF32>(rp, ap, qp, fp, sms, sample, st)
               : launch_all<ScalarF32>(rp, ap, qp, fp, sms, sample, st);
}

}  // namespace

extern "C" {

size_t spec_verify_workspace_size(int B, int Kmax, int V, int dtype) {
    if (B < 0 || Kmax < 0 || V <= 0 || (dtype != SPEC_BF16 && dtype != SPEC_F32)) return 0;
    if (B > SPEC_MAX_BATCH || Kmax > SPEC_MAX_DRAFTS) return 0;
    int sms = 0;
    if (device_sms(&sms)) return 0;
    // the widest vector gives the largest per-warp range, hence the most segments
    return make_layout(B, Kmax, V, sms, 2 * Kmax + 1, 8).total;
}

int spec_verify_greedy(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                       const int32_t *draft_tokens, const int32_t *num_draft, int32_t *out_tokens,
                       int32_t *out_accepted, int32_t *out_status, void *ws, size_t ws_bytes,
                       void *cuda_stream) {
    return verify_impl(target, nullptr, dtype, B, Kmax, V, ld_row, draft_tokens, num_draft, nullptr, 0, 0,
                       out_tokens, out_accepted, nullptr, nullptr, out_status, ws, ws_bytes, cuda_stream,
                       false);
}

int spec_verify_sample(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                       int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                       const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                       int32_t *out_accepted, float *out_p, float *out_q, int32_t *out_status, void *ws,
                       size_t ws_bytes, void *cuda_stream) {
    return verify_impl(target, draft, dtype, B, Kmax, V, ld_row, draft_tokens, num_draft, temperature, seed,
                       step, out_tokens, out_accepted, out_p, out_q, out_status, ws, ws_bytes, cuda_stream,
                       true);
}

const char *spec_error_string(int err) {
    switch (err) {
        case SPEC_OK: return "ok";
        case SPEC_EINVAL: return "invalid argument";
        case SPEC_ECUDA: return "CUDA error";
        case SPEC_EUNSUPPORTED: return "unsupported size or layout";
        case SPEC_EWORKSPACE: return "workspace missing or too small";
        default: return "unknown error";
    }
}

int spec_last_cuda_error(void) { return t_last_cuda_error; }

int spec_profile_enable(int on) {
    g_prof = on != 0;
    return SPEC_OK;
}

int spec_profile_read(float *ms, int n) {
    if (!ms || n < 0) return -SPEC_EINVAL;
    if (!g_prof || g_prof_dev < 0) return 0;
    int k = 0;
    for (; k < g_prof_n && k < n; ++k) {
        cudaError_t e = cudaEventSynchronize(g_prof_ev[2 * k + 1]);
        if (e != cudaSuccess) { t_last_cuda_error = (int)e; return -SPEC_ECUDA; }
        e = cudaEventElapsedTime(&ms[k], g_prof_ev[2 * k], g_prof_ev[2 * k + 1]);
        if (e != cudaSuccess) { t_last_cuda_error = (int)e; return -SPEC_ECUDA; }
    }
    return k;
}

}  // extern "C"
