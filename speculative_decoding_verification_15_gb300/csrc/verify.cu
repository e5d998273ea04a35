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
// Kernels per call (fixed grids, no host synchronisation; the second is a
// programmatic dependent launch):
//  main_kernel    streams the rows of every draft position once -- target and draft
//                 rows of sampling requests, target rows of greedy ones -- with plain
//                 16-byte loads: two 512-thread CTAs per SM take the chunks (at most
//                 64 KB of a row) by dynamic tickets.  Per chunk: max, sum of
//                 2^(x log2e / T - max'), and (greedy rows) the lowest argmax.
//                 HBM-bound.
//  commit_kernel  P CTAs ("pieces") per request: each combines the request's chunk
//                 partials, runs the acceptance scan, and reduces its interleaved
//                 share of the one row still needed -- the correction at the first
//                 rejected row j (Gumbel-max over log(max(0, p - q))), the bonus from
//                 row k_b, or the greedy argmax of row k_b -- staged into shared
//                 memory by bulk copies; the last piece to finish combines the
//                 pieces and writes the request's outputs.
// The early-exit calls launch one kernel (early_exit_kernel, below).
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <atomic>
#include <mutex>
#include <type_traits>

#include "spec_common.cuh"
#include "spec_verify.h"

using namespace specv;

namespace {

// ------------------------------------------------------------------ configuration
constexpr int kCW = 16;                          // warps per main-pass CTA
constexpr int kCT = kCW * 32;                    // threads per main-pass CTA
constexpr int kMainBlocksPerSM = 2;              // main-pass CTAs per SM (64 registers a thread)
constexpr int kVPT = 8;                          // 16-byte loads in flight per thread and chunk
constexpr int kChunkMaxBytes = kCT * kVPT * 16 - 32;  // an aligned superset of a chunk fits kCT x kVPT loads
constexpr uint64_t kWaitNs = 2000000000ull;      // bound on every mbarrier wait (2 s)

struct __align__(16) Part {
    float m;         // raw max of the chunk (NaN-propagating)
    float s;         // sum 2^(x c - fl(m c)) over the chunk (sampling rows)
    int idx;         // lowest index of the max (greedy rows; -1 otherwise)
    uint32_t epoch;  // tag of the call that wrote it
};

// ------------------------------------------------------------------ chunking
// Rows are cut into cpr chunks of ce elements (ce a multiple of 8, at most
// kChunkMaxBytes); chunk k of main-pass row r has the flat index r cpr + k.
struct Chunking {
    int cpr, ce;
};

__host__ __device__ inline Chunking make_chunking(int V, int esz) {
    const int max_e = kChunkMaxBytes / esz;
    int cpr = (V + max_e - 1) / max_e;
    int ce = (V + cpr - 1) / cpr;
    ce = (ce + 7) & ~7;
    cpr = (V + ce - 1) / ce;
    return {cpr, ce};
}


// Global byte window of chunk k of a row: the 16-byte aligned superset [a0, a1) of
// elements [e0, e1); smem element 0 is global element e0 - shift.
struct ChunkWin {
    const char *a0;
    uint32_t bytes;
    int e0, e1, shift;
};

__device__ __forceinline__ ChunkWin chunk_window(const char *row, int esz, int V, const Chunking &ck, int k) {
    ChunkWin w;
    w.e0 = k * ck.ce;
    w.e1 = min(w.e0 + ck.ce, V);
    const uintptr_t g0 = (uintptr_t)(row + (int64_t)w.e0 * esz);
    const uintptr_t g1 = (uintptr_t)(row + (int64_t)w.e1 * esz);
    const uintptr_t a0 = g0 & ~(uintptr_t)15, a1 = (g1 + 15) & ~(uintptr_t)15;
    w.a0 = (const char *)a0;
    w.bytes = (uint32_t)(a1 - a0);
    w.shift = (int)((g0 - a0) / esz);
    return w;
}

// ------------------------------------------------------------------ vectors from smem
template <class Vec>
__device__ __forceinline__ void mask_vec(Vec &d, int64_t first, int e0, int e1);

template <>
__device__ __forceinline__ void mask_vec<VecBF16>(VecBF16 &d, int64_t first, int e0, int e1) {
    uint32_t w[4] = {d.v.x, d.v.y, d.v.z, d.v.w};
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const int64_t g = first + e;
        if (g < e0 || g >= e1) w[e >> 1] = (e & 1) ? ((w[e >> 1] & 0x0000FFFFu) | 0xFF800000u)
                                                   : ((w[e >> 1] & 0xFFFF0000u) | 0x0000FF80u);
    }
    d.v = make_uint4(w[0], w[1], w[2], w[3]);
}

template <>
__device__ __forceinline__ void mask_vec<VecF32>(VecF32 &d, int64_t first, int e0, int e1) {
    uint32_t w[4] = {d.v.x, d.v.y, d.v.z, d.v.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const int64_t g = first + e;
        if (g < e0 || g >= e1) w[e] = 0xFF800000u;
    }
    d.v = make_uint4(w[0], w[1], w[2], w[3]);
}

// Loads this thread's vectors of a chunk straight from global memory (16-byte
// loads that bypass L1); entries outside the chunk's window read as -inf.  Vector
// t of thread ct holds global elements ebase + (ct + kCT t) VE + e.  Only a window
// that does not start and end on 16-byte boundaries needs masking, which is
// decided once per chunk (the branch is uniform across the CTA).
template <class Vec>
__device__ __forceinline__ void load_chunk(Vec (&d)[kVPT], const ChunkWin &w, int ct) {
    const int nvec = (int)(w.bytes >> 4);
    const int64_t ebase = (int64_t)w.e0 - w.shift;
#pragma unroll
    for (int t = 0; t < kVPT; ++t) {
        const int j = ct + kCT * t;
        d[t] = j < nvec ? Vec::load(w.a0, j) : Vec::neg_inf();
    }
    if (w.shift != 0 || ebase + (int64_t)nvec * Vec::VE != w.e1) {
#pragma unroll
        for (int t = 0; t < kVPT; ++t) {
            const int j = ct + kCT * t;
            if (j < nvec && (j == 0 || j == nvec - 1)) mask_vec(d[t], ebase + (int64_t)j * Vec::VE, w.e0, w.e1);
        }
    }
}

template <class Vec, int NV>
__device__ __forceinline__ float chunk_max(const Vec (&d)[NV]) {
    float tm = d[0].vmax();
#pragma unroll
    for (int t = 1; t < NV; ++t) tm = max_nan_f32(tm, d[t].vmax());
    return tm;
}

// First entry equal to x among a thread's vectors; vector t of thread ct holds
// entries ebase + (ct + STRIDE t) VE + e.
template <int STRIDE, class Vec, int NV>
__device__ __forceinline__ int chunk_find(const Vec (&d)[NV], int ebase, int ct, float x) {
    int found = -1;
#pragma unroll
    for (int t = 0; t < NV; ++t)
#pragma unroll
        for (int e = 0; e < Vec::VE; ++e)
            if (found < 0 && d[t].get(e) == x) found = ebase + (ct + STRIDE * t) * Vec::VE + e;
    return found;
}

// sum_e 2^(x_e c - ms) over the thread's vectors, two lanes per instruction.
// Every sum is kept relative to a reference fl(m c) -- the product rounded once,
// with __fmul_rn so that the compiler cannot fuse it into a later FMA -- and every
// later use of that reference (rescaling partials, log p) rounds it the same way:
// at small T, m c is in the thousands and one ulp of it is 5e-4.
template <class Vec, int NV>
__device__ __forceinline__ float chunk_expsum(const Vec (&d)[NV], float c, float ms) {
    const float2 cc = make_float2(c, c), mm = make_float2(-ms, -ms);
    float2 acc = make_float2(0.f, 0.f);  // one pair: the warps of the SM supply the parallelism
#pragma unroll
    for (int t = 0; t < NV; ++t)
#pragma unroll
        for (int e = 0; e < Vec::VE; e += 2) {
            const float2 y = ffma2(make_float2(d[t].get(e), d[t].get(e + 1)), cc, mm);
            acc = fadd2(acc, make_float2(ex2_approx(y.x), ex2_approx(y.y)));
        }
    return acc.x + acc.y;
}

// ------------------------------------------------------------------ per-request rows
// Where request b lives.  Padded layout (cu NULL): draft positions b Kmax + i,
// target rows b (Kmax + 1) + i, k_b = num_draft[b] (NULL: Kmax).  Flattened
// layout: draft positions cu[b] + i, target rows (and output token slots)
// cu[b] + b + i, k_b = cu[b + 1] - cu[b].
struct ReqBase {
    int kb;         // k_b, unchecked
    int64_t d0;     // first draft position: draft row, draft token and p/q index
    int64_t t0;     // first target row and first output token slot
    int ntok, npq;  // output token slots and p/q slots of the request
};

__device__ __forceinline__ ReqBase req_base(const int32_t *cu, const int32_t *num_draft, int Kmax, int b) {
    ReqBase r;
    if (cu) {
        const int c0 = cu[b];
        r.kb = cu[b + 1] - c0;
        r.d0 = c0;
        r.t0 = (int64_t)c0 + b;
        r.ntok = r.kb + 1 > 0 ? r.kb + 1 : 0;
        r.npq = r.kb > 0 ? r.kb : 0;
    } else {
        r.kb = num_draft ? num_draft[b] : Kmax;
        r.d0 = (int64_t)b * Kmax;
        r.t0 = (int64_t)b * (Kmax + 1);
        r.ntok = Kmax + 1;
        r.npq = Kmax;
    }
    return r;
}

__device__ __forceinline__ int request_main_rows(const int32_t *cu, const int32_t *num_draft,
                                                 const float *temperature, int Kmax, int b) {
    const int kb = req_base(cu, num_draft, Kmax, b).kb;
    if (kb < 0 || kb > Kmax) return 0;
    if (temperature) {
        const float T = temperature[b];
        if (!(T >= 0.f) || isinf(T)) return 0;
        return T == 0.f ? kb : 2 * kb;
    }
    return kb;
}

// s[b] = main-pass rows of requests 0..b-1 (s[B] = total), in shared memory.
// Row order inside a request: sampling [target 0..k-1 | draft 0..k-1], greedy
// [target 0..k-1].
__device__ void scan_request_rows(int *s, int B, const int32_t *cu, const int32_t *num_draft,
                                  const float *temperature, int Kmax) {
    __shared__ int warp_tot[32];
    const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int per = (B + nthr - 1) / nthr;
    const int lo = min(tid * per, B), hi = min(lo + per, B);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += request_main_rows(cu, num_draft, temperature, Kmax, i);
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
        run += request_main_rows(cu, num_draft, temperature, Kmax, i);
    }
    if (tid == nthr - 1) s[B] = wbase + incl;
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

// =================================================================== shared by the commit and early-exit kernels
// The job row's exact draws: staged units of a row in shared memory, the pruned
// Gumbel-max over them (live lists, Philox blocks drawn only for groups that can
// still win), CTA reductions.  Everything stays in fp32 and 32-bit integers:
// sm_103a has little fp64 throughput.
constexpr int kCommitThreads = 256;           // early-exit CTA threads
constexpr int kCommitWarps = kCommitThreads / 32;
constexpr int kCommitBlocksPerSM = 4;
constexpr int kMaxCluster = 8;
constexpr int kUnitsPerCTA = kCommitWarps;  // early exit: row units per CTA, one per warp
constexpr int kShareMaxBytes = 36 * 1024;   // early exit: row bytes per CTA before the cluster grows
constexpr int kRoundMaxBytes = 40 * 1024;   // early exit: bytes staged per round
constexpr int kUnitGroups = 4;              // groups of four each lane tests per block
constexpr int kBlockGroups = 32 * kUnitGroups;  // groups per block (the unit of work of a warp)
constexpr int kLiveMax = 64 + kBlockGroups;     // a warp's live list: < 64 carried over + one block
constexpr int kLocalScanMax = 1024;         // B up to which each commit CTA counts rows itself
constexpr int kCommitSmemMax = 64 * 1024;   // dynamic shared memory limit set on the kernels

enum JobKind : int { JOB_NONE = 0, JOB_RESID = 1, JOB_BONUS = 2, JOB_ARGMAX = 3 };

struct CommitParams {
    const void *target;
    const void *draft;
    int dtype;
    int64_t ld_row;
    int B, Kmax, V;
    const int32_t *draft_tokens;
    const int32_t *cu;         // flattened layout offsets [B+1], or NULL (padded)
    const int32_t *num_draft;
    const float *temperature;  // NULL: every request greedy
    uint64_t seed;
    uint32_t step;
    int C, ue, NS, slot;       // cluster size, entries per unit, units per round, bytes per unit slot
    int32_t *out_tokens;
    int32_t *out_accepted;
    float *out_p;
    float *out_q;
    int32_t *out_status;
};

// What the warp of draft position i leaves for the scan.
struct PosRes {
    int rej;          // sampling: draft i rejected; greedy: target argmax != x_i
    int tidx;         // target row argmax
    float shift, Cd;  // log p_v = x_v / T - shift and log q_v = y_v / T - Cd on row i
    float seed;       // best exact correction score known before the draw (-inf: none)
    int seed_idx;     // its index, -1 if none
    int nonfinite;    // a row of position i holds NaN or +inf, or is all -inf
    float pad;
};

struct JobDesc {
    int kind, row, A, token;  // token: the greedy mismatch's argmax (JOB_NONE)
    float invT, shift, Cd;    // z = x invT - shift is log p (correction) or x / T (bonus); q likewise with Cd
    float seed;               // exact score of the correction's best seed candidate (-inf: none)
    int seed_idx;
    int status;               // the request's status so far
    uint32_t epoch;           // tag of the call that decided it
};

struct RowRes {
    float M;    // raw row max (NaN-propagating)
    float l2S;  // log2 sum_v 2^(x_v c - fl(M c)) (sampling rows)
    int idx;    // lowest argmax
};

struct __align__(16) SliceRes {  // one CTA's result of a job row share
    float best;    // best exact score (Gumbel-max) or largest finite value (argmax)
    int idx;       // its lowest index, -1 if none
    float rawmax;  // NaN-propagating max of every raw value the CTA read
    int failed;    // a bounded wait gave up
};

struct __align__(16) PieceRes {  // a commit piece's result, stored for the last piece
    float best;
    int idx;
    float rawmax;
    uint32_t tag;  // the call's tag; its complement when a bounded wait gave up
};

// Exact score of the correction draw at one entry: log(p - q) + g, with p > q.
__device__ __forceinline__ float resid_score(float lp, float lq, uint32_t w) {
    return lp + logf(-expm1f(lq - lp)) + gumbel_of_word(w);
}

// Exact score of entry v of the job row (z = x_v invT - shift); -inf when the
// correction has no mass at v.
__device__ __noinline__ float entry_score(bool resid, float invT, float Cd, const char *drow, int dtype, float z,
                                          int v, uint32_t wd) {
    if (resid) {
        const float lq = fmaf(load_logit(drow, dtype, v), invT, -Cd);
        if (!(lq < z)) return kNegInf;
        return resid_score(z, lq, wd);
    }
    return z + gumbel_of_word(wd);
}

// ------------------------------------------------------------------ staged units
// A unit slot holds the bulk copy of row elements [e0, e1) (its 16-byte aligned
// superset); slot element 0 is row element sbase = e0 - shift.
struct UnitView {
    const unsigned char *slot;
    int sbase, e1;
    int g0, g1;   // groups of four [g0, g1)
    int aligned;  // every group starts on an 8-byte (bf16) / 16-byte (fp32) boundary
};

template <int ESZ>
__device__ __forceinline__ float smem_val(const unsigned char *buf, int i) {
    if (ESZ == 2) return __uint_as_float((uint32_t)(*(const uint16_t *)(buf + 2 * i)) << 16);
    return *(const float *)(buf + 4 * i);
}

// The four raw values of group g (entries 4g .. 4g+3); entries at or past e1 read
// as -inf.
template <int ESZ>
__device__ __forceinline__ void group_vals(const UnitView &u, int g, float (&x)[4]) {
    const int off = 4 * g - u.sbase;
    if (u.aligned) {
        if (ESZ == 2) {
            const uint2 w = *(const uint2 *)(u.slot + 2 * off);
            x[0] = bf16_lo(w.x);
            x[1] = bf16_hi(w.x);
            x[2] = bf16_lo(w.y);
            x[3] = bf16_hi(w.y);
        } else {
            const float4 w = *(const float4 *)(u.slot + 4 * off);
            x[0] = w.x;
            x[1] = w.y;
            x[2] = w.z;
            x[3] = w.w;
        }
        if (4 * g + 3 >= u.e1) {
#pragma unroll
            for (int k = 0; k < 4; ++k)
                if (4 * g + k >= u.e1) x[k] = kNegInf;
        }
    } else {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int v = 4 * g + k;
            x[k] = v < u.e1 ? smem_val<ESZ>(u.slot, v - u.sbase) : kNegInf;
        }
    }
}

// NaN-propagating max of group g's raw values (entries at or past e1 as -inf).
template <int ESZ>
__device__ __forceinline__ float group_max(const UnitView &u, int g) {
    if (ESZ == 2 && u.aligned && 4 * g + 3 < u.e1) {
        const uint2 w = *(const uint2 *)(u.slot + 2 * (4 * g - u.sbase));
        const uint32_t m = max_nan_bf16x2(w.x, w.y);
        return max_nan_f32(bf16_lo(m), bf16_hi(m));
    }
    float x[4];
    group_vals<ESZ>(u, g, x);
    return max_nan_f32(max_nan_f32(x[0], x[1]), max_nan_f32(x[2], x[3]));
}

// Gumbel-max over the staged units with exact pruning.  An entry can beat the
// bound thr -- always the exact score of some entry, or -inf -- only if
// z + 17 >= thr (no word gives more than 16.64 of noise) and
// 1 - u <= 1.001 e^(z - thr) (g >= thr - z needs -log u <= e^(z - thr), and
// -log u >= 1 - u).  A warp tests its blocks' groups by their largest z and
// appends the live ones (group, slot and z) to its list in shared memory; every
// 64 listed groups it draws their Philox blocks, two groups per lane (two
// independent chains), so the Philox work follows the number of live groups and
// every draw slot is used.

// Append the live groups of block [gb, ge) of the unit in slot k; returns the new
// (warp-uniform) list length.  CHECK_RAW: fold every raw value into rawmax (rows
// the main pass did not read); otherwise the row is known to be finite.
template <int ESZ, bool CHECK_RAW>
__device__ __forceinline__ int zfilter_block(const UnitView &u, int k, int gb, int ge, float tz, float invT,
                                             float shift, float &rawmax, uint32_t *lg, float *lz, int nlive) {
    const int lane = threadIdx.x & 31;
    const int gfull = u.e1 >> 2;  // groups below gfull lie entirely before e1
    uint32_t lv = 0;
    float zs[kUnitGroups];
#pragma unroll
    for (int t = 0; t < kUnitGroups; ++t) {
        const int g = gb + lane + 32 * t;
        zs[t] = kNegInf;
        if (g < ge) {
            float gm;
            if (ESZ == 2 && u.aligned && g < gfull) {
                const uint2 w = *(const uint2 *)(u.slot + 2 * (4 * g - u.sbase));
                if (CHECK_RAW) {
                    const uint32_t m = max_nan_bf16x2(w.x, w.y);
                    gm = max_nan_f32(bf16_lo(m), bf16_hi(m));
                } else {
                    const uint32_t m = max_bf16x2(w.x, w.y);
                    gm = fmaxf(bf16_lo(m), bf16_hi(m));
                }
            } else {
                float x[4];
                group_vals<ESZ>(u, g, x);
                gm = CHECK_RAW ? max_nan_f32(max_nan_f32(x[0], x[1]), max_nan_f32(x[2], x[3]))
                               : fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3]));
            }
            if (CHECK_RAW) rawmax = max_nan_f32(rawmax, gm);
            zs[t] = fmaf(gm, invT, -shift);
            if (zs[t] > kNegInf && zs[t] >= tz) lv |= 1u << t;
        }
    }
    const int cnt = __popc(lv);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    int pos = nlive + incl - cnt;
#pragma unroll
    for (int t = 0; t < kUnitGroups; ++t)
        if (lv >> t & 1u) {
            lg[pos] = ((uint32_t)(gb + lane + 32 * t) << 3) | (uint32_t)k;
            lz[pos] = zs[t];
            ++pos;
        }
    __syncwarp();
    return nlive + __shfl_sync(0xffffffffu, incl, 31);
}

// Draw the listed groups [base, base + n), n <= 64, two per lane; update thr to
// the warp's best afterwards.
template <int ESZ>
__device__ __forceinline__ void live_round(const uint32_t *lg, const float *lz, int base, int n,
                                           const UnitView *uvs, const JobDesc &jd, uint64_t seed, uint32_t step,
                                           int dtype, uint32_t b, const char *drow, float &thr, float &best,
                                           int &bidx) {
    const int lane = threadIdx.x & 31;
    const bool resid = jd.kind == JOB_RESID;
    const uint32_t purpose = resid ? PURPOSE_RESIDUAL : PURPOSE_BONUS;
    uint32_t gk[2];
    float zm[2];
    bool has[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int item = lane + 32 * h;
        has[h] = item < n;
        const int e = base + (has[h] ? item : 0);
        gk[h] = lg[e];
        zm[h] = lz[e];
    }
    uint4 r4[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) r4[h] = rand_group(seed, step, b, (uint32_t)jd.row, purpose, gk[h] >> 3);
    uint32_t sv = 0;  // bit 4h + q: entry q of group h passed the per-entry test
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        // any survivor needs 1 - u_k <= e^(z_k - thr) <= e^(zmax - thr); the largest
        // w >> 9 of the group gives the smallest 1 - u
        const uint32_t kmax = max(max(r4[h].x >> 9, r4[h].y >> 9), max(r4[h].z >> 9, r4[h].w >> 9));
        if (has[h] && one_minus_u01(kmax << 9) <= ex2_approx((zm[h] - thr) * kLog2e) * 1.001f) {
            float x[4];
            group_vals<ESZ>(uvs[gk[h] & 7u], (int)(gk[h] >> 3), x);
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (one_minus_u01(word_of(r4[h], q)) <= ex2_approx((fmaf(x[q], jd.invT, -jd.shift) - thr) * kLog2e) *
                                                             1.001f)
                    sv |= 1u << (4 * h + q);
        }
    }
    if (sv) {
        // the survivors' draft logits are loaded together: one memory latency however
        // many entries pass (a low bound lets many through)
        float lq[8];
        if (resid) {
#pragma unroll
            for (int k = 0; k < 8; ++k)
                lq[k] = (sv >> k & 1u) ? fmaf(ld_elem<ESZ>(drow, 4 * (int)(gk[k >> 2] >> 3) + (k & 3)), jd.invT,
                                              -jd.Cd)
                                       : 0.f;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (!(sv >> (4 * h) & 15u)) continue;
            float x[4];
            group_vals<ESZ>(uvs[gk[h] & 7u], (int)(gk[h] >> 3), x);  // z again: fewer live registers
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int k = 4 * h + q;
                if (!(sv >> k & 1u)) continue;
                const int v = 4 * (int)(gk[h] >> 3) + q;
                const float z = fmaf(x[q], jd.invT, -jd.shift);
                const uint32_t wd = word_of(r4[h], q);
                // -inf (no residual mass at v) is never a candidate: a row without any
                // must reach the degenerate fallback
                const float sc = resid ? (lq[k] < z ? resid_score(z, lq[k], wd) : kNegInf) : z + gumbel_of_word(wd);
                if (sc > kNegInf && better(sc, v, best, bidx)) { best = sc; bidx = v; }
            }
        }
    }
    thr = fmaxf(thr, warp_max(best));
    __syncwarp();  // the items drawn here are overwritten by the next appends
}

// Reduce (best, idx) with the lowest index on ties, rawmax NaN-propagating and
// failed as an or over a CTA of nwarps warps; every thread returns the CTA's
// result.
__device__ __forceinline__ SliceRes block_reduce_n(SliceRes r, SliceRes *red, int nwarps) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    warp_argmax(r.best, r.idx);
    r.rawmax = warp_max_nan(r.rawmax);
    r.failed = __any_sync(0xffffffffu, r.failed != 0);
    __syncthreads();  // red may still be read from an earlier use
    if (lane == 0) red[warp] = r;
    __syncthreads();
    SliceRes o = red[0];
    for (int w = 1; w < nwarps; ++w) {
        const SliceRes q = red[w];
        if (better(q.best, q.idx, o.best, o.idx)) { o.best = q.best; o.idx = q.idx; }
        o.rawmax = max_nan_f32(o.rawmax, q.rawmax);
        o.failed |= q.failed;
    }
    return o;
}

__device__ __forceinline__ SliceRes block_reduce(SliceRes r, SliceRes *red) {
    return block_reduce_n(r, red, kCommitWarps);
}

// =================================================================== main_kernel
// commit_kernel's per-request words, one 128-byte line per request
constexpr int kSyncWords = 32;
constexpr int kSyncDone = 0;  // pieces finished
constexpr int kSyncBest = 1;  // the pieces' shared bound

struct MainParams {
    const void *target;
    const void *draft;
    int64_t ld_row;
    int B, Kmax, V;
    const int32_t *cu;         // flattened layout offsets [B+1], or NULL (padded)
    const int32_t *num_draft;
    const float *temperature;  // NULL: every request greedy
    int *row_start;            // [B+1], written by block 0 for commit_kernel
    uint32_t *sync;            // [B][kSyncWords] commit_kernel's per-request words, zeroed here by block 0
    uint32_t *ticket;          // dynamic chunk tickets (0 between calls)
    Part *parts;               // [chunks] one per chunk of every main-pass row
    uint16_t *cand;            // [chunks][kCW] sampling rows: the window vector holding each warp's
                               // maximum (0xffff: none), the correction's seed candidates
    uint32_t epoch;            // tag of this call, stored with every partial
};

// What every thread of a main-pass CTA needs about one chunk (written by thread 0).
struct ChunkDesc {
    const char *a0;  // 16-byte aligned start of the chunk's window
    uint32_t bytes;  // window bytes (a multiple of 16)
    int e0, e1;      // row elements [e0, e1) of the chunk
    int shift;       // window element 0 is row element e0 - shift
    float c;         // log2(e) / T, or 0 for a greedy row
    uint32_t t;      // the chunk (flat index); >= total when the CTA is done
    int req;         // its request
};

// Row r of the main pass (request order; inside a request, sampling rows are
// [target 0..k-1 | draft 0..k-1] and greedy rows [target 0..k-1]).
// sc[b] = log2(e) / T_b (0: greedy), computed once per CTA with the row scan.
template <class Vec, class Params>
__device__ __forceinline__ ChunkDesc chunk_desc(const Params &p, const int *rs, const float *sc,
                                                const Chunking &ck, uint32_t t, uint32_t total) {
    ChunkDesc d;
    d.t = t;
    d.a0 = nullptr;
    d.bytes = 0;
    d.e0 = d.e1 = d.shift = 0;
    d.c = 0.f;
    d.req = 0;
    if (t >= total) return d;
    const int r = (int)(t / (uint32_t)ck.cpr), k = (int)(t - (uint32_t)r * (uint32_t)ck.cpr);
    const int b = find_request(rs, p.B, r);
    const int local = r - rs[b];
    const ReqBase rb = req_base(p.cu, p.num_draft, p.Kmax, b);
    const float c = sc[b];
    const int64_t rowbytes = p.ld_row * Vec::ESIZE;
    const char *row = (c == 0.f || local < rb.kb) ? (const char *)p.target + (rb.t0 + local) * rowbytes
                                                   : (const char *)p.draft + (rb.d0 + (local - rb.kb)) * rowbytes;
    const ChunkWin w = chunk_window(row, Vec::ESIZE, p.V, ck, k);
    d.a0 = w.a0;
    d.bytes = w.bytes;
    d.e0 = w.e0;
    d.e1 = w.e1;
    d.shift = w.shift;
    d.c = c;
    d.req = b;
    return d;
}

struct WarpStat {
    float m;  // NaN-propagating max of the warp's entries
    float s;  // sampling: sum 2^(x c - fl(m c)); greedy: unused
    int idx;  // greedy: lowest index of m (-1: none)
    int pad;
};

// Lowest index of the warp maximum M among a thread group's vectors t0 .. t0+NV-1
// of a chunk (greedy rows).  Entry e of vector t of thread ct is element
// ebase + (ct + kCT t) VE + e, so the first t whose vector maximum equals M, then
// the lowest lane holding it, then that lane's first entry, give the lowest index.
template <int T0, class Vec, int NV>
__device__ __forceinline__ int warp_first_index(const Vec (&d)[NV], const float (&vm)[NV], float M, int ebase,
                                                int ct) {
    if (!(M > kNegInf)) return -1;  // all -inf (or NaN): no argmax here
    int idx = -1;
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        const unsigned bal = __ballot_sync(0xffffffffu, vm[t] == M);
        if (idx < 0 && bal) {
            int e = Vec::VE;
#pragma unroll
            for (int q = Vec::VE - 1; q >= 0; --q)
                if (d[t].get(q) == M) e = q;
            const int mine = ebase + (ct + kCT * (T0 + t)) * Vec::VE + e;
            idx = __shfl_sync(0xffffffffu, mine, __ffs(bal) - 1);
        }
    }
    return idx;
}

// Loads vectors t0 .. t0+NV-1 of this thread's share of a chunk (vector t of thread
// ct is window vector ct + kCT t); entries outside the chunk read as -inf.
template <int T0, class Vec, int NV>
__device__ __forceinline__ void load_half_raw(Vec (&d)[NV], const char *a0, int nvec, int ct) {
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        const int j = ct + kCT * (T0 + t);
        d[t] = j < nvec ? Vec::load(a0, j) : Vec::neg_inf();
    }
}

// The masks of the window's edge vectors that hold entries outside [e0, e1).
template <int T0, class Vec, int NV>
__device__ __forceinline__ void mask_half(Vec (&d)[NV], const ChunkDesc &cd, int ct) {
    const int nvec = (int)(cd.bytes >> 4);
    const int64_t ebase = (int64_t)cd.e0 - cd.shift;
    if (cd.shift != 0 || ebase + (int64_t)nvec * Vec::VE != cd.e1) {
#pragma unroll
        for (int t = 0; t < NV; ++t) {
            const int j = ct + kCT * (T0 + t);
            if (j < nvec && (j == 0 || j == nvec - 1)) mask_vec(d[t], ebase + (int64_t)j * Vec::VE, cd.e0, cd.e1);
        }
    }
}

template <int T0, class Vec, int NV>
__device__ __forceinline__ void load_half(Vec (&d)[NV], const ChunkDesc &cd, int ct) {
    load_half_raw<T0>(d, cd.a0, (int)(cd.bytes >> 4), ct);
    mask_half<T0>(d, cd, ct);
}

// A new maximum tm replaces the running one m when it is larger, or NaN; a NaN m
// is never replaced (a later all -inf window must not hide it).
__device__ __forceinline__ bool raises_max(float tm, float m) { return m == m && (tm > m || tm != tm); }

// A lane's running statistics over one half of a chunk: m its max, mc = fl(m c),
// s = sum 2^(x c - mc) (sampling rows; the max moves, and s is rescaled, only when
// a half holds a larger entry).  Returns the half's lane max (NaN-propagating).
// For sampling rows it also keeps mv, the vector (T0 + t) where the lane's max was
// last raised: a cheap pointer to the warp's argmax, kept as a correction seed.
template <int T0, class Vec, int NV>
__device__ __forceinline__ float half_stats(const Vec (&d)[NV], float (&vm)[NV], float c, float &m, float &mc,
                                            float &s, int &mv) {
#pragma unroll
    for (int t = 0; t < NV; ++t) vm[t] = d[t].vmax();
    float tm = vm[0];
    int tv = 0;
#pragma unroll
    for (int t = 1; t < NV; ++t) {
        if (vm[t] > tm) tv = t;
        tm = max_nan_f32(tm, vm[t]);
    }
    if (c != 0.f) {
        if (raises_max(tm, m)) {
            const float mcn = __fmul_rn(tm, c);
            s = (m == kNegInf) ? 0.f : s * ex2_approx(mc - mcn);
            m = tm;
            mc = mcn;
            mv = T0 + tv;
        }
        if (m != kNegInf) s += chunk_expsum(d, c, mc);
    } else {
        m = max_nan_f32(m, tm);
    }
    return tm;
}

// Every needed row once, in chunks of at most 64 KB handed out by dynamic tickets:
// a CTA's first two chunks are its block index and that plus the grid size, every
// later one comes from an atomic counter, two chunks ahead, so that every thread
// knows the next chunk while it still reduces the current one.  Each thread holds
// a chunk's kVPT 16-byte vectors in two halves and reloads a half with the next
// chunk's as soon as it has reduced it, so its loads never stop for the
// reductions, the barrier and the CTA-level combine that end each chunk.  Per
// chunk: warp maxima and exp-sums (greedy rows: warp maxima and their lowest
// indices), combined across the CTA's warps by warp 0 into one Part per chunk,
// stored at the chunk's index; on sampling rows each warp also leaves a pointer to
// the vector holding its maximum, the correction draw's seed candidates.
template <class Vec>
__global__ void __launch_bounds__(kCT, kMainBlocksPerSM) main_kernel(MainParams p) {
    constexpr int kH = kVPT / 2;  // vectors per half
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ WarpStat s_ws[2][kCW];
    __shared__ ChunkDesc s_desc[3];
    int *s_rs = (int *)smem;                                   // [B+1] first main-pass row of each request
    float *s_c = (float *)(smem + sizeof(int) * (size_t)(p.B + 1));  // [B] log2(e) / T (0: greedy)
    const Chunking ck = make_chunking(p.V, Vec::ESIZE);
    const int ct = threadIdx.x;
    // The first chunk's loads go out before the row scan, on the guess that the batch
    // is padded and full (every request Kmax drafts, and T > 0 when the call samples):
    // chunk blockIdx.x is then row r = blockIdx.x / cpr of request r / R.  Every row
    // of the padded layout exists, so a wrong guess only reads a window that the
    // chunk's real descriptor, once the scan has produced it, does not match; that
    // window is then reloaded.
    Vec a[kH], bv[kH];
    const char *g_a0 = nullptr;
    uint32_t g_bytes = 0u;
    if (p.cu == nullptr && p.Kmax > 0) {
        const int R = p.temperature ? 2 * p.Kmax : p.Kmax;
        const int r = (int)(blockIdx.x / (uint32_t)ck.cpr), kc = (int)(blockIdx.x - (uint32_t)r * (uint32_t)ck.cpr);
        const int b = r / R, local = r - b * R;
        if (b < p.B) {
            const int64_t rowbytes = p.ld_row * Vec::ESIZE;
            const char *row = local < p.Kmax
                                  ? (const char *)p.target + ((int64_t)b * (p.Kmax + 1) + local) * rowbytes
                                  : (const char *)p.draft + ((int64_t)b * p.Kmax + (local - p.Kmax)) * rowbytes;
            const ChunkWin w = chunk_window(row, Vec::ESIZE, p.V, ck, kc);
            g_a0 = w.a0;
            g_bytes = w.bytes;
            load_half_raw<0>(a, g_a0, (int)(g_bytes >> 4), ct);
            load_half_raw<kH>(bv, g_a0, (int)(g_bytes >> 4), ct);
        }
    }
    scan_request_rows(s_rs, p.B, p.cu, p.num_draft, p.temperature, p.Kmax);  // ends with __syncthreads
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        const float T = p.temperature ? p.temperature[i] : 0.f;
        s_c[i] = (T > 0.f && !isinf(T)) ? __fdiv_rn(kLog2e, T) : 0.f;
    }
    if (blockIdx.x == 0) {
        for (int i = threadIdx.x; i <= p.B; i += blockDim.x) p.row_start[i] = s_rs[i];
        for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
            p.sync[(size_t)i * kSyncWords + kSyncDone] = 0u;
            p.sync[(size_t)i * kSyncWords + kSyncBest] = 0u;
        }
    }
    pdl_launch_dependents();
    __syncthreads();

    const uint32_t total = (uint32_t)s_rs[p.B] * (uint32_t)ck.cpr;  // < 2^31 (checked by the host)
    const uint32_t G = gridDim.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        s_desc[0] = chunk_desc<Vec>(p, s_rs, s_c, ck, blockIdx.x, total);
        s_desc[1] = chunk_desc<Vec>(p, s_rs, s_c, ck, G + blockIdx.x, total);
    }
    __syncthreads();
    // the current chunk's index, scale and first window element stay in registers;
    // the next chunk's window is read from shared memory where it is used
    uint32_t t = s_desc[0].t;
    float c = s_desc[0].c;
    int ebase = s_desc[0].e0 - s_desc[0].shift;
    if (t < total) {
        if (g_a0 == s_desc[0].a0 && g_bytes == s_desc[0].bytes) {  // the guessed window is the chunk's
            mask_half<0>(a, s_desc[0], ct);
            mask_half<kH>(bv, s_desc[0], ct);
        } else {
            load_half<0>(a, s_desc[0], ct);
            load_half<kH>(bv, s_desc[0], ct);
        }
    }
    int n = 0;
    while (t < total) {
        if (threadIdx.x == 0)
            s_desc[(n + 2) % 3] = chunk_desc<Vec>(p, s_rs, s_c, ck, 2 * G + atomicAdd(p.ticket, 1u), total);
        const ChunkDesc &nx = s_desc[(n + 1) % 3];
        float m = kNegInf, mc = 0.f, s = 0.f;
        int mv = -1;
        float vma[kH], vmb[kH];
        const float ta = half_stats<0>(a, vma, c, m, mc, s, mv);
        int ia = -1;
        float Ma = kNegInf;
        if (c == 0.f) {
            Ma = warp_max_nan(ta);
            ia = warp_first_index<0>(a, vma, Ma, ebase, ct);
        }
        if (nx.t < total) load_half<0>(a, nx, ct);
        const float tb = half_stats<kH>(bv, vmb, c, m, mc, s, mv);
        WarpStat ws;
        ws.pad = 0;
        if (c != 0.f) {
            // the lanes' sums, each relative to its own fl(m c), rescaled to the warp's
            const float M = warp_max_nan(m);
            const float sc = (m == kNegInf || s == 0.f) ? 0.f : s * ex2_approx(mc - __fmul_rn(M, c));
            ws.m = M;
            ws.s = warp_sum(sc);
            ws.idx = -1;
            // the window vector of the lowest lane that holds the warp maximum
            const unsigned own = __ballot_sync(0xffffffffu, m == M && mv >= 0);
            const int src = own ? __ffs(own) - 1 : 0;
            const int vec = __shfl_sync(0xffffffffu, mv, src);
            if (lane == 0)
                p.cand[(size_t)t * kCW + warp] = own ? (uint16_t)(warp * 32 + src + kCT * vec) : (uint16_t)0xffffu;
        } else {
            // entries of half a precede those of half b: a's index wins a tie
            const float Mb = warp_max_nan(tb);
            const int ib = warp_first_index<kH>(bv, vmb, Mb, ebase, ct);
            ws.m = max_nan_f32(Ma, Mb);
            ws.s = 0.f;
            ws.idx = (Ma >= Mb) ? ia : ib;
        }
        if (nx.t < total) load_half<kH>(bv, nx, ct);
        if (lane == 0) s_ws[n & 1][warp] = ws;
        __syncthreads();
        if (warp == 0) {
            // the CTA's warps combined: max, sum relative to fl(max c), lowest argmax
            const WarpStat q = lane < kCW ? s_ws[n & 1][lane] : WarpStat{kNegInf, 0.f, -1, 0};
            const float Mc = warp_max_nan(q.m);
            Part out;
            out.m = Mc;
            float tl = 0.f;
            if (c != 0.f) tl = (q.m == kNegInf || q.s == 0.f) ? 0.f : q.s * exp2f(__fmul_rn(q.m, c) - __fmul_rn(Mc, c));
            out.s = warp_sum(tl);
            uint32_t v = (q.m == Mc && q.idx >= 0) ? (uint32_t)q.idx : 0xffffffffu;
#pragma unroll
            for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
            out.idx = (int)v;
            out.epoch = p.epoch;
            if (lane == 0) p.parts[t] = out;
        }
        ++n;
        t = nx.t;
        c = nx.c;
        ebase = nx.e0 - nx.shift;
    }
}

// ------------------------------------------------------------------ staged job rows (early exit)
__host__ __device__ inline size_t commit_round_bytes(int NS, int slot) {
    return ((size_t)NS * slot + 127) & ~(size_t)127;
}

// Warp-collective (one whole warp): the unit views of round rd of this CTA's share
// of the job row into uvs, then one bulk copy per lane k < NS into slot k, all on
// one barrier phase.  Unit rank + C k lands in slot k of its round.
template <int ESZ>
__device__ __forceinline__ void issue_job_round(const CommitParams &p, uint32_t rank, const char *jrow, int rd,
                                                unsigned char *buf, uint64_t *bar, UnitView *uvs) {
    const int lane = threadIdx.x & 31;
    const Chunking uk = {p.C * kUnitsPerCTA, p.ue};
    const int nunits = (p.V + p.ue - 1) / p.ue;  // units holding entries
    ChunkWin w;
    w.bytes = 0;
    const int u = (int)rank + p.C * (rd * p.NS + lane);
    UnitView uv;
    uv.slot = buf + (size_t)lane * p.slot;
    uv.sbase = uv.e1 = uv.g0 = uv.g1 = 0;
    uv.aligned = 0;
    if (lane < p.NS && u < nunits) {
        w = chunk_window(jrow, ESZ, p.V, uk, u);
        uv.sbase = w.e0 - w.shift;
        uv.e1 = w.e1;
        uv.g0 = w.e0 >> 2;
        uv.g1 = (w.e1 + 3) >> 2;
        uv.aligned = (w.shift & 3) == 0;
    }
    if (lane < p.NS) uvs[lane] = uv;
    const int bytes = warp_sum_i((int)w.bytes);
    if (lane == 0) mbar_arrive_expect_tx(bar, (uint32_t)bytes);
    __syncwarp();
    if (w.bytes) bulk_g2s(buf + (size_t)lane * p.slot, w.a0, w.bytes, bar);
}

// This CTA's share of the job row, round 0 already in flight: the pruned Gumbel-max
// (correction or bonus) or the argmax, over the staged units.  A round's units are
// cut into blocks of kBlockGroups groups, dealt to the warps round-robin, so every
// warp gets a mix of the units.  Every thread of the CTA calls it; every thread
// gets the CTA's result.
template <int ESZ>
__device__ SliceRes job_row_rounds(const CommitParams &p, const JobDesc &jd, uint32_t b, uint32_t rank,
                                   const char *jrow, const char *drow, unsigned char *buf, uint64_t *bar,
                                   UnitView *uvs, uint32_t (*live_g)[kLiveMax], float (*live_z)[kLiveMax],
                                   SliceRes *red) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nrounds = jd.kind == JOB_NONE ? 0 : kUnitsPerCTA / p.NS;
    const int bpu = (((p.ue + 3) >> 2) + kBlockGroups - 1) / kBlockGroups;  // blocks per full unit
    SliceRes mine;
    mine.best = jd.seed;
    mine.idx = jd.seed_idx;
    mine.rawmax = kNegInf;
    mine.failed = 0;
    float thr = jd.seed;
    uint32_t phase = 0;
    for (int rd = 0; rd < nrounds; ++rd) {
        // one thread waits, so that a CTA whose copies are in flight takes no issue
        // slots from the CTAs sharing its SM; the others then take the completed
        // phase themselves (it completes at once), which makes the bytes visible to them
        bool ok = true;
        if (tid == 0) ok = mbar_wait(bar, phase, kWaitNs);
        if (__syncthreads_or(!ok)) {
            // give up on this request; wait (bounded) for the copies in flight first
            if (tid == 0) mbar_wait(bar, phase, kWaitNs);
            mine.failed = 1;
            break;
        }
        mbar_try_wait(bar, phase);
        phase ^= 1u;
        const int nblk = p.NS * bpu;
        if (jd.kind == JOB_BONUS) {
            // seed the bound with each thread's largest entry (exact score)
            float m = kNegInf;
            int mi = -1;
            for (int bi = warp; bi < nblk; bi += kCommitWarps) {
                const UnitView uv = uvs[bi / bpu];
                const int gb = uv.g0 + (bi % bpu) * kBlockGroups, ge = min(gb + kBlockGroups, uv.g1);
                for (int g = gb + lane; g < ge; g += 32) {
                    float xv[4];
                    group_vals<ESZ>(uv, g, xv);
#pragma unroll
                    for (int q = 0; q < 4; ++q)
                        if (xv[q] > m) { m = xv[q]; mi = 4 * g + q; }
                }
            }
            SliceRes seed;
            seed.best = kNegInf;
            seed.idx = -1;
            seed.rawmax = kNegInf;
            seed.failed = 0;
            if (mi >= 0) {
                const uint4 r4 = rand_group(p.seed, p.step, b, (uint32_t)jd.row, PURPOSE_BONUS,
                                            (uint32_t)mi >> 2);
                seed.best = fmaf(m, jd.invT, -jd.shift) + gumbel_of_word(word_of(r4, mi & 3));
                seed.idx = mi;
            }
            seed = block_reduce(seed, red);
            if (better(seed.best, seed.idx, mine.best, mine.idx)) { mine.best = seed.best; mine.idx = seed.idx; }
            thr = fmaxf(thr, seed.best);
        }
        if (jd.kind == JOB_ARGMAX) {
            for (int bi = warp; bi < nblk; bi += kCommitWarps) {
                const UnitView uv = uvs[bi / bpu];
                const int gb = uv.g0 + (bi % bpu) * kBlockGroups, ge = min(gb + kBlockGroups, uv.g1);
                float m = kNegInf;
                int mi = -1;
                for (int g = gb + lane; g < ge; g += 32) {
                    float xv[4];
                    group_vals<ESZ>(uv, g, xv);
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        mine.rawmax = max_nan_f32(mine.rawmax, xv[q]);
                        if (xv[q] > m) { m = xv[q]; mi = 4 * g + q; }
                    }
                }
                if (better(m, mi, mine.best, mine.idx)) { mine.best = m; mine.idx = mi; }
            }
        } else {
            uint32_t *lg = live_g[warp];
            float *lz = live_z[warp];
            int nlive = 0;
            for (int bi = warp; bi < nblk; bi += kCommitWarps) {
                const int k = bi / bpu;
                const UnitView uv = uvs[k];
                const int gb = uv.g0 + (bi % bpu) * kBlockGroups, ge = min(gb + kBlockGroups, uv.g1);
                if (gb >= ge) continue;
                nlive = jd.kind == JOB_BONUS
                            ? zfilter_block<ESZ, true>(uv, k, gb, ge, thr - kGumbelMax, jd.invT, jd.shift,
                                                       mine.rawmax, lg, lz, nlive)
                            : zfilter_block<ESZ, false>(uv, k, gb, ge, thr - kGumbelMax, jd.invT, jd.shift,
                                                        mine.rawmax, lg, lz, nlive);
                while (nlive >= 64) {  // draw the newest 64; the rest stay listed
                    nlive -= 64;
                    live_round<ESZ>(lg, lz, nlive, 64, uvs, jd, p.seed, p.step, p.dtype, b, drow, thr, mine.best, mine.idx);
                }
            }
            if (nlive > 0)
                live_round<ESZ>(lg, lz, 0, nlive, uvs, jd, p.seed, p.step, p.dtype, b, drow, thr, mine.best, mine.idx);
        }
        __syncthreads();  // every warp is done with the round's slots and views
        if (warp == 0 && rd + 1 < nrounds) issue_job_round<ESZ>(p, rank, jrow, rd + 1, buf, bar, uvs);
    }
    return block_reduce(mine, red);
}

// =================================================================== commit_kernel
// P CTAs ("pieces") per request, each with kJobThreads threads.  Every piece of
// request b
//  1. decides the request -- the same arithmetic on the same data in every piece,
//     so all of them agree: it combines each row's per-chunk partials, runs the
//     acceptance scan and finds the one row still needed (the first rejected
//     target row j for the correction, row k_b for the bonus draw or, greedy, for
//     the argmax when every draft matched);
//  2. stages its units of that row -- units piece, piece + P, piece + 2P, ... of
//     kUnitE entries, so the pieces interleave across the vocabulary and share the
//     work of a Zipf-like head evenly -- into shared memory by bulk copies, and
//     reduces them: the pruned Gumbel-max, or the argmax;
//  3. stores its result and bumps the request's counter; the piece that completes
//     the count combines the P results and writes the request's outputs.
// No CTA waits for another: pieces meet through the counter (last arriver).
constexpr int kJobThreads = 128;
constexpr int kJobWarps = kJobThreads / 32;
constexpr int kJobBlocksPerSM = 8;
constexpr int kUnitE = 1024;       // entries per unit (a multiple of 8)
constexpr int kUnitsPerPiece = 8;  // units a piece stages (a live group's slot index takes 3 bits)
constexpr int kCandPrefetch = 256; // seed-candidate pointers a piece fetches with the partials

struct JobParams {
    const void *target;
    const void *draft;
    int dtype;
    int64_t ld_row;
    int B, Kmax, V;
    const int32_t *draft_tokens;
    const int32_t *cu;         // flattened layout offsets [B+1], or NULL (padded)
    const int32_t *num_draft;
    const float *temperature;  // NULL: every request greedy
    uint64_t seed;
    uint32_t step;
    uint32_t epoch;            // tag the main pass stored with this call's partials
    const int *row_start;      // from main_kernel; read only when B > kLocalScanMax
    const Part *parts;
    const uint16_t *cand;      // [chunks][kCW] the main pass's seed-candidate vectors
    int cpr, ce;               // main pass: chunks per row, entries per chunk
    int P;                     // pieces per request
    int slot;                  // bytes per unit slot
    uint32_t *ticket;          // main_kernel's ticket counter, reset here for the next call
    uint32_t *sync;            // [B][kSyncWords]: pieces finished, and the best exact score any piece
                               // has found (ordered bits; 0: none); zeroed by main_kernel
    PieceRes *pres;            // [B * P]
    int32_t *out_tokens;
    int32_t *out_accepted;
    float *out_p;
    float *out_q;
    int32_t *out_status;
};

// Float <-> unsigned with the same order (for atomicMax over scores); 0 means none.
__device__ __forceinline__ uint32_t ordered_bits(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float ordered_float(uint32_t u) {
    if (u == 0u) return kNegInf;
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}
__device__ __forceinline__ uint32_t ld_relaxed_u32(const uint32_t *p) {
    uint32_t v;
    asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__host__ __device__ inline int job_units(int V) { return (V + kUnitE - 1) / kUnitE; }
__host__ __device__ inline int job_pieces(int V) { return (job_units(V) + kUnitsPerPiece - 1) / kUnitsPerPiece; }
__host__ __device__ inline int job_slot_bytes(int esz) { return ((kUnitE * esz + 32) + 127) & ~127; }
__host__ __device__ inline size_t job_smem_bytes(int esz, int Kmax) {
    return (size_t)kUnitsPerPiece * job_slot_bytes(esz) + sizeof(PosRes) * (size_t)Kmax +
           sizeof(RowRes) * 2 * (size_t)Kmax + 5 * sizeof(float) * (size_t)Kmax;
}

// This piece's share of the job row, staged: the pruned Gumbel-max (correction or
// bonus) or the argmax.  Every thread calls it and gets the CTA's result.
template <int ESZ>
__device__ SliceRes job_piece(const JobParams &p, const JobDesc &jd, uint32_t b, const char *drow,
                              const UnitView *uvs, int nu, uint32_t (*live_g)[kLiveMax],
                              float (*live_z)[kLiveMax], SliceRes *red) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const bool resid = jd.kind == JOB_RESID;
    constexpr int bpu = ((kUnitE / 4) + kBlockGroups - 1) / kBlockGroups;  // blocks per unit
    const int nblk = nu * bpu;
    SliceRes mine;
    mine.best = kNegInf;
    mine.idx = -1;
    mine.rawmax = kNegInf;
    mine.failed = 0;
    if (jd.kind == JOB_ARGMAX) {
        for (int bi = warp; bi < nblk; bi += kJobWarps) {
            const UnitView uv = uvs[bi / bpu];
            const int gb = uv.g0 + (bi % bpu) * kBlockGroups, ge = min(gb + kBlockGroups, uv.g1);
            for (int g = gb + lane; g < ge; g += 32) {
                float xv[4];
                group_vals<ESZ>(uv, g, xv);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    mine.rawmax = max_nan_f32(mine.rawmax, xv[q]);
                    if (better(xv[q], 4 * g + q, mine.best, mine.idx) && xv[q] > kNegInf) {
                        mine.best = xv[q];
                        mine.idx = 4 * g + q;
                    }
                }
            }
        }
        return block_reduce_n(mine, red, kJobWarps);
    }
    // seed: the correction's comes from this piece's share of the main pass's
    // candidates (scored while the copies landed); otherwise the exact score of each
    // thread's largest entry bounds the draw from below.  Either way the pieces of a
    // request share the best bound any of them knows (see below)
    mine.best = jd.seed;
    mine.idx = jd.seed_idx;
    if (jd.kind != JOB_RESID) {
        float m = kNegInf;
        int mi = -1;
        for (int bi = warp; bi < nblk; bi += kJobWarps) {
            const UnitView uv = uvs[bi / bpu];
            const int gb = uv.g0 + (bi % bpu) * kBlockGroups, ge = min(gb + kBlockGroups, uv.g1);
            for (int g = gb + lane; g < ge; g += 32) {
                float xv[4];
                group_vals<ESZ>(uv, g, xv);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    if (xv[q] > m) { m = xv[q]; mi = 4 * g + q; }
            }
        }
        SliceRes seed;
        seed.best = kNegInf;
        seed.idx = -1;
        seed.rawmax = kNegInf;
        seed.failed = 0;
        if (mi >= 0) {
            const uint4 r4 = rand_group(p.seed, p.step, b, (uint32_t)jd.row, resid ? PURPOSE_RESIDUAL : PURPOSE_BONUS,
                                        (uint32_t)mi >> 2);
            const float z = fmaf(m, jd.invT, -jd.shift);
            const float sc = entry_score(resid, jd.invT, jd.Cd, drow, p.dtype, z, mi, word_of(r4, mi & 3));
            if (sc > kNegInf) {
                seed.best = sc;
                seed.idx = mi;
            }
        }
        seed = block_reduce_n(seed, red, kJobWarps);
        mine.best = seed.best;
        mine.idx = seed.idx;
        if (threadIdx.x == 0 && seed.best > kNegInf) atomicMax(p.sync + (size_t)b * kSyncWords + kSyncBest, ordered_bits(seed.best));
    }
    // The bound is shared with the request's other pieces: each publishes the best
    // exact score it knows, and reads theirs one block ahead of using it.  Every
    // published value is the exact score of an entry, so it never exceeds the draw's
    // maximum and the pruning stays exact.
    const bool share = true;
    float thr = mine.best, published = mine.best;
    uint32_t shared_bits = share ? ld_relaxed_u32(p.sync + (size_t)b * kSyncWords + kSyncBest) : 0u;
    uint32_t *lg = live_g[warp];
    float *lz = live_z[warp];
    int nlive = 0;
    for (int bi = warp; bi < nblk; bi += kJobWarps) {
        const int k = bi / bpu;
        const UnitView uv = uvs[k];
        const int gb = uv.g0 + (bi % bpu) * kBlockGroups, ge = min(gb + kBlockGroups, uv.g1);
        if (share) {
            thr = fmaxf(thr, ordered_float(shared_bits));
            shared_bits = ld_relaxed_u32(p.sync + (size_t)b * kSyncWords + kSyncBest);
            if (lane == 0 && thr > published) {
                atomicMax(p.sync + (size_t)b * kSyncWords + kSyncBest, ordered_bits(thr));
                published = thr;
            }
        }
        if (gb >= ge) continue;
        nlive = resid ? zfilter_block<ESZ, false>(uv, k, gb, ge, thr - kGumbelMax, jd.invT, jd.shift, mine.rawmax, lg,
                                                  lz, nlive)
                      : zfilter_block<ESZ, true>(uv, k, gb, ge, thr - kGumbelMax, jd.invT, jd.shift, mine.rawmax, lg,
                                                 lz, nlive);
        while (nlive >= 64) {  // draw the newest 64; the rest stay listed
            nlive -= 64;
            live_round<ESZ>(lg, lz, nlive, 64, uvs, jd, p.seed, p.step, p.dtype, b, drow, thr, mine.best, mine.idx);
        }
    }
    if (nlive > 0)
        live_round<ESZ>(lg, lz, 0, nlive, uvs, jd, p.seed, p.step, p.dtype, b, drow, thr, mine.best, mine.idx);
    return block_reduce_n(mine, red, kJobWarps);
}

// One row's statistics from its cpr per-chunk partials, by one thread.
__device__ __forceinline__ RowRes row_from_parts(const Part *pp, int cpr, float c, bool greedy, uint32_t epoch,
                                                 bool &stale) {
    float M = kNegInf;
    for (int q = 0; q < cpr; ++q) {
        const Part x = pp[q];
        stale |= x.epoch != epoch;
        M = max_nan_f32(M, x.m);
    }
    const float MC = __fmul_rn(M, c);
    float sum = 0.f;
    int bi = -1;
    for (int q = 0; q < cpr; ++q) {
        const Part x = pp[q];
        if (!greedy && x.m != kNegInf && x.s != 0.f) sum += x.s * exp2f(__fmul_rn(x.m, c) - MC);
        if (greedy && x.m == M && x.idx >= 0 && (bi < 0 || x.idx < bi)) bi = x.idx;
    }
    RowRes r;
    r.M = M;
    r.idx = bi;
    r.l2S = greedy ? 0.f : log2f(sum);
    return r;
}

template <int ESZ>
__global__ void __launch_bounds__(kJobThreads, kJobBlocksPerSM) commit_kernel(JobParams p) {
    extern __shared__ __align__(128) unsigned char jdyn[];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_live_g[kJobWarps][kLiveMax];
    __shared__ float s_live_z[kJobWarps][kLiveMax];
    __shared__ SliceRes s_red[kJobWarps];
    __shared__ UnitView s_uv[kUnitsPerPiece];
    __shared__ JobDesc s_job;
    __shared__ int s_sum[2 * kJobWarps];
    __shared__ int s_last;
    __shared__ uint16_t s_cand[kCandPrefetch];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x / p.P, piece = blockIdx.x - b * p.P;
    unsigned char *slots = jdyn;
    PosRes *s_pos = (PosRes *)(jdyn + (size_t)kUnitsPerPiece * p.slot);
    RowRes *s_rows = (RowRes *)(s_pos + p.Kmax);  // [2 Kmax] target rows, then draft rows
    float *s_xt = (float *)(s_rows + 2 * p.Kmax); // target logit at x_i
    float *s_xd = s_xt + p.Kmax;                  // draft logit at x_i
    float *s_l2u = s_xd + p.Kmax;                 // log2 of the acceptance uniform u_i
    float *s_pp = s_l2u + p.Kmax;
    float *s_qq = s_pp + p.Kmax;
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        mbar_init_fence();
    }

    // ---- inputs only: this part overlaps the end of main_kernel
    const ReqBase rbase = req_base(p.cu, p.num_draft, p.Kmax, b);
    const int kb_raw = rbase.kb;
    int status = SPEC_STATUS_OK;
    float T = 0.f;
    if (kb_raw < 0 || kb_raw > p.Kmax) status = SPEC_STATUS_BAD_K;
    if (status == SPEC_STATUS_OK && p.temperature) {
        T = p.temperature[b];
        if (!(T >= 0.f) || isinf(T)) status = SPEC_STATUS_BAD_TEMPERATURE;
    }
    const int kb = status == SPEC_STATUS_BAD_K ? 0 : kb_raw;
    const bool greedy = (T == 0.f);
    const int32_t *x = p.draft_tokens + rbase.d0;
    if (status == SPEC_STATUS_OK) {
        bool bad = false;
        for (int i = tid; i < kb; i += kJobThreads) bad |= (x[i] < 0 || x[i] >= p.V);
        if (__syncthreads_or(bad)) status = SPEC_STATUS_BAD_TOKEN;
    }
    const float c = greedy ? 0.f : __fdiv_rn(kLog2e, T);
    const float invT = greedy ? 0.f : __fdiv_rn(1.f, T);
    const int npos = status == SPEC_STATUS_OK ? kb : 0;
    if (!greedy) {
        for (int i = tid; i < npos; i += kJobThreads) {
            const int xi = x[i];
            s_xt[i] = ld_elem<ESZ>(p.target, (rbase.t0 + i) * p.ld_row + xi);
            s_xd[i] = ld_elem<ESZ>(p.draft, (rbase.d0 + i) * p.ld_row + xi);
            const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)i, PURPOSE_ACCEPT, 0u);
            s_l2u[i] = log2f(u01(r4.x));
        }
    }
    // flat main-pass index of this request's first row
    int r0 = 0;
    if (p.B <= kLocalScanMax) {
        int before = 0;
        for (int bb = tid; bb < b; bb += kJobThreads)
            before += request_main_rows(p.cu, p.num_draft, p.temperature, p.Kmax, bb);
        before = warp_sum_i(before);
        if (lane == 0) s_sum[warp] = before;
        __syncthreads();
        for (int w = 0; w < kJobWarps; ++w) r0 += s_sum[w];
    }
    pdl_wait();
    // ---- main_kernel is complete from here on
    if (blockIdx.x == 0 && tid == 0) *p.ticket = 0u;  // every ticket of this call is taken
    if (p.B > kLocalScanMax) r0 = p.row_start[b];
    const int nrows = greedy ? npos : 2 * npos;  // flat rows r0 .. r0 + nrows - 1
    const int items = nrows * p.cpr;
    const bool staged = (size_t)items * sizeof(Part) <= (size_t)kUnitsPerPiece * p.slot;
    const Part *gparts = p.parts + (int64_t)r0 * p.cpr;
    Part *s_parts = (Part *)slots;  // the unit slots hold the partials until the job is known
    if (staged)
        for (int it = tid; it < items; it += kJobThreads) s_parts[it] = gparts[it];
    // this piece's seed-candidate pointers: slots q = piece + P j (j < nq) of each
    // target row's chunk x warp list, fetched with the partials (row A's are used)
    const int ncand = p.cpr * kCW;
    const int nq = piece < ncand ? (ncand - piece + p.P - 1) / p.P : 0;
    const bool cand_pre = !greedy && npos * nq <= kCandPrefetch;
    if (cand_pre)
        for (int it = tid; it < npos * nq; it += kJobThreads) {
            const int i = it / nq, j = it - i * nq;
            s_cand[it] = p.cand[((int64_t)r0 + i) * ncand + piece + p.P * j];
        }
    __syncthreads();
    const Part *rp = staged ? s_parts : gparts;

    // ---- the decision: one thread per row, then one thread per position
    bool stale = false;
    for (int r = tid; r < nrows; r += kJobThreads)
        s_rows[r] = row_from_parts(rp + (int64_t)r * p.cpr, p.cpr, c, greedy && r < npos, p.epoch, stale);
    stale = __syncthreads_or(stale);
    for (int i = tid; i < npos; i += kJobThreads) {
        const RowRes tr = s_rows[i];
        PosRes pr;
        pr.tidx = tr.idx;
        pr.shift = pr.Cd = 0.f;
        pr.seed = kNegInf;
        pr.seed_idx = -1;
        pr.pad = 0.f;
        if (greedy) {
            pr.nonfinite = !(fabsf(tr.M) < __int_as_float(0x7f800000));
            pr.rej = tr.idx != x[i];
        } else {
            const RowRes dr = s_rows[npos + i];
            // a NaN leaves its chunk's max NaN; +inf makes the sum NaN: both show here
            pr.nonfinite = !(fabsf(tr.M) < __int_as_float(0x7f800000) && fabsf(dr.M) < __int_as_float(0x7f800000) &&
                             fabsf(tr.l2S) < __int_as_float(0x7f800000) &&
                             fabsf(dr.l2S) < __int_as_float(0x7f800000));
            const float l2p = fmaf(s_xt[i], c, -__fmul_rn(tr.M, c)) - tr.l2S;  // log2 p_i(x_i)
            const float l2q = fmaf(s_xd[i], c, -__fmul_rn(dr.M, c)) - dr.l2S;  // log2 q_i(x_i)
            // accept iff u q < p, i.e. log2 u < log2 p - log2 q (Q = 0 < P accepts; P = 0 rejects)
            pr.rej = !(s_l2u[i] < l2p - l2q);
            // log p_v = x_v / T - (fl(M c) + log2 S) ln 2, and q likewise
            pr.shift = (__fmul_rn(tr.M, c) + tr.l2S) * 0.6931471805599453f;
            pr.Cd = (__fmul_rn(dr.M, c) + dr.l2S) * 0.6931471805599453f;
            s_pp[i] = exp2f(l2p);
            s_qq[i] = exp2f(l2q);
        }
        s_pos[i] = pr;
    }
    __syncthreads();

    // ---- the scan (warp 0): A = first rejected position, and the job
    if (warp == 0) {
        JobDesc jd;
        jd.kind = JOB_NONE;
        jd.row = 0;
        jd.A = 0;
        jd.token = -1;
        jd.invT = invT;
        jd.shift = jd.Cd = 0.f;
        jd.seed = kNegInf;
        jd.seed_idx = -1;
        jd.epoch = p.epoch;
        int st = status;
        if (st == SPEC_STATUS_OK && stale) st = SPEC_STATUS_INTERNAL;
        if (st == SPEC_STATUS_OK) {
            bool nf = false;
            for (int i = lane; i < kb; i += 32) nf |= s_pos[i].nonfinite != 0;
            if (__any_sync(0xffffffffu, nf)) st = SPEC_STATUS_NONFINITE;
        }
        if (st == SPEC_STATUS_OK) {
            int A = kb;
            for (int i0 = 0; i0 < kb && A == kb; i0 += 32) {
                const int i = i0 + lane;
                const unsigned msk = __ballot_sync(0xffffffffu, i < kb && s_pos[i].rej != 0);
                if (msk) A = i0 + __ffs(msk) - 1;
            }
            jd.A = A;
            if (greedy) {
                if (A < kb) {
                    jd.token = s_pos[A].tidx;
                } else {
                    jd.kind = JOB_ARGMAX;
                    jd.row = kb;
                }
            } else if (A < kb) {
                const PosRes pr = s_pos[A];
                jd.kind = JOB_RESID;
                jd.row = A;
                jd.shift = pr.shift;
                jd.Cd = pr.Cd;
            } else {
                jd.kind = JOB_BONUS;
                jd.row = kb;
            }
        }
        jd.status = st;
        if (lane == 0) s_job = jd;
    }
    __syncthreads();
    JobDesc jd = s_job;
    status = jd.status;

    int token = jd.token;
    bool writer = piece == 0;
    const int64_t rowbytes = p.ld_row * ESZ;
    if (jd.kind != JOB_NONE) {
        // ---- this piece's units of the job row: one bulk copy each, one barrier phase
        const char *jrow = (const char *)p.target + (rbase.t0 + jd.row) * rowbytes;
        const char *drow = jd.kind == JOB_RESID ? (const char *)p.draft + (rbase.d0 + jd.row) * rowbytes : nullptr;
        const int nunits = job_units(p.V);
        const int nu = min(kUnitsPerPiece, (nunits - piece + p.P - 1) / p.P);
        if (warp == 0) {
            const Chunking uk = {nunits, kUnitE};
            ChunkWin w;
            w.bytes = 0;
            UnitView uv;
            uv.slot = slots + (size_t)lane * p.slot;
            uv.sbase = uv.e1 = uv.g0 = uv.g1 = 0;
            uv.aligned = 0;
            if (lane < nu) {
                w = chunk_window(jrow, ESZ, p.V, uk, piece + p.P * lane);
                uv.sbase = w.e0 - w.shift;
                uv.e1 = w.e1;
                uv.g0 = w.e0 >> 2;
                uv.g1 = (w.e1 + 3) >> 2;
                uv.aligned = (w.shift & 3) == 0;
            }
            if (lane < kUnitsPerPiece) s_uv[lane] = uv;
            const int bytes = warp_sum_i((int)w.bytes);
            if (lane == 0) mbar_arrive_expect_tx(&s_bar, (uint32_t)bytes);
            __syncwarp();
            if (w.bytes) bulk_g2s(slots + (size_t)lane * p.slot, w.a0, w.bytes, &s_bar);
        }
        // correction: this piece's share of the seed candidates of row A (the vector
        // holding each warp's maximum of each main-pass chunk), scored while the
        // copies land; the best one is shared with the other pieces
        if (jd.kind == JOB_RESID) {
            constexpr int VE = 16 / ESZ;
            const Chunking mk = {p.cpr, p.ce};
            SliceRes sd;
            sd.best = kNegInf;
            sd.idx = -1;
            sd.rawmax = kNegInf;
            sd.failed = 0;
            for (int j = tid; j < nq; j += kJobThreads) {
                const int q = piece + p.P * j;
                const uint32_t cv = cand_pre ? s_cand[jd.row * nq + j] : p.cand[((int64_t)r0 + jd.row) * ncand + q];
                const ChunkWin w = chunk_window(jrow, ESZ, p.V, mk, q / kCW);
                if (cv == 0xffffu || (cv + 1) * 16 > w.bytes) continue;
                const int ebase = w.e0 - w.shift + (int)cv * VE;
                // the target vector and the draft logits of its entries, loaded together
                const uint4 raw = ld_stream_v4(w.a0 + 16 * (size_t)cv);
                float lq[VE];
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                    const int v = ebase + e;
                    lq[e] = (v >= w.e0 && v < w.e1) ? ld_elem<ESZ>(drow, v) : 0.f;
                }
                float bx = kNegInf, bq = 0.f;
                int bv = -1;
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                    const int v = ebase + e;
                    const float xv = ESZ == 2 ? VecBF16{raw}.get(e) : VecF32{raw}.get(e);
                    if (v >= w.e0 && v < w.e1 && xv > bx) { bx = xv; bv = v; bq = lq[e]; }
                }
                if (bv < 0) continue;
                const float z = fmaf(bx, jd.invT, -jd.shift);
                const float lqs = fmaf(bq, jd.invT, -jd.Cd);
                if (!(lqs < z)) continue;  // no residual mass at bv
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)jd.row, PURPOSE_RESIDUAL,
                                            (uint32_t)bv >> 2);
                const float sc = resid_score(z, lqs, word_of(r4, bv & 3));
                if (better(sc, bv, sd.best, sd.idx)) { sd.best = sc; sd.idx = bv; }
            }
            sd = block_reduce_n(sd, s_red, kJobWarps);
            jd.seed = sd.best;
            jd.seed_idx = sd.idx;
            if (tid == 0 && sd.best > kNegInf) atomicMax(p.sync + (size_t)b * kSyncWords + kSyncBest, ordered_bits(sd.best));
        }
        // one thread waits (bounded), the others then take the completed phase
        bool ok = true;
        if (tid == 0) ok = mbar_wait(&s_bar, 0, kWaitNs);
        SliceRes res;
        if (__syncthreads_or(!ok)) {
            if (tid == 0) mbar_wait(&s_bar, 0, kWaitNs);  // the copies in flight, bounded
            res.best = kNegInf;
            res.idx = -1;
            res.rawmax = kNegInf;
            res.failed = 1;
        } else {
            mbar_try_wait(&s_bar, 0);
            res = job_piece<ESZ>(p, jd, (uint32_t)b, drow, s_uv, nu, s_live_g, s_live_z, s_red);
        }
        // ---- the pieces meet: the last to finish combines them
        if (tid == 0) {
            PieceRes pr;
            pr.best = res.best;
            pr.idx = res.idx;
            pr.rawmax = res.rawmax;
            pr.tag = res.failed ? ~p.epoch : p.epoch;
            p.pres[(int64_t)b * p.P + piece] = pr;
            __threadfence();
            s_last = atomicAdd(p.sync + (size_t)b * kSyncWords + kSyncDone, 1u) == (uint32_t)(p.P - 1);
        }
        __syncthreads();
        writer = s_last != 0;
        if (!writer) return;
        __threadfence();
        SliceRes o;
        o.best = kNegInf;
        o.idx = -1;
        o.rawmax = kNegInf;
        o.failed = 0;
        for (int q = tid; q < p.P; q += kJobThreads) {
            const uint4 w4 = __ldcg((const uint4 *)(p.pres + (int64_t)b * p.P + q));
            if (better(__uint_as_float(w4.x), (int)w4.y, o.best, o.idx)) {
                o.best = __uint_as_float(w4.x);
                o.idx = (int)w4.y;
            }
            o.rawmax = max_nan_f32(o.rawmax, __uint_as_float(w4.z));
            o.failed |= w4.w != p.epoch;
        }
        o = block_reduce_n(o, s_red, kJobWarps);
        if (status == SPEC_STATUS_OK) {
            if (o.failed) status = SPEC_STATUS_INTERNAL;
            else if (jd.kind != JOB_RESID && !(fabsf(o.rawmax) < __int_as_float(0x7f800000)))
                status = SPEC_STATUS_NONFINITE;
        }
        token = o.idx;
        if (status == SPEC_STATUS_OK && jd.kind == JOB_RESID && o.idx < 0) {
            // p <= q everywhere (only by rounding): draw from p_j with the same noise
            const int64_t trow = (rbase.t0 + jd.row) * p.ld_row;
            SliceRes f;
            f.best = kNegInf;
            f.idx = -1;
            f.rawmax = kNegInf;
            f.failed = 0;
            for (int v = tid; v < p.V; v += kJobThreads) {
                const float lp = fmaf(ld_elem<ESZ>(p.target, trow + v), jd.invT, -jd.shift);
                if (!(lp > kNegInf)) continue;
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)jd.row, PURPOSE_RESIDUAL,
                                            (uint32_t)v >> 2);
                const float sc = lp + gumbel_of_word(word_of(r4, v & 3));
                if (better(sc, v, f.best, f.idx)) { f.best = sc; f.idx = v; }
            }
            token = block_reduce_n(f, s_red, kJobWarps).idx;
        }
    }
    if (!writer) return;

    // ---- outputs of request b
    const bool okst = status == SPEC_STATUS_OK;
    const int A = okst ? jd.A : 0;
    int32_t *tok = p.out_tokens + rbase.t0;
    for (int i = tid; i < rbase.ntok; i += kJobThreads)
        tok[i] = !okst ? -1 : (i < A ? x[i] : (i == A ? token : -1));
    const bool pq = okst && !greedy;
    if (p.out_p)
        for (int i = tid; i < rbase.npq; i += kJobThreads) p.out_p[rbase.d0 + i] = pq && i < kb ? s_pp[i] : -1.f;
    if (p.out_q)
        for (int i = tid; i < rbase.npq; i += kJobThreads) p.out_q[rbase.d0 + i] = pq && i < kb ? s_qq[i] : -1.f;
    if (tid == 0) {
        p.out_status[b] = status;
        p.out_accepted[b] = A;
    }
}

// =================================================================== fused verify (large batches)
// For batches of at least one request per SM, one persistent kernel does the whole
// step: the main pass as main_kernel, then -- in the same CTAs, once the chunk
// tickets run out -- the commit work as items taken by tickets (commit_item).  With
// many requests each SM runs several items, so their dependent chains overlap, and
// the kernel boundary and the wait for the last main CTA go away; with few requests
// the piece layout of commit_kernel overlaps more of them, so the host picks by B.
namespace fused {

// Per-request words of the commit items, in the request's 128-byte line of the
// workspace (the line commit_kernel's pieces use), zeroed with the ticket counters
// before every launch.  Both are 64-bit and carry the call's tag in their high half
// as well, so a word of another call reads as empty.
constexpr int kSyncWords = 16;  // 64-bit words a request: the 128-byte line commit_kernel uses
constexpr int kSyncDone = 0;   // (tag, items of the request finished)
constexpr int kSyncBest = 1;   // (tag, ordered bits of the best exact score an item found)
// Ticket counters at the start of the workspace, zeroed in stream order before every
// launch (so a workspace left in any state by another call serves this one), and
// zero again when the kernel ends: the last CTA to leave resets them, since the
// two-kernel path expects its chunk counter (the same word) at zero.  Every chunk
// and every item is taken by ticket: a ticket is only ever held by a running CTA,
// which finishes its chunks before it waits for anything, so progress never depends
// on a CTA that is not resident.
constexpr int kCntChunk = 0;
constexpr int kCntItem = 1;
constexpr int kCntExit = 2;
constexpr int kSV = 2;             // commit items: vectors a thread holds per slice of a chunk
// a warp's live list: < 64 carried + one vector's groups (2 pieces of 4 entries per
// bf16 vector, each listing 2 groups when the window is not group-aligned)
constexpr int kItemLive = 64 + 32 * 2 * 2;
constexpr int kCandPrefetch = 1024;  // seed-candidate pointers an item fetches with the partials

struct VerifyParams {
    const void *target;
    const void *draft;
    int dtype;
    int64_t ld_row;
    int B, Kmax, V;
    const int32_t *draft_tokens;
    const int32_t *cu;         // flattened layout offsets [B+1], or NULL (padded)
    const int32_t *num_draft;
    const float *temperature;  // NULL: every request greedy
    uint64_t seed;
    uint32_t step;
    uint32_t epoch;            // tag of this call, stored with every partial
    int cpr, ce;               // chunks per row, entries per chunk
    int Q;                     // commit items per request (1 .. cpr)
    uint32_t *counters;        // [kCntChunk, kCntItem, kCntExit], zero at launch and at exit
    unsigned long long *sync;  // [B][kSyncWords]
    Part *parts;               // [chunks] one per chunk of every main-pass row
    uint16_t *cand;            // [chunks][kCW] sampling rows: the window vector holding each warp's
                               // maximum (0xffff: none), the correction's seed candidates
    PieceRes *pres;            // [B][Q] the commit items' results
    int32_t *out_tokens;
    int32_t *out_accepted;
    float *out_p;
    float *out_q;
    int32_t *out_status;
};

// The window of chunk k of a job row (a row the main pass may not have read).
__device__ __forceinline__ ChunkDesc job_chunk(const char *row, int esz, int V, const Chunking &ck, int k) {
    const ChunkWin w = chunk_window(row, esz, V, ck, k);
    ChunkDesc d;
    d.a0 = w.a0;
    d.bytes = w.bytes;
    d.e0 = w.e0;
    d.e1 = w.e1;
    d.shift = w.shift;
    d.c = 0.f;
    d.t = (uint32_t)k;
    d.req = 0;
    return d;
}

__device__ __forceinline__ unsigned long long ld_relaxed_u64(const unsigned long long *p) {
    unsigned long long v;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}

// The shared bound of a request: the best exact score published in this call, or
// -inf (a word of another call).
__device__ __forceinline__ float bound_of(unsigned long long w, uint32_t epoch) {
    return (uint32_t)(w >> 32) == epoch ? ordered_float((uint32_t)w) : kNegInf;
}
__device__ __forceinline__ void publish_bound(unsigned long long *w, uint32_t epoch, float s) {
    atomicMax(w, ((unsigned long long)epoch << 32) | ordered_bits(s));
}

// One thread: the request's arrival count, the word's own or a fresh one for this
// call; returns the items arrived, this one included.
__device__ __forceinline__ uint32_t arrive(unsigned long long *w, uint32_t epoch) {
    unsigned long long cur = ld_relaxed_u64(w);
    for (;;) {
        const unsigned long long nw =
            (uint32_t)(cur >> 32) == epoch ? cur + 1ull : (((unsigned long long)epoch << 32) | 1ull);
        const unsigned long long prev = atomicCAS(w, cur, nw);
        if (prev == cur) return (uint32_t)nw;
        cur = prev;
    }
}

// Whole CTA: wait until the n partials at pp all carry this call's tag (the CTAs
// that write them are running and wait for nothing, so they arrive; a 16-byte
// partial is written and read whole), keeping a copy in stage when n <= cap (the
// last round's copies all carry the tag); false after kWaitNs.
__device__ bool wait_parts(const Part *pp, int n, uint32_t epoch, int *flag, Part *stage, int cap) {
    uint64_t t0 = 0;
    unsigned ns = 64;
    const bool keep = n <= cap;
    for (int round = 0;; ++round) {
        bool miss = false;
        for (int i = threadIdx.x; i < n; i += blockDim.x) {
            const uint4 w = __ldcg((const uint4 *)(pp + i));
            miss |= w.w != epoch;
            if (keep) *(uint4 *)(stage + i) = w;
        }
        if (!__syncthreads_or(miss)) return true;
        if (threadIdx.x == 0) {
            const uint64_t now = global_ns();
            if (round == 0) t0 = now;
            *flag = now - t0 > kWaitNs;
        }
        __syncthreads();
        if (*flag) return false;
        __nanosleep(ns);
        if (ns < 1024) ns <<= 1;
    }
}

// One row's statistics from its cpr per-chunk partials, by one thread: from the
// shared-memory copy, or through L2 (other CTAs wrote them in this call).  stale:
// some partial carries another call's tag.
template <bool STAGED>
__device__ __forceinline__ RowRes row_from_parts_tagged(const Part *pp, int cpr, float c, bool greedy, uint32_t epoch,
                                                 bool &stale) {
    float M = kNegInf;
    for (int q = 0; q < cpr; ++q) {
        const uint4 w = STAGED ? *(const uint4 *)(pp + q) : __ldcg((const uint4 *)(pp + q));
        stale |= w.w != epoch;
        M = max_nan_f32(M, __uint_as_float(w.x));
    }
    const float MC = __fmul_rn(M, c);
    float sum = 0.f;
    int bi = -1;
    for (int q = 0; q < cpr; ++q) {
        const uint4 w = STAGED ? *(const uint4 *)(pp + q) : __ldcg((const uint4 *)(pp + q));
        const float m = __uint_as_float(w.x), s = __uint_as_float(w.y);
        const int idx = (int)w.z;
        if (!greedy && m != kNegInf && s != 0.f) sum += s * exp2f(__fmul_rn(m, c) - MC);
        if (greedy && m == M && idx >= 0 && (bi < 0 || idx < bi)) bi = idx;
    }
    RowRes r;
    r.M = M;
    r.idx = bi;
    r.l2S = greedy ? 0.f : log2f(sum);
    return r;
}

// ------------------------------------------------------------------ commit items
// Item (b, q) of the Q items of request b:
//  1. waits until every chunk partial of b's rows carries this call's tag;
//  2. decides the request -- the same arithmetic on the same partials in every item,
//     so all of them agree: row statistics, p(x_i) and q(x_i), the acceptance scan,
//     and the one row still needed (the first rejected target row j for the
//     correction, row k_b for the bonus draw or, greedy, for the argmax when every
//     draft matched);
//  3. streams chunks q, q + Q, ... of that row into registers, as the main pass
//     does, and reduces them: the pruned Gumbel-max, or the argmax;
//  4. stores its result and bumps the request's counter; the item that completes
//     the count combines the Q results and writes the request's outputs.
// The pruned Gumbel-max is exact.  An entry can beat the bound thr -- always the
// exact score of some entry, or -inf -- only if z + kGumbelMax >= thr (no word gives
// more than 16.64 of noise) and 1 - u <= 1.001 e^(z - thr) (g >= thr - z needs
// -log u <= e^(z - thr), and -log u >= 1 - u).  Each warp lists the groups of four
// whose largest z passes the first test, and every 64 listed groups draws their
// Philox blocks, two groups per lane; only entries passing the second test are
// scored exactly.

struct ItemShared {
    SliceRes red[kCW];
    JobDesc job;
    ReqBase rb;  // the request's layout, kept here through the draw (fewer live registers)
    int kb;
    int greedy;
    int flag;
    int last;
};

__host__ __device__ inline size_t align16(size_t x) { return (x + 15) & ~(size_t)15; }

// Lists the live groups of this thread's vector t of a job chunk in the warp's list
// (a group is live when its largest z = x invT - shift is finite and at least tz);
// returns the new length.  CHECK_RAW folds every raw value into rawmax (rows the
// main pass did not read).  mis: the window is not group-aligned, so each 4-entry
// piece of the vector lists both groups it overlaps, with the piece's max as their
// bound (a group may be listed twice: harmless).
template <bool CHECK_RAW, class Vec>
__device__ __forceinline__ int item_filter(const Vec &d, int t, int ebase, bool mis, float tz, float invT,
                                           float shift, float &rawmax, uint32_t *lg, float *lz, int nlive) {
    constexpr int NG = Vec::VE / 4;  // 4-entry pieces per vector
    const int lane = threadIdx.x & 31;
    const unsigned lt = (1u << lane) - 1u;
    const int per = mis ? 2 : 1;
    const int v0 = ebase + ((int)threadIdx.x + kCT * t) * Vec::VE;
    if (CHECK_RAW) rawmax = max_nan_f32(rawmax, d.vmax());
#pragma unroll
    for (int m = 0; m < NG; ++m) {
        const float z = fmaf(d.gmax(m), invT, -shift);
        const bool live = z > kNegInf && z >= tz;
        const unsigned bal = __ballot_sync(0xffffffffu, live);
        if (live) {
            const int pos = nlive + __popc(bal & lt) * per;
            const int g = (v0 + 4 * m) >> 2;  // floor: v0 + 4m may be -4 .. -1 at a row start
            lg[pos] = (uint32_t)g;
            lz[pos] = z;
            if (mis) {
                lg[pos + 1] = (uint32_t)(g + 1);
                lz[pos + 1] = z;
            }
        }
        nlive += __popc(bal) * per;
    }
    __syncwarp();
    return nlive;
}

// Draws the listed groups [base, base + n), n <= 64, two per lane, and updates thr
// to the warp's best afterwards.  Entries outside [0, V) are skipped.
template <int ESZ>
__device__ __forceinline__ void item_round(const uint32_t *lg, const float *lz, int base, int n,
                                           const JobDesc &jd, const char *jrow, const char *drow,
                                           const VerifyParams &p, uint32_t b, float &thr, float &best, int &bidx) {
    const int lane = threadIdx.x & 31;
    const bool resid = jd.kind == JOB_RESID;
    const uint32_t purpose = resid ? PURPOSE_RESIDUAL : PURPOSE_BONUS;
    int gk[2];
    float zm[2];
    bool has[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        const int item = lane + 32 * h;
        has[h] = item < n;
        const int e = base + (has[h] ? item : 0);
        gk[h] = (int)lg[e];
        zm[h] = lz[e];
    }
    uint4 r4[2];
#pragma unroll
    for (int h = 0; h < 2; ++h) r4[h] = rand_group(p.seed, p.step, b, (uint32_t)jd.row, purpose, (uint32_t)gk[h]);
    uint32_t sv = 0;  // bit 4h + q: entry q of group h passed the per-entry test
#pragma unroll
    for (int h = 0; h < 2; ++h) {
        // any survivor needs 1 - u_k <= e^(z_k - thr) <= e^(zmax - thr); the largest
        // w >> 9 of the group gives the smallest 1 - u
        const uint32_t kmax = max(max(r4[h].x >> 9, r4[h].y >> 9), max(r4[h].z >> 9, r4[h].w >> 9));
        if (has[h] && one_minus_u01(kmax << 9) <= ex2_approx((zm[h] - thr) * kLog2e) * 1.001f) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int v = 4 * gk[h] + q;
                if (v < 0 || v >= p.V) continue;
                const float z = fmaf(ld_elem<ESZ>(jrow, v), jd.invT, -jd.shift);
                if (z > kNegInf && one_minus_u01(word_of(r4[h], q)) <= ex2_approx((z - thr) * kLog2e) * 1.001f)
                    sv |= 1u << (4 * h + q);
            }
        }
    }
    // exact scores of the survivors, one entry at a time (rare: few registers)
    while (sv) {
        const int k = __ffs(sv) - 1;
        sv &= sv - 1;
        const int h = k >> 2, q = k & 3;
        const int v = 4 * (h ? gk[1] : gk[0]) + q;
        const uint32_t wd = word_of(h ? r4[1] : r4[0], q);
        const float z = fmaf(ld_elem<ESZ>(jrow, v), jd.invT, -jd.shift);
        float sc;
        if (resid) {
            // -inf (no residual mass at v) is never a candidate: a row without any
            // must reach the degenerate fallback
            const float zq = fmaf(ld_elem<ESZ>(drow, v), jd.invT, -jd.Cd);
            sc = zq < z ? resid_score(z, zq, wd) : kNegInf;
        } else {
            sc = z + gumbel_of_word(wd);
        }
        if (sc > kNegInf && better(sc, v, best, bidx)) { best = sc; bidx = v; }
    }
    thr = fmaxf(thr, warp_max(best));
    __syncwarp();  // the items drawn here are overwritten by the next appends
}

// One slice of a Gumbel-max job: share the bound with the request's other items
// (each publishes the best exact score it knows and reads theirs one slice ahead of
// using it; every published value is the exact score of an entry, so the pruning
// stays exact), list the live groups, draw every full 64.
template <bool CHECK_RAW, class Vec>
__device__ __forceinline__ void item_slice(const Vec (&d)[kSV], int t0, int ebase, const JobDesc &jd,
                                           const char *jrow, const char *drow, const VerifyParams &p, uint32_t b,
                                           unsigned long long *sy, unsigned long long &shared_bits,
                                           float &published, float &thr,
                                           SliceRes &mine, uint32_t *lg, float *lz, int &nlive) {
    const int lane = threadIdx.x & 31;
    thr = fmaxf(thr, bound_of(shared_bits, p.epoch));
    shared_bits = ld_relaxed_u64(sy + kSyncBest);
    if (lane == 0 && thr > published) {
        publish_bound(sy + kSyncBest, p.epoch, thr);
        published = thr;
    }
#pragma unroll
    for (int t = 0; t < kSV; ++t) {
        nlive = item_filter<CHECK_RAW>(d[t], t0 + t, ebase, (ebase & 3) != 0, thr - kGumbelMax, jd.invT, jd.shift,
                                       mine.rawmax, lg, lz, nlive);
        while (nlive >= 64) {  // draw the newest 64; the rest stay listed
            nlive -= 64;
            item_round<Vec::ESIZE>(lg, lz, nlive, 64, jd, jrow, drow, p, b, thr, mine.best, mine.idx);
        }
    }
}

// One slice of an argmax job: the lowest index of the largest value, every raw
// value folded into rawmax.  Entry e of vector t of thread ct is element
// ebase + (ct + kCT (t0 + t)) VE + e.
template <class Vec>
__device__ __forceinline__ void item_argmax_slice(const Vec (&d)[kSV], int t0, int ebase, SliceRes &mine) {
    float vm[kSV];
    float tm = kNegInf;
#pragma unroll
    for (int t = 0; t < kSV; ++t) {
        vm[t] = d[t].vmax();
        tm = max_nan_f32(tm, vm[t]);
    }
    const float M = warp_max_nan(tm);
    mine.rawmax = max_nan_f32(mine.rawmax, M);
    if (!(M > kNegInf)) return;  // all -inf (or NaN): no argmax here
#pragma unroll
    for (int t = 0; t < kSV; ++t) {
        const unsigned bal = __ballot_sync(0xffffffffu, vm[t] == M);
        if (bal) {
            int e = Vec::VE;
#pragma unroll
            for (int q = Vec::VE - 1; q >= 0; --q)
                if (d[t].get(q) == M) e = q;
            const int mine_idx = ebase + ((int)threadIdx.x + kCT * (t0 + t)) * Vec::VE + e;
            const int idx = __shfl_sync(0xffffffffu, mine_idx, __ffs(bal) - 1);
            if (better(M, idx, mine.best, mine.idx)) {
                mine.best = M;
                mine.idx = idx;
            }
            return;
        }
    }
}

// Loads this thread's vectors t0 .. t0+kSV-1 of a chunk (vector t of thread ct is
// window vector ct + kCT t); entries outside the chunk read as -inf.
template <class Vec>
__device__ __forceinline__ void load_slice(Vec (&d)[kSV], const ChunkDesc &cd, int t0, int ct) {
    const int nvec = (int)(cd.bytes >> 4);
    const int64_t ebase = (int64_t)cd.e0 - cd.shift;
#pragma unroll
    for (int t = 0; t < kSV; ++t) {
        const int j = ct + kCT * (t0 + t);
        d[t] = j < nvec ? Vec::load(cd.a0, j) : Vec::neg_inf();
        if (j < nvec && (j == 0 || j == nvec - 1)) mask_vec(d[t], ebase + (int64_t)j * Vec::VE, cd.e0, cd.e1);
    }
}

template <class Vec>
__device__ __forceinline__ void commit_item(const VerifyParams &p, const int *s_rs, int item, ItemShared &sh) {
    // the item's buffers, sized for the largest Kmax (fixed addresses: no registers)
    // live groups and their largest z (the draw), or the request's partials (the decide)
    __shared__ __align__(16) unsigned char s_buf[kCW * kItemLive * 8];
    constexpr int kStageParts = kCW * kItemLive * 8 / (int)sizeof(Part);
    __shared__ PosRes s_pos[SPEC_MAX_DRAFTS];
    __shared__ RowRes s_rows[2 * SPEC_MAX_DRAFTS];  // target rows, then draft rows
    __shared__ float s_xt[SPEC_MAX_DRAFTS], s_xd[SPEC_MAX_DRAFTS];  // target and draft logit at x_i
    __shared__ float s_l2u[SPEC_MAX_DRAFTS];   // log2 of the acceptance uniform u_i
    __shared__ float s_pp[SPEC_MAX_DRAFTS], s_qq[SPEC_MAX_DRAFTS];  // p(x_i), q(x_i)
    __shared__ uint16_t s_cand[kCandPrefetch];  // seed-candidate pointers of the target rows
    constexpr int ESZ = Vec::ESIZE;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = item / p.Q, q = item - b * p.Q;
    unsigned long long *sy = p.sync + (size_t)b * kSyncWords;

    // ---- the request's inputs
    const ReqBase rbase = req_base(p.cu, p.num_draft, p.Kmax, b);
    const int kb_raw = rbase.kb;
    int status = SPEC_STATUS_OK;
    float T = 0.f;
    if (kb_raw < 0 || kb_raw > p.Kmax) status = SPEC_STATUS_BAD_K;
    if (status == SPEC_STATUS_OK && p.temperature) {
        T = p.temperature[b];
        if (!(T >= 0.f) || isinf(T)) status = SPEC_STATUS_BAD_TEMPERATURE;
    }
    const int kb = status == SPEC_STATUS_BAD_K ? 0 : kb_raw;
    const bool greedy = (T == 0.f);
    const int32_t *x = p.draft_tokens + rbase.d0;
    if (status == SPEC_STATUS_OK) {
        bool bad = false;
        for (int i = tid; i < kb; i += kCT) bad |= (x[i] < 0 || x[i] >= p.V);
        if (__syncthreads_or(bad)) status = SPEC_STATUS_BAD_TOKEN;
    }
    const float c = greedy ? 0.f : __fdiv_rn(kLog2e, T);
    const float invT = greedy ? 0.f : __fdiv_rn(1.f, T);
    const int npos = status == SPEC_STATUS_OK ? kb : 0;
    if (!greedy) {
        for (int i = tid; i < npos; i += kCT) {
            const int xi = x[i];
            s_xt[i] = load_logit(p.target, p.dtype, (rbase.t0 + i) * p.ld_row + xi);
            s_xd[i] = load_logit(p.draft, p.dtype, (rbase.d0 + i) * p.ld_row + xi);
            const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)i, PURPOSE_ACCEPT, 0u);
            s_l2u[i] = log2f(u01(r4.x));
        }
    }
    // ---- wait until the main pass has stored every partial of the request's rows
    const int r0 = s_rs[b];
    const int nparts = (s_rs[b + 1] - r0) * p.cpr;
    Part *stage = (Part *)s_buf;
    const bool counted = wait_parts(p.parts + (int64_t)r0 * p.cpr, nparts, p.epoch, &sh.flag, stage, kStageParts);
    const bool staged = nparts <= kStageParts;
    const int nrows = greedy ? npos : 2 * npos;  // flat rows r0 .. r0 + nrows - 1
    const int ncand = p.cpr * kCW;
    const bool cand_pre = !greedy && counted && npos * ncand <= kCandPrefetch;
    if (cand_pre)
        for (int it = tid; it < npos * ncand; it += kCT) s_cand[it] = __ldcg(p.cand + (size_t)r0 * ncand + it);

    // ---- the decision: one thread per row, then one thread per position
    bool stale = false;
    if (counted)
        for (int r = tid; r < nrows; r += kCT)
            s_rows[r] = staged ? row_from_parts_tagged<true>(stage + (int64_t)r * p.cpr, p.cpr, c, greedy && r < npos,
                                                      p.epoch, stale)
                               : row_from_parts_tagged<false>(p.parts + (int64_t)(r0 + r) * p.cpr, p.cpr, c,
                                                       greedy && r < npos, p.epoch, stale);
    stale = __syncthreads_or(stale);
    if (counted) {
        for (int i = tid; i < npos; i += kCT) {
            const RowRes tr = s_rows[i];
            PosRes pr;
            pr.tidx = tr.idx;
            pr.shift = pr.Cd = 0.f;
            pr.seed = kNegInf;
            pr.seed_idx = -1;
            pr.pad = 0.f;
            if (greedy) {
                pr.nonfinite = !(fabsf(tr.M) < __int_as_float(0x7f800000));
                pr.rej = tr.idx != x[i];
            } else {
                const RowRes dr = s_rows[npos + i];
                // a NaN leaves its chunk's max NaN; +inf makes the sum NaN: both show here
                pr.nonfinite = !(fabsf(tr.M) < __int_as_float(0x7f800000) &&
                                 fabsf(dr.M) < __int_as_float(0x7f800000) &&
                                 fabsf(tr.l2S) < __int_as_float(0x7f800000) &&
                                 fabsf(dr.l2S) < __int_as_float(0x7f800000));
                const float l2p = fmaf(s_xt[i], c, -__fmul_rn(tr.M, c)) - tr.l2S;  // log2 p_i(x_i)
                const float l2q = fmaf(s_xd[i], c, -__fmul_rn(dr.M, c)) - dr.l2S;  // log2 q_i(x_i)
                // accept iff u q < p, i.e. log2 u < log2 p - log2 q (Q = 0 < P accepts; P = 0 rejects)
                pr.rej = !(s_l2u[i] < l2p - l2q);
                // log p_v = x_v / T - (fl(M c) + log2 S) ln 2, and q likewise
                pr.shift = (__fmul_rn(tr.M, c) + tr.l2S) * 0.6931471805599453f;
                pr.Cd = (__fmul_rn(dr.M, c) + dr.l2S) * 0.6931471805599453f;
                s_pp[i] = exp2f(l2p);
                s_qq[i] = exp2f(l2q);
            }
            s_pos[i] = pr;
        }
    }
    __syncthreads();

    // ---- the scan (warp 0): A = first rejected position, and the job
    if (warp == 0) {
        JobDesc jd;
        jd.kind = JOB_NONE;
        jd.row = 0;
        jd.A = 0;
        jd.token = -1;
        jd.invT = invT;
        jd.shift = jd.Cd = 0.f;
        jd.seed = kNegInf;
        jd.seed_idx = -1;
        jd.epoch = p.epoch;
        int st = status;
        if (st == SPEC_STATUS_OK && (!counted || stale)) st = SPEC_STATUS_INTERNAL;
        if (st == SPEC_STATUS_OK) {
            bool nf = false;
            for (int i = lane; i < kb; i += 32) nf |= s_pos[i].nonfinite != 0;
            if (__any_sync(0xffffffffu, nf)) st = SPEC_STATUS_NONFINITE;
        }
        if (st == SPEC_STATUS_OK) {
            int A = kb;
            for (int i0 = 0; i0 < kb && A == kb; i0 += 32) {
                const int i = i0 + lane;
                const unsigned msk = __ballot_sync(0xffffffffu, i < kb && s_pos[i].rej != 0);
                if (msk) A = i0 + __ffs(msk) - 1;
            }
            jd.A = A;
            if (greedy) {
                if (A < kb) {
                    jd.token = s_pos[A].tidx;
                } else {
                    jd.kind = JOB_ARGMAX;
                    jd.row = kb;
                }
            } else if (A < kb) {
                const PosRes pr = s_pos[A];
                jd.kind = JOB_RESID;
                jd.row = A;
                jd.shift = pr.shift;
                jd.Cd = pr.Cd;
            } else {
                jd.kind = JOB_BONUS;
                jd.row = kb;
            }
        }
        jd.status = st;
        if (lane == 0) sh.job = jd;
    }
    if (tid == 0) {
        sh.rb = rbase;
        sh.kb = kb;
        sh.greedy = greedy;
    }
    __syncthreads();
    const JobDesc &jd = sh.job;  // read where used: fewer live registers
    status = jd.status;

    int token = jd.token;
    if (jd.kind != JOB_NONE) {
        const int64_t rowbytes = p.ld_row * ESZ;
        const char *jrow = (const char *)p.target + (sh.rb.t0 + jd.row) * rowbytes;
        const char *drow = jd.kind == JOB_RESID ? (const char *)p.draft + (sh.rb.d0 + jd.row) * rowbytes : nullptr;
        const Chunking ck = {p.cpr, p.ce};
        // the first slice's loads go out before the seeds are scored
        constexpr int kSlices = kVPT / kSV;  // a chunk is kSlices slices of kSV vectors a thread
        Vec cur[kSV], nxt[kSV];
        int k = q, sl = 0, eb_cur = 0;
        if (k < p.cpr) {
            const ChunkDesc cd = job_chunk(jrow, ESZ, p.V, ck, k);
            eb_cur = cd.e0 - cd.shift;
            load_slice(cur, cd, 0, tid);
        }
        SliceRes mine;
        mine.best = kNegInf;
        mine.idx = -1;
        mine.rawmax = kNegInf;
        mine.failed = 0;
        float thr = kNegInf;
        if (jd.kind == JOB_RESID) {
            // seeds: the main pass's candidates of row A (the vector holding each
            // warp's maximum of each chunk), exact scores; the best is shared
            constexpr int VE = 16 / ESZ;
            SliceRes sd;
            sd.best = kNegInf;
            sd.idx = -1;
            sd.rawmax = kNegInf;
            sd.failed = 0;
            for (int j = tid; j < ncand; j += kCT) {
                const uint32_t cv = cand_pre ? s_cand[jd.row * ncand + j]
                                             : __ldcg(p.cand + ((size_t)r0 + jd.row) * ncand + j);
                const ChunkWin w = chunk_window(jrow, ESZ, p.V, ck, j / kCW);
                if (cv == 0xffffu || (cv + 1) * 16 > w.bytes) continue;
                const int eb = w.e0 - w.shift + (int)cv * VE;
                // the target vector and the draft logits of its entries, loaded together
                const uint4 raw = ld_stream_v4(w.a0 + 16 * (size_t)cv);
                float lq[VE];
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                    const int v = eb + e;
                    lq[e] = (v >= w.e0 && v < w.e1) ? ld_elem<ESZ>(drow, v) : 0.f;
                }
                float bx = kNegInf, bq = 0.f;
                int bvi = -1;
#pragma unroll
                for (int e = 0; e < VE; ++e) {
                    const int v = eb + e;
                    const float xv = ESZ == 2 ? VecBF16{raw}.get(e) : VecF32{raw}.get(e);
                    if (v >= w.e0 && v < w.e1 && xv > bx) { bx = xv; bvi = v; bq = lq[e]; }
                }
                if (bvi < 0) continue;
                const float z = fmaf(bx, jd.invT, -jd.shift);
                const float zq = fmaf(bq, jd.invT, -jd.Cd);
                if (!(zq < z)) continue;  // no residual mass at bvi
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)jd.row, PURPOSE_RESIDUAL,
                                            (uint32_t)bvi >> 2);
                const float s = resid_score(z, zq, word_of(r4, bvi & 3));
                if (better(s, bvi, sd.best, sd.idx)) { sd.best = s; sd.idx = bvi; }
            }
            sd = block_reduce_n(sd, sh.red, kCW);
            mine.best = sd.best;
            mine.idx = sd.idx;
            thr = sd.best;
            if (tid == 0 && sd.best > kNegInf) publish_bound(sy + kSyncBest, p.epoch, sd.best);
        }
        uint32_t *lg = (uint32_t *)s_buf + warp * kItemLive;
        float *lz = (float *)(s_buf + kCW * kItemLive * 4) + warp * kItemLive;
        int nlive = 0;
        float published = thr;
        unsigned long long shared_bits = ld_relaxed_u64(sy + kSyncBest);
        bool first = true;
        while (k < p.cpr) {
            // the next slice: the rest of this chunk, then chunk k + Q
            int k2 = k, sl2 = sl + 1;
            if (sl2 == kSlices) {
                sl2 = 0;
                k2 = k + p.Q;
            }
            const bool more = k2 < p.cpr;
            int eb_next = eb_cur;
            if (more) {
                const ChunkDesc nd = job_chunk(jrow, ESZ, p.V, ck, k2);
                eb_next = nd.e0 - nd.shift;
                load_slice(nxt, nd, sl2 * kSV, tid);
            }
            if (jd.kind == JOB_ARGMAX) {
                item_argmax_slice(cur, sl * kSV, eb_cur, mine);
            } else {
                if (jd.kind == JOB_BONUS && first) {
                    // bonus seed: the exact score of each lane's largest entry of the
                    // first slice; the warp's best bounds its draws from below
                    float m = kNegInf;
                    int mi = -1;
#pragma unroll
                    for (int t = 0; t < kSV; ++t)
#pragma unroll
                        for (int e = 0; e < Vec::VE; ++e) {
                            const float xv = cur[t].get(e);
                            if (xv > m) { m = xv; mi = eb_cur + (tid + kCT * t) * Vec::VE + e; }
                        }
                    if (mi >= 0) {
                        const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)jd.row, PURPOSE_BONUS,
                                                    (uint32_t)mi >> 2);
                        const float s = fmaf(m, jd.invT, -jd.shift) + gumbel_of_word(word_of(r4, mi & 3));
                        if (better(s, mi, mine.best, mine.idx)) { mine.best = s; mine.idx = mi; }
                    }
                    thr = warp_max(mine.best);
                }
                first = false;
                if (jd.kind == JOB_RESID)
                    item_slice<false>(cur, sl * kSV, eb_cur, jd, jrow, drow, p, (uint32_t)b, sy, shared_bits,
                                      published, thr, mine, lg, lz, nlive);
                else
                    item_slice<true>(cur, sl * kSV, eb_cur, jd, jrow, drow, p, (uint32_t)b, sy, shared_bits,
                                     published, thr, mine, lg, lz, nlive);
            }
#pragma unroll
            for (int t = 0; t < kSV; ++t) cur[t] = nxt[t];
            k = k2;
            sl = sl2;
            eb_cur = eb_next;
        }
        if (jd.kind != JOB_ARGMAX && nlive > 0)
            item_round<ESZ>(lg, lz, 0, nlive, jd, jrow, drow, p, (uint32_t)b, thr, mine.best, mine.idx);
        const SliceRes res = block_reduce_n(mine, sh.red, kCW);

        // ---- the items meet: the last to finish combines them
        if (tid == 0) {
            PieceRes pr;
            pr.best = res.best;
            pr.idx = res.idx;
            pr.rawmax = res.rawmax;
            pr.tag = p.epoch;
            p.pres[(int64_t)b * p.Q + q] = pr;
            __threadfence();
            sh.last = arrive(sy + kSyncDone, p.epoch) == (uint32_t)p.Q;
        }
        __syncthreads();
        if (!sh.last) return;
        __threadfence();
        SliceRes o;
        o.best = kNegInf;
        o.idx = -1;
        o.rawmax = kNegInf;
        o.failed = 0;
        for (int i = tid; i < p.Q; i += kCT) {
            const uint4 w4 = __ldcg((const uint4 *)(p.pres + (int64_t)b * p.Q + i));
            if (better(__uint_as_float(w4.x), (int)w4.y, o.best, o.idx)) {
                o.best = __uint_as_float(w4.x);
                o.idx = (int)w4.y;
            }
            o.rawmax = max_nan_f32(o.rawmax, __uint_as_float(w4.z));
            o.failed |= w4.w != p.epoch;
        }
        o = block_reduce_n(o, sh.red, kCW);
        if (status == SPEC_STATUS_OK) {
            if (o.failed) status = SPEC_STATUS_INTERNAL;
            else if (jd.kind != JOB_RESID && !(fabsf(o.rawmax) < __int_as_float(0x7f800000)))
                status = SPEC_STATUS_NONFINITE;
        }
        token = o.idx;
        if (status == SPEC_STATUS_OK && jd.kind == JOB_RESID && o.idx < 0) {
            // p <= q everywhere (only by rounding): draw from p_j with the same noise
            const int64_t trow = (sh.rb.t0 + jd.row) * p.ld_row;
            SliceRes f;
            f.best = kNegInf;
            f.idx = -1;
            f.rawmax = kNegInf;
            f.failed = 0;
            for (int v = tid; v < p.V; v += kCT) {
                const float lp = fmaf(load_logit(p.target, p.dtype, trow + v), jd.invT, -jd.shift);
                if (!(lp > kNegInf)) continue;
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)jd.row, PURPOSE_RESIDUAL,
                                            (uint32_t)v >> 2);
                const float s = lp + gumbel_of_word(word_of(r4, v & 3));
                if (better(s, v, f.best, f.idx)) { f.best = s; f.idx = v; }
            }
            token = block_reduce_n(f, sh.red, kCW).idx;
        }
    } else {
        // no row left to reduce: the items only meet
        if (tid == 0) {
            __threadfence();
            sh.last = arrive(sy + kSyncDone, p.epoch) == (uint32_t)p.Q;
        }
        __syncthreads();
        if (!sh.last) return;
    }

    // ---- outputs of request b (the last item)
    const ReqBase ob = sh.rb;
    const int okb = sh.kb;
    const int32_t *ox = p.draft_tokens + ob.d0;
    const bool okst = status == SPEC_STATUS_OK;
    const int A = okst ? jd.A : 0;
    int32_t *tok = p.out_tokens + ob.t0;
    for (int i = tid; i < ob.ntok; i += kCT) tok[i] = !okst ? -1 : (i < A ? ox[i] : (i == A ? token : -1));
    const bool pq = okst && !sh.greedy;
    if (p.out_p)
        for (int i = tid; i < ob.npq; i += kCT) p.out_p[ob.d0 + i] = pq && i < okb ? s_pp[i] : -1.f;
    if (p.out_q)
        for (int i = tid; i < ob.npq; i += kCT) p.out_q[ob.d0 + i] = pq && i < okb ? s_qq[i] : -1.f;
    if (tid == 0) {
        p.out_status[b] = status;
        p.out_accepted[b] = A;
    }
}

// One persistent kernel, kMainBlocksPerSM CTAs of kCT threads per SM.
//  Main pass: every row of every draft position read once -- target and draft rows
//  of sampling requests, target rows of greedy ones -- in chunks of at most 64 KB
//  taken by tickets.  A CTA keeps a chunk's kVPT 16-byte vectors per thread
//  in two halves and reloads a half with the next chunk's as soon as it has reduced
//  it, so its loads never stop for the reductions, the barrier and the CTA-level
//  combine that end each chunk.  Per chunk: warp maxima and exp-sums (greedy rows:
//  warp maxima and their lowest indices), combined by warp 0 into one Part stored at
//  the chunk's index; on sampling rows each warp also leaves a pointer to the vector
//  holding its maximum, the correction draw's seed candidates.
//  Commit: when the chunk tickets run out, the CTA takes commit items by tickets
//  until none are left (commit_item).
template <class Vec>
__global__ void __launch_bounds__(kCT, kMainBlocksPerSM) verify_kernel(VerifyParams p) {
    constexpr int kH = kVPT / 2;  // vectors per half
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ WarpStat s_ws[2][kCW];
    __shared__ ChunkDesc s_desc[3];
    __shared__ uint32_t s_item[2];
    __shared__ ItemShared s_sh;
    int *s_rs = (int *)smem;  // [B+1] first main-pass row of each request
    float *s_c = (float *)(smem + align16(sizeof(int) * (size_t)(p.B + 1)));  // [B] log2(e) / T (0: greedy)
    scan_request_rows(s_rs, p.B, p.cu, p.num_draft, p.temperature, p.Kmax);  // ends with __syncthreads
    for (int i = threadIdx.x; i < p.B; i += blockDim.x) {
        const float T = p.temperature ? p.temperature[i] : 0.f;
        s_c[i] = (T > 0.f && !isinf(T)) ? __fdiv_rn(kLog2e, T) : 0.f;
    }
    __syncthreads();

    const Chunking ck = {p.cpr, p.ce};
    const uint32_t total = (uint32_t)s_rs[p.B] * (uint32_t)ck.cpr;  // < 2^31 (checked by the host)
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, ct = threadIdx.x;
    if (threadIdx.x == 0) {
        const uint32_t t0 = atomicAdd(p.counters + kCntChunk, 2u);
        s_desc[0] = chunk_desc<Vec>(p, s_rs, s_c, ck, t0, total);
        s_desc[1] = chunk_desc<Vec>(p, s_rs, s_c, ck, t0 + 1u, total);
    }
    __syncthreads();
    // the current chunk's index, scale and first window element stay in registers;
    // the next chunk's window is read from shared memory where it is used
    uint32_t t = s_desc[0].t;
    float c = s_desc[0].c;
    int ebase = s_desc[0].e0 - s_desc[0].shift;
    Vec a[kH], bv[kH];
    if (t < total) {
        load_half<0>(a, s_desc[0], ct);
        load_half<kH>(bv, s_desc[0], ct);
    }
    int n = 0;
    while (t < total) {
        if (threadIdx.x == 0)
            s_desc[(n + 2) % 3] = chunk_desc<Vec>(p, s_rs, s_c, ck, atomicAdd(p.counters + kCntChunk, 1u), total);
        const ChunkDesc &nx = s_desc[(n + 1) % 3];
        float m = kNegInf, mc = 0.f, s = 0.f;
        int mv = -1;
        float vma[kH], vmb[kH];
        const float ta = half_stats<0>(a, vma, c, m, mc, s, mv);
        int ia = -1;
        float Ma = kNegInf;
        if (c == 0.f) {
            Ma = warp_max_nan(ta);
            ia = warp_first_index<0>(a, vma, Ma, ebase, ct);
        }
        if (nx.t < total) load_half<0>(a, nx, ct);
        const float tb = half_stats<kH>(bv, vmb, c, m, mc, s, mv);
        WarpStat ws;
        ws.pad = 0;
        if (c != 0.f) {
            // the lanes' sums, each relative to its own fl(m c), rescaled to the warp's
            const float M = warp_max_nan(m);
            const float sc = (m == kNegInf || s == 0.f) ? 0.f : s * ex2_approx(mc - __fmul_rn(M, c));
            ws.m = M;
            ws.s = warp_sum(sc);
            ws.idx = -1;
            // the window vector of the lowest lane that holds the warp maximum
            const unsigned own = __ballot_sync(0xffffffffu, m == M && mv >= 0);
            const int src = own ? __ffs(own) - 1 : 0;
            const int vec = __shfl_sync(0xffffffffu, mv, src);
            if (lane == 0)
                p.cand[(size_t)t * kCW + warp] = own ? (uint16_t)(warp * 32 + src + kCT * vec) : (uint16_t)0xffffu;
        } else {
            // entries of half a precede those of half b: a's index wins a tie
            const float Mb = warp_max_nan(tb);
            const int ib = warp_first_index<kH>(bv, vmb, Mb, ebase, ct);
            ws.m = max_nan_f32(Ma, Mb);
            ws.s = 0.f;
            ws.idx = (Ma >= Mb) ? ia : ib;
        }
        if (nx.t < total) load_half<kH>(bv, nx, ct);
        if (lane == 0) s_ws[n & 1][warp] = ws;
        __syncthreads();
        if (warp == 0) {
            // the CTA's warps combined: max, sum relative to fl(max c), lowest argmax
            const WarpStat q = lane < kCW ? s_ws[n & 1][lane] : WarpStat{kNegInf, 0.f, -1, 0};
            const float Mc = warp_max_nan(q.m);
            Part out;
            out.m = Mc;
            float tl = 0.f;
            if (c != 0.f) tl = (q.m == kNegInf || q.s == 0.f) ? 0.f : q.s * exp2f(__fmul_rn(q.m, c) - __fmul_rn(Mc, c));
            out.s = warp_sum(tl);
            uint32_t v = (q.m == Mc && q.idx >= 0) ? (uint32_t)q.idx : 0xffffffffu;
#pragma unroll
            for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
            out.idx = (int)v;
            out.epoch = p.epoch;
            if (lane == 0) p.parts[t] = out;  // one 16-byte store: the tag and the values arrive together
        }
        ++n;
        t = nx.t;
        c = nx.c;
        ebase = nx.e0 - nx.shift;
    }

    // ---- commit items
    const uint32_t nitems = (uint32_t)p.B * (uint32_t)p.Q;
    for (int it = 0;; ++it) {
        if (threadIdx.x == 0) s_item[it & 1] = atomicAdd(p.counters + kCntItem, 1u);
        __syncthreads();
        const uint32_t item = s_item[it & 1];
        if (item >= nitems) break;
        commit_item<Vec>(p, s_rs, (int)item, s_sh);
    }
    // the last CTA to leave: every ticket of this call is taken
    if (threadIdx.x == 0 && atomicAdd(p.counters + kCntExit, 1u) == gridDim.x - 1) {
        p.counters[kCntChunk] = 0u;
        p.counters[kCntItem] = 0u;
        p.counters[kCntExit] = 0u;
    }
}


}  // namespace fused

// =================================================================== early_exit_kernel
// Early-exit verify ("Accelerating Large-Model Inference ... DSpark", Sec. 1: the
// longest accepted prefix is committed plus one token, so no row after the first
// rejected position is needed; "From draft-then-verify to DSpark": the rejection
// test at each position in order).  One cluster of C CTAs per request walks the
// draft positions in order.  At position i every CTA streams its share of target
// row i (and draft row i) with plain 16-byte loads and reduces it; the shares'
// statistics meet over DSMEM -- every CTA reads all of them, in rank order, so
// every CTA reaches the same decision -- and the walk stops at the first
// rejection (or greedy mismatch, or non-finite row).  The correction is then drawn
// over that row, or the bonus over row k_b, by the same staged Gumbel-max as
// commit_kernel.  No workspace and no global synchronisation: a request's rows
// after its first rejection are never read.
constexpr int kEEVecs = 8;  // 16-byte loads per thread per batch

struct __align__(16) EEPart {
    float mt;   // target share: raw max (NaN-propagating)
    float st;   // target share: sum 2^(x c - fl(mt c))
    int it;     // target share: lowest argmax
    float md;   // draft share: raw max
    float sd;   // draft share: sum 2^(y c - fl(md c))
    float seed; // best exact correction score among the share's warp argmaxes
    int seed_idx;
    int pad;
};

// This thread's vectors of a share window: vector j = j0 + tid + kCommitThreads t.
template <class Vec>
__device__ __forceinline__ void ee_load(Vec (&d)[kEEVecs], const ChunkWin &w, int j0) {
    const int nvec = (int)(w.bytes >> 4);
    const int ebase = w.e0 - w.shift;
#pragma unroll
    for (int t = 0; t < kEEVecs; ++t) {
        const int j = j0 + (int)threadIdx.x + kCommitThreads * t;
        d[t] = j < nvec ? Vec::load(w.a0, j) : Vec::neg_inf();
        if (j < nvec && (j == 0 || j == nvec - 1) && (w.shift != 0 || ebase + nvec * Vec::VE != w.e1))
            mask_vec(d[t], ebase + (int64_t)j * Vec::VE, w.e0, w.e1);
    }
}

// Per-thread running statistics of one share window (as main_kernel's lanes);
// kat: the batch where the thread's running max was last raised.
template <class Vec>
__device__ void ee_thread_stats(const ChunkWin &w, float c, float &m, float &mc, float &s, int &kat,
                                bool &nan_seen) {
    const int nvec = (int)(w.bytes >> 4);
    for (int j0 = 0; j0 < nvec; j0 += kCommitThreads * kEEVecs) {
        Vec d[kEEVecs];
        ee_load(d, w, j0);
        float tm = d[0].vmax();
#pragma unroll
        for (int t = 1; t < kEEVecs; ++t) tm = max_nan_f32(tm, d[t].vmax());
        if (c != 0.f) {
            if (raises_max(tm, m)) {
                const float mcn = __fmul_rn(tm, c);
                s = (m == kNegInf) ? 0.f : s * ex2_approx(mc - mcn);
                m = tm;
                mc = mcn;
                kat = j0;
            }
            if (m != kNegInf) {
                const float2 cc = make_float2(c, c), mm = make_float2(-mc, -mc);
                float2 acc = make_float2(0.f, 0.f);
#pragma unroll
                for (int t = 0; t < kEEVecs; ++t)
#pragma unroll
                    for (int e = 0; e < Vec::VE; e += 2) {
                        const float2 y = ffma2(make_float2(d[t].get(e), d[t].get(e + 1)), cc, mm);
                        acc = fadd2(acc, make_float2(ex2_approx(y.x), ex2_approx(y.y)));
                    }
                s += acc.x + acc.y;
            }
        } else {
            if (tm != tm) {
                nan_seen = true;
            } else if (tm > m) {
                m = tm;
                kat = j0;
            }
        }
    }
}

// Lowest index of the warp's maximum M over the share (the lanes holding it reload
// the batch where their max was raised, as main_kernel's flush does).
template <class Vec>
__device__ int ee_warp_index(const ChunkWin &w, int kat, float m, float M) {
    int idx = -1;
    if (kat >= 0 && m == M) {
        Vec d[kEEVecs];
        ee_load(d, w, kat);
        idx = chunk_find<kCommitThreads>(d, w.e0 - w.shift + kat * Vec::VE, (int)threadIdx.x, M);
    }
    uint32_t v = (uint32_t)idx;
#pragma unroll
    for (int o = 16; o; o >>= 1) v = min(v, __shfl_xor_sync(0xffffffffu, v, o));
    return (int)v;
}

// Block reduction of the threads' statistics of one row; every thread returns the
// CTA's (max, sum relative to fl(max c), lowest argmax).  wm / wi keep the warps'
// maxima and argmaxes (correction seed candidates).  c == 0: max and argmax only,
// with NaN propagated.
__device__ void ee_block_stats(float m, float mc, float s, int widx, bool nan_seen, float c, float *wm, int *wi,
                               float *ws, float &M, float &S, int &I) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    float Mw, Sw = 0.f;
    if (c != 0.f) {
        Mw = warp_max_nan(m);
        const float sc = (m == kNegInf || s == 0.f) ? 0.f : s * ex2_approx(mc - __fmul_rn(Mw, c));
        Sw = warp_sum(sc);
    } else {
        const bool any_nan = __any_sync(0xffffffffu, nan_seen);
        Mw = warp_max_nan(m);
        if (any_nan) Mw = __int_as_float(0x7fc00000);
    }
    __syncthreads();  // wm / wi / ws may still be read from the previous row
    if (lane == 0) {
        wm[warp] = Mw;
        wi[warp] = widx;
        ws[warp] = Sw;
    }
    __syncthreads();
    M = wm[0];
    for (int w = 1; w < kCommitWarps; ++w) M = max_nan_f32(M, wm[w]);
    S = 0.f;
    float ab = kNegInf;
    I = -1;
    for (int w = 0; w < kCommitWarps; ++w) {
        if (c != 0.f && wm[w] != kNegInf && ws[w] != 0.f) S += ws[w] * exp2f(__fmul_rn(wm[w], c) - __fmul_rn(M, c));
        if (better(wm[w], wi[w], ab, I)) { ab = wm[w]; I = wi[w]; }
    }
}

// Every CTA of the cluster writes its part to its own slot, then reads every
// CTA's slot (rank order) into all[]; every thread calls it, the whole cluster
// the same number of times.  Slots alternate by parity, so a slot is rewritten
// only after the next exchange's barrier, which every reader passes after
// reading.
__device__ __forceinline__ void ee_exchange(const EEPart &mine, EEPart *slot, EEPart *all, int C) {
    const int tid = threadIdx.x;
    if (tid == 0) *slot = mine;
    cluster_arrive();
    cluster_wait();
    if (tid < C) {
        const uint32_t local = smem_addr(slot);
        uint32_t remote;
        asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(local), "r"((uint32_t)tid));
        uint4 a, b2;
        asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(a.x), "=r"(a.y), "=r"(a.z), "=r"(a.w) : "r"(remote) : "memory");
        asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                     : "=r"(b2.x), "=r"(b2.y), "=r"(b2.z), "=r"(b2.w) : "r"(remote + 16) : "memory");
        EEPart q;
        q.mt = __uint_as_float(a.x);
        q.st = __uint_as_float(a.y);
        q.it = (int)a.z;
        q.md = __uint_as_float(a.w);
        q.sd = __uint_as_float(b2.x);
        q.seed = __uint_as_float(b2.y);
        q.seed_idx = (int)b2.z;
        q.pad = 0;
        all[tid] = q;
    }
    __syncthreads();
}

__host__ __device__ inline size_t ee_smem_bytes(int NS, int slot, int Kmax) {
    return commit_round_bytes(NS, slot) + 5 * sizeof(float) * (size_t)Kmax;
}

template <int ESZ>
__global__ void __launch_bounds__(kCommitThreads, kCommitBlocksPerSM) early_exit_kernel(CommitParams p) {
    using Vec = typename std::conditional<ESZ == 2, VecBF16, VecF32>::type;
    extern __shared__ __align__(128) unsigned char cdyn[];
    __shared__ uint64_t s_bar;
    __shared__ uint32_t s_live_g[kCommitWarps][kLiveMax];
    __shared__ float s_live_z[kCommitWarps][kLiveMax];
    __shared__ SliceRes s_red[kCommitWarps];
    __shared__ SliceRes s_inbox[kMaxCluster];
    __shared__ UnitView s_uv[kUnitsPerCTA];
    __shared__ EEPart s_slot[3];  // two alternating exchange slots and the seed slot
    __shared__ EEPart s_all[kMaxCluster];
    __shared__ float s_wm[kCommitWarps], s_ws[kCommitWarps];
    __shared__ int s_wi[kCommitWarps];
    __shared__ float s_tm[kCommitWarps];  // target share: per-warp maxima (seed candidates)
    __shared__ int s_ti[kCommitWarps];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    const int b = blockIdx.x / p.C;
    cluster_arrive_relaxed();

    unsigned char *buf = cdyn;
    float *s_xt = (float *)(cdyn + commit_round_bytes(p.NS, p.slot));
    float *s_xd = s_xt + p.Kmax;
    float *s_l2u = s_xd + p.Kmax;
    float *s_pp = s_l2u + p.Kmax;
    float *s_qq = s_pp + p.Kmax;
    if (tid == 0) {
        mbar_init(&s_bar, 1);
        mbar_init_fence();
    }

    const ReqBase rbase = req_base(p.cu, p.num_draft, p.Kmax, b);
    const int kb_raw = rbase.kb;
    int status = SPEC_STATUS_OK;
    float T = 0.f;
    if (kb_raw < 0 || kb_raw > p.Kmax) status = SPEC_STATUS_BAD_K;
    if (status == SPEC_STATUS_OK && p.temperature) {
        T = p.temperature[b];
        if (!(T >= 0.f) || isinf(T)) status = SPEC_STATUS_BAD_TEMPERATURE;
    }
    const int kb = status == SPEC_STATUS_BAD_K ? 0 : kb_raw;
    const bool greedy = (T == 0.f);
    const int32_t *x = p.draft_tokens + rbase.d0;
    if (status == SPEC_STATUS_OK) {
        bool bad = false;
        for (int i = tid; i < kb; i += kCommitThreads) bad |= (x[i] < 0 || x[i] >= p.V);
        if (__syncthreads_or(bad)) status = SPEC_STATUS_BAD_TOKEN;
    }
    const float c = greedy ? 0.f : __fdiv_rn(kLog2e, T);
    const float invT = greedy ? 0.f : __fdiv_rn(1.f, T);
    const int npos = status == SPEC_STATUS_OK ? kb : 0;
    for (int i = tid; i < p.Kmax; i += kCommitThreads) {
        s_pp[i] = -1.f;
        s_qq[i] = -1.f;
        if (i < npos && !greedy) {
            const int xi = x[i];
            s_xt[i] = ld_elem<ESZ>(p.target, (rbase.t0 + i) * p.ld_row + xi);
            s_xd[i] = ld_elem<ESZ>(p.draft, (rbase.d0 + i) * p.ld_row + xi);
            const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)i, PURPOSE_ACCEPT, 0u);
            s_l2u[i] = log2f(u01(r4.x));
        }
    }
    cluster_wait();  // every CTA of the cluster is running
    __syncthreads();

    const int64_t rowbytes = p.ld_row * ESZ;
    const int sh = (((p.V + p.C - 1) / p.C) + 7) & ~7;  // share of a row per CTA
    const Chunking shk = {p.C, sh};
    const bool has_share = (int64_t)rank * sh < p.V;
    auto share_window = [&](const char *row) {
        ChunkWin w;
        if (has_share) {
            w = chunk_window(row, ESZ, p.V, shk, (int)rank);
        } else {
            w.a0 = row;
            w.bytes = 0;
            w.e0 = w.e1 = w.shift = 0;
        }
        return w;
    };
    auto nonfinite = [](float v) { return !(fabsf(v) < __int_as_float(0x7f800000)); };

    JobDesc jd;
    jd.kind = JOB_NONE;
    jd.row = 0;
    jd.A = 0;
    jd.token = -1;
    jd.invT = invT;
    jd.shift = jd.Cd = 0.f;
    jd.seed = kNegInf;
    jd.seed_idx = -1;
    int A = kb;
    int nx = 0;  // exchanges so far (slot parity)
    if (status == SPEC_STATUS_OK) {
        for (int i = 0; i < kb; ++i) {
            // ---- this CTA's share of target row i (and draft row i)
            const char *trow = (const char *)p.target + (rbase.t0 + i) * rowbytes;
            float m = kNegInf, mc = 0.f, s = 0.f;
            int kat = -1;
            bool nan_seen = false;
            const ChunkWin tw = share_window(trow);
            ee_thread_stats<Vec>(tw, c, m, mc, s, kat, nan_seen);
            const int widx = ee_warp_index<Vec>(tw, kat, m, warp_max_nan(m));
            EEPart part;
            ee_block_stats(m, mc, s, widx, nan_seen, c, s_wm, s_wi, s_ws, part.mt, part.st, part.it);
            if (tid < kCommitWarps) {  // the target share's warp argmaxes: correction seed candidates
                s_tm[tid] = s_wm[tid];
                s_ti[tid] = s_wi[tid];
            }
            part.md = 0.f;
            part.sd = 0.f;
            if (!greedy) {
                const char *drow = (const char *)p.draft + (rbase.d0 + i) * rowbytes;
                float m2 = kNegInf, mc2 = 0.f, s2 = 0.f;
                int k2 = -1;
                bool n2 = false;
                ee_thread_stats<Vec>(share_window(drow), c, m2, mc2, s2, k2, n2);
                int i2;  // the draft row's argmax is not needed
                ee_block_stats(m2, mc2, s2, -1, n2, c, s_wm, s_wi, s_ws, part.md, part.sd, i2);
            }
            part.seed = kNegInf;
            part.seed_idx = -1;
            part.pad = 0;
            // ---- the shares meet; every CTA combines them in rank order
            ee_exchange(part, &s_slot[nx & 1], s_all, p.C);
            ++nx;
            float Mt = s_all[0].mt, Md = s_all[0].md;
            for (int r = 1; r < p.C; ++r) {
                Mt = max_nan_f32(Mt, s_all[r].mt);
                Md = max_nan_f32(Md, s_all[r].md);
            }
            float St = 0.f, Sd = 0.f, bm = kNegInf;
            int It = -1;
            for (int r = 0; r < p.C; ++r) {
                const EEPart q = s_all[r];
                if (!greedy && q.mt != kNegInf && q.st != 0.f) St += q.st * exp2f(__fmul_rn(q.mt, c) - __fmul_rn(Mt, c));
                if (!greedy && q.md != kNegInf && q.sd != 0.f) Sd += q.sd * exp2f(__fmul_rn(q.md, c) - __fmul_rn(Md, c));
                if (better(q.mt, q.it, bm, It)) { bm = q.mt; It = q.it; }
            }
            if (nonfinite(Mt) || (!greedy && (nonfinite(Md) || nonfinite(St) || nonfinite(Sd)))) {
                status = SPEC_STATUS_NONFINITE;
                break;
            }
            if (greedy) {
                if (It != x[i]) {
                    A = i;
                    jd.token = It;
                    break;
                }
                continue;
            }
            const float l2St = log2f(St), l2Sd = log2f(Sd);
            const float l2p = fmaf(s_xt[i], c, -__fmul_rn(Mt, c)) - l2St;  // log2 p_i(x_i)
            const float l2q = fmaf(s_xd[i], c, -__fmul_rn(Md, c)) - l2Sd;  // log2 q_i(x_i)
            if (tid == 0) {
                s_pp[i] = exp2f(l2p);
                s_qq[i] = exp2f(l2q);
            }
            // accept iff u q < p, i.e. log2 u < log2 p - log2 q (Q = 0 < P accepts; P = 0 rejects)
            if (s_l2u[i] < l2p - l2q) continue;
            A = i;
            jd.kind = JOB_RESID;
            jd.row = i;
            jd.shift = (__fmul_rn(Mt, c) + l2St) * 0.6931471805599453f;
            jd.Cd = (__fmul_rn(Md, c) + l2Sd) * 0.6931471805599453f;
            // exact correction scores at this CTA's warp argmaxes of target row i; the
            // best over the cluster bounds the draw
            const char *drow = (const char *)p.draft + (rbase.d0 + i) * rowbytes;
            float sb = kNegInf;
            int si = -1;
            if (warp == 0) {
                if (lane < kCommitWarps && s_ti[lane] >= 0) {
                    const int v = s_ti[lane];
                    const float z = fmaf(s_tm[lane], invT, -jd.shift);
                    const float lq = fmaf(ld_elem<ESZ>(drow, v), invT, -jd.Cd);
                    if (lq < z) {
                        const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)i, PURPOSE_RESIDUAL,
                                                    (uint32_t)v >> 2);
                        const float sc = resid_score(z, lq, word_of(r4, v & 3));
                        if (sc > kNegInf) { sb = sc; si = v; }
                    }
                }
                warp_argmax(sb, si);
            }
            EEPart sp;
            sp.mt = sp.st = sp.md = sp.sd = 0.f;
            sp.it = sp.pad = 0;
            sp.seed = __shfl_sync(0xffffffffu, sb, 0);
            sp.seed_idx = __shfl_sync(0xffffffffu, si, 0);
            if (warp == 0 && lane == 0) s_slot[2] = sp;
            __syncthreads();
            ee_exchange(s_slot[2], &s_slot[2], s_all, p.C);
            for (int r = 0; r < p.C; ++r)
                if (better(s_all[r].seed, s_all[r].seed_idx, jd.seed, jd.seed_idx)) {
                    jd.seed = s_all[r].seed;
                    jd.seed_idx = s_all[r].seed_idx;
                }
            break;
        }
        if (status == SPEC_STATUS_OK && A == kb && jd.token < 0 && jd.kind == JOB_NONE) {
            jd.row = kb;
            jd.kind = greedy ? JOB_ARGMAX : JOB_BONUS;
        }
    }
    jd.A = A;

    // ---- the one extra token: staged Gumbel-max over the job row (or argmax)
    const char *jrow = (const char *)p.target + (rbase.t0 + jd.row) * rowbytes;
    const char *jdrow = jd.kind == JOB_RESID ? (const char *)p.draft + (rbase.d0 + jd.row) * rowbytes : nullptr;
    if (warp == 0 && jd.kind != JOB_NONE) issue_job_round<ESZ>(p, rank, jrow, 0, buf, &s_bar, s_uv);
    __syncthreads();
    const SliceRes res = job_row_rounds<ESZ>(p, jd, (uint32_t)b, rank, jrow, jdrow, buf, &s_bar, s_uv, s_live_g,
                                             s_live_z, s_red);
    if (tid == 0) st_cluster_v4(&s_inbox[rank], 0, make_uint4(__float_as_uint(res.best), (uint32_t)res.idx,
                                                               __float_as_uint(res.rawmax), (uint32_t)res.failed));
    cluster_arrive();
    cluster_wait();
    if (rank != 0) return;

    int token = jd.token;
    if (status == SPEC_STATUS_OK && jd.kind != JOB_NONE) {
        SliceRes o = s_inbox[0];
        for (int r = 1; r < p.C; ++r) {
            const SliceRes q = s_inbox[r];
            if (better(q.best, q.idx, o.best, o.idx)) { o.best = q.best; o.idx = q.idx; }
            o.rawmax = max_nan_f32(o.rawmax, q.rawmax);
            o.failed |= q.failed;
        }
        if (o.failed) status = SPEC_STATUS_INTERNAL;
        else if (jd.kind != JOB_RESID && nonfinite(o.rawmax)) status = SPEC_STATUS_NONFINITE;
        token = o.idx;
        if (status == SPEC_STATUS_OK && jd.kind == JOB_RESID && o.idx < 0) {
            // p <= q everywhere (only by rounding): draw from p_j with the same noise
            const int64_t trow = (rbase.t0 + jd.row) * p.ld_row;
            SliceRes f;
            f.best = kNegInf;
            f.idx = -1;
            f.rawmax = kNegInf;
            f.failed = 0;
            for (int v = tid; v < p.V; v += kCommitThreads) {
                const float lp = fmaf(ld_elem<ESZ>(p.target, trow + v), jd.invT, -jd.shift);
                if (!(lp > kNegInf)) continue;
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)jd.row, PURPOSE_RESIDUAL,
                                            (uint32_t)v >> 2);
                const float sc = lp + gumbel_of_word(word_of(r4, v & 3));
                if (better(sc, v, f.best, f.idx)) { f.best = sc; f.idx = v; }
            }
            token = block_reduce(f, s_red).idx;
        }
    }
    const bool ok = status == SPEC_STATUS_OK;
    const int Aout = ok ? A : 0;
    int32_t *tok = p.out_tokens + rbase.t0;
    for (int i = tid; i < rbase.ntok; i += kCommitThreads)
        tok[i] = !ok ? -1 : (i < Aout ? x[i] : (i == Aout ? token : -1));
    const bool pq = ok && !greedy;
    if (p.out_p)
        for (int i = tid; i < rbase.npq; i += kCommitThreads) p.out_p[rbase.d0 + i] = pq && i < kb ? s_pp[i] : -1.f;
    if (p.out_q)
        for (int i = tid; i < rbase.npq; i += kCommitThreads) p.out_q[rbase.d0 + i] = pq && i < kb ? s_qq[i] : -1.f;
    if (tid == 0) {
        p.out_status[b] = status;
        p.out_accepted[b] = Aout;
    }
}

// =================================================================== host side
thread_local int t_last_cuda_error = 0;

std::mutex g_mu;
int g_sms[64];
bool g_attr_set[64][4];

int device_info(int *dev_out, int *sms_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    if (dev < 0 || dev >= 64) return SPEC_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mu);
    if (g_sms[dev] == 0) {
        int sms = 0;
        e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
        g_sms[dev] = sms;
    }
    *dev_out = dev;
    *sms_out = g_sms[dev];
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
            cudaSetDevice(g_prof_dev);
            for (auto &e : g_prof_ev) cudaEventDestroy(e);
            cudaSetDevice(dev);
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
    explicit ProfScope(cudaStream_t st) : s(st), k(-1) {
        if (g_prof && g_prof_n < kMaxProfKernels) {
            k = g_prof_n++;
            cudaEventRecord(g_prof_ev[2 * k], s);
        }
    }
    ~ProfScope() {
        if (k >= 0) cudaEventRecord(g_prof_ev[2 * k + 1], s);
    }
};

// Workspace of the two-kernel verify (caller-owned, 256-byte aligned pieces):
//   ticket     main_kernel's chunk-ticket counter: zero before the first call,
//              and every call leaves it zero (commit_kernel resets it);
//   row_start  [B+1] first main-pass row of each request;
//   sync       [B] 128-byte records, one line per request so that the pieces of
//              different requests never contend for a line: pieces finished and the
//              pieces' shared bound (both zeroed by main_kernel in every call);
//   parts      one Part per chunk of every main-pass row (B * rows * cpr);
//   cand       kCW seed-candidate vectors per chunk (B * rows * cpr * kCW, 16-bit);
//   pres       [B * P] commit pieces' results.
struct Layout {
    size_t off_ticket, off_row_start, off_sync, off_parts, off_cand, off_pres, total;
    int cpr;                 // main pass: chunks per row
    int P, jslot;            // commit: pieces per request, bytes per unit slot
    int C, ue, NS, slot;     // early exit: cluster size, entries per unit, units per round, bytes per slot
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Layout make_layout(int B, int Kmax, int V, int esz, int main_rows_per_request) {
    Layout L;
    const Chunking ck = make_chunking(V, esz);
    L.cpr = ck.cpr;
    L.P = job_pieces(V);
    L.jslot = job_slot_bytes(esz);
    size_t o = 0;
    L.off_ticket = o;
    o = align256(o + 16);
    L.off_row_start = o;
    o = align256(o + sizeof(int) * (size_t)(B + 1));
    L.off_sync = o;
    o = align256(o + sizeof(uint32_t) * kSyncWords * (size_t)B);
    L.off_parts = o;
    o = align256(o + sizeof(Part) * (size_t)B * (size_t)main_rows_per_request * (size_t)ck.cpr);
    L.off_cand = o;
    o = align256(o + sizeof(uint16_t) * kCW * (size_t)B * (size_t)main_rows_per_request * (size_t)ck.cpr);
    L.off_pres = o;
    o = align256(o + sizeof(PieceRes) * (size_t)B * (size_t)L.P);
    L.total = o;
    // early exit: a row splits into 8 C units, C CTAs (one cluster) per request with
    // one unit per warp; a CTA's share stays near kShareMaxBytes, and its units are
    // staged NS at a time (NS a power of two, so that the warps split evenly)
    const int64_t rowb = (int64_t)V * esz;
    const int64_t c_need = (rowb + kShareMaxBytes - 1) / kShareMaxBytes;
    L.C = (int)(c_need < 1 ? 1 : (c_need > kMaxCluster ? kMaxCluster : c_need));
    const int units = L.C * kUnitsPerCTA;
    L.ue = (((V + units - 1) / units) + 7) & ~7;
    L.slot = L.ue * esz + 32;  // an aligned superset of a unit's window fits
    L.NS = kUnitsPerCTA;
    while (L.NS > 1 && (int64_t)L.NS * L.slot > kRoundMaxBytes) L.NS >>= 1;
    return L;
}

int check_launch() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    return SPEC_OK;
}

// Tag of a call: every partial the main pass writes carries it, and the commit pass
// reports status 5 for a request whose partials do not (a chunk the main pass did
// not write in this call, as after a workspace that was not zeroed before first use).
std::atomic<uint32_t> g_epoch{0};

uint32_t next_epoch() {
    uint32_t e;
    do {
        e = g_epoch.fetch_add(1u) + 1u;
    } while (e == 0u || e == 0xffffffffu);
    return e;
}

// The device pointer p must belong to device dev (or be managed memory).
int check_device_pointer(const void *p, int dev) {
    cudaPointerAttributes a;
    const cudaError_t e = cudaPointerGetAttributes(&a, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return SPEC_EINVAL;
    }
    if (a.type == cudaMemoryTypeManaged) return SPEC_OK;
    return (a.type == cudaMemoryTypeDevice && a.device == dev) ? SPEC_OK : SPEC_EINVAL;
}

// Dynamic shared memory of main_kernel: the row scan and the per-request scales.
size_t main_extra(int B) { return sizeof(int) * (size_t)(B + 1) + sizeof(float) * (size_t)B; }

template <class Vec>
int set_smem_attrs(int dev) {
    const int which = Vec::ESIZE == 2 ? 0 : 1;
    if (g_attr_set[dev][which]) return SPEC_OK;
    cudaError_t e = cudaFuncSetAttribute(commit_kernel<Vec::ESIZE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kCommitSmemMax);
    // the largest shared-memory carveout, so that kJobBlocksPerSM pieces fit an SM
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(commit_kernel<Vec::ESIZE>, cudaFuncAttributePreferredSharedMemoryCarveout,
                                 (int)cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(main_kernel<Vec>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)main_extra(SPEC_MAX_BATCH));
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    g_attr_set[dev][which] = true;
    return SPEC_OK;
}

template <class Vec>
int launch_early_exit(int dev, const Layout &L, const CommitParams &cp, cudaStream_t st) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const int which = 2 + (Vec::ESIZE == 2 ? 0 : 1);
        if (!g_attr_set[dev][which]) {
            cudaError_t e = cudaFuncSetAttribute(early_exit_kernel<Vec::ESIZE>,
                                                 cudaFuncAttributeMaxDynamicSharedMemorySize, kCommitSmemMax);
            if (e == cudaSuccess)
                e = cudaFuncSetAttribute(early_exit_kernel<Vec::ESIZE>,
                                         cudaFuncAttributePreferredSharedMemoryCarveout,
                                         (int)cudaSharedmemCarveoutMaxShared);
            if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
            g_attr_set[dev][which] = true;
        }
    }
    ProfScope ps(st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(cp.B * L.C));
    cfg.blockDim = dim3(kCommitThreads);
    cfg.dynamicSmemBytes = ee_smem_bytes(L.NS, L.slot, cp.Kmax);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)L.C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeClusterSchedulingPolicyPreference;
    attr[1].val.clusterSchedulingPolicyPreference = cudaClusterSchedulingPolicyLoadBalancing;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, early_exit_kernel<Vec::ESIZE>, cp);
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    return SPEC_OK;
}

// Dynamic shared memory of the fused verify kernel: the row scan and the scales.
size_t fused_smem(int B) { return fused::align16(sizeof(int) * (size_t)(B + 1)) + sizeof(float) * (size_t)B; }

template <class Vec>
int launch_fused(int dev, int sms, const fused::VerifyParams &vp, size_t zero_bytes, cudaStream_t st) {
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const int which = Vec::ESIZE == 2 ? 0 : 1;
        static bool set[64][2];
        if (!set[dev][which]) {
            // the largest B; no carveout preference: the main loop's loads in flight need L1
            const cudaError_t e = cudaFuncSetAttribute(fused::verify_kernel<Vec>,
                                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                                       (int)fused_smem(SPEC_MAX_BATCH));
            if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
            set[dev][which] = true;
        }
    }
    // the ticket counters and the requests' lines start at zero whatever the workspace held
    const cudaError_t e = cudaMemsetAsync(vp.counters, 0, zero_bytes, st);
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    {
        ProfScope ps(st);
        fused::verify_kernel<Vec><<<kMainBlocksPerSM * sms, kCT, fused_smem(vp.B), st>>>(vp);
    }
    return check_launch();
}

template <class Vec>
int launch_all(int dev, int sms, const Layout &L, const MainParams &mp, const JobParams &jp, cudaStream_t st) {
    int rc;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        rc = set_smem_attrs<Vec>(dev);
    }
    if (rc) return rc;
    {
        ProfScope ps(st);
        main_kernel<Vec><<<kMainBlocksPerSM * sms, kCT, main_extra(mp.B), st>>>(mp);
    }
    if ((rc = check_launch())) return rc;
    ProfScope ps(st);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((int64_t)mp.B * L.P));
    cfg.blockDim = dim3(kJobThreads);
    cfg.dynamicSmemBytes = job_smem_bytes(Vec::ESIZE, mp.Kmax);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, commit_kernel<Vec::ESIZE>, jp);
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    return SPEC_OK;
}

int verify_impl(const void *target, const void *draft, int dtype, int B, int Kmax, int V, int64_t ld_row,
                const int32_t *draft_tokens, const int32_t *cu, const int32_t *num_draft, const float *temperature,
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
    const int esz = dtype == SPEC_BF16 ? 2 : 4;
    if (((uintptr_t)target % esz) || (draft && ((uintptr_t)draft % esz))) return SPEC_EINVAL;
    if ((int64_t)B * (2 * Kmax + 1) * (int64_t)V > ((int64_t)1 << 50)) return SPEC_EUNSUPPORTED;
    int dev = 0, sms = 0;
    int rc = device_info(&dev, &sms);
    if (rc) return rc;
    if ((rc = check_device_pointer(target, dev))) return rc;
    const Layout L = make_layout(B, Kmax, V, esz, sample ? 2 * Kmax : Kmax);
    // chunk indices of the main pass are 32-bit; the commit grid is B * P CTAs
    if ((int64_t)B * 2 * Kmax * L.cpr >= ((int64_t)1 << 31) || (int64_t)B * L.P >= ((int64_t)1 << 31))
        return SPEC_EUNSUPPORTED;
    if (job_smem_bytes(esz, Kmax) > (size_t)kCommitSmemMax) return SPEC_EUNSUPPORTED;
    if (!ws) return SPEC_EWORKSPACE;
    if (ws_bytes < L.total || ((uintptr_t)ws & 255)) return SPEC_EWORKSPACE;
    rc = prof_prepare();
    if (rc) return rc;

    char *w = (char *)ws;
    const float *temps = sample ? temperature : nullptr;
    const uint32_t epoch = next_epoch();

    if (B >= sms && L.cpr <= L.P) {
        // one request or more per SM: the fused kernel (its items' results fit the
        // pieces' array: Q <= cpr <= P)
        fused::VerifyParams vp;
        vp.target = target;
        vp.draft = draft;
        vp.dtype = dtype;
        vp.ld_row = ld_row;
        vp.B = B;
        vp.Kmax = Kmax;
        vp.V = V;
        vp.draft_tokens = draft_tokens;
        vp.cu = cu;
        vp.num_draft = num_draft;
        vp.temperature = temps;
        vp.seed = seed;
        vp.step = (uint32_t)step;
        vp.epoch = epoch;
        vp.cpr = L.cpr;
        vp.ce = make_chunking(V, esz).ce;
        const int G = kMainBlocksPerSM * sms;
        vp.Q = G / B < 1 ? 1 : (G / B > L.cpr ? L.cpr : G / B);
        vp.counters = (uint32_t *)(w + L.off_ticket);
        vp.sync = (unsigned long long *)(w + L.off_sync);
        vp.parts = (Part *)(w + L.off_parts);
        vp.cand = (uint16_t *)(w + L.off_cand);
        vp.pres = (PieceRes *)(w + L.off_pres);
        vp.out_tokens = out_tokens;
        vp.out_accepted = out_accepted;
        vp.out_p = sample ? out_p : nullptr;
        vp.out_q = sample ? out_q : nullptr;
        vp.out_status = out_status;
        cudaStream_t st = (cudaStream_t)cuda_stream;
        // one memset: the counters, row_start (unused here) and the requests' lines
        const size_t zb = L.off_sync + sizeof(uint32_t) * kSyncWords * (size_t)B;
        return dtype == SPEC_BF16 ? launch_fused<VecBF16>(dev, sms, vp, zb, st)
                                  : launch_fused<VecF32>(dev, sms, vp, zb, st);
    }

    MainParams mp;
    mp.target = target;
    mp.draft = draft;
    mp.ld_row = ld_row;
    mp.B = B;
    mp.Kmax = Kmax;
    mp.V = V;
    mp.cu = cu;
    mp.num_draft = num_draft;
    mp.temperature = temps;
    mp.row_start = (int *)(w + L.off_row_start);
    mp.sync = (uint32_t *)(w + L.off_sync);
    mp.ticket = (uint32_t *)(w + L.off_ticket);
    mp.parts = (Part *)(w + L.off_parts);
    mp.cand = (uint16_t *)(w + L.off_cand);
    mp.epoch = epoch;

    JobParams jp;
    jp.target = target;
    jp.draft = draft;
    jp.dtype = dtype;
    jp.ld_row = ld_row;
    jp.B = B;
    jp.Kmax = Kmax;
    jp.V = V;
    jp.draft_tokens = draft_tokens;
    jp.cu = cu;
    jp.num_draft = num_draft;
    jp.temperature = temps;
    jp.seed = seed;
    jp.step = (uint32_t)step;
    jp.epoch = epoch;
    jp.row_start = mp.row_start;
    jp.parts = mp.parts;
    jp.cand = mp.cand;
    jp.cpr = L.cpr;
    jp.ce = make_chunking(V, esz).ce;
    jp.P = L.P;
    jp.slot = L.jslot;
    jp.ticket = mp.ticket;
    jp.sync = mp.sync;
    jp.pres = (PieceRes *)(w + L.off_pres);
    jp.out_tokens = out_tokens;
    jp.out_accepted = out_accepted;
    jp.out_p = sample ? out_p : nullptr;
    jp.out_q = sample ? out_q : nullptr;
    jp.out_status = out_status;

    cudaStream_t st = (cudaStream_t)cuda_stream;
    return dtype == SPEC_BF16 ? launch_all<VecBF16>(dev, sms, L, mp, jp, st)
                              : launch_all<VecF32>(dev, sms, L, mp, jp, st);
}

// Scratch of spec_verify_sample_noalloc: part of this module's device image, one
// copy per device, so that entry point never calls an allocating routine.
static __device__ __align__(256) unsigned char g_static_scratch[SPEC_STATIC_SCRATCH_BYTES];
void *g_static_scratch_ptr[64];

// Address of the current device's copy, looked up once with that device current.
int static_scratch(int dev, void **out) {
    std::lock_guard<std::mutex> lk(g_mu);
    if (!g_static_scratch_ptr[dev]) {
        void *ptr = nullptr;
        cudaError_t e = cudaGetSymbolAddress(&ptr, g_static_scratch);
        if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
        g_static_scratch_ptr[dev] = ptr;
    }
    *out = g_static_scratch_ptr[dev];
    return SPEC_OK;
}

// Early-exit verify: one kernel, no workspace (see early_exit_kernel).
int early_exit_impl(const void *target, const void *draft, int dtype, int B, int Kmax, int V, int64_t ld_row,
                    const int32_t *draft_tokens, const int32_t *num_draft, const float *temperature,
                    uint64_t seed, uint64_t step, int32_t *out_tokens, int32_t *out_accepted, float *out_p,
                    float *out_q, int32_t *out_status, void *cuda_stream, bool sample) {
    if (B < 0 || Kmax < 0 || V <= 0 || ld_row < V) return SPEC_EINVAL;
    if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_EINVAL;
    if (B == 0) return SPEC_OK;
    if (B > SPEC_MAX_BATCH || Kmax > SPEC_MAX_DRAFTS) return SPEC_EUNSUPPORTED;
    if (!target || !out_tokens || !out_accepted || !out_status) return SPEC_EINVAL;
    if (Kmax > 0 && !draft_tokens) return SPEC_EINVAL;
    if (sample && (!temperature || (Kmax > 0 && !draft))) return SPEC_EINVAL;
    const int esz = dtype == SPEC_BF16 ? 2 : 4;
    if (((uintptr_t)target % esz) || (draft && ((uintptr_t)draft % esz))) return SPEC_EINVAL;
    int dev = 0, sms = 0;
    int rc = device_info(&dev, &sms);
    if (rc) return rc;
    if ((rc = check_device_pointer(target, dev))) return rc;
    const Layout L = make_layout(B, Kmax, V, esz, sample ? 2 * Kmax : Kmax);
    if (L.slot > kRoundMaxBytes || ee_smem_bytes(L.NS, L.slot, Kmax) > (size_t)kCommitSmemMax)
        return SPEC_EUNSUPPORTED;
    rc = prof_prepare();
    if (rc) return rc;
    CommitParams cp = {};
    cp.target = target;
    cp.draft = draft;
    cp.dtype = dtype;
    cp.ld_row = ld_row;
    cp.B = B;
    cp.Kmax = Kmax;
    cp.V = V;
    cp.draft_tokens = draft_tokens;
    cp.cu = nullptr;
    cp.num_draft = num_draft;
    cp.temperature = sample ? temperature : nullptr;
    cp.seed = seed;
    cp.step = (uint32_t)step;
    cp.C = L.C;
    cp.ue = L.ue;
    cp.NS = L.NS;
    cp.slot = L.slot;
    cp.out_tokens = out_tokens;
    cp.out_accepted = out_accepted;
    cp.out_p = sample ? out_p : nullptr;
    cp.out_q = sample ? out_q : nullptr;
    cp.out_status = out_status;
    cudaStream_t st = (cudaStream_t)cuda_stream;
    return dtype == SPEC_BF16 ? launch_early_exit<VecBF16>(dev, L, cp, st) : launch_early_exit<VecF32>(dev, L, cp, st);
}

}  // namespace

namespace specv {
void note_cuda_error(int e) { t_last_cuda_error = e; }
}  // namespace specv

extern "C" {

size_t spec_verify_workspace_size(int B, int Kmax, int V, int dtype) {
    if (B < 0 || Kmax < 0 || V <= 0 || (dtype != SPEC_BF16 && dtype != SPEC_F32)) return 0;
    if (B > SPEC_MAX_BATCH || Kmax > SPEC_MAX_DRAFTS) return 0;
    return make_layout(B, Kmax, V, dtype == SPEC_BF16 ? 2 : 4, 2 * Kmax).total;
}

int spec_verify_greedy(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                       const int32_t *draft_tokens, const int32_t *num_draft, int32_t *out_tokens,
                       int32_t *out_accepted, int32_t *out_status, void *ws, size_t ws_bytes,
                       void *cuda_stream) {
    return verify_impl(target, nullptr, dtype, B, Kmax, V, ld_row, draft_tokens, nullptr, num_draft, nullptr, 0, 0,
                       out_tokens, out_accepted, nullptr, nullptr, out_status, ws, ws_bytes, cuda_stream,
                       false);
}

int spec_verify_sample(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                       int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                       const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                       int32_t *out_accepted, float *out_p, float *out_q, int32_t *out_status, void *ws,
                       size_t ws_bytes, void *cuda_stream) {
    return verify_impl(target, draft, dtype, B, Kmax, V, ld_row, draft_tokens, nullptr, num_draft, temperature, seed,
                       step, out_tokens, out_accepted, out_p, out_q, out_status, ws, ws_bytes, cuda_stream,
                       true);
}

int spec_verify_sample_noalloc(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                               int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                               const float *temperature, uint64_t seed, uint64_t step,
                               int32_t *out_tokens, int32_t *out_accepted, float *out_p, float *out_q,
                               int32_t *out_status, void *cuda_stream) {
    if (B < 0 || Kmax < 0 || V <= 0 || ld_row < V) return SPEC_EINVAL;
    if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_EINVAL;
    if (B == 0) return SPEC_OK;
    if (B > SPEC_MAX_BATCH || Kmax > SPEC_MAX_DRAFTS) return SPEC_EUNSUPPORTED;
    int dev = 0, sms = 0;
    int rc = device_info(&dev, &sms);
    if (rc) return rc;
    if (make_layout(B, Kmax, V, dtype == SPEC_BF16 ? 2 : 4, 2 * Kmax).total > SPEC_STATIC_SCRATCH_BYTES)
        return SPEC_ESCRATCH;
    void *ws = nullptr;
    if ((rc = static_scratch(dev, &ws))) return rc;
    return verify_impl(target, draft, dtype, B, Kmax, V, ld_row, draft_tokens, nullptr, num_draft, temperature, seed,
                       step, out_tokens, out_accepted, out_p, out_q, out_status, ws, SPEC_STATIC_SCRATCH_BYTES,
                       cuda_stream, true);
}

int spec_verify_greedy_flat(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                            const int32_t *cu_draft, const int32_t *draft_tokens, int32_t *out_tokens,
                            int32_t *out_accepted, int32_t *out_status, void *ws, size_t ws_bytes,
                            void *cuda_stream) {
    if (B > 0 && !cu_draft) return SPEC_EINVAL;
    return verify_impl(target, nullptr, dtype, B, Kmax, V, ld_row, draft_tokens, cu_draft, nullptr, nullptr, 0, 0,
                       out_tokens, out_accepted, nullptr, nullptr, out_status, ws, ws_bytes, cuda_stream, false);
}

int spec_verify_sample_flat(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                            int64_t ld_row, const int32_t *cu_draft, const int32_t *draft_tokens,
                            const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                            int32_t *out_accepted, float *out_p, float *out_q, int32_t *out_status, void *ws,
                            size_t ws_bytes, void *cuda_stream) {
    if (B > 0 && !cu_draft) return SPEC_EINVAL;
    return verify_impl(target, draft, dtype, B, Kmax, V, ld_row, draft_tokens, cu_draft, nullptr, temperature,
                       seed, step, out_tokens, out_accepted, out_p, out_q, out_status, ws, ws_bytes, cuda_stream,
                       true);
}

int spec_verify_sample_early_exit(const void *target, const void *draft, int dtype, int B, int Kmax, int V,
                                  int64_t ld_row, const int32_t *draft_tokens, const int32_t *num_draft,
                                  const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                                  int32_t *out_accepted, float *out_p, float *out_q, int32_t *out_status,
                                  void *cuda_stream) {
    return early_exit_impl(target, draft, dtype, B, Kmax, V, ld_row, draft_tokens, num_draft, temperature, seed,
                           step, out_tokens, out_accepted, out_p, out_q, out_status, cuda_stream, true);
}

int spec_verify_greedy_early_exit(const void *target, int dtype, int B, int Kmax, int V, int64_t ld_row,
                                  const int32_t *draft_tokens, const int32_t *num_draft, int32_t *out_tokens,
                                  int32_t *out_accepted, int32_t *out_status, void *cuda_stream) {
    return early_exit_impl(target, nullptr, dtype, B, Kmax, V, ld_row, draft_tokens, num_draft, nullptr, 0, 0,
                           out_tokens, out_accepted, nullptr, nullptr, out_status, cuda_stream, false);
}

const char *spec_error_string(int err) {
    switch (err) {
        case SPEC_OK: return "ok";
        case SPEC_EINVAL: return "invalid argument";
        case SPEC_ECUDA: return "CUDA error";
        case SPEC_EUNSUPPORTED: return "unsupported size or layout";
        case SPEC_EWORKSPACE: return "workspace missing or too small";
        case SPEC_ESCRATCH: return "sizes need more than the fixed scratch of spec_verify_sample_noalloc";
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
