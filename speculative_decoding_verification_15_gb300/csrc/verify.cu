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
// Kernels per call (fixed grids, no host synchronisation; each launch after the
// first is a programmatic dependent launch):
//  main_kernel    streams the rows of every draft position once -- target and draft
//                 rows of sampling requests, target rows of greedy ones -- through a
//                 bulk-copy (TMA) ring in shared memory: one persistent CTA per SM, a
//                 producer warp issuing 32 KB cp.async.bulk copies, sixteen consumer
//                 warps reducing them.  Per (CTA, row, warp): max, sum of
//                 2^(x log2e / T - max'), and the lowest argmax.  HBM-bound.
//  accept_kernel  one CTA per request: combines the partials of its rows, sets the
//                 status, computes p(x_i) and q(x_i), runs the acceptance scan,
//                 emits the accepted drafts, and queues one job: the correction at
//                 the first rejected row j (seeded with the segment argmaxes of row
//                 j), the bonus draw on row k_b, or the greedy argmax of row k_b.
//  tail_kernel    one warp per 1024-entry unit of each job's row, loaded with its
//                 own 16-byte loads: Gumbel-max over log(max(0, p - q)) (draft values
//                 gathered only at entries that can still win), Gumbel-max over the
//                 target row, or argmax.
//  final_kernel   one warp per job: combines the tail partials into the token.
#include <cuda_runtime.h>
#include <stdint.h>
#include <string.h>

#include <mutex>

#include "spec_common.cuh"
#include "spec_verify.h"

using namespace specv;

namespace {

// ------------------------------------------------------------------ configuration
constexpr int kCW = 16;                          // consumer warps per CTA (4 per scheduler)
constexpr int kCT = kCW * 32;                    // consumer threads
constexpr int kPipeThreads = kCT + 32;           // + one producer warp
constexpr int kMaxStages = 8;                    // ring depth: as many as shared memory allows
constexpr int kStageBytes = 32768;               // one chunk (plus alignment slack)
constexpr int kChunkMaxBytes = kStageBytes - 32; // payload; an aligned superset fits a stage
constexpr int kVPT = kStageBytes / 16 / kCT;     // 16-byte vectors per consumer thread (4)
constexpr size_t kSmemBudget = 226 * 1024;       // dynamic shared memory per CTA (227 KB minus static)
constexpr uint64_t kWaitNs = 2000000000ull;      // bound on every mbarrier wait (2 s)
constexpr int kAcceptThreads = 512;
constexpr int kFinalThreads = 256;
constexpr int kMaxRowsPerRequest = 2 * SPEC_MAX_DRAFTS;
constexpr int kMaxDesc = 512;                    // per-CTA row descriptors kept in smem
constexpr float kRescaleAt = 1024.f;             // lane chunk sum that moves the reference

enum JobKind : int { JOB_RESID = 0, JOB_BONUS = 1, JOB_ARGMAX = 2 };

struct Part {
    float m;     // raw max of the segment (NaN-propagating)
    float s;     // main pass: sum 2^(x c - fl(m c)); unused in the tail pass
    int idx;     // lowest index of the max (main pass, argmax jobs) or of the best score
    float best;  // tail pass: best Gumbel score
};

struct Job {
    int b, row, kind;
    float invT, Ct, Cd;  // log p_v = x_v invT - Ct, log q_v = y_v invT - Cd (correction)
    float seed_best;     // exact score of the best candidate found by accept_kernel
    int seed_idx;
};

struct Ctrl {
    int err;        // non-zero: a bounded wait gave up
    int job_count;  // jobs queued by accept_kernel
};

// Order-preserving map of a float onto uint32 (for atomicMax on scores).
__device__ __forceinline__ uint32_t ord_of(float f) {
    const uint32_t u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float float_of_ord(uint32_t o) {
    return __uint_as_float((o & 0x80000000u) ? (o & 0x7fffffffu) : ~o);
}

// ------------------------------------------------------------------ chunking
// Rows are cut into cpr chunks of ce elements (ce a multiple of 8, at most
// kChunkMaxBytes); the flattened chunk list of all rows is split into G equal
// contiguous ranges, one per CTA.
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

__host__ __device__ inline int64_t cta_first(int64_t total, int G, int i) { return total * i / G; }
__host__ __device__ inline int cta_of(int64_t total, int G, int64_t c) { return (int)(((c + 1) * G - 1) / total); }

// Rows one CTA can touch, an upper bound.
__host__ inline int segs_per_cta(int64_t total_max, int G, int cpr) {
    const int64_t per = (total_max + G - 1) / G;
    return (int)((per + cpr - 1) / cpr) + 1;
}

__device__ __forceinline__ int64_t part_slot(int cta, int nseg, int seg, int warp) {
    return ((int64_t)cta * nseg + seg) * kCW + warp;
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

// Loads this consumer thread's vectors of a staged chunk; out-of-window entries -inf.
// Vector t of thread ct holds global elements ebase + (ct + kCT t) VE + e.  Only a
// window that does not start and end on 16-byte boundaries needs masking, which
// is decided once per chunk (the branch is uniform across the CTA).
template <class Vec>
__device__ __forceinline__ void load_chunk(Vec (&d)[kVPT], const char *stage, const ChunkWin &w, int ct) {
    const int nvec = (int)(w.bytes >> 4);
    const int64_t ebase = (int64_t)w.e0 - w.shift;
    const bool ragged = w.shift != 0 || ebase + (int64_t)nvec * Vec::VE != w.e1;
    if (!ragged) {
#pragma unroll
        for (int t = 0; t < kVPT; ++t) {
            const int j = ct + kCT * t;
            d[t] = j < nvec ? Vec{lds128(stage + 16 * j)} : Vec::neg_inf();
        }
    } else {
#pragma unroll
        for (int t = 0; t < kVPT; ++t) {
            const int j = ct + kCT * t;
            if (j < nvec) {
                d[t].v = lds128(stage + 16 * j);
                if (j == 0 || j == nvec - 1) mask_vec(d[t], ebase + (int64_t)j * Vec::VE, w.e0, w.e1);
            } else {
                d[t] = Vec::neg_inf();
            }
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
__device__ __forceinline__ int chunk_find(const Vec (&d)[NV], int64_t ebase, int ct, float x) {
    int found = -1;
#pragma unroll
    for (int t = 0; t < NV; ++t)
#pragma unroll
        for (int e = 0; e < Vec::VE; ++e)
            if (found < 0 && d[t].get(e) == x) found = (int)(ebase + (int64_t)(ct + STRIDE * t) * Vec::VE + e);
    return found;
}

// sum_e 2^(x_e c - ms) over the thread's vectors, two lanes per instruction
template <class Vec>
__device__ __forceinline__ float chunk_expsum(const Vec (&d)[kVPT], float c, float ms) {
    const float2 cc = make_float2(c, c), mm = make_float2(-ms, -ms);
    float2 acc[Vec::VE / 2];
#pragma unroll
    for (int e = 0; e < Vec::VE / 2; ++e) acc[e] = make_float2(0.f, 0.f);
#pragma unroll
    for (int t = 0; t < kVPT; ++t)
#pragma unroll
        for (int e = 0; e < Vec::VE; e += 2) {
            const float2 y = ffma2(make_float2(d[t].get(e), d[t].get(e + 1)), cc, mm);
            acc[e / 2] = fadd2(acc[e / 2], make_float2(ex2_approx(y.x), ex2_approx(y.y)));
        }
#pragma unroll
    for (int e = 1; e < Vec::VE / 2; ++e) acc[0] = fadd2(acc[0], acc[e]);
    return acc[0].x + acc[0].y;
}

// ------------------------------------------------------------------ ring
struct Ring {
    char *stages;
    uint64_t *full;
    uint64_t *empty;
    int n;  // stages
};

__host__ __device__ constexpr size_t ring_bytes(int n) {
    return (size_t)n * kStageBytes + 2 * (size_t)kMaxStages * sizeof(uint64_t);
}

__device__ __forceinline__ Ring ring_at(unsigned char *smem, int n) {
    Ring r;
    r.stages = (char *)smem;
    r.full = (uint64_t *)(smem + (size_t)n * kStageBytes);
    r.empty = r.full + kMaxStages;
    r.n = n;
    return r;
}

__device__ __forceinline__ void ring_init(const Ring &r) {
    if (threadIdx.x == 0) {
        for (int s = 0; s < r.n; ++s) {
            mbar_init(&r.full[s], 1);
            mbar_init(&r.empty[s], kCW);
        }
        mbar_init_fence();
    }
}

// Producer (one thread): stage chunks c0 .. c1-1; window(c) gives the source.
template <class Window>
__device__ void ring_produce(const Ring &r, int64_t c0, int64_t c1, Window window, int *err) {
    int s = 0;
    uint32_t ph = 0;
    for (int64_t c = c0; c < c1; ++c) {
        if (!mbar_wait(&r.empty[s], ph ^ 1u, kWaitNs)) {
            atomicOr(err, 1);
            // wait (bounded) for the copies this thread still has in flight
            const int64_t issued = c - c0;
            for (int64_t back = 1; back <= r.n && issued - back >= 0; ++back) {
                const int64_t i2 = issued - back;
                mbar_wait(&r.full[i2 % r.n], (uint32_t)(i2 / r.n) & 1u, kWaitNs);
            }
            return;
        }
        const ChunkWin w = window(c);
        mbar_arrive_expect_tx(&r.full[s], w.bytes);
        bulk_g2s(r.stages + (size_t)s * kStageBytes, w.a0, w.bytes, &r.full[s]);
        if (++s == r.n) {
            s = 0;
            ph ^= 1u;
        }
    }
}

// ------------------------------------------------------------------ per-request rows
__device__ __forceinline__ int request_main_rows(const int32_t *num_draft, const float *temperature, int Kmax,
                                                 int b) {
    const int kb = num_draft ? num_draft[b] : Kmax;
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
__device__ void scan_request_rows(int *s, int B, const int32_t *num_draft, const float *temperature, int Kmax) {
    __shared__ int warp_tot[32];
    const int nthr = blockDim.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    const int per = (B + nthr - 1) / nthr;
    const int lo = min(tid * per, B), hi = min(lo + per, B);
    int local = 0;
    for (int i = lo; i < hi; ++i) local += request_main_rows(num_draft, temperature, Kmax, i);
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
        run += request_main_rows(num_draft, temperature, Kmax, i);
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

// =================================================================== main_kernel
struct MainParams {
    const void *target;
    const void *draft;
    int64_t ld_row;
    int B, Kmax, V;
    const int32_t *num_draft;
    const float *temperature;  // NULL: every request greedy
    int *row_start;            // [B+1], written by block 0 for accept_kernel
    Part *parts;
    int nseg;
    int stages;
    Ctrl *ctrl;
};

struct MainRow {
    const char *ptr;
    float c;      // log2(e) / T, or 0 for a greedy row
};

template <class Vec>
__device__ __forceinline__ MainRow main_row(const MainParams &p, const int *rs, int r) {
    const int b = find_request(rs, p.B, r);
    const int local = r - rs[b];
    const int kb = p.num_draft ? p.num_draft[b] : p.Kmax;
    const float T = p.temperature ? p.temperature[b] : 0.f;
    const int64_t rowbytes = p.ld_row * Vec::ESIZE;
    MainRow m;
    if (T == 0.f || local < kb) {
        m.ptr = (const char *)p.target + ((int64_t)b * (p.Kmax + 1) + local) * rowbytes;
    } else {
        m.ptr = (const char *)p.draft + ((int64_t)b * p.Kmax + (local - kb)) * rowbytes;
    }
    m.c = T == 0.f ? 0.f : __fdiv_rn(kLog2e, T);
    return m;
}

template <class Vec>
__global__ void __launch_bounds__(kPipeThreads, 1) main_kernel(MainParams p) {
    extern __shared__ __align__(128) unsigned char smem[];
    const Ring ring = ring_at(smem, p.stages);
    int *s_rs = (int *)(smem + ring_bytes(p.stages));
    MainRow *s_desc = (MainRow *)(smem + ring_bytes(p.stages) + sizeof(int) * (size_t)(((p.B + 1) + 3) & ~3));
    ring_init(ring);
    scan_request_rows(s_rs, p.B, p.num_draft, p.temperature, p.Kmax);  // ends with __syncthreads
    if (blockIdx.x == 0)
        for (int i = threadIdx.x; i <= p.B; i += blockDim.x) p.row_start[i] = s_rs[i];
    pdl_launch_dependents();

    const Chunking ck = make_chunking(p.V, Vec::ESIZE);
    const int G = gridDim.x;
    const int64_t total = (int64_t)s_rs[p.B] * ck.cpr;
    if (total == 0) return;
    const int64_t c0 = cta_first(total, G, blockIdx.x), c1 = cta_first(total, G, blockIdx.x + 1);
    if (c0 == c1) return;
    const int first_row = (int)(c0 / ck.cpr);
    const int nrows = (int)((c1 - 1) / ck.cpr) - first_row + 1;
    const bool table = nrows <= kMaxDesc;
    if (table)
        for (int i = threadIdx.x; i < nrows; i += blockDim.x) s_desc[i] = main_row<Vec>(p, s_rs, first_row + i);
    __syncthreads();
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int k0 = (int)(c0 - (int64_t)first_row * ck.cpr);

    if (warp == kCW) {  // producer
        if (lane == 0) {
            int r = first_row, k = k0;
            MainRow mr = table ? s_desc[0] : main_row<Vec>(p, s_rs, r);
            ring_produce(ring, c0, c1, [&](int64_t) {
                const ChunkWin w = chunk_window(mr.ptr, Vec::ESIZE, p.V, ck, k);
                if (++k == ck.cpr) {
                    k = 0;
                    ++r;
                    if (r < first_row + nrows) mr = table ? s_desc[r - first_row] : main_row<Vec>(p, s_rs, r);
                }
                return w;
            }, &p.ctrl->err);
        }
        return;
    }

    const int ct = threadIdx.x;  // consumer thread 0 .. kCT-1
    int r = first_row, k = k0;
    MainRow mr = table ? s_desc[0] : main_row<Vec>(p, s_rs, r);
    float m = kNegInf, mc = 0.f, s = 0.f;
    int aidx = -1;
    bool nan_seen = false;
    auto flush = [&]() {
        Part out;
        if (mr.c != 0.f) {
            const float M = warp_max_nan(m);
            const float MC = M * mr.c;
            const float sc = (m == kNegInf || s == 0.f) ? 0.f : s * ex2_approx(mc - MC);
            out.s = (float)warp_sum_d((double)sc);
            float mm = m;
            int ii = aidx;
            warp_argmax(mm, ii);
            out.m = M;
            out.idx = ii;
        } else {
            const bool any_nan = __any_sync(0xffffffffu, nan_seen);
            float mm = m;
            int ii = aidx;
            warp_argmax(mm, ii);
            out.m = any_nan ? __int_as_float(0x7fc00000) : mm;
            out.s = 0.f;
            out.idx = ii;
        }
        out.best = 0.f;
        if (lane == 0) p.parts[part_slot(blockIdx.x, p.nseg, r - first_row, warp)] = out;
    };

    int st = 0;
    uint32_t ph = 0;
    for (int64_t cc = c0; cc < c1; ++cc) {
        if (!mbar_wait(&ring.full[st], ph, kWaitNs)) {
            atomicOr(&p.ctrl->err, 2);
            break;
        }
        const ChunkWin w = chunk_window(mr.ptr, Vec::ESIZE, p.V, ck, k);
        Vec d[kVPT];
        load_chunk(d, ring.stages + (size_t)st * kStageBytes, w, ct);
        __syncwarp();
        if (lane == 0) mbar_arrive(&ring.empty[st]);
        if (++st == ring.n) {
            st = 0;
            ph ^= 1u;
        }
        const int64_t ebase = (int64_t)w.e0 - w.shift;
        if (mr.c != 0.f) {
            // s is kept relative to a per-lane reference entry m (mc = fl(m c)); any
            // reference gives the exact sum, so it only moves when this chunk's terms
            // grow past kRescaleAt (an entry more than 5 log2-units above m), on the
            // first finite chunk, or for NaN / +inf.
            float cs = chunk_expsum(d, mr.c, mc);
            if (m == kNegInf || !(cs < kRescaleAt)) {
                const float tm = chunk_max(d);
                if (!(tm <= m)) {  // new reference, or NaN
                    const float mcn = tm * mr.c;
                    s = (m == kNegInf) ? 0.f : s * ex2_approx(mc - mcn);
                    m = tm;
                    mc = mcn;
                    aidx = chunk_find<kCT>(d, ebase, ct, tm);
                    cs = chunk_expsum(d, mr.c, mc);
                } else if (m == kNegInf) {
                    cs = 0.f;  // every entry so far is -inf
                }
            }
            s += cs;
        } else {
            const float tm = chunk_max(d);
            if (tm != tm) {
                nan_seen = true;
            } else if (tm > m) {
                m = tm;
                aidx = chunk_find<kCT>(d, ebase, ct, tm);
            }
        }
        if (++k == ck.cpr || cc + 1 == c1) {  // row segment ends
            flush();
            k = 0;
            ++r;
            if (r < first_row + nrows) mr = table ? s_desc[r - first_row] : main_row<Vec>(p, s_rs, r);
            m = kNegInf;
            mc = 0.f;
            s = 0.f;
            aidx = -1;
            nan_seen = false;
        }
    }
}

// =================================================================== combine helpers
// Partials of flat row r: CTAs [lo, hi] x kCW warps.
struct RowParts {
    int lo, hi, seg_lo;
    __device__ __forceinline__ int n() const { return (hi - lo + 1) * kCW; }
};

__device__ __forceinline__ RowParts row_parts(int64_t total, int G, int cpr, int r) {
    RowParts rp;
    rp.lo = cta_of(total, G, (int64_t)r * cpr);
    rp.hi = cta_of(total, G, (int64_t)r * cpr + cpr - 1);
    rp.seg_lo = r;
    return rp;
}

// Partial q of row r, or nullptr when its CTA has an empty chunk range (possible
// when there are fewer chunks than CTAs): such CTAs lie between the row's first
// and last CTA but wrote nothing.
__device__ __forceinline__ const Part *part_of(const Part *parts, int64_t total, int G, int cpr, int nseg, int r,
                                                const RowParts &rp, int q) {
    const int cta = rp.lo + q / kCW;
    const int64_t c0 = cta_first(total, G, cta);
    if (c0 == cta_first(total, G, cta + 1)) return nullptr;
    const int seg = r - (int)(c0 / cpr);
    return &parts[part_slot(cta, nseg, seg, q % kCW)];
}

struct RowRes {
    float M;    // raw row max
    float l2S;  // log2 sum_v 2^(x_v c - fl(M c)) (stats rows)
    float xv;   // logit at the draft token (stats rows)
    int idx;    // lowest argmax
};

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
    int nseg, G, cpr;
    int32_t *out_tokens;
    int32_t *out_accepted;
    float *out_p;
    float *out_q;
    int32_t *out_status;
    Job *jobs;
    int *job_list;
    uint32_t *job_best;
    Ctrl *ctrl;
};

// Exact score of the correction draw at one entry: log(p - q) + g, with p > q.
__device__ __forceinline__ float resid_score(float lp, float lq, uint32_t w) {
    return lp + logf(-expm1f(lq - lp)) + gumbel_of_word(w);
}

__global__ void __launch_bounds__(kAcceptThreads) accept_kernel(AcceptParams p) {
    __shared__ RowRes s_rows[kMaxRowsPerRequest];
    pdl_wait();
    pdl_launch_dependents();
    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nwarps = blockDim.x >> 5;
    const int K1 = p.Kmax + 1;
    int32_t *tok = p.out_tokens + (int64_t)b * K1;
    for (int i = tid; i < K1; i += blockDim.x) tok[i] = -1;
    if (p.out_p)
        for (int i = tid; i < p.Kmax; i += blockDim.x) p.out_p[(int64_t)b * p.Kmax + i] = -1.f;
    if (p.out_q)
        for (int i = tid; i < p.Kmax; i += blockDim.x) p.out_q[(int64_t)b * p.Kmax + i] = -1.f;

    // statuses, in order: k_b, temperature, tokens, non-finite rows
    const int kb = p.num_draft ? p.num_draft[b] : p.Kmax;
    int status = SPEC_STATUS_OK;
    float T = 0.f;
    if (kb < 0 || kb > p.Kmax) status = SPEC_STATUS_BAD_K;
    if (status == SPEC_STATUS_OK && p.temperature) {
        T = p.temperature[b];
        if (!(T >= 0.f) || isinf(T)) status = SPEC_STATUS_BAD_TEMPERATURE;
    }
    if (p.ctrl->err) status = SPEC_STATUS_INTERNAL;
    const bool greedy = (T == 0.f);
    const int32_t *x = p.draft_tokens + (int64_t)b * p.Kmax;
    if (status == SPEC_STATUS_OK) {
        bool bad = false;
        for (int i = tid; i < kb; i += blockDim.x) bad |= (x[i] < 0 || x[i] >= p.V);
        if (__syncthreads_or(bad)) status = SPEC_STATUS_BAD_TOKEN;
    }
    const float c = greedy ? 0.f : __fdiv_rn(kLog2e, T);
    const int64_t total = (int64_t)p.row_start[p.B] * p.cpr;
    const int r0 = p.row_start[b];
    const int nrows = status == SPEC_STATUS_OK ? (greedy ? kb : 2 * kb) : 0;

    // combine the partials of every row of this request, one warp per row
    bool nonfinite = false;
    for (int rr = warp; rr < nrows; rr += nwarps) {
        const int r = r0 + rr;
        // the draft token's logit: independent of the partials, so issued first
        float xv = 0.f;
        if (!greedy) {
            const bool is_draft = rr >= kb;
            const int i = is_draft ? rr - kb : rr;
            const int64_t row = is_draft ? ((int64_t)b * p.Kmax + i) : ((int64_t)b * K1 + i);
            xv = load_logit(is_draft ? p.draft : p.target, p.dtype, row * p.ld_row + x[i]);
        }
        const RowParts rp = row_parts(total, p.G, p.cpr, r);
        float m = kNegInf;
        for (int q = lane; q < rp.n(); q += 32) {
            const Part *pt = part_of(p.parts, total, p.G, p.cpr, p.nseg, r, rp, q);
            if (pt) m = max_nan_f32(m, pt->m);
        }
        const float M = warp_max_nan(m);
        double sum = 0.0;
        float bm = kNegInf;
        int bi = -1;
        const float MC = M * c;
        for (int q = lane; q < rp.n(); q += 32) {
            const Part *pt = part_of(p.parts, total, p.G, p.cpr, p.nseg, r, rp, q);
            if (!pt) continue;
            if (!greedy && pt->m != kNegInf && pt->s != 0.f) sum += (double)pt->s * (double)exp2f(pt->m * c - MC);
            if (better(pt->m, pt->idx, bm, bi)) { bm = pt->m; bi = pt->idx; }
        }
        warp_argmax(bm, bi);
        RowRes res;
        res.M = M;
        res.idx = bi;
        res.l2S = 0.f;
        res.xv = 0.f;
        if (!greedy) {
            sum = warp_sum_d(sum);
            res.l2S = log2f((float)sum);
            res.xv = xv;
        }
        nonfinite |= !(fabsf(M) < __int_as_float(0x7f800000));
        if (lane == 0) s_rows[rr] = res;
    }
    if (__syncthreads_or(nonfinite) && status == SPEC_STATUS_OK) status = SPEC_STATUS_NONFINITE;

    if (status != SPEC_STATUS_OK) {
        if (tid == 0) {
            p.out_status[b] = status;
            p.out_accepted[b] = 0;
        }
        return;
    }
    if (warp != 0) return;

    // acceptance scan, 32 positions at a time; A = first rejected position
    int A = kb;
    int token = -1;
    if (greedy) {
        for (int i0 = 0; i0 < kb && A == kb; i0 += 32) {
            const int i = i0 + lane;
            const bool mism = i < kb && s_rows[i].idx != x[i];
            const unsigned msk = __ballot_sync(0xffffffffu, mism);
            if (msk) A = i0 + __ffs(msk) - 1;
        }
        if (A < kb) token = s_rows[A].idx;
    } else {
        for (int i0 = 0; i0 < kb; i0 += 32) {
            const int i = i0 + lane;
            bool rej = false;
            if (i < kb) {
                const RowRes tr = s_rows[i], dr = s_rows[kb + i];
                const float l2p = fmaf(tr.xv, c, -(tr.M * c)) - tr.l2S;  // log2 p_i(x_i)
                const float l2q = fmaf(dr.xv, c, -(dr.M * c)) - dr.l2S;  // log2 q_i(x_i)
                if (p.out_p) p.out_p[(int64_t)b * p.Kmax + i] = exp2f(l2p);
                if (p.out_q) p.out_q[(int64_t)b * p.Kmax + i] = exp2f(l2q);
                // accept iff u q < p, i.e. log2 u < log2 p - log2 q (Q = 0 < P accepts; P = 0 rejects)
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)i, PURPOSE_ACCEPT, 0u);
                rej = !(log2f(u01(r4.x)) < l2p - l2q);
            }
            const unsigned msk = __ballot_sync(0xffffffffu, rej);
            if (msk && A == kb) A = i0 + __ffs(msk) - 1;
        }
    }
    for (int i = lane; i < A; i += 32) tok[i] = x[i];

    if (greedy && A < kb) {
        if (lane == 0) tok[A] = token;
    } else {
        Job job;
        job.b = b;
        job.row = A;
        job.kind = greedy ? JOB_ARGMAX : (A < kb ? JOB_RESID : JOB_BONUS);
        job.invT = greedy ? 0.f : __fdiv_rn(1.f, T);
        job.Ct = job.Cd = 0.f;
        job.seed_best = kNegInf;
        job.seed_idx = -1;
        if (job.kind == JOB_RESID) {
            const int j = A;
            const RowRes tr = s_rows[j], dr = s_rows[kb + j];
            job.Ct = (float)(((double)(tr.M * c) + (double)tr.l2S) * 0.6931471805599453);
            job.Cd = (float)(((double)(dr.M * c) + (double)dr.l2S) * 0.6931471805599453);
            // seed the correction draw with the segment argmaxes of target row j
            const int r = r0 + j;
            const RowParts rp = row_parts(total, p.G, p.cpr, r);
            const int64_t drow = ((int64_t)b * p.Kmax + j) * p.ld_row;
            float best = kNegInf;
            int bidx = -1;
            for (int q = lane; q < rp.n(); q += 32) {
                const Part *pt = part_of(p.parts, total, p.G, p.cpr, p.nseg, r, rp, q);
                if (!pt || pt->idx < 0) continue;
                const int v = pt->idx;
                const float lp = fmaf(pt->m, job.invT, -job.Ct);
                const float lq = fmaf(load_logit(p.draft, p.dtype, drow + v), job.invT, -job.Cd);
                if (!(lq < lp)) continue;
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)j, PURPOSE_RESIDUAL,
                                            (uint32_t)v >> 2);
                const float sc = resid_score(lp, lq, word_of(r4, v & 3));
                if (better(sc, v, best, bidx)) { best = sc; bidx = v; }
            }
            warp_argmax(best, bidx);
            job.seed_best = best;
            job.seed_idx = bidx;
        }
        if (lane == 0) {
            p.jobs[b] = job;
            const int pos = atomicAdd(&p.ctrl->job_count, 1);
            p.job_list[pos] = b;
            p.job_best[pos] = ord_of(job.seed_best);
        }
    }
    if (lane == 0) {
        p.out_status[b] = SPEC_STATUS_OK;
        p.out_accepted[b] = A;
    }
}

// =================================================================== tail_kernel
// Exact score of one entry that survived the bound (rare; kept out of line so the
// hot loop stays small).  Returns -inf when the entry has no residual mass.
struct GumbelRow {
    const char *drow;  // draft row (correction only)
    int dtype;
    bool resid;
    float invT, shift_c, Cd;
};

__device__ __noinline__ float exact_score(const GumbelRow &gr, float z, int v, uint32_t wd) {
    if (gr.resid) {
        const float lq = fmaf(load_logit(gr.drow, gr.dtype, v), gr.invT, -gr.Cd);
        if (!(lq < z)) return kNegInf;
        return resid_score(z, lq, wd);
    }
    return z + gumbel_of_word(wd);
}

// Random word of entry v when the window is not aligned to groups of four.
__device__ __noinline__ uint32_t rand_word_slow(uint64_t seed, uint32_t step, uint32_t b, uint32_t row,
                                                uint32_t purpose, int v) {
    return word_of(rand_group(seed, step, b, row, purpose, (uint32_t)v >> 2), v & 3);
}

// Raw words of group slot s (vector s / G, group s % G) of a thread's chunk data,
// and the four logits they hold.
template <class Vec>
struct GroupWords;

template <>
struct GroupWords<VecBF16> {
    static constexpr int N = 2;  // 4 bf16 = 2 words
    template <int NV>
    __device__ __forceinline__ static void get(const VecBF16 (&d)[NV], int s, uint32_t (&w)[4]) {
        uint32_t w0 = 0, w1 = 0;
#pragma unroll
        for (int t = 0; t < NV; ++t) {
            if (s == 2 * t) { w0 = d[t].v.x; w1 = d[t].v.y; }
            if (s == 2 * t + 1) { w0 = d[t].v.z; w1 = d[t].v.w; }
        }
        w[0] = w0;
        w[1] = w1;
    }
    __device__ __forceinline__ static float value(const uint32_t (&w)[4], int k) {
        return (k & 1) ? bf16_hi(w[k >> 1]) : bf16_lo(w[k >> 1]);
    }
};

template <>
struct GroupWords<VecF32> {
    static constexpr int N = 4;
    template <int NV>
    __device__ __forceinline__ static void get(const VecF32 (&d)[NV], int s, uint32_t (&w)[4]) {
        uint4 v = d[0].v;
#pragma unroll
        for (int t = 1; t < NV; ++t)
            if (s == t) v = d[t].v;
        w[0] = v.x;
        w[1] = v.y;
        w[2] = v.z;
        w[3] = v.w;
    }
    __device__ __forceinline__ static float value(const uint32_t (&w)[4], int k) { return __uint_as_float(w[k]); }
};

// Tail pass: one warp per unit of 32 lanes x kVPT vectors of a row, loaded with its
// own 16-byte loads (one extra vector per lane covers a window that does not start
// on a 16-byte boundary).
constexpr int kTailNV = kVPT + 1;
constexpr int kTailWarps = 8;
constexpr int kTailThreads = kTailWarps * 32;
constexpr int kTailBlocksPerSM = 3;
// Per-warp list of live groups in shared memory (raw words + first index).
constexpr int kLiveMax = 32 * kTailNV * 2;  // groups of four a warp can hold per unit (bf16: 2 per vector)
constexpr size_t kLiveBytesPerWarp = (size_t)kLiveMax * (2 * sizeof(uint32_t) + sizeof(int));
constexpr int kTailJobCache = 256;  // jobs whose descriptors each tail CTA keeps in shared memory

// One staged chunk of a Gumbel-max row: z = x invT - shift_c is log p (correction)
// or x / T (bonus).  Exact pruning, in order: the chunk or group bound
// z + 17 < thr (no word gives more than 16.64 of noise), then per entry
// 1 - u > 1.001 e^(z - thr) (g >= thr - z needs -log u <= e^(z - thr), and
// -log u >= 1 - u).  Each lane appends its live groups of four to the warp's
// list; the warp then draws one Philox block per listed group, 32 at a time, so
// the work follows the number of live groups rather than the busiest lane.
template <int STRIDE, class Vec, int NV>
__device__ __forceinline__ void gumbel_chunk(const Vec (&d)[NV], int64_t ebase, int ct, const GumbelRow &gr,
                                             uint64_t seed, uint32_t step, uint32_t b, uint32_t row,
                                             uint32_t purpose, float tm, float thr, unsigned char *live_buf,
                                             float &best, int &bidx) {
    // thr only ever holds an exact score of some entry (or -inf), so raising it to
    // the warp's best as exact scores come in keeps the pruning exact.
    using GW = GroupWords<Vec>;
    constexpr int G = Vec::VE / 4;  // groups of four per vector
    const int lane = ct & 31;
    uint32_t live = 0;
    if (fmaf(tm, gr.invT, -gr.shift_c) + kGumbelMax >= thr) {
#pragma unroll
        for (int t = 0; t < NV; ++t)
#pragma unroll
            for (int g = 0; g < G; ++g)
                if (fmaf(d[t].gmax(g), gr.invT, -gr.shift_c) + kGumbelMax >= thr) live |= 1u << (t * G + g);
    }
    const int cnt = __popc(live);
    int incl = cnt;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    const int total = __shfl_sync(0xffffffffu, incl, 31);
    if (total == 0) return;
    constexpr int kItems = 32 * NV * G;  // most groups one warp can list per chunk
    static_assert((size_t)kItems * (GW::N * sizeof(uint32_t) + sizeof(int)) <= kLiveBytesPerWarp,
                  "live list exceeds its per-warp region");
    uint32_t *lw = (uint32_t *)live_buf;
    int *lv0 = (int *)(live_buf + (size_t)kItems * GW::N * sizeof(uint32_t));
    const int excl = incl - cnt;
#pragma unroll
    for (int t = 0; t < NV; ++t)
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const int sl = t * G + g;
            if (!(live >> sl & 1u)) continue;
            const int pos = excl + __popc(live & ((1u << sl) - 1u));
            if (GW::N == 2) {
                lw[pos * 2] = g == 0 ? d[t].v.x : d[t].v.z;
                lw[pos * 2 + 1] = g == 0 ? d[t].v.y : d[t].v.w;
            } else {
                lw[pos * GW::N] = d[t].v.x;
                lw[pos * GW::N + 1] = d[t].v.y;
                lw[pos * GW::N + 2] = d[t].v.z;
                lw[pos * GW::N + 3] = d[t].v.w;
            }
            lv0[pos] = (int)(ebase + (int64_t)(ct + STRIDE * t) * Vec::VE + 4 * g);
        }
    __syncwarp();
    const bool aligned = (ebase & 3) == 0;
    // Each lane takes two listed groups per round: their Philox blocks are
    // independent, which keeps the scheduler busy through the 10-round chains.
#pragma unroll 1
    for (int base = 0; base < total; base += 64) {
        if (base) thr = fmaxf(thr, warp_max(best));  // later rounds prune against the best so far
        uint32_t w[2][4];
        int v0[2];
        bool has[2];
        uint4 r4[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            // (the first group of a row that starts off a 16-byte boundary has a
            // negative base index: its leading entries are masked, the rest are real)
            const int item = base + lane + 32 * h;
            has[h] = item < total;
            const int it2 = has[h] ? item : total - 1;
#pragma unroll
            for (int q = 0; q < GW::N; ++q) w[h][q] = lw[it2 * GW::N + q];
            v0[h] = lv0[it2];
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) r4[h] = rand_group(seed, step, b, row, purpose, (uint32_t)v0[h] >> 2);
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            if (!has[h]) continue;
            if (aligned) {
                // any survivor needs 1 - u_k <= e^(z_k - thr) <= e^(zmax - thr); the
                // largest w >> 9 of the group gives the smallest 1 - u
                const uint32_t kmax = max(max(r4[h].x >> 9, r4[h].y >> 9), max(r4[h].z >> 9, r4[h].w >> 9));
                float xm = GW::value(w[h], 0);
#pragma unroll
                for (int k = 1; k < 4; ++k) xm = fmaxf(xm, GW::value(w[h], k));
                const float zm = fmaf(xm, gr.invT, -gr.shift_c);
                if (!(one_minus_u01(kmax << 9) <= ex2_approx((zm - thr) * kLog2e) * 1.001f)) continue;
            }
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                const int v = v0[h] + k;
                const float z = fmaf(GW::value(w[h], k), gr.invT, -gr.shift_c);
                const uint32_t wd = aligned ? word_of(r4[h], k) : rand_word_slow(seed, step, b, row, purpose, v);
                if (one_minus_u01(wd) <= ex2_approx((z - thr) * kLog2e) * 1.001f) {
                    const float sc = exact_score(gr, z, v, wd);
                    // -inf: no residual mass at v, never a candidate (a row without any
                    // must reach the degenerate fallback)
                    if (sc > kNegInf && better(sc, v, best, bidx)) { best = sc; bidx = v; }
                }
            }
        }
    }
    __syncwarp();  // the list is rewritten by the next chunk
}

struct TailParams {
    const void *target;
    const void *draft;
    int dtype;
    int64_t ld_row;
    int Kmax, V;
    uint64_t seed;
    uint32_t step;
    const Job *jobs;
    const int *job_list;
    uint32_t *job_best;  // [jobs] ord_of(best score seen), shared across warps
    Part *parts;         // [job * units per row + unit]
    Ctrl *ctrl;
};

// Loads one unit's window straight from global memory; out-of-window entries -inf.
// Vector t of lane l holds entries ebase + (l + 32 t) VE + e.
template <class Vec, int NV>
__device__ __forceinline__ void load_unit(Vec (&d)[NV], const ChunkWin &w, int lane) {
    const int nvec = (int)(w.bytes >> 4);
    const int64_t ebase = (int64_t)w.e0 - w.shift;
#pragma unroll
    for (int t = 0; t < NV; ++t) {
        const int j = lane + 32 * t;
        d[t] = j < nvec ? Vec::load(w.a0, j) : Vec::neg_inf();
    }
    if (w.shift != 0 || ebase + (int64_t)nvec * Vec::VE != w.e1) {
#pragma unroll
        for (int t = 0; t < NV; ++t) {
            const int j = lane + 32 * t;
            if (j < nvec && (j == 0 || j == nvec - 1)) mask_vec(d[t], ebase + (int64_t)j * Vec::VE, w.e0, w.e1);
        }
    }
}

// One row per job: the correction (Gumbel-max over log(p - q)), the bonus draw
// (Gumbel-max over x / T) or the greedy argmax.  Rows are cut into units of
// 32 x kVPT vectors; every warp takes a contiguous range of units (so it loads a
// job's descriptor about once), loads them itself and writes one partial per
// unit.  The work is latency-bound, so the kernel runs many independent warps
// rather than a shared-memory ring.
template <class Vec>
__global__ void __launch_bounds__(kTailThreads, kTailBlocksPerSM) tail_kernel(TailParams p) {
    __shared__ __align__(16) unsigned char s_live[kTailWarps * kLiveBytesPerWarp];
    __shared__ Job s_jobs[kTailJobCache];
    pdl_wait();
    pdl_launch_dependents();
    constexpr int UE = 32 * kVPT * Vec::VE;  // entries per unit
    const Chunking uk = {(p.V + UE - 1) / UE, UE};
    const int njobs = p.ctrl->job_count;
    const int64_t total = (int64_t)njobs * uk.cpr;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t nw = (int64_t)gridDim.x * kTailWarps, gw = (int64_t)blockIdx.x * kTailWarps + warp;
    const int64_t rowbytes = p.ld_row * Vec::ESIZE;
    unsigned char *live_buf = s_live + kLiveBytesPerWarp * warp;
    const bool cache = njobs <= kTailJobCache;
    if (cache)
        for (int i = threadIdx.x; i < njobs; i += blockDim.x) s_jobs[i] = p.jobs[p.job_list[i]];
    __syncthreads();
    // Units are dealt round-robin: a row's units (whose cost depends on the row)
    // spread over many warps instead of piling onto a few.
    for (int64_t u = gw; u < total; u += nw) {
        const int r = (int)(u / uk.cpr);
        const Job job = cache ? s_jobs[r] : p.jobs[p.job_list[r]];
        const char *trow = (const char *)p.target + ((int64_t)job.b * (p.Kmax + 1) + job.row) * rowbytes;
        const ChunkWin w = chunk_window(trow, Vec::ESIZE, p.V, uk, (int)(u - (int64_t)r * uk.cpr));
        const uint32_t published = p.job_best[r];
        Vec d[kTailNV];
        load_unit(d, w, lane);
        const int64_t ebase = (int64_t)w.e0 - w.shift;
        const float tm = chunk_max(d);
        Part out;
        out.s = 0.f;
        if (job.kind == JOB_ARGMAX) {
            const bool any_nan = __any_sync(0xffffffffu, tm != tm);
            float mm = (tm == tm) ? tm : kNegInf;
            int ii = (tm == tm && tm > kNegInf) ? chunk_find<32>(d, ebase, lane, tm) : -1;
            warp_argmax(mm, ii);
            out.m = any_nan ? __int_as_float(0x7fc00000) : mm;
            out.idx = ii;
            out.best = 0.f;
        } else {
            const bool resid = job.kind == JOB_RESID;
            float best = resid ? job.seed_best : kNegInf;
            int bidx = resid ? job.seed_idx : -1;
            if (!resid && tm == tm && tm > kNegInf) {  // bonus: seed the bound with each lane's largest entry
                const int v = chunk_find<32>(d, ebase, lane, tm);
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)job.b, (uint32_t)job.row, PURPOSE_BONUS,
                                            (uint32_t)v >> 2);
                best = tm * job.invT + gumbel_of_word(word_of(r4, v & 3));
                bidx = v;
            }
            // bound: the best score any warp has published for this job so far
            const float thr = fmaxf(warp_max(best), float_of_ord(published));
            GumbelRow gr;
            gr.drow = (const char *)p.draft + ((int64_t)job.b * p.Kmax + job.row) * rowbytes;
            gr.dtype = p.dtype;
            gr.resid = resid;
            gr.invT = job.invT;
            gr.shift_c = resid ? job.Ct : 0.f;
            gr.Cd = job.Cd;
            gumbel_chunk<32>(d, ebase, lane, gr, p.seed, p.step, (uint32_t)job.b, (uint32_t)job.row,
                             resid ? PURPOSE_RESIDUAL : PURPOSE_BONUS, tm, thr, live_buf, best, bidx);
            out.m = warp_max_nan(tm);
            warp_argmax(best, bidx);
            out.best = best;
            out.idx = bidx;
            if (lane == 0 && bidx >= 0) atomicMax(&p.job_best[r], ord_of(best));
        }
        if (lane == 0) p.parts[u] = out;
    }
}

// =================================================================== final_kernel
struct FinalParams {
    const void *target;
    int dtype;
    int64_t ld_row;
    int Kmax, V, upr;
    uint64_t seed;
    uint32_t step;
    const Job *jobs;
    const int *job_list;
    const Part *parts;
    Ctrl *ctrl;
    int32_t *out_tokens;
    int32_t *out_accepted;
    float *out_p;
    float *out_q;
    int32_t *out_status;
};

__global__ void __launch_bounds__(kFinalThreads) final_kernel(FinalParams p) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int jb = blockIdx.x * (kFinalThreads / 32) + (threadIdx.x >> 5);
    const int njobs = p.ctrl->job_count;
    if (jb >= njobs) return;
    const Job job = p.jobs[p.job_list[jb]];
    float m = kNegInf, best = kNegInf;
    int idx = -1;
    const Part *parts = p.parts + (int64_t)jb * p.upr;
    for (int q = lane; q < p.upr; q += 32) {
        const Part pt = parts[q];
        m = max_nan_f32(m, pt.m);
        const float sc = job.kind == JOB_ARGMAX ? pt.m : pt.best;
        if (better(sc, pt.idx, best, idx)) { best = sc; idx = pt.idx; }
    }
    m = warp_max_nan(m);
    warp_argmax(best, idx);
    const int64_t K1 = p.Kmax + 1;
    int status = SPEC_STATUS_OK;
    if (p.ctrl->err) status = SPEC_STATUS_INTERNAL;
    else if (job.kind != JOB_RESID && !(fabsf(m) < __int_as_float(0x7f800000))) status = SPEC_STATUS_NONFINITE;
    if (status == SPEC_STATUS_OK && job.kind == JOB_RESID && idx < 0) {
        // p <= q everywhere (only by rounding): draw from p_j with the same noise
        const int64_t trow = ((int64_t)job.b * K1 + job.row) * p.ld_row;
        best = kNegInf;
        for (int v = lane; v < p.V; v += 32) {
            const float lp = fmaf(load_logit(p.target, p.dtype, trow + v), job.invT, -job.Ct);
            if (!(lp > kNegInf)) continue;
            const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)job.b, (uint32_t)job.row, PURPOSE_RESIDUAL,
                                        (uint32_t)v >> 2);
            const float sc = lp + gumbel_of_word(word_of(r4, v & 3));
            if (better(sc, v, best, idx)) { best = sc; idx = v; }
        }
        warp_argmax(best, idx);
    }
    if (status != SPEC_STATUS_OK) {
        for (int i = lane; i < K1; i += 32) p.out_tokens[job.b * K1 + i] = -1;
        for (int i = lane; i < p.Kmax; i += 32) {
            if (p.out_p) p.out_p[(int64_t)job.b * p.Kmax + i] = -1.f;
            if (p.out_q) p.out_q[(int64_t)job.b * p.Kmax + i] = -1.f;
        }
        if (lane == 0) {
            p.out_status[job.b] = status;
            p.out_accepted[job.b] = 0;
        }
        return;
    }
    if (lane == 0) p.out_tokens[job.b * K1 + job.row] = idx;
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

struct Layout {
    size_t off_ctrl, off_row_start, off_parts, off_jobs, off_job_list, off_job_best, off_parts2, total;
    int nseg, G, cpr, upr;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

Layout make_layout(int B, int Kmax, int V, int esz, int sms, int main_rows_per_request) {
    Layout L;
    L.G = sms;
    const Chunking ck = make_chunking(V, esz);
    L.cpr = ck.cpr;
    L.nseg = segs_per_cta((int64_t)B * main_rows_per_request * ck.cpr, L.G, ck.cpr);
    size_t o = 0;
    L.off_ctrl = o;
    o = align256(o + sizeof(Ctrl));
    L.off_row_start = o;
    o = align256(o + sizeof(int) * (size_t)(B + 1));
    L.off_parts = o;
    o = align256(o + sizeof(Part) * (size_t)L.G * L.nseg * kCW);
    L.off_jobs = o;
    o = align256(o + sizeof(Job) * (size_t)B);
    L.off_job_list = o;
    o = align256(o + sizeof(int) * (size_t)B);
    L.off_job_best = o;
    o = align256(o + sizeof(uint32_t) * (size_t)B);
    const int ue = 32 * kVPT * (16 / esz);  // entries per tail unit
    L.upr = (V + ue - 1) / ue;
    L.off_parts2 = o;
    o = align256(o + sizeof(Part) * (size_t)B * L.upr);
    L.total = o;
    return L;
}

int check_launch() {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    return SPEC_OK;
}

template <class K, class P>
int launch_pdl(K kernel, dim3 grid, dim3 block, size_t smem, cudaStream_t st, const P &params) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, kernel, params);
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    return SPEC_OK;
}

// Ring depth from the shared-memory budget left after the per-CTA tables.
int stages_for(size_t extra) {
    const size_t avail = kSmemBudget - extra - 2 * (size_t)kMaxStages * sizeof(uint64_t);
    int n = (int)(avail / kStageBytes);
    return n > kMaxStages ? kMaxStages : n;
}
size_t main_extra(int B) { return sizeof(int) * (size_t)(((B + 1) + 3) & ~3) + sizeof(MainRow) * kMaxDesc; }

template <class Vec>
int set_smem_attrs(int dev, size_t main_smem) {
    const int which = Vec::ESIZE == 2 ? 0 : 1;
    if (g_attr_set[dev][which]) return SPEC_OK;
    cudaError_t e = cudaFuncSetAttribute(main_kernel<Vec>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)main_smem);

    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    g_attr_set[dev][which] = true;
    return SPEC_OK;
}

template <class Vec>
int launch_all(int dev, const Layout &L, const MainParams &mp, const AcceptParams &ap, const TailParams &tp,
               const FinalParams &fp, cudaStream_t st) {
    int rc = set_smem_attrs<Vec>(dev, kSmemBudget);
    if (rc) return rc;
    cudaError_t e = cudaMemsetAsync(mp.ctrl, 0, sizeof(Ctrl), st);
    if (e != cudaSuccess) { t_last_cuda_error = (int)e; return SPEC_ECUDA; }
    const size_t main_smem = ring_bytes(mp.stages) + main_extra(mp.B);
    {
        ProfScope ps(st);
        main_kernel<Vec><<<L.G, kPipeThreads, main_smem, st>>>(mp);
    }
    if ((rc = check_launch())) return rc;
    {
        ProfScope ps(st);
        rc = launch_pdl(accept_kernel, dim3(mp.B), dim3(kAcceptThreads), 0, st, ap);
    }
    if (rc) return rc;
    {
        ProfScope ps(st);
        rc = launch_pdl(tail_kernel<Vec>, dim3(L.G * kTailBlocksPerSM), dim3(kTailThreads), 0, st, tp);
    }
    if (rc) return rc;
    {
        ProfScope ps(st);
        const int wpb = kFinalThreads / 32;
        rc = launch_pdl(final_kernel, dim3((mp.B + wpb - 1) / wpb), dim3(kFinalThreads), 0, st, fp);
    }
    return rc;
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
    const int esz = dtype == SPEC_BF16 ? 2 : 4;
    if (((uintptr_t)target % esz) || (draft && ((uintptr_t)draft % esz))) return SPEC_EINVAL;
    if ((int64_t)B * (2 * Kmax + 1) * (int64_t)V > ((int64_t)1 << 50)) return SPEC_EUNSUPPORTED;
    int dev = 0, sms = 0;
    int rc = device_info(&dev, &sms);
    if (rc) return rc;
    const Layout L = make_layout(B, Kmax, V, esz, sms, sample ? 2 * Kmax : Kmax);
    if (!ws) return SPEC_EWORKSPACE;
    if (ws_bytes < L.total) return SPEC_EWORKSPACE;
    rc = prof_prepare();
    if (rc) return rc;

    char *w = (char *)ws;
    Ctrl *ctrl = (Ctrl *)(w + L.off_ctrl);
    const float *temps = sample ? temperature : nullptr;

    MainParams mp;
    mp.target = target;
    mp.draft = draft;
    mp.ld_row = ld_row;
    mp.B = B;
    mp.Kmax = Kmax;
    mp.V = V;
    mp.num_draft = num_draft;
    mp.temperature = temps;
    mp.row_start = (int *)(w + L.off_row_start);
    mp.parts = (Part *)(w + L.off_parts);
    mp.nseg = L.nseg;
    mp.stages = stages_for(main_extra(B));
    mp.ctrl = ctrl;

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
    ap.temperature = temps;
    ap.seed = seed;
    ap.step = (uint32_t)step;
    ap.row_start = mp.row_start;
    ap.parts = mp.parts;
    ap.nseg = L.nseg;
    ap.G = L.G;
    ap.cpr = L.cpr;
    ap.out_tokens = out_tokens;
    ap.out_accepted = out_accepted;
    ap.out_p = sample ? out_p : nullptr;
    ap.out_q = sample ? out_q : nullptr;
    ap.out_status = out_status;
    ap.jobs = (Job *)(w + L.off_jobs);
    ap.job_list = (int *)(w + L.off_job_list);
    ap.job_best = (uint32_t *)(w + L.off_job_best);
    ap.ctrl = ctrl;

    TailParams tp;
    tp.target = target;
    tp.draft = draft;
    tp.dtype = dtype;
    tp.ld_row = ld_row;
    tp.Kmax = Kmax;
    tp.V = V;
    tp.seed = seed;
    tp.step = (uint32_t)step;
    tp.jobs = ap.jobs;
    tp.job_list = ap.job_list;
    tp.parts = (Part *)(w + L.off_parts2);
    tp.job_best = (uint32_t *)(w + L.off_job_best);
    tp.ctrl = ctrl;

    FinalParams fp;
    fp.target = target;
    fp.dtype = dtype;
    fp.ld_row = ld_row;
    fp.Kmax = Kmax;
    fp.V = V;
    fp.upr = L.upr;
    fp.seed = seed;
    fp.step = (uint32_t)step;
    fp.jobs = ap.jobs;
    fp.job_list = ap.job_list;
    fp.parts = tp.parts;
    fp.ctrl = ctrl;
    fp.out_tokens = out_tokens;
    fp.out_accepted = out_accepted;
    fp.out_p = ap.out_p;
    fp.out_q = ap.out_q;
    fp.out_status = out_status;

    cudaStream_t st = (cudaStream_t)cuda_stream;
    return dtype == SPEC_BF16 ? launch_all<VecBF16>(dev, L, mp, ap, tp, fp, st)
                              : launch_all<VecF32>(dev, L, mp, ap, tp, fp, st);
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

}  // namespace

extern "C" {

size_t spec_verify_workspace_size(int B, int Kmax, int V, int dtype) {
    if (B < 0 || Kmax < 0 || V <= 0 || (dtype != SPEC_BF16 && dtype != SPEC_F32)) return 0;
    if (B > SPEC_MAX_BATCH || Kmax > SPEC_MAX_DRAFTS) return 0;
    int dev = 0, sms = 0;
    if (device_info(&dev, &sms)) return 0;
    return make_layout(B, Kmax, V, dtype == SPEC_BF16 ? 2 : 4, sms, 2 * Kmax).total;
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
    if (make_layout(B, Kmax, V, dtype == SPEC_BF16 ? 2 : 4, sms, 2 * Kmax).total > SPEC_STATIC_SCRATCH_BYTES)
        return SPEC_ESCRATCH;
    void *ws = nullptr;
    if ((rc = static_scratch(dev, &ws))) return rc;
    return verify_impl(target, draft, dtype, B, Kmax, V, ld_row, draft_tokens, num_draft, temperature, seed,
                       step, out_tokens, out_accepted, out_p, out_q, out_status, ws, SPEC_STATIC_SCRATCH_BYTES,
                       cuda_stream, true);
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
