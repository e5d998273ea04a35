// markov.cu -- Markov-head drafting on GB300 (sm_103a).
//
// "Accelerating Large-Model Inference ... DSpark", drafting-engine table, layer 2
// (Markov head): the backbone's logits U_k of a draft block are corrected left to
// right by a low-rank bias chosen by the token already drawn at the previous
// position; "DSpark paper review" Sec. 4.1 (the head runs once per position, in
// sequence; default rank 256).  For request b and position k:
//   prev = anchor[b] (k = 0) or x_{k-1};
//   z_v  = U[b, k, v] + sum_j emb[prev, j] * proj[v, j]      (emb, proj: [V, r]);
//   x_k  = argmax_v z_v (T_b = 0), else argmax_v z_v / T_b + g_v, g_v from the
//          library's Philox stream with purpose 3 at row k.
//
// Kernels per position (2 K launches per call, no host synchronisation):
//  markov_bias_kernel    one CTA per 32 vocabulary entries: stages those entries'
//                        projection rows in shared memory once, then one warp per
//                        request computes the 32 dot products with the request's
//                        embedding row (fp32, products of the stored values exact)
//                        and writes z.  Every projection row is read once per
//                        position (from L2 after the first position: r x V x 2 B =
//                        78 MB at V = 151936, r = 256 in bf16, fits the 129 MB L2).
//  markov_sample_kernel  one CTA per request: Gumbel-max (or argmax) over z_k,
//                        status, and the token that the next position's bias uses.
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_common.cuh"
#include "spec_verify.h"

using namespace specv;

namespace {

constexpr int kMkCols = 32;        // vocabulary entries per bias CTA
constexpr int kMkThreads = 256;    // 8 warps: one request at a time each
constexpr int kMkWarps = kMkThreads / 32;
constexpr int kMkSampleThreads = 1024;

struct MarkovParams {
    const void *base;  // [B, K, ld_row] backbone logits
    const void *emb;   // [V, r]
    const void *proj;  // [V, r]
    int dtype, B, K, V, r;
    int64_t ld_row;
    const int32_t *anchor;      // [B]
    const float *temperature;   // [B] or NULL (greedy)
    uint64_t seed;
    uint32_t step;
    int32_t *tokens;  // [B, K]
    float *z;         // [B, K, V] corrected logits
    int32_t *status;  // [B]
};

__host__ __device__ inline size_t bias_smem_bytes(int r) {
    // projection tile [32][r + 4] (the +4 keeps 16-byte rows and spreads the lanes'
    // rows over the banks) and one embedding row per warp
    return sizeof(float) * ((size_t)kMkCols * (r + 4) + (size_t)kMkWarps * r);
}

__global__ void __launch_bounds__(kMkThreads) markov_bias_kernel(MarkovParams p, int k) {
    extern __shared__ __align__(16) float msm[];
    const int rs = p.r + 4;
    float *tile = msm;                         // [32][rs]
    float *hrow = msm + (size_t)kMkCols * rs;  // [8][r]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v0 = blockIdx.x * kMkCols;
    const int ncol = min(kMkCols, p.V - v0);
    // the 32 projection rows: ncol * r contiguous elements
    for (int i = tid; i < kMkCols * p.r; i += kMkThreads) {
        const int c = i / p.r, j = i - c * p.r;
        tile[c * rs + j] = c < ncol ? load_logit(p.proj, p.dtype, (int64_t)(v0 + c) * p.r + j) : 0.f;
    }
    __syncthreads();
    const int v = v0 + lane;
    const float4 *trow = reinterpret_cast<const float4 *>(tile + lane * rs);
    float *h = hrow + warp * p.r;
    for (int b = warp; b < p.B; b += kMkWarps) {
        const int prev = k == 0 ? p.anchor[b] : p.tokens[(int64_t)b * p.K + k - 1];
        const bool ok = prev >= 0 && prev < p.V;
        if (ok)
            for (int j = lane; j < p.r; j += 32) h[j] = load_logit(p.emb, p.dtype, (int64_t)prev * p.r + j);
        __syncwarp();
        float acc = 0.f;
        if (ok) {
            const float4 *h4 = reinterpret_cast<const float4 *>(h);
            for (int j4 = 0; j4 < (p.r >> 2); ++j4) {
                const float4 a = h4[j4], t = trow[j4];
                acc = fmaf(a.x, t.x, acc);
                acc = fmaf(a.y, t.y, acc);
                acc = fmaf(a.z, t.z, acc);
                acc = fmaf(a.w, t.w, acc);
            }
        }
        if (lane < ncol) {
            const int64_t row = (int64_t)b * p.K + k;
            // a request whose previous token is not a token (it failed earlier) gets NaN
            p.z[row * p.V + v] = ok ? load_logit(p.base, p.dtype, row * p.ld_row + v) + acc : __int_as_float(0x7fc00000);
        }
        __syncwarp();  // h is rewritten for the warp's next request
    }
}

// bf16 factors: the same z through bf16 tensor-core products with fp32 accumulation
// (mma.sync m16n8k16; the products of bf16 values are exact).  One CTA per 64
// vocabulary entries, all requests in chunks of 64: the chunk's embedding rows H
// [64][r] and the entries' projection rows P [64][r] sit in shared memory as bf16
// with rows padded by 8 elements (the fragment loads of a warp then hit 32
// different banks).  Warp w owns entries 8w .. 8w+7 and all four 16-request
// tiles; per 16-wide slice of r it loads one B fragment and four A fragments.
constexpr int kMmCols = 64;
constexpr int kMmReqs = 64;

__host__ __device__ inline size_t mma_smem_bytes(int r) {
    return sizeof(uint16_t) * (size_t)(kMmCols + kMmReqs) * (r + 8) + sizeof(int) * kMmReqs;
}

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

__global__ void __launch_bounds__(kMkThreads) markov_bias_mma_kernel(MarkovParams p, int k) {
    extern __shared__ __align__(16) uint16_t mms[];
    const int rs = p.r + 8;  // row stride in elements (16-byte rows)
    uint16_t *Ps = mms;                        // [64 entries][rs]
    uint16_t *Hs = mms + (size_t)kMmCols * rs;  // [64 requests][rs]
    int *okv = reinterpret_cast<int *>(Hs + (size_t)kMmReqs * rs);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int v0 = blockIdx.x * kMmCols;
    const int ncol = min(kMmCols, p.V - v0);
    const int vpr = p.r >> 3;  // 16-byte vectors per row
    for (int i = tid; i < kMmCols * vpr; i += kMkThreads) {
        const int c = i / vpr, q = i - c * vpr;
        uint4 x = make_uint4(0, 0, 0, 0);
        if (c < ncol) x = *reinterpret_cast<const uint4 *>((const uint16_t *)p.proj + (int64_t)(v0 + c) * p.r + 8 * q);
        *reinterpret_cast<uint4 *>(Ps + c * rs + 8 * q) = x;
    }
    const int g = lane >> 2, t2 = (lane & 3) * 2;
    for (int b0 = 0; b0 < p.B; b0 += kMmReqs) {
        __syncthreads();  // Hs and okv of the previous chunk are no longer read
        if (tid < kMmReqs) {
            const int b = b0 + tid;
            int ok = 0;
            if (b < p.B) {
                const int prev = k == 0 ? p.anchor[b] : p.tokens[(int64_t)b * p.K + k - 1];
                ok = (prev >= 0 && prev < p.V) ? prev + 1 : 0;  // 1 + the row to gather, 0: none
            }
            okv[tid] = ok;
        }
        __syncthreads();
        for (int i = tid; i < kMmReqs * vpr; i += kMkThreads) {
            const int m = i / vpr, q = i - m * vpr;
            const int ok = okv[m];
            uint4 x = make_uint4(0, 0, 0, 0);
            if (ok) x = *reinterpret_cast<const uint4 *>((const uint16_t *)p.emb + (int64_t)(ok - 1) * p.r + 8 * q);
            *reinterpret_cast<uint4 *>(Hs + m * rs + 8 * q) = x;
        }
        __syncthreads();
        float acc[4][4];
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[mt][e] = 0.f;
        const uint16_t *pb = Ps + (warp * 8 + g) * rs + t2;
        for (int kk = 0; kk < p.r; kk += 16) {
            uint32_t bf[2];
            bf[0] = *reinterpret_cast<const uint32_t *>(pb + kk);
            bf[1] = *reinterpret_cast<const uint32_t *>(pb + kk + 8);
#pragma unroll
            for (int mt = 0; mt < 4; ++mt) {
                const uint16_t *pa = Hs + (mt * 16 + g) * rs + kk + t2;
                uint32_t af[4];
                af[0] = *reinterpret_cast<const uint32_t *>(pa);
                af[1] = *reinterpret_cast<const uint32_t *>(pa + 8 * rs);
                af[2] = *reinterpret_cast<const uint32_t *>(pa + 8);
                af[3] = *reinterpret_cast<const uint32_t *>(pa + 8 * rs + 8);
                mma_bf16_16816(acc[mt], af, bf);
            }
        }
        // C fragment: rows (requests) g and g + 8 of each tile, entries t2, t2 + 1 of the warp's 8
#pragma unroll
        for (int mt = 0; mt < 4; ++mt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int m = mt * 16 + g + (e >= 2 ? 8 : 0);
                const int n = warp * 8 + t2 + (e & 1);
                const int b = b0 + m;
                if (b < p.B && n < ncol) {
                    const int64_t row = (int64_t)b * p.K + k;
                    const int v = v0 + n;
                    p.z[row * p.V + v] = okv[m] ? load_logit(p.base, p.dtype, row * p.ld_row + v) + acc[mt][e]
                                                : __int_as_float(0x7fc00000);
                }
            }
    }
}

// One CTA per request.  k = -1: the status of a block with no positions (K = 0).
__global__ void __launch_bounds__(kMkSampleThreads) markov_sample_kernel(MarkovParams p, int k) {
    __shared__ float red_s[kMkSampleThreads / 32];
    __shared__ int red_i[kMkSampleThreads / 32];
    const int b = blockIdx.x, tid = threadIdx.x;
    int st;
    float T = 0.f;
    if (k <= 0) {
        const int a = p.anchor[b];
        st = (a < 0 || a >= p.V) ? SPEC_STATUS_BAD_TOKEN : SPEC_STATUS_OK;
        if (st == SPEC_STATUS_OK && p.temperature) {
            T = p.temperature[b];
            if (!(T >= 0.f) || isinf(T)) st = SPEC_STATUS_BAD_TEMPERATURE;
        }
    } else {
        st = p.status[b];
        if (p.temperature) T = p.temperature[b];
    }
    if (k < 0) {
        if (tid == 0) p.status[b] = st;
        return;
    }
    float best = kNegInf;
    int bi = -1;
    bool bad = false;
    if (st == SPEC_STATUS_OK) {
        const float *zr = p.z + ((int64_t)b * p.K + k) * p.V;
        const float invT = T == 0.f ? 0.f : __fdiv_rn(1.f, T);
        // thread tid takes the groups of 4 entries tid, tid + 1024, ... (one Philox
        // block per group)
        for (int g = tid; 4 * g < p.V; g += kMkSampleThreads) {
            const uint4 r4 = T == 0.f ? make_uint4(0, 0, 0, 0)
                                      : rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)k, PURPOSE_DRAFT, (uint32_t)g);
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int v = 4 * g + e;
                if (v >= p.V) break;
                const float zv = zr[v];
                if (zv != zv || zv == __int_as_float(0x7f800000)) bad = true;
                if (!(zv > kNegInf)) continue;
                const float sc = T == 0.f ? zv : fmaf(zv, invT, gumbel_of_word(word_of(r4, e)));
                if (better(sc, v, best, bi)) {
                    best = sc;
                    bi = v;
                }
            }
        }
    }
    bad = __syncthreads_or(bad);
    warp_argmax(best, bi);
    if ((tid & 31) == 0) {
        red_s[tid >> 5] = best;
        red_i[tid >> 5] = bi;
    }
    __syncthreads();
    if (tid < 32) {
        best = red_s[tid];
        bi = red_i[tid];
        warp_argmax(best, bi);
    }
    if (tid == 0) red_i[0] = bi;
    __syncthreads();
    bi = red_i[0];
    if (st == SPEC_STATUS_OK && (bad || bi < 0)) st = SPEC_STATUS_NONFINITE;
    if (st == SPEC_STATUS_OK) {
        if (tid == 0) p.tokens[(int64_t)b * p.K + k] = bi;
    } else {
        // a failed request has every token -1 (later positions write their own)
        for (int i = tid; i <= k; i += kMkSampleThreads) p.tokens[(int64_t)b * p.K + i] = -1;
    }
    if (tid == 0) p.status[b] = st;
}

int markov_impl(const MarkovParams &p, cudaStream_t stream) {
    const size_t smem = bias_smem_bytes(p.r);
    cudaError_t e = cudaSuccess;
    if (smem > 48 * 1024) {  // ranks above 348: opt in to the larger shared memory
        e = cudaFuncSetAttribute(markov_bias_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) {
            note_cuda_error((int)e);
            return SPEC_ECUDA;
        }
    }
    // bf16 factors with 16-byte rows (r a multiple of 16, aligned bases): tensor cores
    const bool mma = p.dtype == SPEC_BF16 && (p.r % 16) == 0 && ((uintptr_t)p.emb % 16) == 0 &&
                     ((uintptr_t)p.proj % 16) == 0;
    const size_t msmem = mma_smem_bytes(p.r);
    if (mma && msmem > 48 * 1024) {
        e = cudaFuncSetAttribute(markov_bias_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)msmem);
        if (e != cudaSuccess) {
            note_cuda_error((int)e);
            return SPEC_ECUDA;
        }
    }
    if (p.K == 0) {
        markov_sample_kernel<<<p.B, kMkSampleThreads, 0, stream>>>(p, -1);
    } else {
        const int nb = (p.V + kMkCols - 1) / kMkCols, nbm = (p.V + kMmCols - 1) / kMmCols;
        for (int k = 0; k < p.K; ++k) {
            if (mma)
                markov_bias_mma_kernel<<<nbm, kMkThreads, msmem, stream>>>(p, k);
            else
                markov_bias_kernel<<<nb, kMkThreads, smem, stream>>>(p, k);
            markov_sample_kernel<<<p.B, kMkSampleThreads, 0, stream>>>(p, k);
        }
    }
    e = cudaGetLastError();
    if (e != cudaSuccess) {
        note_cuda_error((int)e);
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

}  // namespace

extern "C" int spec_markov_draft(const void *base, int dtype, int B, int K, int V, int64_t ld_row,
                                 const int32_t *anchor, const void *emb, const void *proj, int rank,
                                 const float *temperature, uint64_t seed, uint64_t step, int32_t *out_tokens,
                                 float *out_logits, int32_t *out_status, void *cuda_stream) {
    if (B < 0 || K < 0 || V <= 0 || ld_row < V || rank <= 0) return SPEC_EINVAL;
    if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_EINVAL;
    if (B == 0) return SPEC_OK;
    if (B > SPEC_MAX_BATCH || K > SPEC_MAX_DRAFTS || rank > SPEC_MARKOV_MAX_RANK || (rank & 3))
        return SPEC_EUNSUPPORTED;
    if (!anchor || !emb || !proj || !out_status) return SPEC_EINVAL;
    if (K > 0 && (!base || !out_tokens || !out_logits)) return SPEC_EINVAL;
    const int esz = dtype == SPEC_BF16 ? 2 : 4;
    if (((uintptr_t)base % esz) || ((uintptr_t)emb % esz) || ((uintptr_t)proj % esz) || ((uintptr_t)out_logits % 4))
        return SPEC_EINVAL;
    MarkovParams p;
    p.base = base;
    p.emb = emb;
    p.proj = proj;
    p.dtype = dtype;
    p.B = B;
    p.K = K;
    p.V = V;
    p.r = rank;
    p.ld_row = ld_row;
    p.anchor = anchor;
    p.temperature = temperature;
    p.seed = seed;
    p.step = (uint32_t)step;
    p.tokens = out_tokens;
    p.z = out_logits;
    p.status = out_status;
    return markov_impl(p, (cudaStream_t)cuda_stream);
}
