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
//  bias                  z for every request and entry.  bf16 factors (rank a
//                        multiple of 16): the tensor cores, markov_bias_ws_kernel
//                        (r <= 256, one CTA per SM split by role) or
//                        markov_bias_tma_kernel (two CTAs per SM); otherwise
//                        markov_bias_kernel, fp32 dot products, one CTA per 32
//                        entries.  Every projection row is read once per position.
//  markov_sample_kernel  one cluster of 4 CTAs per request, each over a quarter of
//                        the row: the pruned exact Gumbel-max (or the argmax) over
//                        z_k, status, and the token that the next position's bias
//                        uses.
// Top-K drafting: markov_topk_select_kernel (every row's candidates, one launch),
// then markov_topk_draw_kernel (the walk over the positions, a CTA per request).
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>
#include <stdint.h>

#include <mutex>
#include <type_traits>

#include "spec_common.cuh"
#include "spec_verify.h"

using namespace specv;

namespace {

constexpr int kMkCols = 32;        // vocabulary entries per bias CTA
constexpr int kMkThreads = 256;    // 8 warps: one request at a time each
constexpr int kMkWarps = kMkThreads / 32;
constexpr int kSmC = 4;           // sample pass: CTAs (one cluster) per request
constexpr int kSmThreads = 512;   // sample pass: threads per CTA
constexpr int kSmBatch = 8;       // sample pass: 4-entry groups a thread has in flight
constexpr uint64_t kWaitNs = 2000000000ull;  // bound on every mbarrier wait (2 s)

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

// fp32 (or unaligned / odd-rank bf16) factors: one CTA per 32 vocabulary entries
// stages those entries' projection rows in shared memory once, then one warp per
// request computes the 32 dot products with the request's embedding row (fp32; the
// products of the stored values are exact) and writes z.
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
// (mma.sync m16n8k16; the products of bf16 values are exact), over tiles of 64
// vocabulary entries and chunks of 64 requests.
constexpr int kMmCols = 64;
constexpr int kMmReqs = 64;

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b[0]), "r"(b[1]));
}

// bf16 factors, the same products with the projection rows streamed: a persistent
// grid (two CTAs per SM at r = 256) walks the 64-entry column tiles; for each chunk
// of 64 requests a CTA keeps their embedding rows H in shared memory (rows padded by
// 8 elements) and brings each tile's projection rows in by 8 bulk copies of 8 rows,
// block j at j (16 r + 16) bytes: the 16 bytes between blocks put rows 8 j + beta,
// j = 0 .. 7, on different banks, so that the tensor cores' B operand for the
// entries {8 j + beta} (n-block beta) loads without conflicts by ldmatrix.  Two
// tiles are in flight while a third is multiplied.  Warp w forms requests
// 32 (w / 4) .. +31 and n-blocks 2 (w % 4), 2 (w % 4) + 1 (mma.sync m16n8k16, bf16
// in, fp32 accumulate); the products then pass through shared memory (the stage just
// consumed), so that U is read and z written with 16-byte accesses along the rows;
// z = U + (emb . proj), U added after the products.  A bulk-copy wait is bounded: if
// one gives up, the CTA waits (bounded) for its copies in flight and writes NaN for
// the rest of its tiles, so those requests report status 4.
constexpr int kCtStride = 68;  // floats a row of the staged product tile (64 + 4)

__host__ __device__ inline size_t tma_stage_bytes(int r) {
    const size_t rows = (size_t)8 * (16 * (size_t)r + 16);
    const size_t ctile = sizeof(float) * (size_t)kMmReqs * kCtStride;
    return rows > ctile ? rows : ctile;
}
__host__ __device__ inline size_t tma_smem_bytes(int r) {
    return sizeof(uint16_t) * (size_t)kMmReqs * (r + 8) + 2 * tma_stage_bytes(r) + sizeof(int) * kMmReqs;
}

__device__ __forceinline__ void ldsm_x4(uint32_t (&d)[4], uint32_t addr) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(d[0]), "=r"(d[1]), "=r"(d[2]), "=r"(d[3])
                 : "r"(addr));
}

// VEC: U rows 8-byte aligned (ld_row % 4 == 0, base 8-byte aligned) and z rows
// 16-byte aligned (V % 4 == 0, z 16-byte aligned): the epilogue's vector accesses.
template <bool VEC>
__global__ void __launch_bounds__(kMkThreads, 2) markov_bias_tma_kernel(MarkovParams p, int k) {
    extern __shared__ __align__(128) unsigned char tsm[];
    __shared__ __align__(8) uint64_t s_bar[2];
    const int r = p.r, rs = r + 8;
    const size_t sb = tma_stage_bytes(r);
    const uint32_t blk = 16u * (uint32_t)r + 16u;  // bytes from one block of 8 rows to the next
    const uint32_t rowbytes = (uint32_t)r * 2u;
    uint16_t *Hs = reinterpret_cast<uint16_t *>(tsm);                // [64 requests][rs]
    unsigned char *stages = tsm + sizeof(uint16_t) * (size_t)kMmReqs * rs;  // [2][sb]
    int *okv = reinterpret_cast<int *>(stages + 2 * sb);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int mh = warp >> 2, nq = warp & 3;
    const int li = lane >> 3, l8 = lane & 7;  // ldmatrix: this lane's matrix and row
    const int g = lane >> 2, t4 = lane & 3;   // mma fragments: row group, column pair
    const int ntiles = (p.V + kMmCols - 1) / kMmCols;
    const int vpr = r >> 3;
    if (tid == 0) {
        mbar_init(&s_bar[0], 1);
        mbar_init(&s_bar[1], 1);
        mbar_init_fence();
    }
    __syncthreads();
    uint32_t used[2] = {0u, 0u};  // phases of each stage waited on so far (the same in every thread)
    bool pend[2] = {false, false};
    bool failed = false;
    for (int b0 = 0; b0 < p.B; b0 += kMmReqs) {
        // tile t into stage st: warp 0 registers the bytes, lanes 0..7 copy a block each
        auto issue = [&](int t, int st) {
            if (failed || t >= ntiles) return;
            pend[st] = true;
            if (warp != 0) return;
            const int v0 = t * kMmCols, nc = min(kMmCols, p.V - v0);
            if (lane == 0) mbar_arrive_expect_tx(&s_bar[st], (uint32_t)nc * rowbytes);
            __syncwarp();
            const int rows = min(8, nc - 8 * lane);
            if (lane < 8 && rows > 0)
                bulk_g2s(stages + (size_t)st * sb + (size_t)lane * blk,
                         (const uint16_t *)p.proj + (int64_t)(v0 + 8 * lane) * r, (uint32_t)rows * rowbytes,
                         &s_bar[st]);
        };
        // the first two tiles' copies go out before the embedding rows are gathered
        // (the stages are free: no copy is pending between chunks of requests)
        int i = 0;
        issue(blockIdx.x, 0);
        issue(blockIdx.x + gridDim.x, 1);
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
        for (int j = tid; j < kMmReqs * vpr; j += kMkThreads) {
            const int m = j / vpr, q = j - m * vpr;
            const int ok = okv[m];
            uint4 x = make_uint4(0, 0, 0, 0);
            if (ok) x = *reinterpret_cast<const uint4 *>((const uint16_t *)p.emb + (int64_t)(ok - 1) * r + 8 * q);
            *reinterpret_cast<uint4 *>(Hs + m * rs + 8 * q) = x;
        }
        __syncthreads();  // H and okv are in
        for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
            const int st = i & 1;
            unsigned char *sbase = stages + (size_t)st * sb;
            bool ok = !failed;
            if (ok) {
                if (tid == 0) ok = mbar_wait(&s_bar[st], used[st] & 1u, kWaitNs);
                ok = !__syncthreads_or(!ok);
                if (ok) mbar_try_wait(&s_bar[st], used[st] & 1u);  // every thread observes the completed phase
                used[st] += 1u;
                pend[st] = false;
                if (!ok) {
                    failed = true;
                    // the copies in flight still land: wait for them (bounded) before the
                    // CTA can leave
                    if (tid == 0) {
                        mbar_wait(&s_bar[st], (used[st] - 1u) & 1u, kWaitNs);
                        if (pend[st ^ 1]) mbar_wait(&s_bar[st ^ 1], used[st ^ 1] & 1u, kWaitNs);
                    }
                    pend[st ^ 1] = false;
                    __syncthreads();
                }
            }
            const int v0 = t * kMmCols, ncol = min(kMmCols, p.V - v0);
            // the epilogue's backbone logits, loaded before the products: request row
            // 16 pass + tid / 16, entries 4 (tid % 16) .. +3 of the tile
            const int eq = 4 * (tid & 15);
            uint2 upk[4];
#pragma unroll
            for (int ps = 0; ps < 4; ++ps) {
                const int m = 16 * ps + (tid >> 4), b = b0 + m;
                upk[ps] = make_uint2(0u, 0u);
                if (b < p.B && eq < ncol) {
                    const unsigned short *ur =
                        (const unsigned short *)p.base + ((int64_t)b * p.K + k) * p.ld_row + v0 + eq;
                    if (VEC && eq + 4 <= ncol) {
                        upk[ps] = __ldg(reinterpret_cast<const uint2 *>(ur));
                    } else {
                        uint32_t h[4];
#pragma unroll
                        for (int e = 0; e < 4; ++e) h[e] = eq + e < ncol ? (uint32_t)__ldg(ur + e) : 0u;
                        upk[ps] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
                    }
                }
            }
            float acc[2][2][4];
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int c = 0; c < 2; ++c)
#pragma unroll
                    for (int e = 0; e < 4; ++e) acc[a][c][e] = 0.f;
            if (ok) {
                const uint32_t a_addr = smem_addr(Hs + (size_t)(32 * mh + (li & 1) * 8 + l8) * rs + (li >> 1) * 8);
                const uint32_t a_step = 16u * (uint32_t)rs * 2u;  // the next 16-request tile
                const uint32_t b_addr = smem_addr(sbase) + (uint32_t)l8 * blk +
                                        (uint32_t)(2 * nq + (li >> 1)) * rowbytes + (uint32_t)(li & 1) * 16u;
                // fragments of the next 16-wide slice of r load while this one multiplies
                uint32_t fa[2][4], fb[2][4], fc[2][4];  // [buffer]: A tile 0, A tile 1, B
                auto frag = [&](int kk, uint32_t (&x)[4], uint32_t (&y)[4], uint32_t (&z)[4]) {
                    ldsm_x4(x, a_addr + 2u * kk);
                    ldsm_x4(y, a_addr + a_step + 2u * kk);
                    ldsm_x4(z, b_addr + 2u * kk);
                };
                auto mma4 = [&](const uint32_t (&x)[4], const uint32_t (&y)[4], const uint32_t (&z)[4]) {
                    const uint32_t bn0[2] = {z[0], z[1]}, bn1[2] = {z[2], z[3]};
                    mma_bf16_16816(acc[0][0], x, bn0);
                    mma_bf16_16816(acc[0][1], x, bn1);
                    mma_bf16_16816(acc[1][0], y, bn0);
                    mma_bf16_16816(acc[1][1], y, bn1);
                };
                frag(0, fa[0], fb[0], fc[0]);
                for (int kk = 0; kk < r; kk += 32) {
                    if (kk + 16 < r) frag(kk + 16, fa[1], fb[1], fc[1]);
                    mma4(fa[0], fb[0], fc[0]);
                    if (kk + 32 < r) frag(kk + 32, fa[0], fb[0], fc[0]);
                    if (kk + 16 < r) mma4(fa[1], fb[1], fc[1]);
                }
            }
            __syncthreads();  // every warp is done with the stage's rows
            // products into the stage as C [64 requests][kCtStride]: column c of n-block
            // beta is tile entry 8 c + beta
            float *Cs = reinterpret_cast<float *>(sbase);
#pragma unroll
            for (int a = 0; a < 2; ++a)
#pragma unroll
                for (int c = 0; c < 2; ++c) {
                    const int m = 32 * mh + 16 * a + g, beta = 2 * nq + c;
                    Cs[m * kCtStride + 16 * t4 + beta] = acc[a][c][0];
                    Cs[m * kCtStride + 16 * t4 + 8 + beta] = acc[a][c][1];
                    Cs[(m + 8) * kCtStride + 16 * t4 + beta] = acc[a][c][2];
                    Cs[(m + 8) * kCtStride + 16 * t4 + 8 + beta] = acc[a][c][3];
                }
            __syncthreads();
#pragma unroll
            for (int ps = 0; ps < 4; ++ps) {
                const int m = 16 * ps + (tid >> 4), b = b0 + m;
                if (b >= p.B || eq >= ncol) continue;
                const float4 cv = *reinterpret_cast<const float4 *>(Cs + m * kCtStride + eq);
                const bool good = ok && okv[m] != 0;
                const uint32_t w[2] = {upk[ps].x, upk[ps].y};
                float o[4];
                const float cc[4] = {cv.x, cv.y, cv.z, cv.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const uint32_t h = (e & 1) ? (w[e >> 1] & 0xffff0000u) : (w[e >> 1] << 16);
                    o[e] = good ? __uint_as_float(h) + cc[e] : __int_as_float(0x7fc00000);
                }
                float *zp = p.z + ((int64_t)b * p.K + k) * p.V + v0 + eq;
                if (VEC && eq + 4 <= ncol) {
                    *reinterpret_cast<float4 *>(zp) = make_float4(o[0], o[1], o[2], o[3]);
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (eq + e < ncol) zp[e] = o[e];
                }
            }
            __syncthreads();  // stage st is free
            issue(t + 2 * (int)gridDim.x, st);
        }
        // the next chunk of requests rewrites H and okv; no copy is pending here
        __syncthreads();
    }
}

// The same products with the work split by roles (one CTA per SM, 14 warps): warp 12
// issues the projection copies into kWsStages stages; warps 0..7 multiply, in two
// groups of four that take alternate tiles (warp (group, w) forms requests 32 (w / 2)
// .. +31 and n-blocks 4 (w % 2) .. +3: eight independent accumulators), and write the
// products into the group's staged tile; warps 8..11 add the backbone logits and write
// z.  The backbone logits are loaded by the write-back warps themselves three tiles
// ahead, or (TM) copied by warp 13 through a tensor map into one of two slots.  The
// roles meet on mbarriers (stage full / stage released, tile staged / tile written
// back, logits in / slot released), so the tensor cores work on the next tile while
// the previous one is written out and the tile after it is copied in.  Every wait is
// bounded; after one gives up the roles stop waiting, the tiles not multiplied are
// written as NaN (status 4), and the copies still in flight are waited for (bounded)
// before the CTA leaves.
constexpr int kWsStages = 4;
constexpr int kWsMma = 8;  // multiplying warps
constexpr int kWsEpi = 4;  // write-back warps
constexpr int kWsThreads = 32 * (kWsMma + kWsEpi + 2);  // + the copy warp, + (TM) the backbone-logit copy warp

__host__ __device__ inline size_t ws_stage_bytes(int r) { return (size_t)8 * (16 * (size_t)r + 16); }
__host__ __device__ inline size_t ws_smem_bytes(int r) {
    return sizeof(uint16_t) * (size_t)kMmReqs * (r + 8) + kWsStages * ws_stage_bytes(r) +
           2 * sizeof(float) * (size_t)kMmReqs * kCtStride + sizeof(int) * kMmReqs;
}

// TM (r a multiple of 64): each tile's projection rows arrive as r / 64 tensor-map
// copies of a 64-entry x 64-element box (8 KB), 128-byte swizzled, into 1024-byte
// aligned stages; the dynamic shared memory then carries 1 KB of alignment slack.
__host__ __device__ inline size_t ws_stage_bytes_tm(int r) { return (size_t)(r / 64) * 8192; }
// The backbone logits come the same way: a 3-D tensor map over base [B, K, ld_row],
// one box of 64 entries x 64 requests of position k a tile, into two 8 KB slots filled
// by a warp of their own.
constexpr int kUSlotBytes = 64 * 64 * 2;
__host__ __device__ inline size_t ws_smem_bytes_tm(int r) {
    return sizeof(uint16_t) * (size_t)kMmReqs * (r + 8) + 1024 + kWsStages * ws_stage_bytes_tm(r) +
           2 * (size_t)kUSlotBytes + 2 * sizeof(float) * (size_t)kMmReqs * kCtStride + sizeof(int) * kMmReqs;
}

// One 2-D tensor-map copy of box {x, y} into shared memory, completed on an mbarrier.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int x, int y, int z, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::
            "r"(smem_addr(dst)),
        "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(z), "r"(smem_addr(bar))
        : "memory");
}

__device__ __forceinline__ bool ws_failed(const int *f) { return *(volatile const int *)f != 0; }

template <bool VEC, bool TM>
__global__ void __launch_bounds__(kWsThreads, 1) markov_bias_ws_kernel(MarkovParams p, int k,
                                                                      const __grid_constant__ CUtensorMap tmap,
                                                                      const __grid_constant__ CUtensorMap umap) {
    extern __shared__ __align__(128) unsigned char wsm[];
    __shared__ __align__(8) uint64_t s_full[kWsStages], s_empty[kWsStages], s_cfull[2], s_cempty[2];
    __shared__ int s_fail;
    __shared__ uint32_t s_cons[kWsStages];  // copies of each stage the multiplying warps have waited for
    __shared__ __align__(8) uint64_t s_ufull[2], s_uempty[2];  // TM: the backbone-logit slots
    __shared__ uint32_t s_ucons[2];
    const int r = p.r, rs = r + 8;
    const size_t sb = TM ? ws_stage_bytes_tm(r) : ws_stage_bytes(r);
    const uint32_t blk = 16u * (uint32_t)r + 16u;
    const uint32_t rowbytes = (uint32_t)r * 2u;
    uint16_t *Hs = reinterpret_cast<uint16_t *>(wsm);                          // [64][rs]
    unsigned char *stages = wsm + sizeof(uint16_t) * (size_t)kMmReqs * rs;      // [kWsStages][sb]
    if (TM) stages += (1024u - (smem_addr(stages) & 1023u)) & 1023u;         // the swizzle's 1 KB atoms
    unsigned char *ubuf = stages + kWsStages * sb;                            // TM: [2][64 requests][64] bf16
    float *Cb = reinterpret_cast<float *>(ubuf + (TM ? 2 * kUSlotBytes : 0));   // [2][64][kCtStride]
    int *okv = reinterpret_cast<int *>(Cb + 2 * kMmReqs * kCtStride);
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int ntiles = (p.V + kMmCols - 1) / kMmCols;
    const int nmine = (int)blockIdx.x < ntiles ? (ntiles - 1 - (int)blockIdx.x) / (int)gridDim.x + 1 : 0;
    const int vpr = r >> 3;
    if (tid == 0) {
        for (int s2 = 0; s2 < kWsStages; ++s2) {
            mbar_init(&s_full[s2], 1);
            mbar_init(&s_empty[s2], kWsMma / 2);
            s_cons[s2] = 0u;
        }
        for (int c = 0; c < 2; ++c) {
            mbar_init(&s_cfull[c], kWsMma / 2);
            mbar_init(&s_cempty[c], kWsEpi);
            mbar_init(&s_ufull[c], 1);
            mbar_init(&s_uempty[c], kWsEpi);
            s_ucons[c] = 0u;
        }
        s_fail = 0;
        mbar_init_fence();
    }
    __syncthreads();
    uint32_t issued[kWsStages] = {};  // producer: copies issued into each stage
    uint32_t uissued[2] = {0u, 0u};   // backbone-logit copy warp (TM): copies issued into each slot
    int gi = 0;  // tiles of this CTA before the current chunk of requests (phase bookkeeping)
    for (int b0 = 0; b0 < p.B; b0 += kMmReqs) {
        // producer: one tile's copies into stage gt % kWsStages, once the multiplying
        // warps have released the stage's previous tile
        auto produce = [&](int i) {
            const int gt = gi + i, st = gt % kWsStages;
            bool ok = !ws_failed(&s_fail);
            if (ok && gt >= kWsStages && lane == 0) ok = mbar_wait(&s_empty[st], (uint32_t)((gt / kWsStages - 1) & 1), kWaitNs);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) s_fail = 1;
                return;
            }
            const int t = (int)blockIdx.x + i * (int)gridDim.x;
            const int v0 = t * kMmCols, nc = min(kMmCols, p.V - v0);
            if (TM) {
                // whole boxes (the rows past V are filled with zeros and counted)
                if (lane == 0) {
                    mbar_arrive_expect_tx(&s_full[st], (uint32_t)sb);
                    for (int c = 0; c < r / 64; ++c)
                        tma_load_2d(stages + (size_t)st * sb + (size_t)c * 8192, &tmap, 64 * c, v0, &s_full[st]);
                }
                __syncwarp();
                issued[st] += 1u;
                return;
            }
            if (lane == 0) mbar_arrive_expect_tx(&s_full[st], (uint32_t)nc * rowbytes);
            __syncwarp();
            const int rows = min(8, nc - 8 * lane);
            if (lane < 8 && rows > 0)
                bulk_g2s(stages + (size_t)st * sb + (size_t)lane * blk,
                         (const uint16_t *)p.proj + (int64_t)(v0 + 8 * lane) * r, (uint32_t)rows * rowbytes,
                         &s_full[st]);
            issued[st] += 1u;
        };
        // TM: tile i's backbone logits into slot gt % 2, once the write-back warps are
        // done with the slot's previous tile (the backbone-logit copy warp)
        auto produce_u = [&](int i) {
            const int gt = gi + i, us = gt & 1;
            bool ok = !ws_failed(&s_fail);
            if (ok && gt >= 2 && lane == 0) ok = mbar_wait(&s_uempty[us], (uint32_t)((gt / 2 - 1) & 1), kWaitNs);
            ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
            if (!ok) {
                if (lane == 0) s_fail = 1;
                return;
            }
            const int t = (int)blockIdx.x + i * (int)gridDim.x;
            if (lane == 0) {
                mbar_arrive_expect_tx(&s_ufull[us], (uint32_t)kUSlotBytes);
                tma_load_3d(ubuf + (size_t)us * kUSlotBytes, &umap, t * kMmCols, k, b0, &s_ufull[us]);
            }
            __syncwarp();
            uissued[us] += 1u;
        };
        const int first = min(nmine, kWsStages);
        if (warp == kWsMma + kWsEpi)
            for (int i = 0; i < first; ++i) produce(i);
        if (TM && warp == kWsMma + kWsEpi + 1)
            for (int i = 0; i < min(nmine, 2); ++i) produce_u(i);
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
        for (int j = tid; j < kMmReqs * vpr; j += kWsThreads) {
            const int m = j / vpr, q = j - m * vpr;
            const int ok = okv[m];
            uint4 x = make_uint4(0, 0, 0, 0);
            if (ok) x = *reinterpret_cast<const uint4 *>((const uint16_t *)p.emb + (int64_t)(ok - 1) * r + 8 * q);
            *reinterpret_cast<uint4 *>(Hs + m * rs + 8 * q) = x;
        }
        __syncthreads();  // H and okv are in
        if (warp < kWsMma) {
            // ---- multiply: warps 4 grp .. 4 grp + 3 take the tiles gt with gt % 2 == grp;
            // warp (grp, wg) forms requests 32 (wg / 2) .. +31 and n-blocks 4 (wg % 2) .. +3
            // (eight independent accumulators a warp)
            const int grp = warp >> 2, wg = warp & 3, mh = wg >> 1, nh = wg & 1;
            const int li = lane >> 3, l8 = lane & 7, g = lane >> 2, t4 = lane & 3;
            const uint32_t a_addr = smem_addr(Hs + (size_t)(32 * mh + (li & 1) * 8 + l8) * rs + (li >> 1) * 8);
            const uint32_t a_step = 16u * (uint32_t)rs * 2u;
            for (int i = (grp - gi) & 1; i < nmine; i += 2) {
                const int gt = gi + i, st = gt % kWsStages, cb = gt & 1;
                if (ws_failed(&s_fail)) break;
                if (!mbar_wait(&s_full[st], (uint32_t)((gt / kWsStages) & 1), kWaitNs)) {
                    s_fail = 1;
                    break;
                }
                if (wg == 0 && lane == 0) atomicAdd(&s_cons[st], 1u);
                float acc[2][4][4];
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int c = 0; c < 4; ++c)
#pragma unroll
                        for (int e = 0; e < 4; ++e) acc[a][c][e] = 0.f;
                // B: n-blocks 4 nh + 2 hb + (li >> 1), k half (li & 1), for hb = 0, 1.
                // Block copies: entries {8 j + beta} of n-block beta, block j at j blk.
                // Tensor copies: entries 8 beta .. 8 beta + 7 of n-block beta, box c of
                // elements 64 c .. 64 c + 63, row n at n * 128 with 16-byte chunk q stored
                // at q ^ (n % 8) (n % 8 = l8 for this lane's row)
                const uint32_t b_addr = smem_addr(stages + (size_t)st * sb) + (uint32_t)l8 * blk +
                                        (uint32_t)(4 * nh + (li >> 1)) * rowbytes + (uint32_t)(li & 1) * 16u;
                const uint32_t b_step = 2u * rowbytes;  // the next two n-blocks
                const uint32_t t_row = smem_addr(stages + (size_t)st * sb) + (uint32_t)(8 * (4 * nh + (li >> 1)) + l8) * 128u;
                uint32_t fa[2][4], fb[2][4], fc[2][4], fd[2][4];
                auto frag = [&](int kk, int q) {
                    ldsm_x4(fa[q], a_addr + 2u * kk);
                    ldsm_x4(fb[q], a_addr + a_step + 2u * kk);
                    if (TM) {
                        const uint32_t off = (uint32_t)(kk >> 6) * 8192u +
                                             ((uint32_t)((((kk & 63) >> 3) + (li & 1)) ^ l8) << 4);
                        ldsm_x4(fc[q], t_row + off);
                        ldsm_x4(fd[q], t_row + 16u * 128u + off);
                    } else {
                        ldsm_x4(fc[q], b_addr + 2u * kk);
                        ldsm_x4(fd[q], b_addr + b_step + 2u * kk);
                    }
                };
                auto mma8 = [&](int q) {
                    const uint32_t bn[4][2] = {{fc[q][0], fc[q][1]}, {fc[q][2], fc[q][3]},
                                               {fd[q][0], fd[q][1]}, {fd[q][2], fd[q][3]}};
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        mma_bf16_16816(acc[0][c], fa[q], bn[c]);
                        mma_bf16_16816(acc[1][c], fb[q], bn[c]);
                    }
                };
                frag(0, 0);
                for (int kk = 0; kk < r; kk += 32) {
                    if (kk + 16 < r) frag(kk + 16, 1);
                    mma8(0);
                    if (kk + 32 < r) frag(kk + 32, 0);
                    if (kk + 16 < r) mma8(1);
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_empty[st]);  // this warp is done with the stage
                if (gt >= 2 && !mbar_wait(&s_cempty[cb], (uint32_t)((gt / 2 - 1) & 1), kWaitNs)) {
                    s_fail = 1;
                    break;
                }
                float *Cs = Cb + (size_t)cb * kMmReqs * kCtStride;
#pragma unroll
                for (int a = 0; a < 2; ++a)
#pragma unroll
                    for (int c = 0; c < 4; ++c) {
                        const int m = 32 * mh + 16 * a + g, beta = 4 * nh + c;
                        // column j of n-block beta: entry 8 j + beta (blocks), 8 beta + j (boxes)
                        const int e0 = TM ? 8 * beta + 2 * t4 : 16 * t4 + beta;
                        const int e1 = TM ? e0 + 1 : e0 + 8;
                        Cs[m * kCtStride + e0] = acc[a][c][0];
                        Cs[m * kCtStride + e1] = acc[a][c][1];
                        Cs[(m + 8) * kCtStride + e0] = acc[a][c][2];
                        Cs[(m + 8) * kCtStride + e1] = acc[a][c][3];
                    }
                __syncwarp();
                if (lane == 0) mbar_arrive(&s_cfull[cb]);
            }
        } else if (warp < kWsMma + kWsEpi) {
            // ---- write back: 128 threads, request row 8 pass + e / 16, entries 4 (e % 16) .. +3;
            // the backbone logits load three tiles ahead of their use
            const int e = tid - 32 * kWsMma, eq = 4 * (e & 15);
            auto load_u = [&](int i, uint2 (&upk)[8]) {
                const int t = (int)blockIdx.x + i * (int)gridDim.x;
                const int v0 = t * kMmCols, ncol = min(kMmCols, p.V - v0);
#pragma unroll
                for (int ps = 0; ps < 8; ++ps) {
                    const int m = 8 * ps + (e >> 4), b = b0 + m;
                    upk[ps] = make_uint2(0u, 0u);
                    if (i < nmine && b < p.B && eq < ncol) {
                        const unsigned short *ur =
                            (const unsigned short *)p.base + ((int64_t)b * p.K + k) * p.ld_row + v0 + eq;
                        if (VEC && eq + 4 <= ncol) {
                            upk[ps] = __ldg(reinterpret_cast<const uint2 *>(ur));
                        } else {
                            uint32_t h[4];
#pragma unroll
                            for (int q = 0; q < 4; ++q) h[q] = eq + q < ncol ? (uint32_t)__ldg(ur + q) : 0u;
                            upk[ps] = make_uint2(h[0] | (h[1] << 16), h[2] | (h[3] << 16));
                        }
                    }
                }
            };
            uint2 u1[8], u2[8], u3[8];  // tiles i + 1 .. i + 3, loaded three tiles ahead
            if (!TM) {
                load_u(0, u1);
                load_u(1, u2);
                load_u(2, u3);
            }
            for (int i = 0; i < nmine; ++i) {
                const int gt = gi + i, cb = gt & 1;
                const int t = (int)blockIdx.x + i * (int)gridDim.x;
                const int v0 = t * kMmCols, ncol = min(kMmCols, p.V - v0);
                uint2 upk[8];
                const int us = gt & 1;
                bool uok = true;
                if (TM) {
                    uok = !ws_failed(&s_fail) && mbar_wait(&s_ufull[us], (uint32_t)((gt / 2) & 1), kWaitNs);
                    if (!uok) s_fail = 1;
                    if (uok && e == 0) atomicAdd(&s_ucons[us], 1u);
                    const unsigned char *ur = ubuf + (size_t)us * kUSlotBytes + 2 * eq;
#pragma unroll
                    for (int ps = 0; ps < 8; ++ps)
                        upk[ps] = uok ? *reinterpret_cast<const uint2 *>(ur + 128 * (8 * ps + (e >> 4)))
                                      : make_uint2(0u, 0u);
                } else {
#pragma unroll
                    for (int ps = 0; ps < 8; ++ps) {
                        upk[ps] = u1[ps];
                        u1[ps] = u2[ps];
                        u2[ps] = u3[ps];
                    }
                    load_u(i + 3, u3);
                }
                bool ok = uok && !ws_failed(&s_fail);
                if (ok && !mbar_wait(&s_cfull[cb], (uint32_t)((gt / 2) & 1), kWaitNs)) {
                    s_fail = 1;
                    ok = false;
                }
                const float *Cs = Cb + (size_t)cb * kMmReqs * kCtStride;
#pragma unroll
                for (int ps = 0; ps < 8; ++ps) {
                    const int m = 8 * ps + (e >> 4), b = b0 + m;
                    if (b >= p.B || eq >= ncol) continue;
                    const bool good = ok && okv[m] != 0;
                    const float4 cv = good ? *reinterpret_cast<const float4 *>(Cs + m * kCtStride + eq)
                                           : make_float4(0.f, 0.f, 0.f, 0.f);
                    const uint32_t w[2] = {upk[ps].x, upk[ps].y};
                    const float cc[4] = {cv.x, cv.y, cv.z, cv.w};
                    float o[4];
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        const uint32_t h = (q & 1) ? (w[q >> 1] & 0xffff0000u) : (w[q >> 1] << 16);
                        o[q] = good ? __uint_as_float(h) + cc[q] : __int_as_float(0x7fc00000);
                    }
                    float *zp = p.z + ((int64_t)b * p.K + k) * p.V + v0 + eq;
                    if (VEC && eq + 4 <= ncol) {
                        *reinterpret_cast<float4 *>(zp) = make_float4(o[0], o[1], o[2], o[3]);
                    } else {
#pragma unroll
                        for (int q = 0; q < 4; ++q)
                            if (eq + q < ncol) zp[q] = o[q];
                    }
                }
                __syncwarp();
                if (ok && lane == 0) mbar_arrive(&s_cempty[cb]);
                if (TM && uok && lane == 0) mbar_arrive(&s_uempty[us]);
            }
        } else if (warp == kWsMma + kWsEpi) {
            // ---- copies of the remaining tiles
            for (int i = first; i < nmine; ++i) produce(i);
        } else if (TM) {
            // ---- backbone-logit copies of the remaining tiles
            for (int i = 2; i < nmine; ++i) produce_u(i);
        }
        __syncthreads();
        // after a give-up: the copies issued but not waited for still land; wait for
        // them (bounded) before the shared memory is reused or the CTA leaves
        if (tid == 32 * (kWsMma + kWsEpi) && ws_failed(&s_fail))
            for (int s2 = 0; s2 < kWsStages; ++s2)
                for (uint32_t ph = s_cons[s2]; ph < issued[s2]; ++ph) mbar_wait(&s_full[s2], ph & 1u, kWaitNs);
        if (TM && tid == 32 * (kWsMma + kWsEpi + 1) && ws_failed(&s_fail))
            for (int s2 = 0; s2 < 2; ++s2)
                for (uint32_t ph = s_ucons[s2]; ph < uissued[s2]; ++ph) mbar_wait(&s_ufull[s2], ph & 1u, kWaitNs);
        __syncthreads();
        gi += nmine;
        if (ws_failed(&s_fail)) {
            // the rest of the requests' rows: NaN (their requests report status 4)
            for (int bb = b0 + kMmReqs; bb < p.B; ++bb)
                for (int t = (int)blockIdx.x; t < ntiles; t += (int)gridDim.x) {
                    const int v0 = t * kMmCols, ncol = min(kMmCols, p.V - v0);
                    for (int q = tid; q < ncol; q += kWsThreads)
                        p.z[((int64_t)bb * p.K + k) * p.V + v0 + q] = __int_as_float(0x7fc00000);
                }
            break;
        }
    }
}

// Status of a block with no positions (K = 0): the anchors and temperatures checked.
__global__ void markov_status_kernel(MarkovParams p) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= p.B) return;
    const int a = p.anchor[b];
    int st = (a < 0 || a >= p.V) ? SPEC_STATUS_BAD_TOKEN : SPEC_STATUS_OK;
    if (st == SPEC_STATUS_OK && p.temperature) {
        const float T = p.temperature[b];
        if (!(T >= 0.f) || isinf(T)) st = SPEC_STATUS_BAD_TEMPERATURE;
    }
    p.status[b] = st;
}

// Groups g of 4 entries of row zr (float4 loads when rows are 16-byte aligned; the
// entries past V read as -inf).
template <bool VEC>
__device__ __forceinline__ float4 load_group(const float *zr, int g, int V) {
    if constexpr (VEC) {
        return reinterpret_cast<const float4 *>(zr)[g];
    } else {
        float q[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) q[e] = 4 * g + e < V ? zr[4 * g + e] : kNegInf;
        return make_float4(q[0], q[1], q[2], q[3]);
    }
}

// CTA argmax (lowest index among equal scores) of the threads' (s, i); every thread
// gets the result.
__device__ __forceinline__ void block_argmax_sm(float &s, int &i, float *red_s, int *red_i) {
    warp_argmax(s, i);
    const int tid = threadIdx.x;
    if ((tid & 31) == 0) {
        red_s[tid >> 5] = s;
        red_i[tid >> 5] = i;
    }
    __syncthreads();
    s = red_s[0];
    i = red_i[0];
    for (int w = 1; w < kSmThreads / 32; ++w)
        if (better(red_s[w], red_i[w], s, i)) {
            s = red_s[w];
            i = red_i[w];
        }
    __syncthreads();  // red_s and red_i are reused
}

// One cluster of kSmC CTAs per request, CTA c reading the c-th contiguous share of
// the row's 4-entry groups.  The draw argmax_v z_v / T + g_v is pruned exactly (as
// the verify's draws): a group of 4 entries can only beat a known exact score thr if
// z_max / T + 17 >= thr (no word gives more than 16.64 of noise), and an entry only
// if 1 - u <= 1.001 e^(z / T - thr).  Pass 1 finds each thread's largest entry (and
// checks the row); thr starts at the best exact score of those entries over the
// whole cluster, exchanged through distributed shared memory; pass 2 draws the groups
// that can still win.  The CTAs' results meet the same way and are combined in rank
// order (lowest index among equal scores), so the token does not depend on the split.
// T = 0: pass 1 alone gives the argmax.
template <bool VEC>
__global__ void __launch_bounds__(kSmThreads, 2) markov_sample_kernel(MarkovParams p, int k) {
    __shared__ float red_s[kSmThreads / 32];
    __shared__ int red_i[kSmThreads / 32];
    __shared__ __align__(16) uint4 s_ex[2][kSmC];  // the two exchanges' slots, one per rank
    const uint32_t rank = cluster_ctarank();
    const int b = blockIdx.x / kSmC, tid = threadIdx.x;
    cluster_arrive_relaxed();
    int st;
    float T = 0.f;
    if (k == 0) {
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
    const bool greedy = T == 0.f;
    const float invT = greedy ? 0.f : __fdiv_rn(1.f, T);
    const float *zr = p.z + ((int64_t)b * p.K + k) * p.V;
    const int ng = (p.V + 3) >> 2;
    const int g_lo = (int)((int64_t)ng * rank / kSmC), g_hi = (int)((int64_t)ng * (rank + 1) / kSmC);
    constexpr int kStride = kSmBatch * kSmThreads;

    // ---- pass 1: each thread's largest entry (the lowest index among equal ones)
    float m = kNegInf;
    int mi = -1;
    bool bad = false;
    if (st == SPEC_STATUS_OK) {
        for (int g0 = g_lo + tid; g0 < g_hi; g0 += kStride) {
            float4 q[kSmBatch];
#pragma unroll
            for (int u = 0; u < kSmBatch; ++u) {
                const int g = g0 + u * kSmThreads;
                q[u] = g < g_hi ? load_group<VEC>(zr, g, p.V) : make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
            }
#pragma unroll
            for (int u = 0; u < kSmBatch; ++u) {
                const int g = g0 + u * kSmThreads;
                const float zq[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    if (zq[e] != zq[e] || zq[e] == __int_as_float(0x7f800000)) bad = true;
                    if (zq[e] > m) {
                        m = zq[e];
                        mi = 4 * g + e;
                    }
                }
            }
        }
    }
    float best = kNegInf;  // greedy: z itself; sampling: the exact score
    int bi = -1;
    if (mi >= 0) {
        bi = mi;
        if (greedy) {
            best = m;
        } else {
            const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)k, PURPOSE_DRAFT, (uint32_t)mi >> 2);
            best = fmaf(m, invT, gumbel_of_word(word_of(r4, mi & 3)));
        }
    }
    bad = __syncthreads_or(bad);
    float s1 = best;
    int i1 = bi;
    block_argmax_sm(s1, i1, red_s, red_i);
    cluster_wait();  // every CTA of the cluster is running
    if (tid == 0)
        for (uint32_t c = 0; c < kSmC; ++c)
            st_cluster_v4(&s_ex[0][rank], c, make_uint4(__float_as_uint(s1), (uint32_t)i1, bad ? 1u : 0u, 0u));
    cluster_arrive();
    cluster_wait();
    {
        const uint4 x0 = s_ex[0][0];
        s1 = __uint_as_float(x0.x);
        i1 = (int)x0.y;
        bad = x0.z != 0u;
        for (int c = 1; c < kSmC; ++c) {
            const uint4 x = s_ex[0][c];
            bad |= x.z != 0u;
            if (better(__uint_as_float(x.x), (int)x.y, s1, i1)) {
                s1 = __uint_as_float(x.x);
                i1 = (int)x.y;
            }
        }
    }

    // ---- pass 2 (sampling): the groups that can beat thr
    if (st == SPEC_STATUS_OK && !greedy && !bad && i1 >= 0) {
        float thr = s1;
        for (int g0 = g_lo + tid; g0 < g_hi; g0 += kStride) {
            float4 q[kSmBatch];
#pragma unroll
            for (int u = 0; u < kSmBatch; ++u) {
                const int g = g0 + u * kSmThreads;
                q[u] = g < g_hi ? load_group<VEC>(zr, g, p.V) : make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
            }
#pragma unroll
            for (int u = 0; u < kSmBatch; ++u) {
                const int g = g0 + u * kSmThreads;
                const float zq[4] = {q[u].x, q[u].y, q[u].z, q[u].w};
                const float zmax = fmaxf(fmaxf(zq[0], zq[1]), fmaxf(zq[2], zq[3]));
                if (!(zmax > kNegInf) || fmaf(zmax, invT, kGumbelMax) < thr) continue;
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)k, PURPOSE_DRAFT, (uint32_t)g);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int v = 4 * g + e;
                    if (v >= p.V || !(zq[e] > kNegInf)) continue;
                    const uint32_t wd = word_of(r4, e);
                    if (one_minus_u01(wd) > ex2_approx((fmaf(zq[e], invT, 0.f) - thr) * kLog2e) * 1.001f) continue;
                    const float sc = fmaf(zq[e], invT, gumbel_of_word(wd));
                    if (better(sc, v, best, bi)) {
                        best = sc;
                        bi = v;
                        thr = fmaxf(thr, sc);
                    }
                }
            }
        }
    }
    block_argmax_sm(best, bi, red_s, red_i);
    if (tid == 0)
        for (uint32_t c = 0; c < kSmC; ++c)
            st_cluster_v4(&s_ex[1][rank], c, make_uint4(__float_as_uint(best), (uint32_t)bi, 0u, 0u));
    cluster_arrive();
    cluster_wait();  // no shared memory of another CTA is touched after this
    if (rank != 0) return;
    if (greedy) {
        bi = i1;
    } else {
        best = __uint_as_float(s_ex[1][0].x);
        bi = (int)s_ex[1][0].y;
        for (int c = 1; c < kSmC; ++c) {
            const uint4 x = s_ex[1][c];
            if (better(__uint_as_float(x.x), (int)x.y, best, bi)) {
                best = __uint_as_float(x.x);
                bi = (int)x.y;
            }
        }
    }
    if (st == SPEC_STATUS_OK && (bad || bi < 0)) st = SPEC_STATUS_NONFINITE;
    if (st == SPEC_STATUS_OK) {
        if (tid == 0) p.tokens[(int64_t)b * p.K + k] = bi;
    } else {
        // a failed request has every token -1 (later positions write their own)
        for (int i = tid; i <= k; i += kSmThreads) p.tokens[(int64_t)b * p.K + i] = -1;
    }
    if (tid == 0) p.status[b] = st;
}

// ------------------------------------------------------------------ top-K drafting
// "Bringing DSpark to vLLM Metal" -- "Making the draft cheaper": correct only the
// top-K candidates of each position.  The candidates of row (b, k) are the topk
// largest backbone logits U[b, k, .] (a NaN counts as +inf, so that it is seen;
// lower v first among equal values); z_v = U + bias for them, -inf elsewhere, and
// the draw runs over them alone.  The candidates do not depend on the token drawn
// before, so all B K rows are selected at once, in parallel, before the sequential
// walk over the positions.
constexpr int kTkThreads = 512;     // selection CTA: one per row
constexpr int kTkDrawThreads = 256; // draw CTA: one per request

// Order-preserving key of a logit: NaN largest, -0 as +0 (equal values, equal keys).
__device__ __forceinline__ uint32_t topk_key(float x) {
    if (x != x) return 0xffffffffu;
    const uint32_t u = __float_as_uint(x == 0.f ? 0.f : x);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exact selection of row blockIdx.x by radix: the ncand-th largest key over four
// 8-bit digits (each pass histograms the entries whose higher digits match), then
// one pass in index order that lists the entries above that key and the
// lowest-index entries equal to it (and fills the corrected row with -inf when
// fill).  Five reads of the row: the fallback of the one-pass selection below.
template <int ESZ>
__device__ __noinline__ void topk_radix(const MarkovParams &p, int ncand, int32_t *cands, bool fill) {
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_pick[2];  // the digit, the entries above it
    __shared__ int s_scan[kTkThreads / 32];
    constexpr int VE = 16 / ESZ;  // entries a thread reads per step (consecutive)
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t row = blockIdx.x;  // b * K + k
    const char *u = (const char *)p.base + row * p.ld_row * ESZ;
    uint32_t prefix = 0u, pmask = 0u;
    int rem = ncand;
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        for (int i = tid; i < 256; i += kTkThreads) hist[i] = 0u;
        __syncthreads();
        for (int v0 = tid * VE; v0 < p.V; v0 += kTkThreads * VE) {
#pragma unroll
            for (int e = 0; e < VE; ++e) {
                const int v = v0 + e;
                if (v >= p.V) break;
                const uint32_t key = topk_key(ld_elem<ESZ>(u, v));
                if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
            }
        }
        __syncthreads();
        if (warp == 0) {
            // lane l holds bins 255 - 8 l .. 248 - 8 l; counts from the top down
            uint32_t c[8], tot = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = hist[255 - 8 * lane - i];
                tot += c[i];
            }
            uint32_t incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t above = incl - tot;  // entries in the bins above this lane's
            const bool mine = above < (uint32_t)rem && incl >= (uint32_t)rem;
            if (mine) {
                uint32_t run = above;
                for (int i = 0; i < 8; ++i) {
                    if (run + c[i] >= (uint32_t)rem) {
                        s_pick[0] = 255u - 8u * lane - i;
                        s_pick[1] = run;
                        break;
                    }
                    run += c[i];
                }
            }
        }
        __syncthreads();
        prefix |= s_pick[0] << shift;
        pmask |= 0xffu << shift;
        rem -= (int)s_pick[1];
        __syncthreads();  // s_pick is rewritten by the next pass
    }
    // prefix: the ncand-th largest key; rem: entries equal to it that are taken
    float *zrow = (fill && p.z) ? p.z + row * p.V : nullptr;
    int32_t *out = cands + row * ncand;
    int eq_base = 0, out_base = 0;
    for (int blk = 0; blk * kTkThreads * VE < p.V; ++blk) {
        const int v0 = (blk * kTkThreads + tid) * VE;
        uint32_t keys[VE];
        int neq = 0, ngt = 0;
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            const int v = v0 + e;
            keys[e] = v < p.V ? topk_key(ld_elem<ESZ>(u, v)) : 0u;
            if (v < p.V) {
                neq += keys[e] == prefix;
                ngt += keys[e] > prefix;
                if (zrow) zrow[v] = kNegInf;
            }
        }
        // exclusive scans (index order) of the equal entries and of the listed ones
        // (at most 8 each a thread: packed in one word)
        const int packed = (neq << 16) | ngt;
        int incl = packed;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, incl, o);
            if (lane >= o) incl += y;
        }
        if (lane == 31) s_scan[warp] = incl;
        __syncthreads();
        int wbase = 0, total = 0;
        for (int w = 0; w < kTkThreads / 32; ++w) {
            const int t = s_scan[w];
            if (w < warp) wbase += t;
            total += t;
        }
        __syncthreads();  // s_scan is rewritten by the next block
        const int excl = wbase + incl - packed;
        int eq_rank = eq_base + (excl >> 16);
        int gt_seen = excl & 0xffff, eq_seen = excl >> 16;
        // the position of an entry in the list: the listed entries before it
        // (above-key ones, and equal ones taken) -- equal ones are taken while
        // their rank is below rem
        int pos = out_base + gt_seen + min(eq_base + eq_seen, rem) - min(eq_base, rem);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
            const int v = v0 + e;
            if (v >= p.V) break;
            if (keys[e] > prefix) {
                out[pos++] = v;
            } else if (keys[e] == prefix) {
                if (eq_rank < rem) out[pos++] = v;
                ++eq_rank;
            }
        }
        const int beq = total >> 16, bgt = total & 0xffff;
        out_base += bgt + min(eq_base + beq, rem) - min(eq_base, rem);
        eq_base += beq;
    }
}

constexpr int kTkGather = 4096;  // entries the fast selection gathers at most
constexpr int kTkTieMax = 1024;  // entries equal to the threshold key ranked by index in the fast path

// Block (kTkThreads threads): the k-th largest of the n keys at keys (k <= n), by
// radix over four 8-bit digits; returns it, with *take = how many of the keys equal
// to it belong to the k largest.  Scratch: hist[256], pick[2].
__device__ uint32_t radix_kth(const uint32_t *keys, int n, int k, uint32_t *hist, uint32_t *pick, int *take) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t prefix = 0u, pmask = 0u;
    int rem = k;
    for (int pass = 0; pass < 4; ++pass) {
        const int sh = 24 - 8 * pass;
        for (int i = tid; i < 256; i += blockDim.x) hist[i] = 0u;
        __syncthreads();
        for (int i = tid; i < n; i += blockDim.x) {
            const uint32_t key = keys[i];
            if ((key & pmask) == prefix) atomicAdd(&hist[(key >> sh) & 255u], 1u);
        }
        __syncthreads();
        if (warp == 0) {
            uint32_t c[8], tot = 0u;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                c[i] = hist[255 - 8 * lane - i];
                tot += c[i];
            }
            uint32_t incl = tot;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t y = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += y;
            }
            const uint32_t above = incl - tot;
            if (above < (uint32_t)rem && incl >= (uint32_t)rem) {
                uint32_t run = above;
                for (int i = 0; i < 8; ++i) {
                    if (run + c[i] >= (uint32_t)rem) {
                        pick[0] = 255u - 8u * lane - i;
                        pick[1] = run;
                        break;
                    }
                    run += c[i];
                }
            }
        }
        __syncthreads();
        prefix |= pick[0] << sh;
        pmask |= 0xffu << sh;
        rem -= (int)pick[1];
        __syncthreads();
    }
    *take = rem;
    return prefix;
}

// One CTA per row (b, k).  Entry v is thread v mod kTkThreads's (neighbouring
// entries -- where a Zipf-like head puts the largest logits -- go to different
// threads).  Pass 1: each thread's largest key; the ncand-th largest of those
// maxima is a lower bound t0 of the row's ncand-th largest key (they are ncand
// distinct entries).  Pass 2: every entry with key >= t0 is gathered into shared
// memory (typically a few hundred).  The ncand-th largest key of the gathered set
// (radix) is the row's; the entries above it are listed, and those equal to it
// ranked by index.  Exact; when more than kTkGather entries pass t0 (or ncand
// exceeds the thread count, or too many tie), the row is selected again by radix
// over the whole row (topk_radix).
// VEC: rows 16-byte aligned; the passes then read 16-byte vectors (8 bf16 or 4 fp32
// entries, vector j of the row is thread j mod kTkThreads's), take each vector's
// NaN-propagating maximum, and look at single entries only in the vectors whose
// maximum reaches the bound.
template <int ESZ, bool VEC>
__global__ void __launch_bounds__(kTkThreads) markov_topk_select_kernel(MarkovParams p, int ncand, int32_t *cands) {
    __shared__ uint32_t s_key[kTkGather];
    __shared__ int s_idx[kTkGather];
    __shared__ uint32_t hist[256];
    __shared__ uint32_t s_pick[2];
    __shared__ int s_cnt[3];
    __shared__ int s_tie[kTkTieMax];
    const int tid = threadIdx.x;
    const int64_t row = blockIdx.x;
    const char *u = (const char *)p.base + row * p.ld_row * ESZ;
    if (p.z) {  // the corrected row: -inf outside the candidates (they are written later)
        float *zrow = p.z + row * p.V;
        if ((p.V & 3) == 0) {
            const float4 ni = make_float4(kNegInf, kNegInf, kNegInf, kNegInf);
            for (int i = tid; i < (p.V >> 2); i += kTkThreads) reinterpret_cast<float4 *>(zrow)[i] = ni;
        } else {
            for (int i = tid; i < p.V; i += kTkThreads) zrow[i] = kNegInf;
        }
    }
    if (ncand > kTkThreads) {
        topk_radix<ESZ>(p, ncand, cands, false);
        return;
    }
    constexpr int kU = 8;  // loads in flight per thread
    using Vv = typename std::conditional<ESZ == 2, VecBF16, VecF32>::type;
    constexpr int VE = Vv::VE;
    const int nfull = VEC ? p.V / VE : 0;  // whole vectors; the entries after them are read one by one
    uint32_t tmax = 0u;    // below every key (0 is the key of no value: NaN maps to the top)
    if (VEC) {
        float m = kNegInf;
        bool have = false;
        for (int j0 = tid; j0 < nfull; j0 += kTkThreads * kU) {
            Vv x[kU];
#pragma unroll
            for (int e = 0; e < kU; ++e) {
                const int j = j0 + e * kTkThreads;
                x[e] = j < nfull ? Vv::load(u, j) : Vv::neg_inf();
            }
#pragma unroll
            for (int e = 0; e < kU; ++e) m = max_nan_f32(m, x[e].vmax());
            have = true;
        }
        for (int v = nfull * VE + tid; v < p.V; v += kTkThreads) {
            m = max_nan_f32(m, ld_elem<ESZ>(u, v));
            have = true;
        }
        tmax = have ? topk_key(m) : 0u;
    } else {
        for (int v0 = tid; v0 < p.V; v0 += kTkThreads * kU) {
            float x[kU];
#pragma unroll
            for (int e = 0; e < kU; ++e) {
                const int v = v0 + e * kTkThreads;
                x[e] = v < p.V ? ld_elem<ESZ>(u, v) : 0.f;
            }
#pragma unroll
            for (int e = 0; e < kU; ++e)
                if (v0 + e * kTkThreads < p.V) tmax = max(tmax, topk_key(x[e]));
        }
    }
    s_key[tid] = tmax;
    if (tid == 0) {
        s_cnt[0] = 0;
        s_cnt[1] = 0;
        s_cnt[2] = 0;
    }
    int take;
    const uint32_t t0 = radix_kth(s_key, kTkThreads, ncand, hist, s_pick, &take);
    // pass 2: gather every entry at or above t0
    if (VEC) {
        // a vector can hold such an entry only if its maximum is NaN or >= the value
        // of t0 (t0 == 0: every entry; t0 the NaN key: NaN entries only)
        const uint32_t tu = (t0 & 0x80000000u) ? (t0 & 0x7fffffffu) : ~t0;
        const float tv = __uint_as_float(tu);
        auto keep = [&](float x, int v) {
            const uint32_t key = topk_key(x);
            if (key >= t0) {
                const int slot = atomicAdd(&s_cnt[0], 1);
                if (slot < kTkGather) {
                    s_key[slot] = key;
                    s_idx[slot] = v;
                }
            }
        };
        for (int j0 = tid; j0 < nfull; j0 += kTkThreads * kU) {
            Vv x[kU];
#pragma unroll
            for (int e = 0; e < kU; ++e) {
                const int j = j0 + e * kTkThreads;
                x[e] = j < nfull ? Vv::load(u, j) : Vv::neg_inf();
            }
#pragma unroll
            for (int e = 0; e < kU; ++e) {
                const int j = j0 + e * kTkThreads;
                const float vm = x[e].vmax();
                const bool maybe = t0 == 0u || vm != vm || (t0 != 0xffffffffu && vm >= tv);
                if (j < nfull && maybe)
                    for (int q = 0; q < VE; ++q) keep(x[e].get(q), j * VE + q);
            }
        }
        for (int v = nfull * VE + tid; v < p.V; v += kTkThreads) keep(ld_elem<ESZ>(u, v), v);
    }
    const int lane = tid & 31;
    for (int w0 = tid - lane; !VEC && w0 < p.V; w0 += kTkThreads * kU) {
        const int v0 = w0 + lane;
        float x[kU];
#pragma unroll
        for (int e = 0; e < kU; ++e) {
            const int v = v0 + e * kTkThreads;
            x[e] = v < p.V ? ld_elem<ESZ>(u, v) : 0.f;
        }
#pragma unroll
        for (int e = 0; e < kU; ++e) {
            const int v = v0 + e * kTkThreads;
            const uint32_t key = v < p.V ? topk_key(x[e]) : 0u;
            const bool in = v < p.V && key >= t0;
            const unsigned bal = __ballot_sync(0xffffffffu, in);
            if (bal) {
                int base = 0;
                if (lane == 0) base = atomicAdd(&s_cnt[0], __popc(bal));
                base = __shfl_sync(0xffffffffu, base, 0);
                const int slot = base + __popc(bal & ((1u << lane) - 1u));
                if (in && slot < kTkGather) {
                    s_key[slot] = key;
                    s_idx[slot] = v;
                }
            }
        }
    }
    __syncthreads();
    const int ng = s_cnt[0];
    if (ng > kTkGather) {
        topk_radix<ESZ>(p, ncand, cands, false);
        return;
    }
    // the row's ncand-th largest key: that of the gathered set, which holds every
    // entry at or above t0 <= it
    int rem;
    const uint32_t thr = radix_kth(s_key, ng, ncand, hist, s_pick, &rem);
    int32_t *out = cands + row * ncand;
    for (int i = tid; i < ng; i += kTkThreads) {
        if (s_key[i] > thr) {
            out[atomicAdd(&s_cnt[1], 1)] = s_idx[i];
        } else if (s_key[i] == thr) {
            const int slot = atomicAdd(&s_cnt[2], 1);
            if (slot < kTkTieMax) s_tie[slot] = s_idx[i];
        }
    }
    __syncthreads();
    const int ne = s_cnt[2];
    if (ne > kTkTieMax) {
        topk_radix<ESZ>(p, ncand, cands, false);
        return;
    }
    // the equal entries ranked by index (bitonic sort of at most kTkTieMax)
    int n2 = 1;
    while (n2 < ne) n2 <<= 1;
    for (int i = ne + tid; i < n2; i += kTkThreads) s_tie[i] = 0x7fffffff;
    __syncthreads();
    for (int k2 = 2; k2 <= n2; k2 <<= 1)
        for (int jj = k2 >> 1; jj > 0; jj >>= 1) {
            for (int i = tid; i < n2; i += kTkThreads) {
                const int x = i ^ jj;
                if (x > i) {
                    const int a = s_tie[i], c = s_tie[x];
                    const bool up = (i & k2) == 0;
                    if (up ? (a > c) : (a < c)) {
                        s_tie[i] = c;
                        s_tie[x] = a;
                    }
                }
            }
            __syncthreads();
        }
    const int base = ncand - rem;
    for (int i = tid; i < rem; i += kTkThreads) out[base + i] = s_tie[i];
}

// One CTA per request: the positions in order; at position k the bias of each of
// the row's ncand candidates (four threads a candidate, fp32), then the draw over
// them.  The loads a position needs that do not depend on the token drawn before it
// (its candidates' projection rows and backbone logits) go out together with the
// one that does (the embedding row of that token), so that a position waits for
// one round of loads.  FAST (bf16, r a multiple of 32, 16-byte aligned factor rows):
// a candidate's four threads each hold every fourth 16-byte vector of its
// projection row in registers; the candidate indices of the next position are read
// while this one is drawn.
template <int ESZ, bool FAST>
__global__ void __launch_bounds__(kTkDrawThreads) markov_topk_draw_kernel(MarkovParams p, int ncand,
                                                                       const int32_t *cands) {
    __shared__ float s_h[SPEC_MARKOV_MAX_RANK];
    __shared__ float s_z[SPEC_MARKOV_MAX_TOPK];
    __shared__ float red_s[kTkDrawThreads / 32];
    __shared__ int red_i[kTkDrawThreads / 32];
    __shared__ int s_tok;
    constexpr int kPV = SPEC_MARKOV_MAX_RANK / 32;  // FAST: vectors a thread holds (r / 32 used)
    const int b = blockIdx.x, tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NW = kTkDrawThreads / 32;
    int prev = p.anchor[b];
    int st = (prev < 0 || prev >= p.V) ? SPEC_STATUS_BAD_TOKEN : SPEC_STATUS_OK;
    float T = 0.f;
    if (st == SPEC_STATUS_OK && p.temperature) {
        T = p.temperature[b];
        if (!(T >= 0.f) || isinf(T)) st = SPEC_STATUS_BAD_TEMPERATURE;
    }
    const float invT = T == 0.f ? 0.f : __fdiv_rn(1.f, T);
    const int part = tid & 3, nv = p.r >> 5;  // FAST: this thread's vectors part, part + 4, ... (nv of them)
    int vnext = (FAST && (tid >> 2) < ncand && p.K > 0) ? cands[(int64_t)b * p.K * ncand + (tid >> 2)] : 0;
    for (int k = 0; k < p.K && st == SPEC_STATUS_OK; ++k) {
        const int64_t row = (int64_t)b * p.K + k;
        const int32_t *cl = cands + row * ncand;
        const char *u = (const char *)p.base + row * p.ld_row * ESZ;
        if (FAST) {
            // round 0's candidate (the most common case: ncand <= kTkDrawThreads / 4):
            // its projection vectors and backbone logit load with the embedding row
            const int ci0 = tid >> 2;
            const int v0 = vnext;
            uint4 pv[kPV];
            float u0 = 0.f;
            if (ci0 < ncand) {
                const uint4 *pr = reinterpret_cast<const uint4 *>((const uint16_t *)p.proj + (int64_t)v0 * p.r);
#pragma unroll
                for (int i = 0; i < kPV; ++i)
                    if (i < nv) pv[i] = __ldg(pr + part + 4 * i);
                if (part == 0) u0 = ld_elem<ESZ>(u, v0);
            }
            for (int j = tid; j < p.r; j += kTkDrawThreads) s_h[j] = ld_elem<ESZ>(p.emb, (int64_t)prev * p.r + j);
            __syncthreads();
            for (int c0 = 0; c0 < ncand; c0 += kTkDrawThreads / 4) {
                const int ci = c0 + (tid >> 2);
                int v = v0;
                if (c0 > 0 && ci < ncand) {
                    v = cl[ci];
                    const uint4 *pr = reinterpret_cast<const uint4 *>((const uint16_t *)p.proj + (int64_t)v * p.r);
#pragma unroll
                    for (int i = 0; i < kPV; ++i)
                        if (i < nv) pv[i] = __ldg(pr + part + 4 * i);
                    if (part == 0) u0 = ld_elem<ESZ>(u, v);
                }
                float acc = 0.f;
                if (ci < ncand) {
#pragma unroll
                    for (int i = 0; i < kPV; ++i) {
                        if (i >= nv) break;
                        const float *h = s_h + 8 * (part + 4 * i);
                        const uint32_t w[4] = {pv[i].x, pv[i].y, pv[i].z, pv[i].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            acc = fmaf(h[2 * e], bf16_lo(w[e]), acc);
                            acc = fmaf(h[2 * e + 1], bf16_hi(w[e]), acc);
                        }
                    }
                }
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                if (ci < ncand && part == 0) {
                    const float z = u0 + acc;
                    s_z[ci] = z;
                    if (p.z) p.z[row * p.V + v] = z;
                }
            }
            // the next position's first candidates, read while this one is drawn
            if (k + 1 < p.K && ci0 < ncand) vnext = cl[(int64_t)ncand + ci0];
        } else {
            for (int j = tid; j < p.r; j += kTkDrawThreads) s_h[j] = ld_elem<ESZ>(p.emb, (int64_t)prev * p.r + j);
            __syncthreads();
            // four threads a candidate, each a quarter of the rank (interleaved), the
            // loads unrolled so that they are in flight together
            for (int c0 = 0; c0 < ncand; c0 += kTkDrawThreads / 4) {
                const int ci = c0 + (tid >> 2);
                float acc = 0.f;
                int v = 0;
                if (ci < ncand) {
                    v = cl[ci];
                    const char *pr = (const char *)p.proj + (int64_t)v * p.r * ESZ;
#pragma unroll 8
                    for (int j = part; j < p.r; j += 4) acc = fmaf(s_h[j], ld_elem<ESZ>(pr, j), acc);
                }
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                if (ci < ncand && part == 0) {
                    const float z = ld_elem<ESZ>(u, v) + acc;
                    s_z[ci] = z;
                    if (p.z) p.z[row * p.V + v] = z;
                }
            }
        }
        __syncthreads();
        float best = kNegInf;
        int bi = -1;
        bool bad = false;
        for (int ci = tid; ci < ncand; ci += kTkDrawThreads) {
            const int v = cl[ci];
            const float z = s_z[ci];
            if (z != z || z == __int_as_float(0x7f800000)) bad = true;
            if (!(z > kNegInf)) continue;
            float sc = z;
            if (T != 0.f) {
                const uint4 r4 = rand_group(p.seed, p.step, (uint32_t)b, (uint32_t)k, PURPOSE_DRAFT, (uint32_t)v >> 2);
                sc = fmaf(z, invT, gumbel_of_word(word_of(r4, v & 3)));
            }
            if (better(sc, v, best, bi)) {
                best = sc;
                bi = v;
            }
        }
        bad = __syncthreads_or(bad);
        warp_argmax(best, bi);
        if (lane == 0) {
            red_s[warp] = best;
            red_i[warp] = bi;
        }
        __syncthreads();
        if (tid == 0) {
            float bs = red_s[0];
            int bx = red_i[0];
            for (int w = 1; w < NW; ++w)
                if (better(red_s[w], red_i[w], bs, bx)) {
                    bs = red_s[w];
                    bx = red_i[w];
                }
            s_tok = bx;
        }
        __syncthreads();
        prev = s_tok;
        if (bad || prev < 0) st = SPEC_STATUS_NONFINITE;
        else if (tid == 0) p.tokens[row] = prev;
        __syncthreads();  // s_h, s_z and s_tok are rewritten at the next position
    }
    if (st != SPEC_STATUS_OK)
        for (int i = tid; i < p.K; i += kTkDrawThreads) p.tokens[(int64_t)b * p.K + i] = -1;
    if (tid == 0) p.status[b] = st;
}

// The sample pass of position k: one cluster of kSmC CTAs per request.
cudaError_t launch_sample(const MarkovParams &p, int k, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(p.B * kSmC));
    cfg.blockDim = dim3(kSmThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kSmC;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return (p.V & 3) == 0 ? cudaLaunchKernelEx(&cfg, markov_sample_kernel<true>, p, k)
                          : cudaLaunchKernelEx(&cfg, markov_sample_kernel<false>, p, k);
}

int markov_topk_impl(const MarkovParams &p, int ncand, int32_t *cands, cudaStream_t stream) {
    const int esz = p.dtype == SPEC_BF16 ? 2 : 4;
    const bool tvec = ((uintptr_t)p.base % 16) == 0 && ((p.ld_row * esz) % 16) == 0;
    if (p.K == 0) {
        markov_status_kernel<<<(p.B + 255) / 256, 256, 0, stream>>>(p);
    } else if (p.dtype == SPEC_BF16) {
        if (tvec)
            markov_topk_select_kernel<2, true><<<p.B * p.K, kTkThreads, 0, stream>>>(p, ncand, cands);
        else
            markov_topk_select_kernel<2, false><<<p.B * p.K, kTkThreads, 0, stream>>>(p, ncand, cands);
        const bool fast = (p.r % 32) == 0 && ((uintptr_t)p.proj % 16) == 0;
        if (fast)
            markov_topk_draw_kernel<2, true><<<p.B, kTkDrawThreads, 0, stream>>>(p, ncand, cands);
        else
            markov_topk_draw_kernel<2, false><<<p.B, kTkDrawThreads, 0, stream>>>(p, ncand, cands);
    } else {
        if (tvec)
            markov_topk_select_kernel<4, true><<<p.B * p.K, kTkThreads, 0, stream>>>(p, ncand, cands);
        else
            markov_topk_select_kernel<4, false><<<p.B * p.K, kTkThreads, 0, stream>>>(p, ncand, cands);
        markov_topk_draw_kernel<4, false><<<p.B, kTkDrawThreads, 0, stream>>>(p, ncand, cands);
    }
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        note_cuda_error((int)e);
        return SPEC_ECUDA;
    }
    return SPEC_OK;
}

// Per device, set up once: the bias kernels' shared-memory limits (what the largest
// rank each one serves needs) and the SM count; per rank, the occupancy of the two-CTA
// bias kernel, queried the first time that rank is drawn.
struct MarkovDevice {
    bool ready = false;
    int sms = 0;
    int per[SPEC_MARKOV_MAX_RANK / 16 + 1];  // CTAs per SM of markov_bias_tma_kernel by r / 16; -1: not yet known
};
std::mutex g_mk_mu;
MarkovDevice g_mk[64];

int markov_device(int r, int *sms, int *per) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess && (dev < 0 || dev >= 64)) return SPEC_EUNSUPPORTED;
    std::lock_guard<std::mutex> lk(g_mk_mu);
    MarkovDevice &d = g_mk[dev];
    if (e == cudaSuccess && !d.ready) {
        e = cudaFuncSetAttribute(markov_bias_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bias_smem_bytes(SPEC_MARKOV_MAX_RANK));
        const int tmax = (int)tma_smem_bytes(SPEC_MARKOV_MAX_RANK), wmax = (int)ws_smem_bytes(256);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(markov_bias_tma_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, tmax);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(markov_bias_tma_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, tmax);
        const int wtm = (int)ws_smem_bytes_tm(256);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(markov_bias_ws_kernel<true, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     wmax);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(markov_bias_ws_kernel<false, false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     wmax);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(markov_bias_ws_kernel<true, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, wtm);
        if (e == cudaSuccess)
            e = cudaFuncSetAttribute(markov_bias_ws_kernel<false, true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     wtm);
        if (e == cudaSuccess) e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev);
        if (e == cudaSuccess) {
            for (int &x : d.per) x = -1;
            d.ready = true;
        }
    }
    if (e == cudaSuccess && (r % 16) == 0 && d.per[r / 16] < 0) {
        int n = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, markov_bias_tma_kernel<true>, kMkThreads,
                                                          tma_smem_bytes(r));
        if (e == cudaSuccess) d.per[r / 16] = n;
    }
    if (e != cudaSuccess) {
        note_cuda_error((int)e);
        return SPEC_ECUDA;
    }
    *sms = d.sms;
    *per = (r % 16) == 0 ? d.per[r / 16] : 0;
    return SPEC_OK;
}

// The driver's tensor-map encoder, looked up once (null if the driver has none).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        cudaGetLastError();
    });
    return fn;
}

// The projection rows [V, r] (bf16, r a multiple of 64) as a 2-D tensor map of
// 64 x 64 boxes, 128-byte swizzled; false if it cannot be made.
bool proj_tensor_map(const MarkovParams &p, CUtensorMap *map) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || (p.r % 64) != 0 || ((uintptr_t)p.proj % 16) != 0) return false;
    const cuuint64_t dims[2] = {(cuuint64_t)p.r, (cuuint64_t)p.V};
    const cuuint64_t strides[1] = {(cuuint64_t)p.r * 2};
    const cuuint32_t box[2] = {64, 64};
    const cuuint32_t estr[2] = {1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(p.proj), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The backbone logits [B, K, ld_row] (bf16) as a 3-D tensor map {V, K, B} of
// 64 x 1 x 64 boxes (a tile's entries of one position for a chunk of requests); false
// if it cannot be made (rows not 16-byte aligned).
bool base_tensor_map(const MarkovParams &p, CUtensorMap *map) {
    const PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || (p.ld_row % 8) != 0 || ((uintptr_t)p.base % 16) != 0) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)p.V, (cuuint64_t)p.K, (cuuint64_t)p.B};
    const cuuint64_t strides[2] = {(cuuint64_t)p.ld_row * 2, (cuuint64_t)p.ld_row * 2 * (cuuint64_t)p.K};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(p.base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int markov_impl(const MarkovParams &p, cudaStream_t stream) {
    int sms = 0, per = 0;
    const int rc = markov_device(p.r, &sms, &per);
    if (rc) return rc;
    cudaError_t e = cudaSuccess;
    const size_t smem = bias_smem_bytes(p.r);
    // bf16 factors with 16-byte rows (r a multiple of 16, aligned bases): tensor cores,
    // the role-split kernel where its stages and two staged tiles fit (r <= 256), else
    // the two-CTA kernel; vector accesses in the epilogue where U and z rows allow them
    const bool mma = p.dtype == SPEC_BF16 && (p.r % 16) == 0 && ((uintptr_t)p.emb % 16) == 0 &&
                     ((uintptr_t)p.proj % 16) == 0;
    const bool tvec = (p.ld_row % 4) == 0 && ((uintptr_t)p.base % 8) == 0 && (p.V % 4) == 0 &&
                      ((uintptr_t)p.z % 16) == 0;
    const int ntiles = (p.V + kMmCols - 1) / kMmCols;
    const size_t tsmem = tma_smem_bytes(p.r), wsmem = ws_smem_bytes(p.r);
    const int tgrid = mma && per > 0 ? min(ntiles, per * sms) : 0;
    const int wgrid = mma && p.r <= 256 ? min(ntiles, sms) : 0;
    alignas(64) CUtensorMap tmap = {}, umap = {};
    const bool tm = wgrid > 0 && p.K > 0 && proj_tensor_map(p, &tmap) && base_tensor_map(p, &umap);
    const size_t wsmem_tm = ws_smem_bytes_tm(p.r);
    if (p.K == 0) {
        markov_status_kernel<<<(p.B + 255) / 256, 256, 0, stream>>>(p);
    } else {
        const int nb = (p.V + kMkCols - 1) / kMkCols;
        for (int k = 0; k < p.K; ++k) {
            if (tm && tvec)
                markov_bias_ws_kernel<true, true><<<wgrid, kWsThreads, wsmem_tm, stream>>>(p, k, tmap, umap);
            else if (tm)
                markov_bias_ws_kernel<false, true><<<wgrid, kWsThreads, wsmem_tm, stream>>>(p, k, tmap, umap);
            else if (wgrid > 0 && tvec)
                markov_bias_ws_kernel<true, false><<<wgrid, kWsThreads, wsmem, stream>>>(p, k, tmap, umap);
            else if (wgrid > 0)
                markov_bias_ws_kernel<false, false><<<wgrid, kWsThreads, wsmem, stream>>>(p, k, tmap, umap);
            else if (mma && tgrid > 0 && tvec)
                markov_bias_tma_kernel<true><<<tgrid, kMkThreads, tsmem, stream>>>(p, k);
            else if (mma && tgrid > 0)
                markov_bias_tma_kernel<false><<<tgrid, kMkThreads, tsmem, stream>>>(p, k);
            else
                markov_bias_kernel<<<nb, kMkThreads, smem, stream>>>(p, k);
            e = launch_sample(p, k, stream);
            if (e != cudaSuccess) {
                note_cuda_error((int)e);
                return SPEC_ECUDA;
            }
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

extern "C" size_t spec_markov_topk_workspace_size(int B, int K, int V, int topk) {
    if (B < 0 || K < 0 || V <= 0 || topk <= 0 || topk > SPEC_MARKOV_MAX_TOPK) return 0;
    const size_t ncand = (size_t)(topk < V ? topk : V);
    return (sizeof(int32_t) * (size_t)B * (size_t)K * ncand + 255) & ~(size_t)255;
}

extern "C" int spec_markov_draft_topk(const void *base, int dtype, int B, int K, int V, int64_t ld_row,
                                      const int32_t *anchor, const void *emb, const void *proj, int rank,
                                      const float *temperature, uint64_t seed, uint64_t step, int topk,
                                      int32_t *out_tokens, float *out_logits, int32_t *out_status, void *ws,
                                      size_t ws_bytes, void *cuda_stream) {
    if (B < 0 || K < 0 || V <= 0 || ld_row < V || rank <= 0 || topk <= 0) return SPEC_EINVAL;
    if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_EINVAL;
    if (B == 0) return SPEC_OK;
    if (B > SPEC_MAX_BATCH || K > SPEC_MAX_DRAFTS || rank > SPEC_MARKOV_MAX_RANK || (rank & 3) ||
        topk > SPEC_MARKOV_MAX_TOPK)
        return SPEC_EUNSUPPORTED;
    if ((int64_t)B * K >= ((int64_t)1 << 31)) return SPEC_EUNSUPPORTED;
    if (!anchor || !emb || !proj || !out_status) return SPEC_EINVAL;
    if (K > 0 && (!base || !out_tokens)) return SPEC_EINVAL;
    const int esz = dtype == SPEC_BF16 ? 2 : 4;
    if (((uintptr_t)base % esz) || ((uintptr_t)emb % esz) || ((uintptr_t)proj % esz) || ((uintptr_t)out_logits % 4))
        return SPEC_EINVAL;
    const size_t need = spec_markov_topk_workspace_size(B, K, V, topk);
    if (K > 0 && (!ws || ws_bytes < need || ((uintptr_t)ws & 15))) return SPEC_EWORKSPACE;
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
    return markov_topk_impl(p, topk < V ? topk : V, (int32_t *)ws, (cudaStream_t)cuda_stream);
}
