// spec_common.cuh -- device building blocks of the verify/commit kernels (sm_103a).
//
// Counter-based RNG: Philox4x32-10 as defined by Salmon, Moraes, Dror and Shaw,
// "Parallel random numbers: as easy as 1, 2, 3" (SC'11): ten rounds of the 4x32
// S-box with multipliers 0xD2511F53 / 0xCD9E8D57 and the Weyl key increments
// 0x9E3779B9 / 0xBB67AE85.  Stream layout of this library: key = (seed lo, seed hi),
// counter = (v >> 2, b, (row << 4) | purpose, step lo), word v & 3.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace specv {

constexpr float kLog2e = 1.4426950408889634f;
constexpr float kNegInf = -__builtin_huge_valf();
// Largest Gumbel noise a 32-bit word can give is -ln(-ln(1 - 2^-24)) = 16.64; pruning
// bounds use 17 so that rounding can never make a pruned element win.
constexpr float kGumbelMax = 17.0f;

enum Purpose : uint32_t { PURPOSE_ACCEPT = 0, PURPOSE_RESIDUAL = 1, PURPOSE_BONUS = 2, PURPOSE_DRAFT = 3 };

// Records the CUDA error that spec_last_cuda_error() reports (host; defined in verify.cu).
void note_cuda_error(int e);

// ------------------------------------------------------------------ Philox
__device__ __forceinline__ uint4 philox4x32_10(uint4 x, uint32_t k0, uint32_t k1) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
        // one 32x32 -> 64-bit product per multiplier gives both halves
        const uint64_t pa = (uint64_t)x.x * 0xD2511F53u;
        const uint64_t pc = (uint64_t)x.z * 0xCD9E8D57u;
        x = make_uint4((uint32_t)(pc >> 32) ^ x.y ^ k0, (uint32_t)pc, (uint32_t)(pa >> 32) ^ x.w ^ k1, (uint32_t)pa);
        k0 += 0x9E3779B9u;
        k1 += 0xBB67AE85u;
    }
    return x;
}

// The four words of the group holding vocabulary entries 4*grp .. 4*grp+3.
__device__ __forceinline__ uint4 rand_group(uint64_t seed, uint32_t step, uint32_t b, uint32_t row,
                                            uint32_t purpose, uint32_t grp) {
    return philox4x32_10(make_uint4(grp, b, (row << 4) | purpose, step), (uint32_t)seed,
                         (uint32_t)(seed >> 32));
}

__device__ __forceinline__ uint32_t word_of(const uint4 &r, int k) {
    return k == 0 ? r.x : (k == 1 ? r.y : (k == 2 ? r.z : r.w));
}

// u = (2 (w >> 9) + 1) 2^-24, exact in fp32; and 1 - u, also exact.
__device__ __forceinline__ float u01(uint32_t w) {
    return __uint2float_rn(((w >> 9) << 1) | 1u) * 5.9604644775390625e-8f;
}
__device__ __forceinline__ float one_minus_u01(uint32_t w) {
    return __uint2float_rn(((0x7FFFFFu - (w >> 9)) << 1) | 1u) * 5.9604644775390625e-8f;
}

// Gumbel noise g = -log(-log u) from the word, accurate for u near 1 (where the
// winners of a Gumbel-max draw come from): -log u = -log1p(-(1 - u)) with 1 - u exact.
static __device__ __noinline__ float gumbel_of_word(uint32_t w) {
    const float e = -log1pf(-one_minus_u01(w));
    return -logf(e);
}

// ------------------------------------------------------------------ loads
__device__ __forceinline__ uint4 ld_stream_v4(const void *p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "l"(p));
    return r;
}

__device__ __forceinline__ uint32_t max_nan_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// max of two bf16 pairs; a NaN lane yields the other operand
__device__ __forceinline__ uint32_t max_bf16x2(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ float max_nan_f32(float a, float b) {
    float d;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(d) : "f"(a), "f"(b));
    return d;
}

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// ------------------------------------------------------------------ vector views
// A "vector" is 16 bytes of a row: 8 bf16 or 4 fp32 logits.
struct VecBF16 {
    static constexpr int VE = 8;
    static constexpr int ESIZE = 2;
    uint4 v;
    __device__ __forceinline__ static VecBF16 load(const void *row, int64_t vi) {
        return {ld_stream_v4((const uint4 *)row + vi)};
    }
    __device__ __forceinline__ static VecBF16 neg_inf() {
        return {make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)};
    }
    __device__ __forceinline__ float get(int e) const {
        const uint32_t w = (e >> 1) == 0 ? v.x : ((e >> 1) == 1 ? v.y : ((e >> 1) == 2 ? v.z : v.w));
        return (e & 1) ? bf16_hi(w) : bf16_lo(w);
    }
    __device__ __forceinline__ float vmax() const {
        const uint32_t m = max_nan_bf16x2(max_nan_bf16x2(v.x, v.y), max_nan_bf16x2(v.z, v.w));
        return max_nan_f32(bf16_lo(m), bf16_hi(m));
    }
    // max over elements 4g .. 4g+3
    __device__ __forceinline__ float gmax(int g) const {
        const uint32_t m = g == 0 ? max_nan_bf16x2(v.x, v.y) : max_nan_bf16x2(v.z, v.w);
        return max_nan_f32(bf16_lo(m), bf16_hi(m));
    }
};

struct VecF32 {
    static constexpr int VE = 4;
    static constexpr int ESIZE = 4;
    uint4 v;
    __device__ __forceinline__ static VecF32 load(const void *row, int64_t vi) {
        return {ld_stream_v4((const uint4 *)row + vi)};
    }
    __device__ __forceinline__ static VecF32 neg_inf() {
        return {make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u)};
    }
    __device__ __forceinline__ float get(int e) const {
        return __uint_as_float(e == 0 ? v.x : (e == 1 ? v.y : (e == 2 ? v.z : v.w)));
    }
    __device__ __forceinline__ float vmax() const {
        return max_nan_f32(max_nan_f32(get(0), get(1)), max_nan_f32(get(2), get(3)));
    }
    __device__ __forceinline__ float gmax(int) const { return vmax(); }
};

// Scalar read of one logit (token gathers).
__device__ __forceinline__ float load_logit(const void *base, int dtype, int64_t idx) {
    if (dtype == 0) return __uint_as_float((uint32_t)__ldg((const unsigned short *)base + idx) << 16);
    return __ldg((const float *)base + idx);
}

// The same with the element size fixed at compile time: no branch between
// consecutive gathers, so they issue back to back.
template <int ESZ>
__device__ __forceinline__ float ld_elem(const void *base, int64_t idx) {
    if (ESZ == 2) return __uint_as_float((uint32_t)__ldg((const unsigned short *)base + idx) << 16);
    return __ldg((const float *)base + idx);
}

// ------------------------------------------------------------------ async copies
// Bulk (TMA) copies global -> shared, completed on an mbarrier, and bounded waits.
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count));
}

__device__ __forceinline__ void mbar_init_fence() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
                 : "memory");
}

// try_wait with a suspend-time hint: a thread whose phase is not complete sleeps in
// the barrier (up to the hint, in ns) instead of spinning and taking issue slots
// from the warps that compute.
constexpr uint32_t kSuspendHintNs = 100000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_addr(bar)), "r"(parity), "r"(kSuspendHintNs)
        : "memory");
    return done != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for the phase of the given parity to complete; false after limit_ns.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (!mbar_try_wait(bar, parity))
        if (global_ns() - t0 > limit_ns) return false;
    return true;
}

// cp.async.bulk: `bytes` (multiple of 16) from 16-byte aligned global to shared memory.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Programmatic dependent launch: let the next kernel in the stream start its
// launch early, and wait for the previous kernel's results.
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;"); }
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(smem_addr(p)));
    return r;
}

// Packed fp32 pair arithmetic (sm_100 family): two lanes of work per instruction.
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    unsigned long long d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)),
          "l"(*reinterpret_cast<unsigned long long *>(&c)));
    return *reinterpret_cast<float2 *>(&d);
}

__device__ __forceinline__ float2 fadd2(float2 a, float2 b) {
    unsigned long long d;
    asm("add.f32x2 %0, %1, %2;"
        : "=l"(d)
        : "l"(*reinterpret_cast<unsigned long long *>(&a)), "l"(*reinterpret_cast<unsigned long long *>(&b)));
    return *reinterpret_cast<float2 *>(&d);
}

// ------------------------------------------------------------------ warp reductions
__device__ __forceinline__ float warp_max_nan(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = max_nan_f32(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x = fmaxf(x, __shfl_xor_sync(0xffffffffu, x, o));
    return x;
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

__device__ __forceinline__ int warp_sum_i(int x) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) x += __shfl_xor_sync(0xffffffffu, x, o);
    return x;
}

// (score, idx) argmax with the lowest idx on equal scores; idx < 0 means "none".
__device__ __forceinline__ bool better(float s1, int i1, float s2, int i2) {
    if (i2 < 0) return i1 >= 0;
    if (i1 < 0) return false;
    return s1 > s2 || (s1 == s2 && i1 < i2);
}

__device__ __forceinline__ void warp_argmax(float &s, int &i) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        const float s2 = __shfl_xor_sync(0xffffffffu, s, o);
        const int i2 = __shfl_xor_sync(0xffffffffu, i, o);
        if (better(s2, i2, s, i)) { s = s2; i = i2; }
    }
}

// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// Split cluster barrier.  Every thread of every CTA of the cluster executes each
// call, in the order arrive, wait, arrive, wait, ... (the .aligned forms need the
// whole warp).  arrive_relaxed orders nothing; arrive releases this thread's
// earlier memory operations and wait acquires the other CTAs' released ones.
__device__ __forceinline__ void cluster_arrive_relaxed() {
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
}
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.aligned;" ::: "memory"); }

// 16-byte store into the shared memory of CTA `rank` of this cluster, at the
// address that `local` has in this CTA's shared memory.
__device__ __forceinline__ void st_cluster_v4(void *local, uint32_t rank, uint4 v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(remote), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

}  // namespace specv
