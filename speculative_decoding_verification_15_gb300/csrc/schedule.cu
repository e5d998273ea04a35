// schedule.cu -- confidence-scheduled verify lengths on sm_103a.
//
// "DSpark paper review" (vllmbangkok.com), Sec. 4.2.1: prefix survival
// c_1 x ... x c_k, which never increases along a draft.  Sec. 4.2.2: rank the draft
// tokens of every request by survival, grant them one at a time, read the step
// time of each total from a table profiled at startup, and keep the total with the
// best expected throughput -- searching the whole table, since a step-shaped table
// can drop before its real peak.
//
// One CTA: survival products per request (fp64, left to right), a bitonic sort of
// all candidate slots in shared memory (survival descending, then request, then
// position), an inclusive scan of the sorted survivals, the throughput of every
// admissible total, its argmax (smallest total on ties), and per-request counts.
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace {

constexpr int kSchedThreads = 1024;

__device__ __forceinline__ bool before(double ka, int ia, double kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const float *conf, const int32_t *max_len, int B,
                                                                 int Kmax, const float *tau, int n_table,
                                                                 int budget, int min_len, int npow2,
                                                                 int32_t *out_len, double *out_info) {
    extern __shared__ __align__(16) unsigned char smem[];
    double *key = (double *)smem;                     // [npow2]  survival, later prefix sums
    int *id = (int *)(key + npow2);                   // [npow2]  b * Kmax + i
    int *cnt = id + npow2;                            // [B]
    __shared__ int s_n0, s_ncand;
    __shared__ double s_E0;
    __shared__ double s_redF[kSchedThreads / 32];
    __shared__ int s_redN[kSchedThreads / 32];
    __shared__ double s_wsum[kSchedThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

    if (tid == 0) {
        s_n0 = 0;
        s_ncand = 0;
        s_E0 = 0.0;
    }
    for (int i = tid; i < npow2; i += kSchedThreads) {
        key[i] = -1.0;  // padding sorts after every survival (>= 0)
        id[i] = 0x7fffffff;
    }
    __syncthreads();

    // survival products and candidate slots
    for (int b = tid; b < B; b += kSchedThreads) {
        int ml = max_len ? max_len[b] : Kmax;
        ml = ml < 0 ? 0 : (ml > Kmax ? Kmax : ml);
        const int mand = min_len < ml ? min_len : ml;
        double surv = 1.0, e0 = 0.0;
        for (int i = 0; i < Kmax; ++i) {
            double c = (double)conf[(int64_t)b * Kmax + i];
            if (!(c >= 0.0)) c = 0.0;  // negative or NaN
            if (c > 1.0) c = 1.0;
            surv = surv * c;
            if (i < mand) {
                e0 += surv;
            } else if (i < ml) {
                key[b * Kmax + i] = surv;
                id[b * Kmax + i] = b * Kmax + i;
            }
        }
        cnt[b] = 0;
        atomicAdd(&s_n0, mand);
        atomicAdd(&s_ncand, ml - mand);
        atomicAdd(&s_E0, e0);
    }
    __syncthreads();

    // bitonic sort: `before` order (survival descending, then b, then i)
    for (int k = 2; k <= npow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < npow2; i += kSchedThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const bool up = (i & k) == 0;
                    const bool ordered = before(key[i], id[i], key[ixj], id[ixj]);
                    if (up != ordered) {
                        const double tk = key[i];
                        key[i] = key[ixj];
                        key[ixj] = tk;
                        const int ti = id[i];
                        id[i] = id[ixj];
                        id[ixj] = ti;
                    }
                }
            }
            __syncthreads();
        }
    }

    // inclusive scan of the sorted survivals (padding contributes 0)
    const int per = (npow2 + kSchedThreads - 1) / kSchedThreads;
    const int lo = tid * per < npow2 ? tid * per : npow2;
    const int hi = lo + per < npow2 ? lo + per : npow2;
    double local = 0.0;
    for (int i = lo; i < hi; ++i) local += key[i] > 0.0 ? key[i] : 0.0;
    double incl = local;
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[wid] = incl;
    __syncthreads();
    double base = 0.0;
    for (int w = 0; w < wid; ++w) base += s_wsum[w];
    double run = base + incl - local;
    for (int i = lo; i < hi; ++i) {
        run += key[i] > 0.0 ? key[i] : 0.0;
        key[i] = run;
    }
    __syncthreads();

    // throughput of every admissible total, best over the whole table
    const int n0 = s_n0;
    int nhi = n0 + s_ncand;
    if (budget < nhi) nhi = budget;
    if (n_table - 1 < nhi) nhi = n_table - 1;
    double bestF = -__longlong_as_double(0x7ff0000000000000LL);
    int bestN = n0;
    for (int n = n0 + tid; n <= nhi; n += kSchedThreads) {
        const double E = s_E0 + (n > n0 ? key[n - n0 - 1] : 0.0);
        const double t = (double)tau[n];
        const double F = (t > 0.0 && isfinite(t)) ? ((double)B + E) / t : -__longlong_as_double(0x7ff0000000000000LL);
        if (F > bestF || (F == bestF && n < bestN)) {
            bestF = F;
            bestN = n;
        }
    }
    for (int o = 16; o > 0; o >>= 1) {
        const double F2 = __shfl_xor_sync(0xffffffffu, bestF, o);
        const int N2 = __shfl_xor_sync(0xffffffffu, bestN, o);
        if (F2 > bestF || (F2 == bestF && N2 < bestN)) {
            bestF = F2;
            bestN = N2;
        }
    }
    if (lane == 0) {
        s_redF[wid] = bestF;
        s_redN[wid] = bestN;
    }
    __syncthreads();
    if (tid == 0) {
        for (int w = 1; w < kSchedThreads / 32; ++w)
            if (s_redF[w] > s_redF[0] || (s_redF[w] == s_redF[0] && s_redN[w] < s_redN[0])) {
                s_redF[0] = s_redF[w];
                s_redN[0] = s_redN[w];
            }
    }
    __syncthreads();
    const int nstar = s_redN[0];
    const int take = nstar - n0 > 0 ? nstar - n0 : 0;
    for (int t = tid; t < take; t += kSchedThreads) atomicAdd(&cnt[id[t] / Kmax], 1);
    __syncthreads();
    for (int b = tid; b < B; b += kSchedThreads) {
        int ml = max_len ? max_len[b] : Kmax;
        ml = ml < 0 ? 0 : (ml > Kmax ? Kmax : ml);
        out_len[b] = (min_len < ml ? min_len : ml) + cnt[b];
    }
    if (tid == 0 && out_info) {
        const double E = s_E0 + (take > 0 ? key[take - 1] : 0.0);
        out_info[0] = (double)nstar;
        out_info[1] = (double)B + E;
        const double t = (nstar >= 0 && nstar < n_table) ? (double)tau[nstar] : 0.0;
        out_info[2] = t > 0.0 ? ((double)B + E) / t : 0.0;
    }
}

}  // namespace

extern "C" int spec_schedule_verify_len(const float *conf, const int32_t *max_len, int B, int Kmax,
                                        const float *step_time_us, int n_table, int budget, int min_len,
                                        int32_t *out_len, double *out_info, void *cuda_stream) {
    if (B < 0 || Kmax < 0 || min_len < 0 || n_table < 1 || budget < 0) return SPEC_EINVAL;
    if ((int64_t)budget < (int64_t)B * min_len || (int64_t)n_table - 1 < (int64_t)B * min_len) return SPEC_EINVAL;
    if (!step_time_us || (B > 0 && !out_len) || (B > 0 && Kmax > 0 && !conf)) return SPEC_EINVAL;
    if ((int64_t)B * Kmax > SPEC_MAX_SCHED_ITEMS || B > SPEC_MAX_BATCH) return SPEC_EUNSUPPORTED;
    int npow2 = 2;
    while (npow2 < B * Kmax) npow2 <<= 1;
    const size_t smem = (size_t)npow2 * (sizeof(double) + sizeof(int)) + sizeof(int) * (size_t)(B > 0 ? B : 1);
    cudaError_t e = cudaFuncSetAttribute(schedule_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return SPEC_ECUDA;
    schedule_kernel<<<1, kSchedThreads, smem, (cudaStream_t)cuda_stream>>>(
        conf, max_len, B, Kmax, step_time_us, n_table, budget, min_len, npow2, out_len, out_info);
    e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}
