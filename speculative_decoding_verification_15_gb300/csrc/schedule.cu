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
//
// Variants:
//  * two-step-stale sizing (Sec. 4.2.2, production): the engine prepares the next
//    batch while the GPU still runs, so the total comes from the scores of two
//    steps earlier and the slots from the latest scores -- the same kernel sorts
//    twice;
//  * static threshold truncation ("Accelerating Large-Model Inference ... DSpark",
//    prefix scheduler; the review's Sec. 3 fixed cutoff): each draft stops at the
//    first position whose confidence is below a threshold -- one thread a request.
#include <cuda_runtime.h>
#include <stdint.h>

#include "spec_verify.h"

namespace {

constexpr int kSchedThreads = 1024;

// Survivals are non-negative doubles, so their bit patterns order like their values:
// the sort compares 64-bit integers (sm_103a's fp64 compare rate is a small fraction
// of its integer rate).
__device__ __forceinline__ bool before(unsigned long long ka, int ia, unsigned long long kb, int ib) {
    return ka > kb || (ka == kb && ia < ib);
}

// Survival products of conf and the candidate slots: key[b Kmax + i] = the bits of
// S_{b,i} for the slots a request may add (m_b <= i < maxlen_b), 0 with the largest
// id elsewhere (after every survival, zeros included); returns n0 = sum m_b, the
// number of candidates and E0 = sum of the mandatory survivals through shared
// memory.  Every thread of the CTA calls it.
__device__ void build_keys(const float *conf, const int32_t *max_len, int B, int Kmax, int min_len, int npow2,
                           unsigned long long *key, int *id, int *s_n0, int *s_ncand, double *s_E0,
                           double *s_wsum) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    if (tid == 0) {
        *s_n0 = 0;
        *s_ncand = 0;
    }
    for (int i = tid; i < npow2; i += kSchedThreads) {
        key[i] = 0ull;
        id[i] = 0x7fffffff;
    }
    __syncthreads();
    double e0sum = 0.0;
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
                key[b * Kmax + i] = (unsigned long long)__double_as_longlong(surv);
                id[b * Kmax + i] = b * Kmax + i;
            }
        }
        atomicAdd(s_n0, mand);
        atomicAdd(s_ncand, ml - mand);
        e0sum += e0;
    }
    // E0 summed in request order: each thread's requests, then the threads in order
    double incl = e0sum;
    for (int o = 1; o < 32; o <<= 1) {
        const double y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
    }
    if (lane == 31) s_wsum[wid] = incl;
    __syncthreads();
    if (tid == 0) {
        double tot = 0.0;
        for (int w = 0; w < kSchedThreads / 32; ++w) tot += s_wsum[w];
        *s_E0 = tot;
    }
    __syncthreads();
}

// Bitonic sort of (key, id) in the `before` order (survival descending, then b,
// then i), then key[j] = the sum of the j+1 largest survivals (padding adds 0).
__device__ void sort_and_scan(unsigned long long *key, int *id, int npow2, double *s_wsum) {
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    for (int k = 2; k <= npow2; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = tid; i < npow2; i += kSchedThreads) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const bool up = (i & k) == 0;
                    const bool ordered = before(key[i], id[i], key[ixj], id[ixj]);
                    if (up != ordered) {
                        const unsigned long long tk = key[i];
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
    const int per = (npow2 + kSchedThreads - 1) / kSchedThreads;
    const int lo = tid * per < npow2 ? tid * per : npow2;
    const int hi = lo + per < npow2 ? lo + per : npow2;
    double local = 0.0;
    for (int i = lo; i < hi; ++i) local += __longlong_as_double((long long)key[i]);
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
        run += __longlong_as_double((long long)key[i]);
        key[i] = (unsigned long long)__double_as_longlong(run);  // from here on: the prefix sums
    }
    __syncthreads();
}

__device__ __forceinline__ double prefix_at(const unsigned long long *key, int j) {
    return __longlong_as_double((long long)key[j]);
}

// One CTA.  conf sizes the batch: the total n* with the best expected throughput
// over the whole table.  conf_alloc (NULL: conf) ranks the slots that fill it.
__global__ void __launch_bounds__(kSchedThreads) schedule_kernel(const float *conf, const float *conf_alloc,
                                                                 const int32_t *max_len, int B, int Kmax,
                                                                 const float *tau, int n_table, int budget,
                                                                 int min_len, int npow2, int32_t *out_len,
                                                                 double *out_info) {
    extern __shared__ __align__(16) unsigned char smem[];
    unsigned long long *key = (unsigned long long *)smem;  // [npow2]  survival bits, later prefix-sum bits
    int *id = (int *)(key + npow2);                   // [npow2]  b * Kmax + i
    int *cnt = id + npow2;                            // [B]
    __shared__ int s_n0, s_ncand;
    __shared__ double s_E0;
    __shared__ double s_redF[kSchedThreads / 32];
    __shared__ int s_redN[kSchedThreads / 32];
    __shared__ double s_wsum[kSchedThreads / 32];
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;

    for (int b = tid; b < B; b += kSchedThreads) cnt[b] = 0;
    build_keys(conf, max_len, B, Kmax, min_len, npow2, key, id, &s_n0, &s_ncand, &s_E0, s_wsum);
    sort_and_scan(key, id, npow2, s_wsum);

    // throughput of every admissible total, best over the whole table
    const int n0 = s_n0;
    int nhi = n0 + s_ncand;
    if (budget < nhi) nhi = budget;
    if (n_table - 1 < nhi) nhi = n_table - 1;
    double bestF = -__longlong_as_double(0x7ff0000000000000LL);
    int bestN = n0;
    for (int n = n0 + tid; n <= nhi; n += kSchedThreads) {
        const double E = s_E0 + (n > n0 ? prefix_at(key, n - n0 - 1) : 0.0);
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
    if (conf_alloc) {  // the latest scores pick the n* slots (same mandatory slots and candidates)
        build_keys(conf_alloc, max_len, B, Kmax, min_len, npow2, key, id, &s_n0, &s_ncand, &s_E0, s_wsum);
        sort_and_scan(key, id, npow2, s_wsum);
    }
    const int take = nstar - n0 > 0 ? nstar - n0 : 0;
    for (int t = tid; t < take; t += kSchedThreads) atomicAdd(&cnt[id[t] / Kmax], 1);
    __syncthreads();
    for (int b = tid; b < B; b += kSchedThreads) {
        int ml = max_len ? max_len[b] : Kmax;
        ml = ml < 0 ? 0 : (ml > Kmax ? Kmax : ml);
        out_len[b] = (min_len < ml ? min_len : ml) + cnt[b];
    }
    if (tid == 0 && out_info) {
        const double E = s_E0 + (take > 0 ? prefix_at(key, take - 1) : 0.0);
        out_info[0] = (double)nstar;
        out_info[1] = (double)B + E;
        const double t = (nstar >= 0 && nstar < n_table) ? (double)tau[nstar] : 0.0;
        out_info[2] = t > 0.0 ? ((double)B + E) / t : 0.0;
    }
}

// Static threshold truncation: one thread per request scans its confidences left
// to right and stops at the first one below the threshold (NaN counts as below).
__global__ void threshold_kernel(const float *conf, const int32_t *max_len, int B, int Kmax, float threshold,
                                 int32_t *out_len) {
    const int b = blockIdx.x * blockDim.x + threadIdx.x;
    if (b >= B) return;
    int ml = max_len ? max_len[b] : Kmax;
    ml = ml < 0 ? 0 : (ml > Kmax ? Kmax : ml);
    int L = ml;
    for (int i = 0; i < ml; ++i)
        if (!(conf[(int64_t)b * Kmax + i] >= threshold)) {
            L = i;
            break;
        }
    out_len[b] = L;
}

}  // namespace

namespace {

int launch_schedule(const float *conf, const float *conf_alloc, const int32_t *max_len, int B, int Kmax,
                    const float *step_time_us, int n_table, int budget, int min_len, int32_t *out_len,
                    double *out_info, void *cuda_stream) {
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
        conf, conf_alloc, max_len, B, Kmax, step_time_us, n_table, budget, min_len, npow2, out_len, out_info);
    e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}

}  // namespace

extern "C" int spec_schedule_verify_len(const float *conf, const int32_t *max_len, int B, int Kmax,
                                        const float *step_time_us, int n_table, int budget, int min_len,
                                        int32_t *out_len, double *out_info, void *cuda_stream) {
    return launch_schedule(conf, nullptr, max_len, B, Kmax, step_time_us, n_table, budget, min_len, out_len,
                           out_info, cuda_stream);
}

extern "C" int spec_schedule_verify_len_stale(const float *conf_stale, const float *conf, const int32_t *max_len,
                                              int B, int Kmax, const float *step_time_us, int n_table,
                                              int budget, int min_len, int32_t *out_len, double *out_info,
                                              void *cuda_stream) {
    if (B > 0 && Kmax > 0 && (!conf || !conf_stale)) return SPEC_EINVAL;
    return launch_schedule(conf_stale, conf, max_len, B, Kmax, step_time_us, n_table, budget, min_len, out_len,
                           out_info, cuda_stream);
}

extern "C" int spec_schedule_threshold(const float *conf, const int32_t *max_len, int B, int Kmax,
                                       float threshold, int32_t *out_len, void *cuda_stream) {
    if (B < 0 || Kmax < 0 || threshold != threshold) return SPEC_EINVAL;
    if (B == 0) return SPEC_OK;
    if (!out_len || (Kmax > 0 && !conf)) return SPEC_EINVAL;
    if (B > SPEC_MAX_BATCH) return SPEC_EUNSUPPORTED;
    threshold_kernel<<<(B + 255) / 256, 256, 0, (cudaStream_t)cuda_stream>>>(conf, max_len, B, Kmax, threshold,
                                                                           out_len);
    const cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? SPEC_OK : SPEC_ECUDA;
}
