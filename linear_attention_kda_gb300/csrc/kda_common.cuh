// Device helpers shared by the libkda kernels (sm_103a).
#pragma once
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/kda.h"

namespace kda {

using bf16 = __nv_bfloat16;

template <typename T> __device__ __forceinline__ float ld(const T *p);
template <> __device__ __forceinline__ float ld<float>(const float *p) { return *p; }
template <> __device__ __forceinline__ float ld<bf16>(const bf16 *p) { return __bfloat162float(*p); }

template <typename T> __device__ __forceinline__ void st(T *p, float x);
template <> __device__ __forceinline__ void st<float>(float *p, float x) { *p = x; }
template <> __device__ __forceinline__ void st<bf16>(bf16 *p, float x) { *p = __float2bfloat16_rn(x); }

// Eq. 5 of the Kimi K3 report with the bias inside the logit:
// g = g_min * Sigmoid(exp(A) * (z + b)).  expA = exp(A_log[h]) precomputed.
__device__ __forceinline__ float gate_logdecay(float z, float b, float expA, float g_min) {
    const float x = expA * (z + b);
    return g_min / (1.0f + expf(-x));
}

// The gate selected by kind (kda_gate_kind_t): Eq. 5 above, or the unbounded softplus gate of the
// earlier design, g = -expA * Softplus(z + b) with Softplus(x) = max(x, 0) + ln(1 + e^{-|x|})
// (= ln(1 + e^x), no overflow for any x).
__device__ __forceinline__ float gate_log(int kind, float z, float b, float expA, float g_min) {
    if (kind == KDA_GATE_SOFTPLUS) {
        const float x = z + b;
        return -expA * (fmaxf(x, 0.f) + log1pf(expf(-fabsf(x))));
    }
    return gate_logdecay(z, b, expA, g_min);
}

// 16-byte asynchronous copy global -> shared memory (cached in L2 only): many can be in flight per
// thread without holding registers; cp_async_wait_all() waits for this thread's copies.
__device__ __forceinline__ void cp_async16(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;"
                 :: "r"((uint32_t)__cvta_generic_to_shared(smem_dst)), "l"(gsrc) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }
// Closes this thread's current group of cp.async copies (an empty group is allowed); wait_group1 waits
// until at most the newest group is still in flight.
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_group1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }
// 4-byte asynchronous copy global -> shared memory (both 4-byte aligned).
__device__ __forceinline__ void cp_async4(void *smem_dst, const void *gsrc) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;"
                 :: "r"((uint32_t)__cvta_generic_to_shared(smem_dst)), "l"(gsrc) : "memory");
}
// The executing thread's earlier cp.async copies arrive (once, when all have landed) on an mbarrier whose
// expected count includes this arrival.
__device__ __forceinline__ void cp_async_arrive_noinc(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];"
                 :: "r"((uint32_t)__cvta_generic_to_shared(bar)) : "memory");
}

// rows x cols fp32 block from global (row pitch gp floats) to shared memory (row pitch sp floats) by
// 16-byte copies spread over nt threads; cols, gp, sp multiples of 4 and both bases 16-byte aligned
__device__ __forceinline__ void tile_async(float *s, int sp, const float *g, int64_t gp, int rows, int cols,
                                           int tid, int nt) {
    const int q4 = cols >> 2;
    for (int e = tid; e < rows * q4; e += nt) {
        const int r = e / q4, c = (e - r * q4) << 2;
        cp_async16(s + r * sp + c, g + r * gp + c);
    }
}

// Asks L2 to fetch [p, p + bytes) ahead of use (16-byte aligned address, size a multiple of 16).
__device__ __forceinline__ void prefetch_l2(const void *p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(p), "r"(bytes) : "memory");
}

// First device-detected error wins; later ones are dropped.
__device__ __forceinline__ void set_error(int *err, int code) {
    if (err) atomicCAS(err, 0, code);
}

// Sequence n containing token t: largest n with cu[n] <= t (cu has N + 1 entries).
__device__ __forceinline__ int find_seq(const int32_t *cu, int N, int64_t t) {
    int lo = 0, hi = N;  // invariant: cu[lo] <= t, answer in [lo, hi)
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if ((int64_t)cu[mid] <= t) lo = mid; else hi = mid;
    }
    return lo;
}

}  // namespace kda

// Host-side helpers (defined in kda_api.cu).
int *kda_device_error_ptr();  // device address of this device's error word
