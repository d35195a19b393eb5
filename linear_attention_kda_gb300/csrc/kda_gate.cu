// kda_gate: Eq. 5 (bounded gate) and the chunk-local cumulative log-decay of
// Eq. 3 (Kimi K3 report, section 2.1.1), as a standalone operation.
//
// Elementwise mode (chunk_size == 0): one thread per (token, head, channel).
// Cumulative mode: one CTA per (window of chunk_size tokens, head, block of
// 128 channels).  A window's tokens belong to at most two chunks; the CTA
// scans from the first token of the earliest of them, restarting the sum at
// every chunk start (chunk starts are sequence starts plus multiples of
// chunk_size), and writes only its own window.  Loads are coalesced along
// channels.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

template <typename T>
__global__ void gate_elementwise_kernel(const T *__restrict__ z, const float *__restrict__ bias,
                                        const float *__restrict__ A_log, float g_min, int kind, int64_t total,
                                        int H, int dk, float *__restrict__ out) {
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i % dk);
        const int h = (int)((i / dk) % H);
        const float b = bias ? bias[h * dk + c] : 0.f;
        const float eA = A_log ? expf(A_log[h]) : 1.f;
        out[i] = gate_log(kind, ld(z + i), b, eA, g_min);
    }
}

// Chunk start of token t (chunks aligned to each sequence start).
__device__ __forceinline__ int64_t chunk_start_of(const int32_t *cu, int N, int64_t seq_len_eq,
                                                  int64_t t, int C) {
    int64_t s;
    if (cu) s = cu[find_seq(cu, N, t)];
    else s = (t / seq_len_eq) * seq_len_eq;
    s = max((int64_t)0, min(s, t));  // keeps reads in [0, T) even if cu_seqlens is corrupt
    return s + ((t - s) / C) * C;
}

template <typename T>
__global__ void gate_cumsum_kernel(const T *__restrict__ z, const float *__restrict__ bias,
                                   const float *__restrict__ A_log, float g_min, int kind, int64_t Ttot,
                                   int N, const int32_t *__restrict__ cu, int H, int dk, int C,
                                   float *__restrict__ out, int *err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *is_start = smem_raw;  // [2C]
    const int64_t w0 = (int64_t)blockIdx.x * C;
    const int h = blockIdx.y;
    const int c = blockIdx.z * blockDim.x + threadIdx.x;
    const int64_t seq_len_eq = cu ? 0 : Ttot / N;

    if (cu && blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0) {
        // device-side validation of cu_seqlens: 0 = c_0 <= ... <= c_N = T
        bool bad = false;
        for (int n = threadIdx.x; n <= N; n += blockDim.x) {
            const int64_t x = cu[n];
            if (n == 0 && x != 0) bad = true;
            if (n == N && x != Ttot) bad = true;
            if (n > 0 && x < (int64_t)cu[n - 1]) bad = true;
        }
        if (bad) set_error(err, KDA_ERR_BAD_SEQLENS);
    }
    const int64_t s0 = chunk_start_of(cu, N, seq_len_eq, w0, C);  // earliest chunk start needed
    const int64_t t_end = min(Ttot, w0 + C);
    const int span = (int)(t_end - s0);
    for (int i = threadIdx.x; i < span; i += blockDim.x) {
        const int64_t t = s0 + i;
        is_start[i] = (chunk_start_of(cu, N, seq_len_eq, t, C) == t) ? 1 : 0;
    }
    __syncthreads();
    if (c >= dk) return;
    const float b = bias ? bias[h * dk + c] : 0.f;
    const float eA = A_log ? expf(A_log[h]) : 1.f;
    float G = 0.f;
    for (int i = 0; i < span; ++i) {
        const int64_t t = s0 + i;
        if (is_start[i]) G = 0.f;
        const int64_t idx = (t * H + h) * (int64_t)dk + c;
        G += gate_log(kind, ld(z + idx), b, eA, g_min);
        if (t >= w0) out[idx] = G;
    }
}

}  // namespace kda

using namespace kda;

kda_status_t kda_launch_gate(const kda_gate_args *a, cudaStream_t stream) {
    if (a->T == 0) return KDA_OK;
    int *err = kda_device_error_ptr();
    if (!err) return KDA_ERR_CUDA;
    if (a->chunk_size == 0) {
        const int64_t total = a->T * a->H * (int64_t)a->dk;
        const int threads = 256;
        const int64_t want = (total + threads - 1) / threads;
        const int blocks = (int)(want < 152 * 32 ? want : 152 * 32);
        if (a->dtype == KDA_BF16)
            gate_elementwise_kernel<bf16><<<blocks, threads, 0, stream>>>(
                (const bf16 *)a->z, a->dt_bias, a->A_log, a->g_min, a->gate_kind, total, a->H, a->dk, a->out);
        else
            gate_elementwise_kernel<float><<<blocks, threads, 0, stream>>>(
                (const float *)a->z, a->dt_bias, a->A_log, a->g_min, a->gate_kind, total, a->H, a->dk, a->out);
    } else {
        const int C = a->chunk_size;
        const int threads = a->dk < 128 ? ((a->dk + 31) / 32) * 32 : 128;
        dim3 grid((unsigned)((a->T + C - 1) / C), (unsigned)a->H, (unsigned)((a->dk + threads - 1) / threads));
        const size_t smem = 2 * (size_t)C;
        if (a->dtype == KDA_BF16)
            gate_cumsum_kernel<bf16><<<grid, threads, smem, stream>>>(
                (const bf16 *)a->z, a->dt_bias, a->A_log, a->g_min, a->gate_kind, a->T, (int)a->N, a->cu_seqlens,
                a->H, a->dk, C, a->out, err);
        else
            gate_cumsum_kernel<float><<<grid, threads, smem, stream>>>(
                (const float *)a->z, a->dt_bias, a->A_log, a->g_min, a->gate_kind, a->T, (int)a->N, a->cu_seqlens,
                a->H, a->dk, C, a->out, err);
    }
    return kda_cuda_status(cudaGetLastError());
}
