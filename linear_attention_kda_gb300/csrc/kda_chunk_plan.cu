// Chunk planning for kda_chunk_fwd: workspace layout (host) and the
// per-sequence chunk offsets (device).
//
// Chunks of C tokens start at each sequence's first token (the last chunk of a
// sequence may be shorter).  Chunk slots are numbered sequence by sequence:
// sequence n owns slots [chunk_start[n], chunk_start[n + 1]).  The number of
// slots is bounded on the host without reading cu_seqlens:
//     sum_n ceil(len_n / C) <= floor((T + N (C - 1)) / C),
// so kernels are launched over that bound and slots past chunk_start[N] exit.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

__global__ void __launch_bounds__(1024)
chunk_plan_kernel(const int32_t *__restrict__ cu, int64_t T, int N, int C,
                  int32_t *__restrict__ chunk_start, int *err) {
    __shared__ int s_bad;
    __shared__ int s_warp[32];
    __shared__ int s_carry;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) { s_bad = 0; s_carry = 0; }
    __syncthreads();
    if (cu) {
        for (int n = tid; n <= N; n += blockDim.x) {
            const int64_t x = cu[n];
            bool bad = (n == 0 && x != 0) || (n == N && x != T) || (n > 0 && x < (int64_t)cu[n - 1]);
            if (bad) atomicOr(&s_bad, 1);
        }
    }
    __syncthreads();
    if (s_bad) {
        if (tid == 0) set_error(err, KDA_ERR_BAD_SEQLENS);
        for (int n = tid; n <= N; n += blockDim.x) chunk_start[n] = 0;  // no chunk runs
        return;
    }
    const int64_t len_eq = cu ? 0 : T / N;
    for (int base = 0; base < N; base += blockDim.x) {
        const int n = base + tid;
        int cnt = 0;
        if (n < N) {
            const int64_t len = cu ? (int64_t)cu[n + 1] - cu[n] : len_eq;
            cnt = (int)((len + C - 1) / C);
        }
        int x = cnt;  // inclusive scan across the block
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, off);
            if (lane >= off) x += y;
        }
        if (lane == 31) s_warp[warp] = x;
        __syncthreads();
        if (warp == 0) {
            int w = (lane < (int)(blockDim.x >> 5)) ? s_warp[lane] : 0;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, w, off);
                if (lane >= off) w += y;
            }
            s_warp[lane] = w;
        }
        __syncthreads();
        const int incl = x + (warp > 0 ? s_warp[warp - 1] : 0) + s_carry;
        if (n < N) chunk_start[n + 1] = incl;
        __syncthreads();
        if (tid == blockDim.x - 1) s_carry = incl;
        __syncthreads();
    }
    if (tid == 0) chunk_start[0] = 0;
}

}  // namespace kda

static size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool kda_make_chunk_plan(int64_t T, int64_t N, int H, int dk, int dv, kda_dtype_t dtype, int C,
                         kda_chunk_plan *p) {
    if (T < 0 || N < 1 || H < 1 || C < 1) return false;
    p->T = T; p->N = N; p->H = H; p->dk = dk; p->dv = dv; p->C = C;
    p->max_chunks = (T + N * (int64_t)(C - 1)) / C;
    // bf16 with d_k = d_v = 128 runs on the tensor cores; everything else on the fp32 CUDA-core path
    p->path = (dtype == KDA_BF16 && dk == 128 && dv == 128 && C == 64) ? 1 : 0;
    if (p->path == 1) {
        p->record_bytes = kda_tc_packet_stride();  // bf16 operand images + gamma^C
    } else {
        // fp32 CUDA-core records: W, Q^, K~ [C, dk]; U [C, dv]; A [C, C]; gamma^C [dk]
        p->record_bytes = align_up(sizeof(float) * ((size_t)C * (3 * dk + dv) + (size_t)C * C + dk), 256);
    }
    p->off_chunk_start = 0;
    p->off_records = align_up(sizeof(int32_t) * (size_t)(N + 1), 256);
    p->total_bytes = p->off_records + p->record_bytes * (size_t)p->max_chunks * (size_t)H;
    return true;
}

kda_status_t kda_launch_chunk_plan(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                   cudaStream_t stream) {
    int *err = kda_device_error_ptr();
    if (!err) return KDA_ERR_CUDA;
    int32_t *chunk_start = (int32_t *)((char *)ws + p.off_chunk_start);
    kda::chunk_plan_kernel<<<1, 1024, 0, stream>>>(a->cu_seqlens, a->T, (int)a->N, p.C, chunk_start, err);
    return cudaGetLastError() == cudaSuccess ? KDA_OK : KDA_ERR_CUDA;
}
