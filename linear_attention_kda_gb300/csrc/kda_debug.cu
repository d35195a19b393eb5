// Optional numeric checks (kda_set_debug_checks): after an entry point's kernels, one more pass over
// what it wrote sets KDA_ERR_NUMERIC in the device error word if any value is NaN or infinite.  Off
// by default; the checks read every output once more, so they cost one extra HBM pass.
#include <atomic>

#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

// Grid-stride scan for a non-finite value: 16-byte loads over the 16-byte-aligned body, scalars for
// the tail.  bf16 is checked on its bit pattern (exponent all ones).
template <typename T>
__global__ void __launch_bounds__(256) check_finite_kernel(const T *__restrict__ p, int64_t n, int *err) {
    constexpr int PER = 16 / sizeof(T);
    const int64_t nv = n / PER;
    const int64_t stride = (int64_t)gridDim.x * blockDim.x;
    bool bad = false;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < nv; i += stride) {
        const uint4 u = reinterpret_cast<const uint4 *>(p)[i];
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            if (sizeof(T) == 4) bad |= (w[j] & 0x7F800000u) == 0x7F800000u;
            else bad |= ((w[j] & 0x7F80u) == 0x7F80u) || ((w[j] & 0x7F800000u) == 0x7F800000u);
        }
    }
    for (int64_t i = nv * PER + (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
        uint32_t x;
        if (sizeof(T) == 4) x = reinterpret_cast<const uint32_t *>(p)[i] & 0x7F800000u, bad |= x == 0x7F800000u;
        else x = reinterpret_cast<const uint16_t *>(p)[i] & 0x7F80u, bad |= x == 0x7F80u;
    }
    if (__syncthreads_or(bad) && threadIdx.x == 0) set_error(err, KDA_ERR_NUMERIC);
}

}  // namespace kda

namespace {
std::atomic<int32_t> g_debug_flags{0};
}

int32_t kda_debug_flags() { return g_debug_flags.load(std::memory_order_relaxed); }

kda_status_t kda_check_finite(const void *p, int64_t n, kda_dtype_t dtype, cudaStream_t stream) {
    if (!p || n <= 0) return KDA_OK;
    int *err = kda_device_error_ptr();
    if (!err) return KDA_ERR_CUDA;
    int dev = 0, sms = 152;
    if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int64_t per = dtype == KDA_BF16 ? 8 : 4;
    const int64_t want = (n / per + 255) / 256;
    const unsigned grid = (unsigned)(want < 4 * (int64_t)sms ? (want > 0 ? want : 1) : 4 * sms);
    if (dtype == KDA_BF16)
        kda::check_finite_kernel<kda::bf16><<<grid, 256, 0, stream>>>((const kda::bf16 *)p, n, err);
    else
        kda::check_finite_kernel<float><<<grid, 256, 0, stream>>>((const float *)p, n, err);
    return kda_cuda_status(cudaGetLastError());
}

extern "C" kda_status_t kda_set_debug_checks(int32_t flags) {
    if (flags & ~KDA_CHECK_FINITE) return KDA_ERR_INVALID_ARG;
    g_debug_flags.store(flags, std::memory_order_relaxed);
    return KDA_OK;
}
