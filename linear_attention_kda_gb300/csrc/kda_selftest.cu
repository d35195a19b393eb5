// kda_selftest_bounded_wait: failure-detection self-test of the bounded waits every kernel uses.
// One CTA waits on an mbarrier that nothing ever arrives at, with the same bounded wait
// (mbar_wait: ~1 s of globaltimer, then give up) as the tensor-core prefill and replay kernels;
// it must return, record KDA_ERR_DEVICE_TIMEOUT in the device error word, and leave the context
// usable.  Nothing faults, traps or hangs.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {
namespace selftest {

using namespace kda::tc;

__global__ void bounded_wait_kernel(int *err, unsigned long long *elapsed_ns) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) mbar_init(&bar, 1);
    __syncthreads();
    const uint64_t t0 = globaltimer_ns();
    const bool ok = mbar_wait(&bar, 0);  // no thread arrives: the phase never completes
    const bool all = __syncthreads_and(ok ? 1 : 0) != 0;
    if (threadIdx.x == 0) {
        if (!all) set_error(err, KDA_ERR_DEVICE_TIMEOUT);
        if (elapsed_ns) *elapsed_ns = globaltimer_ns() - t0;
    }
}

}  // namespace selftest
}  // namespace kda

extern "C" kda_status_t kda_selftest_bounded_wait(unsigned long long *elapsed_ns, struct CUstream_st *stream) {
    if (elapsed_ns && (((uintptr_t)elapsed_ns) & 7u)) return KDA_ERR_MISALIGNED;
    int *err = kda_device_error_ptr();
    if (!err) return KDA_ERR_CUDA;
    kda::selftest::bounded_wait_kernel<<<1, 32, 0, (cudaStream_t)stream>>>(err, elapsed_ns);
    return kda_cuda_status(cudaGetLastError());
}
