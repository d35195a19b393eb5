// kda_chunk_fwd_static_ws: the prefill entry point for callers that cannot
// allocate device memory.
//
// Some hosts hand a kernel library nothing but input and output pointers:
// inference-engine plugins whose engine owns and accounts every byte of device
// memory, runtimes built on a pooled allocator that forbids raw cudaMalloc, or
// code that must never trigger the implicit device synchronisation a
// cudaMalloc/cudaFree can cause.  Such callers cannot provide the scratch that
// kda_chunk_fwd asks for.  This entry point takes the same arguments minus the
// workspace and uses a fixed buffer that lives inside the library instead.
//
// The buffer is a file-scope __device__ array of KDA_STATIC_WORKSPACE_BYTES.
// Every GPU that loads the library holds it until the process exits.  In host
// code the array's name is only a host-side stand-in, so its device address is
// looked up with cudaGetSymbolAddress once per device (on the first call made
// while that device is current) and kept in an atomic per-device slot.  Nothing
// here calls cudaMalloc, cudaFree or any allocating routine.
#include <atomic>

#include "kda_common.cuh"
#include "kda_internal.h"

static __device__ __align__(256) unsigned char g_kda_static_ws[KDA_STATIC_WORKSPACE_BYTES];

namespace {
constexpr int kMaxDev = 64;
std::atomic<void *> g_static_ws_ptr[kMaxDev];  // device address of g_kda_static_ws, per device
}  // namespace

extern "C" kda_status_t kda_chunk_fwd_static_ws(const kda_chunk_args *args, struct CUstream_st *stream) {
    if (!args) return KDA_ERR_INVALID_ARG;
    // sized for the path the call takes: the softplus gate, and the bounded gate below
    // KDA_TC_MIN_G_MIN, run on the fp32 path, whose records are larger
    const size_t need = kda_chunk_fwd_workspace_size_gate(args->T, args->N, args->H, args->dk, args->dv,
                                                          args->dtype, args->chunk_size, args->cu_seqlens_host,
                                                          kda_workspace_gate(args->gate_kind, args->g_min));
    if (need == 0) return kda_chunk_fwd(args, nullptr, 0, stream);  // invalid sizes: same status as kda_chunk_fwd
    if (need > (size_t)KDA_STATIC_WORKSPACE_BYTES) return KDA_ERR_WORKSPACE;  // problem too large for the buffer
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return KDA_ERR_NO_DEVICE;
    if (dev >= kMaxDev) return KDA_ERR_NO_DEVICE;
    void *ws = g_static_ws_ptr[dev].load(std::memory_order_acquire);
    if (!ws) {
        // concurrent first calls on one device look up the same address; the last store wins harmlessly
        if (cudaGetSymbolAddress(&ws, g_kda_static_ws) != cudaSuccess || !ws) return KDA_ERR_CUDA;
        g_static_ws_ptr[dev].store(ws, std::memory_order_release);
    }
    // The prefill scratch needs no clearing: each call writes every byte of it that it later
    // reads (chunk offsets and per-chunk records), so stale contents of an earlier call are harmless.
    return kda_chunk_fwd(args, ws, (size_t)KDA_STATIC_WORKSPACE_BYTES, stream);
}
