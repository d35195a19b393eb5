// C ABI of libkda: host-side validation and dispatch.  Nothing here allocates
// device memory; failing validation launches nothing and returns a status.
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "kda_common.cuh"
#include "kda_internal.h"

// One error word per device that loads this library (set by kernels with
// atomicCAS, first error wins; read and cleared by kda_get_device_error).
static __device__ int g_kda_device_error;

namespace {

constexpr int kMaxDevices = 64;
std::atomic<int *> g_err_ptr[kMaxDevices];  // device address of g_kda_device_error, per device

// gate_kind is a kda_gate_kind_t; g_min matters (finite, < 0) for the bounded gate only
bool gate_ok(int32_t kind, float g_min) {
    if (kind == KDA_GATE_SOFTPLUS) return true;
    return kind == KDA_GATE_LOWER_BOUND && g_min < 0.f && isfinite(g_min);
}
bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }
bool aligned_to(const void *p, size_t a) { return ((uintptr_t)p & (a - 1)) == 0; }

kda_status_t check_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess) return KDA_ERR_NO_DEVICE;
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return KDA_ERR_NO_DEVICE;
    if (major != 10 || minor != 3) return KDA_ERR_NO_DEVICE;
    return KDA_OK;
}

bool dtype_ok(kda_dtype_t t) { return t == KDA_F32 || t == KDA_BF16; }
size_t dtype_size(kda_dtype_t t) { return t == KDA_BF16 ? 2 : 4; }

}  // namespace

namespace {
constexpr int kMaxProfileEvents = 16;
cudaEvent_t g_prof_events[kMaxProfileEvents];
int g_prof_n = 0;
}  // namespace

void kda_profile_mark(int i, cudaStream_t stream) {
    if (i < g_prof_n && g_prof_events[i]) cudaEventRecord(g_prof_events[i], stream);
}

int *kda_device_error_ptr() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    int *e = g_err_ptr[dev].load(std::memory_order_acquire);
    if (!e) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_kda_device_error) != cudaSuccess) return nullptr;
        e = (int *)p;
        g_err_ptr[dev].store(e, std::memory_order_release);
    }
    return e;
}

static thread_local int g_last_cuda_error = 0;

kda_status_t kda_cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return KDA_OK;
    g_last_cuda_error = (int)e;
    return KDA_ERR_CUDA;
}

extern "C" {

int kda_abi_version(void) { return KDA_ABI_VERSION; }

kda_status_t kda_set_profile_events(void *const *events, int32_t n_events) {
    if (n_events < 0 || n_events > kMaxProfileEvents || (n_events > 0 && !events))
        return KDA_ERR_INVALID_ARG;
    for (int i = 0; i < n_events; ++i) g_prof_events[i] = (cudaEvent_t)events[i];
    g_prof_n = n_events;
    return KDA_OK;
}

int32_t kda_chunk_fwd_kernel_count(const kda_chunk_args *a) {
    if (!a) return 0;
    kda_chunk_plan p;
    if (!kda_make_chunk_plan(a->T, a->N > 0 ? a->N : 1, a->H > 0 ? a->H : 1, a->dk, a->dv, a->dtype, 64, &p,
                             a->cu_seqlens_host, a->gate_kind, kda_gate_needs_fp32_path(a->gate_kind, a->g_min)))
        return 0;
    // either one fused launch (intra-chunk transform and output pass together) or the chunk plan,
    // then intra-chunk transform, [segment summaries, fold,] output pass; an empty batch (T = 0)
    // runs the chunk plan and the output pass alone, which passes the states through
    if (a->T == 0) return 2;
    const int extra = (a->out_gate && !(p.path == 1 && p.epi_fused)) ? 1 : 0;  // the output epilogue's own pass
    if (p.fused || p.team) return 1 + extra;
    return (p.split ? 5 : 3) + extra;
}

kda_status_t kda_chunk_fwd_schedule(const kda_chunk_args *a, int64_t *out) {
    if (!a || !out || a->T < 0 || a->N < 1 || a->H < 1) return KDA_ERR_INVALID_ARG;
    kda_chunk_plan p;
    if (!kda_make_chunk_plan(a->T, a->N, a->H, a->dk, a->dv, a->dtype, 64, &p, a->cu_seqlens_host, a->gate_kind,
                             kda_gate_needs_fp32_path(a->gate_kind, a->g_min)))
        return KDA_ERR_INVALID_ARG;
    out[0] = p.fused ? 1 : (p.team ? 2 : 0);
    out[1] = p.fused ? p.kpre : (p.team ? p.team_k : 0);
    out[2] = p.split ? p.seg_len : 0;
    out[3] = kda_chunk_fwd_kernel_count(a);
    return KDA_OK;
}

const char *kda_status_string(kda_status_t s) {
    switch (s) {
        case KDA_OK: return "ok";
        case KDA_ERR_INVALID_ARG: return "invalid argument";
        case KDA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape (head size or chunk size)";
        case KDA_ERR_UNSUPPORTED_DTYPE: return "unsupported dtype";
        case KDA_ERR_MISALIGNED: return "tensor pointer not 16-byte aligned";
        case KDA_ERR_WORKSPACE: return "workspace missing or too small";
        case KDA_ERR_CUDA: return "CUDA runtime error";
        case KDA_ERR_BAD_SEQLENS: return "cu_seqlens is not 0 = c_0 <= ... <= c_N = T";
        case KDA_ERR_BAD_STATE_INDEX: return "state index outside [0, num_slots)";
        case KDA_ERR_NO_DEVICE: return "no current CUDA device of compute capability 10.3";
        case KDA_ERR_DEVICE_TIMEOUT: return "bounded wait inside a kernel gave up";
        case KDA_ERR_BAD_TOKEN_COUNT: return "n_replay or n_commit entry outside its range";
        case KDA_ERR_NUMERIC: return "an output holds a NaN or an infinity (debug checks)";
    }
    return "unknown status";
}

int32_t kda_last_cuda_error(void) {
    const int v = g_last_cuda_error;
    g_last_cuda_error = 0;
    return v;
}

kda_status_t kda_get_device_error(struct CUstream_st *stream) {
    int *p = kda_device_error_ptr();
    if (!p) return KDA_ERR_CUDA;
    if (cudaStreamSynchronize((cudaStream_t)stream) != cudaSuccess) return KDA_ERR_CUDA;
    int v = 0;
    if (cudaMemcpyFromSymbol(&v, g_kda_device_error, sizeof(int)) != cudaSuccess) return KDA_ERR_CUDA;
    const int zero = 0;
    if (v != 0 && cudaMemcpyToSymbol(g_kda_device_error, &zero, sizeof(int)) != cudaSuccess)
        return KDA_ERR_CUDA;
    return (kda_status_t)v;
}

kda_status_t kda_gate(const kda_gate_args *a, struct CUstream_st *stream) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->T < 0 || a->H < 1 || a->dk < 1 || a->chunk_size < 0 || a->chunk_size > 256)
        return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (!gate_ok(a->gate_kind, a->g_min)) return KDA_ERR_INVALID_ARG;
    if (a->T == 0) return KDA_OK;
    if (!a->z || !a->out) return KDA_ERR_INVALID_ARG;
    if (a->chunk_size > 0) {
        if (a->N < 1) return KDA_ERR_INVALID_ARG;
        if (!a->cu_seqlens && a->T % a->N != 0) return KDA_ERR_INVALID_ARG;
        if (a->cu_seqlens && !aligned_to(a->cu_seqlens, 4)) return KDA_ERR_MISALIGNED;
    }
    if (!aligned16(a->z) || !aligned16(a->out) || (a->dt_bias && !aligned16(a->dt_bias)) ||
        (a->A_log && !aligned_to(a->A_log, 4)))
        return KDA_ERR_MISALIGNED;
    kda_status_t st = check_device();
    if (st != KDA_OK) return st;
    st = kda_launch_gate(a, (cudaStream_t)stream);
    if (st == KDA_OK && (kda_debug_flags() & KDA_CHECK_FINITE))
        st = kda_check_finite(a->out, a->T * a->H * (int64_t)a->dk, KDA_F32, (cudaStream_t)stream);
    return st;
}

static kda_status_t validate_chunk(const kda_chunk_args *a) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->T < 0 || a->N < 1 || a->H < 1) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (a->dk != a->dv || (a->dk != 64 && a->dk != 128)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (a->chunk_size != 0 && a->chunk_size != 64) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!gate_ok(a->gate_kind, a->g_min) || !isfinite(a->scale)) return KDA_ERR_INVALID_ARG;
    if (!a->cu_seqlens && a->T % a->N != 0) return KDA_ERR_INVALID_ARG;
    if (a->T > INT32_MAX) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (a->T > 0) {
        if (!a->q || !a->k || !a->v || !a->z || !a->beta || !a->o) return KDA_ERR_INVALID_ARG;
        if (a->o == a->q || a->o == a->k || a->o == a->v || a->o == a->z) return KDA_ERR_INVALID_ARG;
        if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->z) ||
            !aligned16(a->o) || !aligned_to(a->beta, dtype_size(a->dtype)))
            return KDA_ERR_MISALIGNED;
    }
    if ((a->initial_state && !aligned16(a->initial_state)) ||
        (a->final_state && !aligned16(a->final_state)) ||
        (a->dt_bias && !aligned16(a->dt_bias)) || (a->A_log && !aligned_to(a->A_log, 4)) ||
        (a->cu_seqlens && !aligned_to(a->cu_seqlens, 4)))
        return KDA_ERR_MISALIGNED;
    if (a->out_gate) {  // output epilogue (Eq. 6)
        if (!(a->out_norm_eps > 0.f) || !isfinite(a->out_norm_eps)) return KDA_ERR_INVALID_ARG;
        if (a->out_gate == a->o) return KDA_ERR_INVALID_ARG;
        if (!aligned16(a->out_gate) || (a->out_norm_weight && !aligned16(a->out_norm_weight)))
            return KDA_ERR_MISALIGNED;
    }
    if (a->cu_seqlens_host) {
        const int32_t *cu = a->cu_seqlens_host;
        if (cu[0] != 0 || cu[a->N] != a->T) return KDA_ERR_INVALID_ARG;
        for (int64_t n = 0; n < a->N; ++n)
            if (cu[n + 1] < cu[n]) return KDA_ERR_INVALID_ARG;
    }
    return KDA_OK;
}

size_t kda_chunk_fwd_workspace_size_gate(int64_t T, int64_t N, int32_t H, int32_t dk, int32_t dv,
                                         kda_dtype_t dtype, int32_t chunk_size,
                                         const int32_t *cu_seqlens_host, int32_t gate_kind) {
    if (T < 0 || N < 1 || H < 1 || !dtype_ok(dtype)) return 0;
    if (dk != dv || (dk != 64 && dk != 128)) return 0;
    if (chunk_size != 0 && chunk_size != 64) return 0;
    if (gate_kind != KDA_GATE_LOWER_BOUND && gate_kind != KDA_GATE_SOFTPLUS) return 0;
    kda_chunk_plan p;
    if (!kda_make_chunk_plan(T, N, H, dk, dv, dtype, 64, &p, cu_seqlens_host, gate_kind)) return 0;
    return p.total_bytes;
}

size_t kda_chunk_fwd_workspace_size(int64_t T, int64_t N, int32_t H, int32_t dk, int32_t dv,
                                    kda_dtype_t dtype, int32_t chunk_size,
                                    const int32_t *cu_seqlens_host) {
    return kda_chunk_fwd_workspace_size_gate(T, N, H, dk, dv, dtype, chunk_size, cu_seqlens_host,
                                             KDA_GATE_LOWER_BOUND);
}

kda_status_t kda_chunk_fwd(const kda_chunk_args *a, void *workspace, size_t workspace_bytes,
                           struct CUstream_st *stream) {
    kda_status_t st = validate_chunk(a);
    if (st != KDA_OK) return st;
    kda_chunk_plan p;
    if (!kda_make_chunk_plan(a->T, a->N, a->H, a->dk, a->dv, a->dtype, 64, &p, a->cu_seqlens_host, a->gate_kind,
                             kda_gate_needs_fp32_path(a->gate_kind, a->g_min)))
        return KDA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < p.total_bytes) return KDA_ERR_WORKSPACE;
    if (!aligned_to(workspace, 256)) return KDA_ERR_MISALIGNED;
    st = check_device();
    if (st != KDA_OK) return st;
    st = p.path == 1 ? kda_launch_chunk_tc(a, p, workspace, (cudaStream_t)stream)
                     : kda_launch_chunk_simt(a, p, workspace, (cudaStream_t)stream);
    if (st == KDA_OK && a->out_gate && !(p.path == 1 && p.epi_fused)) {
        // the output epilogue as its own HBM-bound pass over o, in place, on all SMs: the fp32 path, and
        // the fused launch on short chains (inside their output pass it would lengthen the latency-bound
        // chain more than the round trip of o costs)
        kda_output_gate_args og{a->T, a->H, a->dv, a->dtype, a->o, a->out_gate, a->out_norm_weight,
                                a->out_norm_eps, a->o};
        st = kda_launch_output_gate(&og, (cudaStream_t)stream);
    }
    if (st == KDA_OK && (kda_debug_flags() & KDA_CHECK_FINITE)) {
        st = kda_check_finite(a->o, a->T * a->H * (int64_t)a->dv, a->dtype, (cudaStream_t)stream);
        if (st == KDA_OK)
            st = kda_check_finite(a->final_state, a->N * a->H * (int64_t)a->dk * a->dv, KDA_F32,
                                  (cudaStream_t)stream);
    }
    return st;
}

size_t kda_chunk_bwd_workspace_size(int64_t T, int64_t N, int32_t H, int32_t dk, int32_t dv,
                                    int32_t chunk_size) {
    if (T < 0 || N < 1 || H < 1 || dk != dv || (dk != 64 && dk != 128)) return 0;
    if (chunk_size != 0 && chunk_size != 64) return 0;
    return kda_chunk_bwd_layout_bytes(T, N, H, dk, dv);
}

size_t kda_chunk_bwd_workspace_size_min(int64_t T, int64_t N, int32_t H, int32_t dk, int32_t dv,
                                        int32_t chunk_size) {
    if (T < 0 || N < 1 || H < 1 || dk != dv || (dk != 64 && dk != 128)) return 0;
    if (chunk_size != 0 && chunk_size != 64) return 0;
    return kda_chunk_bwd_min_layout_bytes(T, N, H, dk, dv);
}

kda_status_t kda_chunk_bwd(const kda_chunk_bwd_args *a, void *workspace, size_t workspace_bytes,
                           struct CUstream_st *stream) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->T < 0 || a->N < 1 || a->H < 1) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (a->dk != a->dv || (a->dk != 64 && a->dk != 128)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (a->chunk_size != 0 && a->chunk_size != 64) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!gate_ok(a->gate_kind, a->g_min) || !isfinite(a->scale)) return KDA_ERR_INVALID_ARG;
    if (!a->cu_seqlens && a->T % a->N != 0) return KDA_ERR_INVALID_ARG;
    if (a->T > INT32_MAX || a->N * (int64_t)a->H > INT32_MAX) return KDA_ERR_UNSUPPORTED_SHAPE;
    const size_t es = dtype_size(a->dtype);
    if (a->T > 0) {
        const void *in[] = {a->q, a->k, a->z, a->v, a->beta, a->grad_o};
        const void *out[] = {a->grad_q, a->grad_k, a->grad_z, a->grad_v, a->grad_beta};
        for (const void *p : in)
            if (!p) return KDA_ERR_INVALID_ARG;
        for (const void *p : out) {
            if (!p) return KDA_ERR_INVALID_ARG;
            for (const void *x : in)
                if (p == x) return KDA_ERR_INVALID_ARG;
        }
        for (int i = 0; i < 5; ++i)
            for (int j = i + 1; j < 5; ++j)
                if (out[i] == out[j]) return KDA_ERR_INVALID_ARG;
        if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->z) || !aligned16(a->v) ||
            !aligned16(a->grad_o) || !aligned16(a->grad_q) || !aligned16(a->grad_k) || !aligned16(a->grad_z) ||
            !aligned16(a->grad_v) || !aligned_to(a->beta, es) || !aligned_to(a->grad_beta, es))
            return KDA_ERR_MISALIGNED;
    }
    if ((a->initial_state && !aligned16(a->initial_state)) ||
        (a->grad_final_state && !aligned16(a->grad_final_state)) ||
        (a->grad_initial_state && !aligned16(a->grad_initial_state)) ||
        (a->dt_bias && !aligned16(a->dt_bias)) || (a->A_log && !aligned_to(a->A_log, 4)) ||
        (a->grad_dt_bias && !aligned_to(a->grad_dt_bias, 4)) || (a->grad_A_log && !aligned_to(a->grad_A_log, 4)) ||
        (a->cu_seqlens && !aligned_to(a->cu_seqlens, 4)))
        return KDA_ERR_MISALIGNED;
    const size_t need = kda_chunk_bwd_min_layout_bytes(a->T, a->N, a->H, a->dk, a->dv);
    if (need == 0) return KDA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < need) return KDA_ERR_WORKSPACE;
    if (!aligned_to(workspace, 256)) return KDA_ERR_MISALIGNED;
    kda_status_t st = check_device();
    if (st != KDA_OK) return st;
    st = kda_launch_chunk_bwd(a, workspace, workspace_bytes, (cudaStream_t)stream);
    if (st == KDA_OK && (kda_debug_flags() & KDA_CHECK_FINITE)) {
        const int64_t tk = a->T * a->H * (int64_t)a->dk, tv = a->T * a->H * (int64_t)a->dv;
        const struct { const void *p; int64_t n; kda_dtype_t t; } outs[] = {
            {a->grad_q, tk, a->dtype}, {a->grad_k, tk, a->dtype}, {a->grad_z, tk, a->dtype},
            {a->grad_v, tv, a->dtype}, {a->grad_beta, a->T * a->H, a->dtype},
            {a->grad_dt_bias, (int64_t)a->H * a->dk, KDA_F32}, {a->grad_A_log, a->H, KDA_F32},
            {a->grad_initial_state, a->N * a->H * (int64_t)a->dk * a->dv, KDA_F32}};
        for (const auto &x : outs)
            if (st == KDA_OK && aligned16(x.p)) st = kda_check_finite(x.p, x.n, x.t, (cudaStream_t)stream);
    }
    return st;
}

kda_status_t kda_output_gate(const kda_output_gate_args *a, struct CUstream_st *stream) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->T < 0 || a->H < 1) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (a->dv != 32 && a->dv != 64 && a->dv != 128 && a->dv != 256) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!(a->eps > 0.f) || !isfinite(a->eps)) return KDA_ERR_INVALID_ARG;
    if (a->T == 0) return KDA_OK;
    if (!a->o || !a->g || !a->y || a->y == a->g) return KDA_ERR_INVALID_ARG;
    if (a->T * (int64_t)a->H > ((int64_t)INT32_MAX) * 8) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!aligned16(a->o) || !aligned16(a->g) || !aligned16(a->y) ||
        (a->norm_weight && !aligned16(a->norm_weight)))
        return KDA_ERR_MISALIGNED;
    kda_status_t st = check_device();
    if (st != KDA_OK) return st;
    st = kda_launch_output_gate(a, (cudaStream_t)stream);
    if (st == KDA_OK && (kda_debug_flags() & KDA_CHECK_FINITE))
        st = kda_check_finite(a->y, a->T * a->H * (int64_t)a->dv, a->dtype, (cudaStream_t)stream);
    return st;
}

kda_status_t kda_recurrent_step(const kda_step_args *a, struct CUstream_st *stream) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->N < 0 || a->H < 1 || a->num_slots < 0) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (a->dk != a->dv || (a->dk != 64 && a->dk != 128)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!gate_ok(a->gate_kind, a->g_min) || !isfinite(a->scale)) return KDA_ERR_INVALID_ARG;
    if (a->N == 0) return KDA_OK;
    if (a->N * (int64_t)a->H > INT32_MAX) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!a->q || !a->k || !a->v || !a->z || !a->beta || !a->o || !a->state) return KDA_ERR_INVALID_ARG;
    if (!a->state_indices && a->num_slots != 0 && a->num_slots < a->N) return KDA_ERR_INVALID_ARG;
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->z) ||
        !aligned16(a->o) || !aligned16(a->state) || !aligned_to(a->beta, dtype_size(a->dtype)) ||
        (a->dt_bias && !aligned16(a->dt_bias)) || (a->A_log && !aligned_to(a->A_log, 4)) ||
        (a->state_indices && !aligned_to(a->state_indices, 4)))
        return KDA_ERR_MISALIGNED;
    kda_status_t st = check_device();
    if (st != KDA_OK) return st;
    st = kda_launch_decode(a, (cudaStream_t)stream);
    if (st == KDA_OK && (kda_debug_flags() & KDA_CHECK_FINITE)) {
        const int64_t slots = a->num_slots ? a->num_slots : a->N;
        st = kda_check_finite(a->o, a->N * a->H * (int64_t)a->dv, a->dtype, (cudaStream_t)stream);
        if (st == KDA_OK)
            st = kda_check_finite(a->state, slots * a->H * (int64_t)a->dk * a->dv, KDA_F32, (cudaStream_t)stream);
    }
    return st;
}

kda_status_t kda_recurrent_replay(const kda_replay_args *a, struct CUstream_st *stream) {
    if (!a) return KDA_ERR_INVALID_ARG;
    if (a->N < 0 || a->H < 1 || a->num_slots < 0 || a->R < 0 || a->M < 1) return KDA_ERR_INVALID_ARG;
    if (!dtype_ok(a->dtype)) return KDA_ERR_UNSUPPORTED_DTYPE;
    if (a->dk != a->dv || (a->dk != 64 && a->dk != 128)) return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!gate_ok(a->gate_kind, a->g_min) || !isfinite(a->scale)) return KDA_ERR_INVALID_ARG;
    if (a->N == 0) return KDA_OK;
    if (a->N * (int64_t)a->H > INT32_MAX || a->N * (int64_t)(a->R > a->M ? a->R : a->M) * a->H > INT32_MAX)
        return KDA_ERR_UNSUPPORTED_SHAPE;
    if (!a->q || !a->k || !a->v || !a->z || !a->beta || !a->o || !a->state || !a->n_commit)
        return KDA_ERR_INVALID_ARG;
    if (a->R > 0 && (!a->rq || !a->rk || !a->rv || !a->rz || !a->rbeta || !a->n_replay))
        return KDA_ERR_INVALID_ARG;
    if (!a->state_indices && a->num_slots != 0 && a->num_slots < a->N) return KDA_ERR_INVALID_ARG;
    const size_t es = dtype_size(a->dtype);
    if (!aligned16(a->q) || !aligned16(a->k) || !aligned16(a->v) || !aligned16(a->z) || !aligned16(a->o) ||
        !aligned16(a->state) || !aligned_to(a->beta, es) || !aligned_to(a->n_commit, 4) ||
        (a->dt_bias && !aligned16(a->dt_bias)) || (a->A_log && !aligned_to(a->A_log, 4)) ||
        (a->state_indices && !aligned_to(a->state_indices, 4)))
        return KDA_ERR_MISALIGNED;
    if (a->R > 0 && (!aligned16(a->rq) || !aligned16(a->rk) || !aligned16(a->rv) || !aligned16(a->rz) ||
                     !aligned_to(a->rbeta, es) || !aligned_to(a->n_replay, 4)))
        return KDA_ERR_MISALIGNED;
    kda_status_t st = check_device();
    if (st != KDA_OK) return st;
    st = kda_launch_replay(a, (cudaStream_t)stream);
    if (st == KDA_OK && (kda_debug_flags() & KDA_CHECK_FINITE)) {
        const int64_t slots = a->num_slots ? a->num_slots : a->N;
        st = kda_check_finite(a->o, a->N * (int64_t)a->M * a->H * a->dv, a->dtype, (cudaStream_t)stream);
        if (st == KDA_OK)
            st = kda_check_finite(a->state, slots * a->H * (int64_t)a->dk * a->dv, KDA_F32, (cudaStream_t)stream);
    }
    return st;
}

}  // extern "C"
