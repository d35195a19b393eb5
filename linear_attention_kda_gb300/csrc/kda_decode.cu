// kda_recurrent_step: one decode token per sequence, Eq. 1 of the Kimi K3
// report (section 2.1.1) applied in place to every (sequence, head) state, as
// section 5.4.2 describes for KDA decode.
//
// The step is bound by HBM traffic on the fp32 state (read once, written
// once: 2 * 4 * D * D bytes per head).  One CTA owns one (sequence, head)
// state; 2 * D threads; warp w holds rows [16 w, 16 w + 16) and lane l holds
// D / 32 consecutive columns, so every warp-wide access of a state row is one
// fully coalesced 128-bit (D = 128) or 64-bit (D = 64) transaction.  The whole
// state stays in registers between the read and the write, which lets the
// step use the single-read form
//     S' = Diag(alpha) S,  p = S'^T k,  r = S'^T q,  e = beta (v - p),
//     S <- S' + k e^T,     o = scale (r + (k . q) e)
// (algebraically Eq. 1 with o_t = S_t^T q_t).  Column sums over the 16 rows of
// a warp stay in registers; the cross-warp sums go through shared memory.
// State traffic uses streaming (evict-first) cache hints: each state is read
// and written exactly once per step.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {

template <int VW> struct vec;
template <> struct vec<4> {
    using T = float4;
    __device__ static void scale(T &x, float a) { x.x *= a; x.y *= a; x.z *= a; x.w *= a; }
    __device__ static float get(const T &x, int i) { return i == 0 ? x.x : i == 1 ? x.y : i == 2 ? x.z : x.w; }
    __device__ static void add(T &x, int i, float a) {
        if (i == 0) x.x += a; else if (i == 1) x.y += a; else if (i == 2) x.z += a; else x.w += a;
    }
};
template <> struct vec<2> {
    using T = float2;
    __device__ static void scale(T &x, float a) { x.x *= a; x.y *= a; }
    __device__ static float get(const T &x, int i) { return i == 0 ? x.x : x.y; }
    __device__ static void add(T &x, int i, float a) { if (i == 0) x.x += a; else x.y += a; }
};

template <int D, typename Tio>
__global__ void __launch_bounds__(2 * D)
decode_step_kernel(const Tio *__restrict__ q, const Tio *__restrict__ k, const Tio *__restrict__ v,
                   const Tio *__restrict__ z, const Tio *__restrict__ beta,
                   const float *__restrict__ bias, const float *__restrict__ A_log, float g_min,
                   int kind, float scale, float *__restrict__ state, const int32_t *__restrict__ state_idx,
                   int64_t num_slots, int H, Tio *__restrict__ o, int *err) {
    constexpr int NT = 2 * D;
    constexpr int NW = NT / 32;   // warps
    constexpr int RPW = D / NW;   // rows per warp (16)
    constexpr int VW = D / 32;    // columns per lane
    using V = vec<VW>;
    using VT = typename V::T;
    static_assert(RPW == 16, "layout assumes 16 rows per warp");

    __shared__ float s_alpha[D], s_k[D], s_q[D], s_v[D], s_e[D];
    __shared__ float s_p[NW][D], s_r[NW][D];
    __shared__ float s_kq;

    const int64_t bid = blockIdx.x;
    const int64_t n = bid / H;
    const int h = (int)(bid % H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    int64_t slot = n;
    if (state_idx) {
        slot = state_idx[n];
        if (slot < 0 || slot >= num_slots) {  // uniform across the block
            if (tid == 0) set_error(err, KDA_ERR_BAD_STATE_INDEX);
            return;
        }
    }
    float *Sh = state + (slot * H + h) * (int64_t)(D * D);
    const int row0 = warp * RPW;
    const int col0 = lane * VW;

    // Issue the 16 state-row loads first; the gate math below overlaps them.
    VT s[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i)
        s[i] = __ldcs(reinterpret_cast<const VT *>(Sh + (row0 + i) * D + col0));

    const int64_t tok = n * H + h;
    if (tid < D) {
        const float eA = A_log ? expf(A_log[h]) : 1.f;
        const float b = bias ? bias[h * D + tid] : 0.f;
        const float g = gate_log(kind, ld(z + tok * D + tid), b, eA, g_min);
        s_alpha[tid] = expf(g);
        s_k[tid] = ld(k + tok * D + tid);
        s_q[tid] = ld(q + tok * D + tid);
        s_v[tid] = ld(v + tok * D + tid);
    }
    const float bt = ld(beta + tok);
    __syncthreads();

    if (warp == 0) {  // k . q
        float acc = 0.f;
#pragma unroll
        for (int i = lane; i < D; i += 32) acc += s_k[i] * s_q[i];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
        if (lane == 0) s_kq = acc;
    }
    float p[VW], r[VW];
#pragma unroll
    for (int j = 0; j < VW; ++j) p[j] = r[j] = 0.f;
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int row = row0 + i;
        V::scale(s[i], s_alpha[row]);
        const float kr = s_k[row], qr = s_q[row];
#pragma unroll
        for (int j = 0; j < VW; ++j) {
            const float x = V::get(s[i], j);
            p[j] += x * kr;
            r[j] += x * qr;
        }
    }
#pragma unroll
    for (int j = 0; j < VW; ++j) {
        s_p[warp][col0 + j] = p[j];
        s_r[warp][col0 + j] = r[j];
    }
    __syncthreads();
    if (tid < D) {
        float P = 0.f, R = 0.f;
#pragma unroll
        for (int w = 0; w < NW; ++w) {
            P += s_p[w][tid];
            R += s_r[w][tid];
        }
        const float e = bt * (s_v[tid] - P);
        s_e[tid] = e;
        st(o + tok * D + tid, scale * (R + s_kq * e));
    }
    __syncthreads();
    float e[VW];
#pragma unroll
    for (int j = 0; j < VW; ++j) e[j] = s_e[col0 + j];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const float kr = s_k[row0 + i];
#pragma unroll
        for (int j = 0; j < VW; ++j) V::add(s[i], j, kr * e[j]);
        __stcs(reinterpret_cast<VT *>(Sh + (row0 + i) * D + col0), s[i]);
    }
}

template <int D, typename Tio>
static void launch(const kda_step_args *a, cudaStream_t stream, int *err) {
    const int64_t slots = a->num_slots > 0 ? a->num_slots : a->N;
    decode_step_kernel<D, Tio><<<(unsigned)(a->N * a->H), 2 * D, 0, stream>>>(
        (const Tio *)a->q, (const Tio *)a->k, (const Tio *)a->v, (const Tio *)a->z,
        (const Tio *)a->beta, a->dt_bias, a->A_log, a->g_min, a->gate_kind, a->scale, a->state,
        a->state_indices, slots, a->H, (Tio *)a->o, err);
}

}  // namespace kda

using namespace kda;

kda_status_t kda_launch_decode(const kda_step_args *a, cudaStream_t stream) {
    if (a->N == 0) return KDA_OK;
    int *err = kda_device_error_ptr();
    if (!err) return KDA_ERR_CUDA;
    const bool b16 = a->dtype == KDA_BF16;
    kda_profile_mark(0, stream);
    if (a->dk == 128) { if (b16) launch<128, bf16>(a, stream, err); else launch<128, float>(a, stream, err); }
    else { if (b16) launch<64, bf16>(a, stream, err); else launch<64, float>(a, stream, err); }
    kda_profile_mark(1, stream);
    return kda_cuda_status(cudaGetLastError());
}
