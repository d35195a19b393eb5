// kda_recurrent_replay: speculative decoding with replay, as the Kimi K3 technical report describes
// the KDA decode kernel (section 5.4).  The state of any accepted draft prefix is a function of the
// committed state and the drafts' projected inputs, which are far smaller than the state; so only the
// inputs are cached, the accepted drafts are replayed on chip, and the replayed tokens, the bonus token
// and the next draft window share one token loop.
//
// Layout and per-token algebra are those of the decode step (kda_decode.cu): one CTA per (sequence,
// head) state, 2 D threads, warp w holding rows [16 w, 16 w + 16), lane l holding D / 32 consecutive
// columns.  The inputs of up to 8 tokens at a time (they do not depend on the state) are staged in
// shared memory with all their loads in flight together; per token
//     S' = Diag(alpha) S,  p = S'^T k,  r = S'^T q,  e = beta (v - p),
//     S <- S' + k e^T,     o = scale (r + (k . q) e)
// (Eq. 1, section 2.1.1).  The state is read once and written at most once per call, after the last
// committed token, so a window of m tokens costs one state round trip instead of m.
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace rp {

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

template <typename Tio> struct Tokens {
    const Tio *q, *k, *z, *v, *beta;
    int L;  // tokens per sequence in this buffer
};

template <int D, typename Tio>
__global__ void __launch_bounds__(2 * D, 2)
replay_kernel(Tokens<Tio> rt, const int32_t *__restrict__ n_replay, Tokens<Tio> nt,
              const int32_t *__restrict__ n_commit, const float *__restrict__ bias,
              const float *__restrict__ A_log, float g_min, float scale, float *__restrict__ state,
              const int32_t *__restrict__ state_idx, int64_t num_slots, int H, Tio *__restrict__ o, int *err) {
    constexpr int NT = 2 * D;
    constexpr int NW = NT / 32;   // warps
    constexpr int RPW = D / NW;   // rows per warp (16)
    constexpr int VW = D / 32;    // columns per lane
    using V = vec<VW>;
    using VT = typename V::T;
    static_assert(RPW == 16, "layout assumes 16 rows per warp");

    constexpr int G = 8;          // tokens whose inputs are staged at a time
    constexpr int IT = G * D / NT;  // staging iterations: thread t holds channel t % D of tokens 2 i + t / D
    constexpr int KQP = D / 32;     // per-warp partial sums of k . q per token
    __shared__ float s_alpha[G][D], s_k[G][D], s_q[G][D], s_v[G][D], s_beta[G], s_kqp[G][KQP];
    __shared__ float s_p[NW][D], s_r[NW][D], s_e[D];

    const int64_t bid = blockIdx.x;
    const int64_t n = bid / H;
    const int h = (int)(bid % H);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

    const int nr = n_replay ? n_replay[n] : 0;
    const int nc = n_commit[n];
    if (nr < 0 || nr > rt.L || nc < 0 || nc > nt.L) {  // uniform across the block
        if (tid == 0) set_error(err, KDA_ERR_BAD_TOKEN_COUNT);
        return;
    }
    int64_t slot = n;
    if (state_idx) {
        slot = state_idx[n];
        if (slot < 0 || slot >= num_slots) {
            if (tid == 0) set_error(err, KDA_ERR_BAD_STATE_INDEX);
            return;
        }
    }
    float *Sh = state + (slot * H + h) * (int64_t)(D * D);
    const int row0 = warp * RPW;
    const int col0 = lane * VW;
    const int c_in = tid % D;  // the channel this thread stages
    const float b_in = bias ? bias[h * D + c_in] : 0.f;
    const float eA = A_log ? expf(A_log[h]) : 1.f;
    const int total = nr + nt.L, last_commit = nr + nc - 1;

    // raw inputs of one group, all loads issued before any is used
    float zr[IT], kr_[IT], qr_[IT], vr[IT], br = 0.f;
    auto fetch = [&](int g0) {
        const int gn = min(G, total - g0);
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int jj = it * (NT / D) + tid / D, j = g0 + jj;
            if (jj < gn) {
                const bool is_new = j >= nr;
                const int64_t tok = (n * (is_new ? nt.L : rt.L) + (is_new ? j - nr : j)) * H + h;  // [N, L, H]
                zr[it] = ld((is_new ? nt.z : rt.z) + tok * D + c_in);
                kr_[it] = ld((is_new ? nt.k : rt.k) + tok * D + c_in);
                qr_[it] = ld((is_new ? nt.q : rt.q) + tok * D + c_in);
                vr[it] = ld((is_new ? nt.v : rt.v) + tok * D + c_in);
            }
        }
        if (tid < gn) {
            const int j = g0 + tid;
            const bool is_new = j >= nr;
            const int64_t tok = (n * (is_new ? nt.L : rt.L) + (is_new ? j - nr : j)) * H + h;
            br = ld((is_new ? nt.beta : rt.beta) + tok);
        }
    };
    auto stage = [&](int g0) {
        const int gn = min(G, total - g0);
#pragma unroll
        for (int it = 0; it < IT; ++it) {
            const int jj = it * (NT / D) + tid / D;
            if (jj < gn) {  // warp-uniform: D is a multiple of 32
                s_alpha[jj][c_in] = expf(gate_logdecay(zr[it], b_in, eA, g_min));
                s_k[jj][c_in] = kr_[it];
                s_q[jj][c_in] = qr_[it];
                s_v[jj][c_in] = vr[it];
                float kq = kr_[it] * qr_[it];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
                if (lane == 0) s_kqp[jj][c_in / 32] = kq;
            }
        }
        if (tid < gn) s_beta[tid] = br;
    };

    if (total > 0) fetch(0);  // the first group's inputs are in flight with the state
    VT s[RPW];
#pragma unroll
    for (int i = 0; i < RPW; ++i)
        s[i] = __ldcs(reinterpret_cast<const VT *>(Sh + (row0 + i) * D + col0));

    for (int g0 = 0; g0 < total; g0 += G) {
        const int gn = min(G, total - g0);
        if (g0 > 0) fetch(g0);
        stage(g0);
        __syncthreads();
        for (int jj = 0; jj < gn; ++jj) {
            const int j = g0 + jj;
            const bool is_new = j >= nr;
            float p[VW], r[VW];
#pragma unroll
            for (int c = 0; c < VW; ++c) p[c] = r[c] = 0.f;
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const int row = row0 + i;
                V::scale(s[i], s_alpha[jj][row]);
                const float kr = s_k[jj][row], qr = s_q[jj][row];
#pragma unroll
                for (int c = 0; c < VW; ++c) {
                    const float x = V::get(s[i], c);
                    p[c] += x * kr;
                    r[c] += x * qr;
                }
            }
#pragma unroll
            for (int c = 0; c < VW; ++c) {
                s_p[warp][col0 + c] = p[c];
                s_r[warp][col0 + c] = r[c];
            }
            __syncthreads();  // partial sums of token j complete
            if (tid < D) {
                float P = 0.f, R = 0.f;
#pragma unroll
                for (int w = 0; w < NW; ++w) {
                    P += s_p[w][tid];
                    R += s_r[w][tid];
                }
                const float e = s_beta[jj] * (s_v[jj][tid] - P);
                s_e[tid] = e;
                if (is_new) {
                    float kq = 0.f;
#pragma unroll
                    for (int w = 0; w < KQP; ++w) kq += s_kqp[jj][w];
                    const int64_t tok = (n * nt.L + (j - nr)) * H + h;
                    st(o + tok * D + tid, scale * (R + kq * e));
                }
            }
            __syncthreads();  // e of token j complete; the partial sums were all read before it
            float e[VW];
#pragma unroll
            for (int c = 0; c < VW; ++c) e[c] = s_e[col0 + c];
#pragma unroll
            for (int i = 0; i < RPW; ++i) {
                const float kr = s_k[jj][row0 + i];
#pragma unroll
                for (int c = 0; c < VW; ++c) V::add(s[i], c, kr * e[c]);
            }
            if (j == last_commit) {  // the committed state: accepted drafts and the committed new tokens
#pragma unroll
                for (int i = 0; i < RPW; ++i) __stcs(reinterpret_cast<VT *>(Sh + (row0 + i) * D + col0), s[i]);
            }
        }
        __syncthreads();  // the group's staged inputs and e are read before the next group overwrites them
    }
}

template <int D, typename Tio>
static void launch(const kda_replay_args *a, cudaStream_t stream, int *err) {
    const int64_t slots = a->num_slots > 0 ? a->num_slots : a->N;
    Tokens<Tio> rt{(const Tio *)a->rq, (const Tio *)a->rk, (const Tio *)a->rz, (const Tio *)a->rv,
                   (const Tio *)a->rbeta, a->R};
    Tokens<Tio> nt{(const Tio *)a->q, (const Tio *)a->k, (const Tio *)a->z, (const Tio *)a->v,
                   (const Tio *)a->beta, a->M};
    replay_kernel<D, Tio><<<(unsigned)(a->N * a->H), 2 * D, 0, stream>>>(
        rt, a->R > 0 ? a->n_replay : nullptr, nt, a->n_commit, a->dt_bias, a->A_log, a->g_min, a->scale,
        a->state, a->state_indices, slots, a->H, (Tio *)a->o, err);
}

}  // namespace rp
}  // namespace kda

using namespace kda;

kda_status_t kda_launch_replay(const kda_replay_args *a, cudaStream_t stream) {
    if (a->N == 0) return KDA_OK;
    int *err = kda_device_error_ptr();
    if (!err) return KDA_ERR_CUDA;
    const bool b16 = a->dtype == KDA_BF16;
    if (a->dk == 128) { if (b16) rp::launch<128, bf16>(a, stream, err); else rp::launch<128, float>(a, stream, err); }
    else { if (b16) rp::launch<64, bf16>(a, stream, err); else rp::launch<64, float>(a, stream, err); }
    return kda_cuda_status(cudaGetLastError());
}
