// kda_recurrent_replay: speculative decoding with replay, as the Kimi K3 technical report describes
// the KDA decode kernel (section 5.4).  The state of any accepted draft prefix is a function of the
// committed state and the drafts' projected inputs, which are far smaller than the state; so only the
// inputs are cached, the accepted drafts are replayed on chip, and the replayed tokens, the bonus token
// and the next draft window share one token loop.
//
// Per (sequence, head) state, the layout of the decode step (kda_decode.cu): 2 D threads, warp w
// holding rows [16 w, 16 w + 16) in registers, lane l holding D / 32 consecutive columns.  The kernel
// is persistent (two CTAs per SM, each looping over states) and software-pipelined: while a CTA runs
// the tokens of one state from registers, one warp has already issued the 1-D bulk copies (TMA) that
// bring the next state and its first 8 tokens' q, k, z, v rows into shared memory, so the state
// traffic of one item overlaps the arithmetic of the previous one instead of alternating with it.
// Per token
//     S' = Diag(alpha) S,  p = S'^T k,  r = S'^T q,  e = beta (v - p),
//     S <- S' + k e^T,     o = scale (r + (k . q) e)
// (Eq. 1, section 2.1.1).  The state is read once and written at most once per call, after the last
// committed token, so a window of m tokens costs one state round trip instead of m.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

namespace kda {
namespace rp {

using namespace kda::tc;

// one thread's VP column pairs of a state row
template <int VP>
__device__ __forceinline__ void ld_row(const float *p, float2 (&x)[VP]) {  // shared memory
    if constexpr (VP == 2) {
        const float4 v = *reinterpret_cast<const float4 *>(p);
        x[0] = make_float2(v.x, v.y);
        x[1] = make_float2(v.z, v.w);
    } else {
        x[0] = *reinterpret_cast<const float2 *>(p);
    }
}
template <int VP>
__device__ __forceinline__ void st_row(float *p, const float2 (&x)[VP]) {  // global, streamed
    if constexpr (VP == 2)
        __stcs(reinterpret_cast<float4 *>(p), make_float4(x[0].x, x[0].y, x[1].x, x[1].y));
    else
        __stcs(reinterpret_cast<float2 *>(p), x[0]);
}

__device__ __forceinline__ float to_f(float x) { return x; }
__device__ __forceinline__ float to_f(bf16 x) { return __bfloat162float(x); }

template <typename Tio> struct Tokens {
    const Tio *q, *k, *z, *v, *beta;
    int L;  // tokens per sequence in this buffer
};

// Dynamic shared memory of one CTA (byte offsets).
template <int D, typename Tio> struct Smem {
    static constexpr int G = 8;                             // tokens staged at a time
    static constexpr int NT = 2 * D, NW = NT / 32, KQP = D / 32;
    static constexpr int SB = 0;                            // next state, D x D fp32 (bulk copy target)
    static constexpr int RAW = SB + D * D * 4;              // its first G tokens' rows: [4][G][D] Tio, q k z v
    static constexpr int FA = RAW + 4 * G * D * (int)sizeof(Tio);  // alpha, k, q, v of the group, [4][G][D] fp32
    static constexpr int PR = FA + 4 * G * D * 4;           // per-warp partial sums p and r, [2][NW][D]
    static constexpr int E = PR + 2 * NW * D * 4;           // e, [D]
    static constexpr int BETA = E + D * 4;                  // [G]
    static constexpr int KQ = BETA + G * 4;                 // per-warp partial sums of k . q, [G][KQP]
    static constexpr int META = KQ + G * KQP * 4;           // n_replay, n_commit, valid, pad, slot (int64)
    static constexpr int BAR = META + 24;                   // one mbarrier (8-byte aligned: META is)
    static constexpr int BYTES = BAR + 8;
    static_assert(META % 8 == 0, "slot and barrier need 8-byte alignment");
};

template <int D, typename Tio>
__global__ void __launch_bounds__(2 * D, 2)
replay_kernel(Tokens<Tio> rt, const int32_t *__restrict__ n_replay, Tokens<Tio> nt,
              const int32_t *__restrict__ n_commit, const float *__restrict__ bias,
              const float *__restrict__ A_log, float g_min, int kind, float scale, float *__restrict__ state,
              const int32_t *__restrict__ state_idx, int64_t num_slots, int64_t n_items, int H,
              Tio *__restrict__ o, int *err) {
    using L = Smem<D, Tio>;
    constexpr int G = L::G, NT = L::NT, NW = L::NW, KQP = L::KQP;
    constexpr int RPW = D / NW;     // rows per warp (16)
    constexpr int VW = D / 32;      // columns per lane
    constexpr int VP = VW / 2;      // column pairs per lane
    constexpr int IT = G * D / NT;  // staging passes: thread t takes channel t % D of tokens 2 i + t / D
    static_assert(RPW == 16, "layout assumes 16 rows per warp");

    extern __shared__ __align__(128) unsigned char smem[];
    float *SB = reinterpret_cast<float *>(smem + L::SB);
    Tio *RAW = reinterpret_cast<Tio *>(smem + L::RAW);
    float(*FA)[G][D] = reinterpret_cast<float(*)[G][D]>(smem + L::FA);  // alpha, k, q, v
    float(*s_p)[D] = reinterpret_cast<float(*)[D]>(smem + L::PR);
    float(*s_r)[D] = s_p + NW;
    float *s_e = reinterpret_cast<float *>(smem + L::E);
    float *s_beta = reinterpret_cast<float *>(smem + L::BETA);
    float(*s_kqp)[KQP] = reinterpret_cast<float(*)[KQP]>(smem + L::KQ);
    int *meta = reinterpret_cast<int *>(smem + L::META);
    int64_t *meta_slot = reinterpret_cast<int64_t *>(smem + L::META + 16);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::BAR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = warp * RPW, col0 = lane * VW;
    const int c_in = tid % D;  // the channel this thread converts
    const int64_t step = gridDim.x;

    // token j of sequence n: replayed (cached buffer) for j < nr, new otherwise; [N, L, H] row index
    auto tok_row = [&](int64_t n, int h, int j, int nr) -> int64_t {
        return j < nr ? (n * rt.L + j) * H + h : (n * nt.L + (j - nr)) * H + h;
    };
    // one staged channel of token jj of the group: the decay alpha = exp(g) (Eq. 5), k, q, v, and the
    // warp's partial sum of k . q (a warp covers 32 channels of one token)
    auto convert = [&](int jj, float zv, float kv, float qv, float vv, float b, float eA) {
        FA[0][jj][c_in] = expf(gate_log(kind, zv, b, eA, g_min));
        FA[1][jj][c_in] = kv;
        FA[2][jj][c_in] = qv;
        FA[3][jj][c_in] = vv;
        float kq = kv * qv;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) kq += __shfl_xor_sync(0xffffffffu, kq, off);
        if (lane == 0) s_kqp[jj][c_in / 32] = kq;
    };

    // warp 0 prefetches: counts and slot of the next item to issue (loaded one item ahead of use)
    int q_nr = 0, q_nc = 0, q_si = 0;  // raw loads: nothing consumes them before the next issue
    Tio br = Tio(0.f);  // warp 0, lane jj: beta of token jj of the item in flight (converted when used)
    auto load_meta = [&](int64_t item) {
        const int64_t n = item / H;
        if (n_replay) q_nr = n_replay[n];
        q_nc = n_commit[n];
        if (state_idx) q_si = state_idx[n];
    };
    // bulk copies of the state and of the first G tokens' q, k, z, v rows of `item` into SB / RAW,
    // completing one phase of `bar`; an item with bad counts or slot is flagged and copies nothing
    auto issue = [&](int64_t item) {
        const int64_t n = item / H;
        const int h = (int)(item % H);
        const int nr = q_nr, nc = q_nc;
        const int64_t slot = state_idx ? (int64_t)q_si : n;
        const bool counts_ok = nr >= 0 && nr <= rt.L && nc >= 0 && nc <= nt.L;
        const bool slot_ok = slot >= 0 && slot < num_slots;
        const bool valid = counts_ok && slot_ok;
        if (lane == 0) {
            meta[0] = nr;
            meta[1] = nc;
            meta[2] = valid;
            *meta_slot = slot;
            if (!counts_ok) set_error(err, KDA_ERR_BAD_TOKEN_COUNT);
            else if (!slot_ok) set_error(err, KDA_ERR_BAD_STATE_INDEX);
        }
        if (!valid) {
            if (lane == 0) mbar_arrive(bar);
            return;
        }
        const int gn = min(G, nr + nt.L);
        constexpr uint32_t row_bytes = D * (uint32_t)sizeof(Tio);
        if (lane == 0) mbar_arrive_expect_tx(bar, D * D * 4 + 4 * gn * row_bytes);
        __syncwarp();
        for (int u = lane; u < 1 + 4 * gn; u += 32) {
            if (u == 0) {
                bulk_g2s(SB, state + (slot * H + h) * (int64_t)(D * D), D * D * 4, bar);
            } else {
                const int t = (u - 1) & 3, jj = (u - 1) >> 2;
                const bool is_new = jj >= nr;
                const Tio *src = t == 0 ? (is_new ? nt.q : rt.q)
                               : t == 1 ? (is_new ? nt.k : rt.k)
                               : t == 2 ? (is_new ? nt.z : rt.z)
                                        : (is_new ? nt.v : rt.v);
                bulk_g2s(RAW + (t * G + jj) * D, src + tok_row(n, h, jj, nr) * D, row_bytes, bar);
            }
        }
        if (lane < gn) br = (lane >= nr ? nt.beta : rt.beta)[tok_row(n, h, lane, nr)];
    };
    // dt_bias of this thread's channel and A_log for the head of the item in flight; nothing here
    // waits for these loads: they are used by the next item
    float b_nx = 0.f, a_nx = 0.f;
    auto load_gate = [&](int64_t item) {
        const int h = (int)(item % H);
        b_nx = bias ? bias[h * D + c_in] : 0.f;
        a_nx = A_log ? A_log[h] : 0.f;
    };

    if (tid == 0) {
        mbar_init(bar, 1);
        fence_proxy_async();
    }
    __syncthreads();
    int64_t item = blockIdx.x;
    if (item < n_items) {
        if (warp == 0) {
            load_meta(item);
            issue(item);
            if (item + step < n_items) load_meta(item + step);
        }
        load_gate(item);
    }

    uint32_t parity = 0;
    for (; item < n_items; item += step, parity ^= 1u) {
        const int64_t n = item / H;
        const int h = (int)(item % H);
        if (!__syncthreads_and(mbar_wait(bar, parity))) {  // bounded: a lost copy cannot hang the GPU
            if (tid == 0) {
                set_error(err, KDA_ERR_DEVICE_TIMEOUT);
                mbar_wait(bar, parity);  // give copies still in flight their time before the CTA exits
            }
            return;
        }
        const int nr = meta[0], nc = meta[1];
        const bool valid = meta[2] != 0;
        const int64_t slot = *meta_slot;
        const float b_in = b_nx, eA = expf(a_nx);  // A_log = 0 without A_log: exp(A) = 1
        const int total = nr + nt.L, last_commit = nr + nc - 1;

        float2 s[RPW][VP];  // column pairs: the per-token arithmetic runs on packed fp32 pairs
        if (valid) {
#pragma unroll
            for (int i = 0; i < RPW; ++i) ld_row(SB + (row0 + i) * D + col0, s[i]);
            const int gn = min(G, total);
#pragma unroll
            for (int it = 0; it < IT; ++it) {
                const int jj = it * (NT / D) + tid / D;
                if (jj < gn)  // warp-uniform: D is a multiple of 32
                    convert(jj, ld(RAW + (2 * G + jj) * D + c_in), ld(RAW + (G + jj) * D + c_in),
                            ld(RAW + jj * D + c_in), ld(RAW + (3 * G + jj) * D + c_in), b_in, eA);
            }
            if (warp == 0 && lane < gn) s_beta[lane] = to_f(br);
        }
        __syncthreads();  // SB and RAW consumed: the next item's copies may land there
        if (item + step < n_items) {
            if (warp == 0) {
                issue(item + step);
                if (item + 2 * step < n_items) load_meta(item + 2 * step);
            }
            load_gate(item + step);
        }
        if (!valid) continue;
        float *Sh = state + (slot * H + h) * (int64_t)(D * D);

        for (int g0 = 0; g0 < total; g0 += G) {
            const int gn = min(G, total - g0);
            if (g0 > 0) {  // windows longer than G tokens: later groups through plain loads, all in flight
                float zr[IT], kr[IT], qr[IT], vr[IT], bb = 0.f;
#pragma unroll
                for (int it = 0; it < IT; ++it) {
                    const int jj = it * (NT / D) + tid / D, j = g0 + jj;
                    if (jj < gn) {
                        const bool is_new = j >= nr;
                        const int64_t off = tok_row(n, h, j, nr) * D + c_in;
                        zr[it] = ld((is_new ? nt.z : rt.z) + off);
                        kr[it] = ld((is_new ? nt.k : rt.k) + off);
                        qr[it] = ld((is_new ? nt.q : rt.q) + off);
                        vr[it] = ld((is_new ? nt.v : rt.v) + off);
                    }
                }
                if (tid < gn) bb = ld((g0 + tid >= nr ? nt.beta : rt.beta) + tok_row(n, h, g0 + tid, nr));
#pragma unroll
                for (int it = 0; it < IT; ++it) {
                    const int jj = it * (NT / D) + tid / D;
                    if (jj < gn) convert(jj, zr[it], kr[it], qr[it], vr[it], b_in, eA);
                }
                if (tid < gn) s_beta[tid] = bb;
                __syncthreads();
            }
            for (int jj = 0; jj < gn; ++jj) {
                const int j = g0 + jj;
                const bool is_new = j >= nr;
                float2 p[VP], r[VP];
#pragma unroll
                for (int c = 0; c < VP; ++c) p[c] = r[c] = make_float2(0.f, 0.f);
#pragma unroll
                for (int i4 = 0; i4 < RPW; i4 += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(&FA[0][jj][row0 + i4]);
                    const float4 k4 = *reinterpret_cast<const float4 *>(&FA[1][jj][row0 + i4]);
                    const float4 q4 = *reinterpret_cast<const float4 *>(&FA[2][jj][row0 + i4]);
                    const float av[4] = {a4.x, a4.y, a4.z, a4.w}, kv[4] = {k4.x, k4.y, k4.z, k4.w},
                                qv[4] = {q4.x, q4.y, q4.z, q4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 a2 = make_float2(av[u], av[u]), k2 = make_float2(kv[u], kv[u]),
                                     q2 = make_float2(qv[u], qv[u]);
#pragma unroll
                        for (int c = 0; c < VP; ++c) {
                            s[i4 + u][c] = __fmul2_rn(s[i4 + u][c], a2);  // S' = Diag(alpha) S
                            p[c] = __ffma2_rn(s[i4 + u][c], k2, p[c]);    // S'^T k
                            r[c] = __ffma2_rn(s[i4 + u][c], q2, r[c]);    // S'^T q
                        }
                    }
                }
#pragma unroll
                for (int c = 0; c < VP; ++c) {
                    *reinterpret_cast<float2 *>(&s_p[warp][col0 + 2 * c]) = p[c];
                    *reinterpret_cast<float2 *>(&s_r[warp][col0 + 2 * c]) = r[c];
                }
                __syncthreads();  // partial sums of token j complete
                // threads [0, D) reduce p and form e; threads [D, 2 D) reduce r for the output
                float Rv = 0.f;
                if (tid < D) {
                    float P = 0.f;
#pragma unroll
                    for (int w = 0; w < NW; ++w) P += s_p[w][tid];
                    s_e[tid] = s_beta[jj] * (FA[3][jj][tid] - P);
                } else if (is_new) {
#pragma unroll
                    for (int w = 0; w < NW; ++w) Rv += s_r[w][tid - D];
                }
                __syncthreads();  // e of token j complete; the partial sums were all read before it
                if (tid >= D && is_new) {
                    float kq = 0.f;
#pragma unroll
                    for (int w = 0; w < KQP; ++w) kq += s_kqp[jj][w];
                    const int c = tid - D;
                    st(o + tok_row(n, h, j, nr) * D + c, scale * (Rv + kq * s_e[c]));
                }
                float2 e[VP];
#pragma unroll
                for (int c = 0; c < VP; ++c) e[c] = *reinterpret_cast<const float2 *>(&s_e[col0 + 2 * c]);
#pragma unroll
                for (int i4 = 0; i4 < RPW; i4 += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&FA[1][jj][row0 + i4]);
                    const float kv[4] = {k4.x, k4.y, k4.z, k4.w};
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const float2 k2 = make_float2(kv[u], kv[u]);
#pragma unroll
                        for (int c = 0; c < VP; ++c) s[i4 + u][c] = __ffma2_rn(k2, e[c], s[i4 + u][c]);  // + k e^T
                    }
                }
                if (j == last_commit) {  // the committed state: accepted drafts and the committed new tokens
#pragma unroll
                    for (int i = 0; i < RPW; ++i) st_row(Sh + (row0 + i) * D + col0, s[i]);
                }
            }
            __syncthreads();  // the group's staged values and e are read before anything overwrites them
        }
    }
}

template <int D, typename Tio>
static kda_status_t launch(const kda_replay_args *a, cudaStream_t stream, int *err) {
    using L = Smem<D, Tio>;
    auto kern = replay_kernel<D, Tio>;
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::BYTES) != cudaSuccess)
        return kda_cuda_status(cudaGetLastError());
    int dev = 0, sms = 0, per_sm = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 2 * D, L::BYTES) != cudaSuccess)
        return kda_cuda_status(cudaGetLastError());
    const int64_t n_items = a->N * (int64_t)a->H;
    const int64_t resident = (int64_t)sms * (per_sm > 0 ? per_sm : 1);
    const unsigned grid = (unsigned)(n_items < resident ? n_items : resident);
    const int64_t slots = a->num_slots > 0 ? a->num_slots : a->N;
    Tokens<Tio> rt{(const Tio *)a->rq, (const Tio *)a->rk, (const Tio *)a->rz, (const Tio *)a->rv,
                   (const Tio *)a->rbeta, a->R};
    Tokens<Tio> nt{(const Tio *)a->q, (const Tio *)a->k, (const Tio *)a->z, (const Tio *)a->v,
                   (const Tio *)a->beta, a->M};
    kern<<<grid, 2 * D, L::BYTES, stream>>>(rt, a->R > 0 ? a->n_replay : nullptr, nt, a->n_commit, a->dt_bias,
                                             a->A_log, a->g_min, a->gate_kind, a->scale, a->state, a->state_indices, slots,
                                             n_items, a->H, (Tio *)a->o, err);
    return kda_cuda_status(cudaGetLastError());
}

}  // namespace rp
}  // namespace kda

using namespace kda;

kda_status_t kda_launch_replay(const kda_replay_args *a, cudaStream_t stream) {
    if (a->N == 0) return KDA_OK;
    int *err = kda_device_error_ptr();
    if (!err) return KDA_ERR_CUDA;
    const bool b16 = a->dtype == KDA_BF16;
    if (a->dk == 128) return b16 ? rp::launch<128, bf16>(a, stream, err) : rp::launch<128, float>(a, stream, err);
    return b16 ? rp::launch<64, bf16>(a, stream, err) : rp::launch<64, float>(a, stream, err);
}
