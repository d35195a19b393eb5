// kda_recurrent_replay: speculative decoding with replay, as the Kimi K3 technical report describes
// the KDA decode kernel (section 5.4).  The state of any accepted draft prefix is a function of the
// committed state and the drafts' projected inputs, which are far smaller than the state; so only the
// inputs are cached, the accepted drafts are replayed on chip, and the replayed tokens, the bonus token
// and the next draft window share one token loop.
//
// Per (sequence, head) state, the layout of the decode step (kda_decode.cu): 2 D threads, warp w
// holding rows [16 w, 16 w + 16) in registers, lane l holding D / 32 consecutive columns.  The kernel
// is persistent (two CTAs per SM, each taking a contiguous run of (head, sequence) states in
// head-major order) and software-pipelined: while a CTA runs the tokens of one state from
// registers, the next state is on its way by a 1-D bulk copy (TMA) and its first 8 tokens' q, k, z,
// v rows by 16-byte cp.async copies from every thread, all completing one mbarrier phase, so the
// state traffic of one item overlaps the arithmetic of the previous one.  Small per-item values
// (counts, slot, first-group beta) are staged for 32 items at a time and the gate parameters are
// reloaded only when the head changes: no global load waits on the per-item critical path.
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
    // a CTA's items' counts, validity, slot and first-group beta, staged MAXI items at a time
    static constexpr int MAXI = 32;
    static constexpr int BNR = KQ + G * KQP * 4;            // int [MAXI]
    static constexpr int BNC = BNR + MAXI * 4;              // int [MAXI]
    static constexpr int BVAL = BNC + MAXI * 4;             // int [MAXI]
    static constexpr int BSLOT = BVAL + MAXI * 4;           // int64 [MAXI]
    static constexpr int BBETA = BSLOT + MAXI * 8;          // float [MAXI][G]
    static constexpr int BAR = BBETA + MAXI * G * 4;        // one mbarrier
    static constexpr int BYTES = BAR + 8;
    static_assert(BSLOT % 8 == 0 && BAR % 8 == 0, "slots and the barrier need 8-byte alignment");
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
    constexpr int MAXI = L::MAXI;
    int *b_nr = reinterpret_cast<int *>(smem + L::BNR);
    int *b_nc = reinterpret_cast<int *>(smem + L::BNC);
    int *b_val = reinterpret_cast<int *>(smem + L::BVAL);
    int64_t *b_slot = reinterpret_cast<int64_t *>(smem + L::BSLOT);
    float(*b_beta)[G] = reinterpret_cast<float(*)[G]>(smem + L::BBETA);
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + L::BAR);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int row0 = warp * RPW, col0 = lane * VW;
    const int c_in = tid % D;  // the channel this thread converts
    // items (head h, sequence n) numbered h-major, it = h N + n; this CTA takes a contiguous run, so its
    // head (dt_bias, A_log) changes rarely and its sequences' counts and slots can be staged at once
    const int64_t N_seq = n_items / H;
    const int64_t base = n_items / gridDim.x, rem = n_items % gridDim.x;
    const int64_t first = blockIdx.x * base + min((int64_t)blockIdx.x, rem);
    const int64_t count = base + ((int64_t)blockIdx.x < rem ? 1 : 0);

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

    // counts, validity, slot and first-group beta of items first + k0 .. + MAXI - 1 (two rounds of loads)
    auto load_batch = [&](int64_t k0) {
        const int nb = (int)min((int64_t)MAXI, count - k0);
        if (tid < nb) {
            const int64_t it = first + k0 + tid, n = it % N_seq;
            const int nr = n_replay ? n_replay[n] : 0, nc = n_commit[n];
            const int64_t slot = state_idx ? (int64_t)state_idx[n] : n;
            const bool counts_ok = nr >= 0 && nr <= rt.L && nc >= 0 && nc <= nt.L;
            const bool slot_ok = slot >= 0 && slot < num_slots;
            if (!counts_ok) set_error(err, KDA_ERR_BAD_TOKEN_COUNT);
            else if (!slot_ok) set_error(err, KDA_ERR_BAD_STATE_INDEX);
            b_nr[tid] = nr;
            b_nc[tid] = nc;
            b_val[tid] = counts_ok && slot_ok;
            b_slot[tid] = slot;
        }
        __syncthreads();
        for (int e = tid; e < nb * G; e += NT) {
            const int kk = e / G, jj = e % G;
            const int64_t it = first + k0 + kk, n = it % N_seq;
            const int h = (int)(it / N_seq), nr = b_nr[kk];
            if (b_val[kk] && jj < min(G, nr + nt.L))
                b_beta[kk][jj] = ld((jj >= nr ? nt.beta : rt.beta) + tok_row(n, h, jj, nr));
        }
        __syncthreads();
    };
    // the state (one 1-D bulk copy by thread 0) and the first G tokens' q, k, z, v rows (16-byte cp.async
    // granules spread over all threads) of item k, completing one phase of `bar`, which counts thread 0's
    // arrival with the state's bytes and every thread's cp.async completion; an invalid item copies nothing
    constexpr int CPR = D * (int)sizeof(Tio) / 16;  // granules per row
    auto issue = [&](int64_t k) {
        const int kb = (int)(k % MAXI);
        const int64_t it = first + k, n = it % N_seq;
        const int h = (int)(it / N_seq);
        if (b_val[kb]) {
            const int nr = b_nr[kb], gn = min(G, nr + nt.L);
            if (tid == 0) {
                mbar_arrive_expect_tx(bar, D * D * 4);
                bulk_g2s(SB, state + (b_slot[kb] * H + h) * (int64_t)(D * D), D * D * 4, bar);
            }
            for (int u = tid; u < 4 * gn * CPR; u += NT) {
                const int t = u / (gn * CPR), r2 = u - t * (gn * CPR), jj = r2 / CPR, part = r2 - jj * CPR;
                const bool is_new = jj >= nr;
                const Tio *src = t == 0 ? (is_new ? nt.q : rt.q)
                               : t == 1 ? (is_new ? nt.k : rt.k)
                               : t == 2 ? (is_new ? nt.z : rt.z)
                                        : (is_new ? nt.v : rt.v);
                cp_async16(RAW + (t * G + jj) * D + part * (16 / (int)sizeof(Tio)),
                           src + tok_row(n, h, jj, nr) * D + part * (16 / (int)sizeof(Tio)));
            }
        } else if (tid == 0) {
            mbar_arrive(bar);
        }
        asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
    };

    if (tid == 0) {
        mbar_init(bar, 1 + NT);  // thread 0's arrival (with the state's bytes) + every thread's cp.async arrival
        fence_proxy_async();
    }
    __syncthreads();
    if (count > 0) {
        load_batch(0);
        issue(0);
    }
    int h_cur = -1;
    float b_in = 0.f, eA = 1.f;  // dt_bias of this thread's channel and exp(A) of the current head

    uint32_t parity = 0;
    for (int64_t kx = 0; kx < count; ++kx, parity ^= 1u) {
        const int64_t item = first + kx, n = item % N_seq;
        const int h = (int)(item / N_seq), kb = (int)(kx % MAXI);
        if (!__syncthreads_and(mbar_wait(bar, parity))) {  // bounded: a lost copy cannot hang the GPU
            if (tid == 0) {
                set_error(err, KDA_ERR_DEVICE_TIMEOUT);
                mbar_wait(bar, parity);  // give copies still in flight their time before the CTA exits
            }
            return;
        }
        const int nr = b_nr[kb], nc = b_nc[kb];
        const bool valid = b_val[kb] != 0;
        const int64_t slot = b_slot[kb];
        if (h != h_cur) {  // a new head: its gate parameters (rare within a CTA's run)
            h_cur = h;
            b_in = bias ? bias[h * D + c_in] : 0.f;
            eA = A_log ? expf(A_log[h]) : 1.f;
        }
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
            if (tid < gn) s_beta[tid] = b_beta[kb][tid];
        }
        __syncthreads();  // SB and RAW consumed: the next item's copies may land there
        if (kx + 1 < count) {
            if ((kx + 1) % MAXI == 0) load_batch(kx + 1);  // (this item's staged values are in registers)
            issue(kx + 1);
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
