// Backward pass of the chunked prefill (kda_chunk_bwd).  The Kimi K3 report (section 2.1.1, Eq. 3
// and Eq. 4) gives the forward only; the gradients here are the exact derivatives of that chunkwise
// form.  Per chunk (rows r of c tokens, state S entering it, Lambda = dL/dS leaving it), with the
// forward quantities of the fp32 path (G the in-chunk cumulative log-decay, E_ric = e^{G_rc - G_ic},
// A, L, T = (I + L)^{-1}, W = T diag(b)(Gamma K), U = T diag(b) V, Q^, K~, gamma):
//     V~ = U - W S,                     dV~ = K~ Lambda + scale A^T dO,
//     dS_in = Diag(gamma) Lambda + scale Q^^T dO - W^T dV~           (reverse recurrence),
//     dQ^ = scale dO S^T,  dA = scale dO V~^T,  dK~ = V~ Lambda^T,  dW = -dV~ S^T,
//     dX_W = T^T dW,  dX_U = T^T dV~,  dL = -(dX_W W^T + dX_U U^T)   (strictly lower),
// and the elementwise and pairwise derivatives of X_W = diag(b)(Gamma K), X_U = diag(b) V, Q^, K~,
// gamma, A and L with respect to q, k, v, beta and G; dg is the reverse cumulative sum of dG, and
// the gate's derivative gives dz, d dt_bias and d A_log.
//
// Kernels.  The forward is recomputed by the fp32 path's intra-chunk kernel, which also writes L; the
// state entering every chunk comes from its chain or, for bf16 at d = 128, from
// chunk_chain_ckpt_tc_kernel (S^T in tensor memory).  Then:
//   chunk_rev_chain_kernel   one CTA per (sequence, head, 32 value columns): Lambda over the chunks
//                            in reverse (columns of Lambda evolve independently, as those of S),
//                            storing the Lambda leaving each chunk; for bf16 at d = 128
//                            chunk_rev_chain_tc_kernel instead, Lambda^T in tensor memory;
//   chunk_bwd_value_kernel_t one CTA of 512 threads per (chunk, head), the value channels 32 at a
//                            time: V~, dV~, dX_U (T^T by back substitution), dv, and the contractions
//                            over the value channels (dQ^, dW, dK~, dA, the X_U part of dL, d gamma,
//                            the X_U part of d beta), accumulated in registers and written once;
//                            it also solves dX_W = T^T dW and adds dL's X_W part at the end; for bf16
//                            at d = 128 chunk_bwd_value_tc_kernel instead (tcgen05 products);
//   chunk_bwd_key_kernel     one CTA per (chunk, head): reads those sums, then per (row, channel)
//                            the pairwise A and L terms, dq, dk, dG; the reverse cumulative sum;
//                            dz, d beta and per-chunk sums for d dt_bias, d A_log;
//   bwd_gate_param_kernel    sums the per-chunk gate-parameter gradients per head.
#include "kda_common.cuh"
#include <algorithm>
#include "kda_internal.h"
#include "kda_f32_records.cuh"
#include "tc_util.cuh"

namespace kda {
namespace bw {

constexpr int NT = 256;   // threads per CTA
constexpr int TILE = 32;  // value columns per CTA (one per lane)

// The chunk-local sums the value side writes for the key side, per (chunk slot, head), in floats.
struct Part {
    int C, dk;
    __host__ __device__ int dQ() const { return 0; }
    __host__ __device__ int dW() const { return C * dk; }
    __host__ __device__ int dK() const { return 2 * C * dk; }
    __host__ __device__ int dA() const { return 3 * C * dk; }
    __host__ __device__ int dLu() const { return 3 * C * dk + C * C; }
    __host__ __device__ int dgam() const { return 3 * C * dk + 2 * C * C; }
    __host__ __device__ int dbu() const { return 3 * C * dk + 2 * C * C + dk; }
    __host__ __device__ int size() const { return 3 * C * dk + 2 * C * C + dk + C; }
};

// ------------------------------------------------------------------ reverse chain over the chunks
template <typename Tio, int DK>
__global__ void __launch_bounds__(NT)
chunk_rev_chain_kernel(int64_t T, int N, const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_start,
                       int H, int dv, const char *__restrict__ records, size_t rec_bytes,
                       float scale, const Tio *__restrict__ d_o, const float *__restrict__ d_final,
                       float *__restrict__ lam_end, float *__restrict__ d_init, int staged) {
    extern __shared__ float sm[];
    constexpr int C = 64, dk = DK;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const int j0 = blockIdx.y * TILE;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NWARP = NT / 32;
    constexpr int RW = C / NWARP, CW = DK / NWARP;  // rows of dV~ and of Lambda per warp
    // 16-byte rows (asynchronous copies, 16-byte broadcast reads); lane-indexed operands are contiguous
    constexpr int PK = dk + 4, PC = C + 4, PS = TILE + 4;
    constexpr int RAW = TILE * (int)sizeof(Tio) / 16;  // 16-byte pieces of a row of dO's slice
    float *Ws = sm;               // [C][PK]
    float *Qs = Ws + C * PK;      // [C][PK]
    float *Kt = Qs + C * PK;      // [C][PK]
    float *As = Kt + C * PK;      // [C][PC]
    float *dOs = As + C * PC;     // [C][PS]
    float *dVt = dOs + C * PS;    // [C][PS]
    float *Lm = dVt + C * PS;     // [dk][PS]
    float *gam = Lm + dk * PS;    // [dk]
    Tio *dOraw = reinterpret_cast<Tio *>(gam + dk);  // [C][TILE] dO as stored, the next chunk's

    const size_t sbase = ((size_t)n * H + h) * (size_t)dk * dv;
    const int64_t s_tok = cu ? (int64_t)cu[n] : (T / N) * n;
    const int64_t e_tok = cu ? (int64_t)cu[n + 1] : s_tok + T / N;
    const int c0 = chunk_start[n], c1 = chunk_start[n + 1];
    auto first_tok = [&](int cix) { return s_tok + (int64_t)(cix - c0) * C; };
    auto length = [&](int cix) { return (int)min((int64_t)C, e_tok - first_tok(cix)); };
    // A chunk's tiles come in three groups of asynchronous copies, each issued as soon as the previous
    // chunk's copy has been read for the last time: its dO slice (as stored), K~ and A after the dV~
    // phase, Q^, W and gamma after the Lambda phase.
    auto issue_do = [&](int cix) {
        if (!staged) return;
        const int64_t t0 = first_tok(cix);
        const int len = length(cix);
        for (int e = tid; e < len * RAW; e += NT) {
            const int r = e / RAW, pc = e % RAW;
            cp_async16(reinterpret_cast<char *>(dOraw) + (r * RAW + pc) * 16,
                       reinterpret_cast<const char *>(d_o + ((t0 + r) * H + h) * (int64_t)dv + j0) + pc * 16);
        }
    };
    auto issue_ka = [&](int cix) {
        const F32Record rec = f32_record(records, rec_bytes, cix, H, h, C, dk, dv);
        tile_async(Kt, PK, rec.K, dk, C, dk, tid, NT);
        tile_async(As, PC, rec.A, C, C, C, tid, NT);
    };
    auto issue_qw = [&](int cix) {
        const F32Record rec = f32_record(records, rec_bytes, cix, H, h, C, dk, dv);
        tile_async(Ws, PK, rec.W, dk, C, dk, tid, NT);
        tile_async(Qs, PK, rec.Q, dk, C, dk, tid, NT);
        tile_async(gam, dk, rec.gam, dk, 1, dk, tid, NT);
    };
    if (d_final) {
        tile_async(Lm, PS, d_final + sbase + j0, dv, dk, TILE, tid, NT);
    } else {
        for (int e = tid; e < dk * TILE; e += NT) Lm[(e / TILE) * PS + e % TILE] = 0.f;
    }
    if (c1 > c0) {
        issue_do(c1 - 1);
        issue_ka(c1 - 1);
    }
    cp_async_commit();
    if (c1 > c0) issue_qw(c1 - 1);
    cp_async_commit();
    for (int cix = c1 - 1; cix >= c0; --cix) {
        const int64_t t0 = first_tok(cix);
        const int len = length(cix);
        if (tid == 0 && cix > c0)  // the next record in this (reverse) order, into L2 meanwhile
            prefetch_l2(records + ((size_t)(cix - 1) * H + h) * rec_bytes, (uint32_t)rec_bytes);
        cp_async_wait_group1();  // this chunk's dO, K~ and A (and, the first time, d final_state)
        __syncthreads();         // the previous chunk is done with dOs; Lambda is final
        float *lg = lam_end + ((size_t)cix * H + h) * (size_t)dk * dv;
        for (int e = tid; e < dk * TILE; e += NT) {
            const int c = e / TILE, j = e % TILE;
            lg[(size_t)c * dv + j0 + j] = Lm[c * PS + j];
        }
#pragma unroll 8
        for (int e = tid; e < C * TILE; e += NT) {
            const int r = e / TILE, j = e % TILE;
            dOs[r * PS + j] = r >= len ? 0.f
                              : staged ? ld(dOraw + r * TILE + j)
                                       : ld(d_o + ((t0 + r) * H + h) * (int64_t)dv + j0 + j);
        }
        __syncthreads();  // dO converted: the staging buffer is free
        if (cix > c0) issue_do(cix - 1);
        // Register-blocked: warp w owns rows [RW w, RW w + RW) of dV~ and rows [CW w, CW w + CW) of
        // Lambda; lane-indexed operands are read once per reduction index, row operands as 16-byte
        // broadcasts.
        const int r0 = warp * RW, cb = warp * CW;
        {  // dV~ = K~ Lambda + scale A^T dO   (A is zero above its diagonal; rows past len are zero)
            float acc[RW], acca[RW];
#pragma unroll
            for (int i = 0; i < RW; ++i) acc[i] = acca[i] = 0.f;
            for (int c = 0; c < dk; c += 4) {
                const float l0 = Lm[c * PS + lane], l1 = Lm[(c + 1) * PS + lane];
                const float l2 = Lm[(c + 2) * PS + lane], l3 = Lm[(c + 3) * PS + lane];
#pragma unroll
                for (int i = 0; i < RW; ++i) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&Kt[(r0 + i) * PK + c]);
                    acc[i] += k4.x * l0 + k4.y * l1 + k4.z * l2 + k4.w * l3;
                }
            }
            for (int i2 = r0; i2 < len; ++i2) {
                const float d = dOs[i2 * PS + lane];
                const float4 a0 = *reinterpret_cast<const float4 *>(&As[i2 * PC + r0]);
                const float4 a1 = *reinterpret_cast<const float4 *>(&As[i2 * PC + r0 + 4]);
                acca[0] += a0.x * d; acca[1] += a0.y * d; acca[2] += a0.z * d; acca[3] += a0.w * d;
                acca[4] += a1.x * d; acca[5] += a1.y * d; acca[6] += a1.z * d; acca[7] += a1.w * d;
            }
#pragma unroll
            for (int i = 0; i < RW; ++i) dVt[(r0 + i) * PS + lane] = acc[i] + scale * acca[i];
        }
        __syncthreads();  // K~ and A are free
        if (cix > c0) issue_ka(cix - 1);
        cp_async_commit();
        cp_async_wait_group1();  // this chunk's Q^, W and gamma (the group just closed may still fly)
        __syncthreads();
        {  // Lambda <- Diag(gamma) Lambda + scale Q^^T dO - W^T dV~
            float lm[CW];
#pragma unroll
            for (int i = 0; i < CW; ++i) lm[i] = gam[cb + i] * Lm[(cb + i) * PS + lane];
            for (int r = 0; r < len; ++r) {
                const float d = scale * dOs[r * PS + lane], dv2 = dVt[r * PS + lane];
#pragma unroll
                for (int j = 0; j < CW; j += 4) {
                    const float4 q4 = *reinterpret_cast<const float4 *>(&Qs[r * PK + cb + j]);
                    const float4 w4 = *reinterpret_cast<const float4 *>(&Ws[r * PK + cb + j]);
                    lm[j] += q4.x * d - w4.x * dv2;
                    lm[j + 1] += q4.y * d - w4.y * dv2;
                    lm[j + 2] += q4.z * d - w4.z * dv2;
                    lm[j + 3] += q4.w * d - w4.w * dv2;
                }
            }
#pragma unroll
            for (int i = 0; i < CW; ++i) Lm[(cb + i) * PS + lane] = lm[i];
        }
        __syncthreads();  // Q^, W and gamma are free
        if (cix > c0) issue_qw(cix - 1);
        cp_async_commit();
    }
    cp_async_wait_all();  // a sequence without chunks: the copy of d final_state
    __syncthreads();
    if (d_init) {
        for (int e = tid; e < dk * TILE; e += NT) {
            const int c = e / TILE, j = e % TILE;
            d_init[sbase + (size_t)c * dv + j0 + j] = Lm[c * PS + j];
        }
    }
}

// ------------------------------------------------------------------ value side, per (chunk, head)
// 512 threads; the value channels are taken 32 at a time.  Thread t owns rows 4 (t / 32) + [0, 4)
// and columns t % 32 + 32 j of the contractions over the value channels (dQ^, dW, dK~ [C][dk]; dA
// and dL [C][C]) and keeps them in registers across the tiles: per reduction index it reads four
// row values (broadcasts) and its column values (lane-strided rows at an odd pitch: no bank
// conflicts).  After the last tile it solves dX_W = T^T dW and adds dL's X_W part, -dX_W W^T,
// while W and L are still in shared memory, and writes every sum once.
constexpr int NTV = 512;
template <int DK>
__global__ void __launch_bounds__(NTV, 1)
chunk_bwd_value_kernel_t(int64_t T, int N, const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_start,
                         int H, int dv, const char *__restrict__ records, size_t rec_bytes,
                         const float *__restrict__ Lbuf, const float *__restrict__ ckpt,
                         const float *__restrict__ lam_end, float scale, const void *__restrict__ v_,
                         const void *__restrict__ beta_, const void *__restrict__ d_o_, void *__restrict__ grad_v_,
                         int bf16_io, float *__restrict__ part) {
    constexpr int C = 64, dk = DK;
    constexpr int CB = DK / 32, IB = C / 32;  // columns per thread of the [C][dk] and [C][C] sums
    constexpr int NWARP = NTV / 32, RW = C / NWARP;  // rows of V~ / dV~ per warp (4)
    extern __shared__ float sm[];
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    int n, len;
    int64_t t0;
    if (!locate_chunk(chunk_start, cu, T, N, C, slot, n, t0, len)) return;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int PK = dk + 4, PC = C + 4, PS = TILE + 1, PW = dk + 1;
    float *Ws = sm;               // [C][PK]
    float *Kt = Ws + C * PK;      // [C][PK]
    float *As = Kt + C * PK;      // [C][PC]
    float *Ls = As + C * PC;      // [C][PC]
    float *Ss = Ls + C * PC;      // [dk][PS]
    float *Lm = Ss + dk * PS;     // [dk][PS]
    float *dOs = Lm + dk * PS;    // [C][PS]
    float *Vs = dOs + C * PS;     // [C][PS]  v
    float *Us = Vs + C * PS;      // [C][PS]
    float *Vt = Us + C * PS;      // [C][PS]  V~
    float *dVt = Vt + C * PS;     // [C][PS]  dV~, then dX_U
    float *bet = dVt + C * PS;    // [C]
    float *dWs = Ss;              // [C][PW] after the tiles: dW, then dX_W (reuses the tile buffers)

    const F32Record rec = f32_record(records, rec_bytes, slot, H, h, C, dk, dv);
    const size_t mbase = ((size_t)slot * H + h) * (size_t)dk * dv;
    tile_async(Ws, PK, rec.W, dk, C, dk, tid, NTV);
    tile_async(Kt, PK, rec.K, dk, C, dk, tid, NTV);
    tile_async(As, PC, rec.A, C, C, C, tid, NTV);
    tile_async(Ls, PC, Lbuf + ((size_t)slot * H + h) * (size_t)C * C, C, C, C, tid, NTV);
    for (int r = tid; r < C; r += NTV)
        bet[r] = r < len ? (bf16_io ? ld((const bf16 *)beta_ + (t0 + r) * H + h) : ld((const float *)beta_ + (t0 + r) * H + h)) : 0.f;

    const int rb = (tid >> 5) * 4;  // this thread's rows of the sums; its columns are lane + 32 j
    float aq[4][CB], aw[4][CB], ak[4][CB], aa[4][IB], al[4][IB], agam = 0.f, abu = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
#pragma unroll
        for (int j = 0; j < CB; ++j) aq[i][j] = aw[i][j] = ak[i][j] = 0.f;
#pragma unroll
        for (int j = 0; j < IB; ++j) aa[i][j] = al[i][j] = 0.f;
    }

    for (int j0 = 0; j0 < dv; j0 += TILE) {
        __syncthreads();  // the previous tile is done with the tile buffers
#pragma unroll 4
        for (int e = tid; e < dk * TILE; e += NTV) {
            const int c = e / TILE, j = e % TILE;
            Ss[c * PS + j] = ckpt[mbase + (size_t)c * dv + j0 + j];
            Lm[c * PS + j] = lam_end[mbase + (size_t)c * dv + j0 + j];
        }
#pragma unroll 4
        for (int e = tid; e < C * TILE; e += NTV) {
            const int r = e / TILE, j = e % TILE;
            const bool ok = r < len;
            const int64_t idx = ((t0 + r) * H + h) * (int64_t)dv + j0 + j;
            if (bf16_io) {
                dOs[r * PS + j] = ok ? ld((const bf16 *)d_o_ + idx) : 0.f;
                Vs[r * PS + j] = ok ? ld((const bf16 *)v_ + idx) : 0.f;
            } else {
                dOs[r * PS + j] = ok ? ld((const float *)d_o_ + idx) : 0.f;
                Vs[r * PS + j] = ok ? ld((const float *)v_ + idx) : 0.f;
            }
            Us[r * PS + j] = rec.U[r * dv + j0 + j];
        }
        cp_async_wait_all();
        __syncthreads();
        {  // V~ = U - W S and dV~ = K~ Lambda + scale A^T dO, rows RW w + [0, RW) at column lane
            const int r0 = warp * RW;
            float vt[RW], dvt[RW], da[RW];
#pragma unroll
            for (int i = 0; i < RW; ++i) {
                vt[i] = Us[(r0 + i) * PS + lane];
                dvt[i] = da[i] = 0.f;
            }
            for (int c = 0; c < dk; c += 4) {
                const float s0 = Ss[c * PS + lane], s1 = Ss[(c + 1) * PS + lane];
                const float s2 = Ss[(c + 2) * PS + lane], s3 = Ss[(c + 3) * PS + lane];
                const float l0 = Lm[c * PS + lane], l1 = Lm[(c + 1) * PS + lane];
                const float l2 = Lm[(c + 2) * PS + lane], l3 = Lm[(c + 3) * PS + lane];
#pragma unroll
                for (int i = 0; i < RW; ++i) {
                    const float4 w = *reinterpret_cast<const float4 *>(&Ws[(r0 + i) * PK + c]);
                    const float4 k4 = *reinterpret_cast<const float4 *>(&Kt[(r0 + i) * PK + c]);
                    vt[i] -= w.x * s0 + w.y * s1 + w.z * s2 + w.w * s3;
                    dvt[i] += k4.x * l0 + k4.y * l1 + k4.z * l2 + k4.w * l3;
                }
            }
            for (int i2 = r0; i2 < len; ++i2) {  // A is zero above its diagonal
                const float d = dOs[i2 * PS + lane];
                const float4 a4 = *reinterpret_cast<const float4 *>(&As[i2 * PC + r0]);
                da[0] += a4.x * d; da[1] += a4.y * d; da[2] += a4.z * d; da[3] += a4.w * d;
            }
#pragma unroll
            for (int i = 0; i < RW; ++i) {
                Vt[(r0 + i) * PS + lane] = vt[i];
                dVt[(r0 + i) * PS + lane] = dvt[i] + scale * da[i];
            }
        }
        __syncthreads();
        // this tile's share of the contractions over value channels
#pragma unroll 4
        for (int l = 0; l < TILE; ++l) {
            float xo[4], xd[4], xv[4], ys[CB], yl[CB], yv[IB];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                xo[i] = dOs[(rb + i) * PS + l];
                xd[i] = dVt[(rb + i) * PS + l];
                xv[i] = Vt[(rb + i) * PS + l];
            }
#pragma unroll
            for (int j = 0; j < CB; ++j) {
                ys[j] = Ss[(lane + 32 * j) * PS + l];
                yl[j] = Lm[(lane + 32 * j) * PS + l];
            }
#pragma unroll
            for (int j = 0; j < IB; ++j) yv[j] = Vt[(lane + 32 * j) * PS + l];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
#pragma unroll
                for (int j = 0; j < CB; ++j) {
                    aq[i][j] += xo[i] * ys[j];
                    aw[i][j] -= xd[i] * ys[j];
                    ak[i][j] += xv[i] * yl[j];
                }
#pragma unroll
                for (int j = 0; j < IB; ++j) aa[i][j] += xo[i] * yv[j];
            }
        }
        if (tid < dk) {
            float dg = 0.f;
            for (int l = 0; l < TILE; ++l) dg += Ss[tid * PS + l] * Lm[tid * PS + l];
            agam += dg;
        }
        __syncthreads();
        // dX_U = T^T dV~: back substitution x_r = b_r - sum_{i > r} L_ir x_i, 8 threads per column
        if (tid < 8 * TILE) {
            const int col = tid >> 3, part8 = tid & 7;
            for (int r = C - 2; r >= 0; --r) {
                float acc = 0.f;
                for (int i = r + 1 + part8; i < C; i += 8) acc += Ls[i * PC + r] * dVt[i * PS + col];
                acc += __shfl_xor_sync(0xffffffffu, acc, 4);
                acc += __shfl_xor_sync(0xffffffffu, acc, 2);
                acc += __shfl_xor_sync(0xffffffffu, acc, 1);
                if (part8 == 0) dVt[r * PS + col] -= acc;
                __syncwarp();
            }
        }
        __syncthreads();
        // dv = beta dX_U;  X_U parts of d beta and dL
        for (int e = tid; e < len * TILE; e += NTV) {
            const int r = e / TILE, j = e % TILE;
            const int64_t idx = ((t0 + r) * H + h) * (int64_t)dv + j0 + j;
            if (bf16_io) st((bf16 *)grad_v_ + idx, bet[r] * dVt[r * PS + j]);
            else st((float *)grad_v_ + idx, bet[r] * dVt[r * PS + j]);
        }
        if (tid < C) {
            float db = 0.f;
            for (int l = 0; l < TILE; ++l) db += dVt[tid * PS + l] * Vs[tid * PS + l];
            abu += db;
        }
#pragma unroll 4
        for (int l = 0; l < TILE; ++l) {
            float xu[4], yu[IB];
#pragma unroll
            for (int i = 0; i < 4; ++i) xu[i] = dVt[(rb + i) * PS + l];
#pragma unroll
            for (int j = 0; j < IB; ++j) yu[j] = Us[(lane + 32 * j) * PS + l];
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < IB; ++j) al[i][j] -= xu[i] * yu[j];
        }
    }
    // dX_W = T^T dW (columns back-substituted, NTV / dk threads per column), then dL -= dX_W W^T
    __syncthreads();
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < CB; ++j) dWs[(rb + i) * PW + lane + 32 * j] = aw[i][j];
    __syncthreads();
    {
        constexpr int TPC = NTV / DK;
        const int col = tid / TPC, sub = tid % TPC;
        for (int r = C - 2; r >= 0; --r) {
            float acc = 0.f;
            for (int i = r + 1 + sub; i < C; i += TPC) acc += Ls[i * PC + r] * dWs[i * PW + col];
#pragma unroll
            for (int off = TPC >> 1; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
            if (sub == 0) dWs[r * PW + col] -= acc;
            __syncwarp();
        }
    }
    __syncthreads();
    for (int c = 0; c < dk; c += 4) {  // rows of dX_W broadcast, rows of W lane-strided (16-byte reads)
        float x[4][4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
#pragma unroll
            for (int u = 0; u < 4; ++u) x[i][u] = dWs[(rb + i) * PW + c + u];
#pragma unroll
        for (int j = 0; j < IB; ++j) {
            const float4 w = *reinterpret_cast<const float4 *>(&Ws[(lane + 32 * j) * PK + c]);
#pragma unroll
            for (int i = 0; i < 4; ++i) al[i][j] -= x[i][0] * w.x + x[i][1] * w.y + x[i][2] * w.z + x[i][3] * w.w;
        }
    }
    const Part P{C, dk};
    float *pp = part + ((size_t)slot * H + h) * (size_t)P.size();
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int r = rb + i;
#pragma unroll
        for (int j = 0; j < CB; ++j) {
            const int e = r * dk + lane + 32 * j;
            pp[P.dQ() + e] = scale * aq[i][j];
            pp[P.dW() + e] = dWs[r * PW + lane + 32 * j];  // dX_W
            pp[P.dK() + e] = ak[i][j];
        }
#pragma unroll
        for (int j = 0; j < IB; ++j) {
            const int c2 = lane + 32 * j, e = r * C + c2;
            pp[P.dA() + e] = c2 <= r ? scale * aa[i][j] : 0.f;
            pp[P.dLu() + e] = c2 < r ? al[i][j] : 0.f;  // the whole dL
        }
    }
    if (tid < dk) pp[P.dgam() + tid] = agam;
    if (tid < C) pp[P.dbu() + tid] = abu;
}

// ------------------------------------------------------------------ value side on the tensor cores
// bf16 I/O with d_k = d_v = 128: one 256-thread CTA per (chunk, head); the value-channel contractions
// are tcgen05 products (bf16 operand images in shared memory, fp32 accumulators in tensor memory),
// each computed transposed so that its 128 rows are channels (one TMEM lane each) and its 64
// columns the chunk's tokens:
//   first:  V~^T = U^T - S^T W^T,  dV~^T = Lambda^T K~^T + dO^T (scale A),  dQ^^T = S dO^T
//   second: dW^T = -S dV~^T,  dK~^T = Lambda V~^T,  [V~; U] dO^T,  [V~; U] dX_U^T
//   third:  [K~; W] dX_W^T accumulated onto the last one
// The stacked products give dA^T (the rows of V~) and the X_U and X_W parts of dL^T (the rows of U
// and W); their other halves are not used.  A thread that owns a channel (a TMEM lane) holds one
// column of dV~ or dW in registers, so both solves with T^T = (I + L^T)^{-1} are back substitutions
// in registers, and it writes the solved column as one 128-byte row of an MN-major operand image.
// S and Lambda are stored once: an image with rows c and K-blocks of 64 value channels is also the
// MN-major image of S^T (rows k = c holding 64 consecutive value channels).
namespace vt {
constexpr uint32_t SIMG = 0;          // S: rows c (128) x 128 value channels, K-major, blocks of 16 KB
constexpr uint32_t LIMG = 32768;      // Lambda, the same
constexpr uint32_t KWIMG = 65536;     // rows 0..63 K~, rows 64..127 W (x 128 key channels), K-major
constexpr uint32_t DOIMG = 98304;     // dO: rows r (64) x 128 value channels, K-major, blocks of 8 KB
constexpr uint32_t AIMG = 114688;     // scale A: rows i (64) x 64 tokens r
constexpr uint32_t VUIMG = 122880;    // MN-major over tokens: group 0 V~, group 1 U, rows j (128), 16 KB each
constexpr uint32_t DVIMG = 155648;    // dV~: rows j (128) x 64 tokens
constexpr uint32_t DXUIMG = 172032;   // dX_U: rows j x 64 tokens
constexpr uint32_t DXWIMG = 188416;   // dX_W: rows c x 64 tokens
constexpr uint32_t LF = 204800;       // L, fp32 [64][64], strictly lower
constexpr uint32_t BET = LF + 16384;  // beta [64]
constexpr uint32_t RED = BET + 256;   // [4][64] the channel warps' shares of d beta (X_U part)
constexpr uint32_t DGAM = RED + 1024; // d gamma [128]
constexpr uint32_t BAR = DGAM + 512;  // 3 mbarriers
constexpr uint32_t TSLOT = BAR + 32;  // TMEM base
constexpr uint32_t TOTAL = TSLOT + 16 + 1024;  // + alignment of the base to 1024 bytes
}  // namespace vt

__device__ __forceinline__ unsigned char *vt_align1024(unsigned char *p) {
    const uint32_t s = tc::smem_u32(p);
    return p + ((1024u - (s & 1023u)) & 1023u);
}
__device__ __forceinline__ uint4 vt_pack8(const float *f) {
    return make_uint4(tc::pack_bf16(f[0], f[1]), tc::pack_bf16(f[2], f[3]), tc::pack_bf16(f[4], f[5]),
                      tc::pack_bf16(f[6], f[7]));
}
__device__ __forceinline__ void vt_load8(const float *p, float *f) {
    const float4 a = *reinterpret_cast<const float4 *>(p), b = *reinterpret_cast<const float4 *>(p + 4);
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w; f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
}
__device__ __forceinline__ void vt_sync() {
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
}
// Waits on an mbarrier from every thread (bounded); a CTA-uniform "all ok".
__device__ __forceinline__ bool vt_wait(uint64_t *bar, uint32_t parity) {
    const bool ok = tc::mbar_wait(bar, parity);
    const bool all = __syncthreads_and(ok ? 1 : 0) != 0;
    tc::fence_after_sync();
    return all;
}
// x <- (I + L^T)^{-1} x for L strictly lower ([64][64] fp32, shared memory), x the 64 fp32 columns
// [tcol, tcol + 64) of this thread's TMEM lane, in place: x_r -= sum_{i > r} L_ir x_i, by blocks of 16 rows
// from the last up (a block's own triangle in registers, then its updates of the earlier blocks).  The
// block loops run at run time, so the code stays small; the warp executes it together.
__device__ __forceinline__ void vt_solve_ut_tmem(uint32_t tcol, const float *L) {
    for (int b = 3; b >= 0; --b) {
        float xb[16];
        tc::tmem_ld16(tcol + 16 * b, xb);
        const float *Lb = L + 16 * b * 64 + 16 * b;  // L[16 b + ii][16 b + rr]
#pragma unroll
        for (int ii = 15; ii >= 1; --ii) {
            const float xi = xb[ii];
#pragma unroll
            for (int rr = 0; rr < ii; rr += 4) {
                const float4 l4 = *reinterpret_cast<const float4 *>(Lb + ii * 64 + rr);
                xb[rr] -= l4.x * xi;
                if (rr + 1 < ii) xb[rr + 1] -= l4.y * xi;
                if (rr + 2 < ii) xb[rr + 2] -= l4.z * xi;
                if (rr + 3 < ii) xb[rr + 3] -= l4.w * xi;
            }
        }
        tc::tmem_st16(tcol + 16 * b, xb);
#pragma unroll 1
        for (int b2 = 0; b2 < b; ++b2) {
            float xc[16];
            tc::tmem_ld16(tcol + 16 * b2, xc);
            const float *Lc = L + 16 * b * 64 + 16 * b2;  // L[16 b + ii][16 b2 + rr]
#pragma unroll
            for (int ii = 0; ii < 16; ++ii) {
#pragma unroll
                for (int rr = 0; rr < 16; rr += 4) {
                    const float4 l4 = *reinterpret_cast<const float4 *>(Lc + ii * 64 + rr);
                    xc[rr] -= l4.x * xb[ii];
                    xc[rr + 1] -= l4.y * xb[ii];
                    xc[rr + 2] -= l4.z * xb[ii];
                    xc[rr + 3] -= l4.w * xb[ii];
                }
            }
            tc::tmem_st16(tcol + 16 * b2, xc);
        }
        tc::tmem_st_wait();
    }
}
// Sums x[0..63] over the warp's lanes by halving exchanges; returns b such that x[0], x[1] then hold
// the sums of entries b, b + 1 (each lane a different pair).
__device__ __forceinline__ int vt_reduce_scatter64(float *x, int lane) {
    int b = 0;
#pragma unroll
    for (int step = 0; step < 5; ++step) {
        const int o = 16 >> step, half = 32 >> step;
        const bool up = (lane & o) != 0;
#pragma unroll
        for (int k = 0; k < half; ++k) {
            const float send = up ? x[k] : x[k + half];
            const float keep = up ? x[k + half] : x[k];
            x[k] = keep + __shfl_xor_sync(0xffffffffu, send, o);
        }
        if (up) b += half;
    }
    return b;
}

// Asks L2 for what item (slot, h) reads: S, Lambda, L, the record's W, U, K~ and A, and its rows of
// dO and v (warp 0; the item is in the sequence table).
__device__ __forceinline__ void vt_prefetch_item(int64_t slot, int h, int64_t t0, int len, int H,
                                                 const char *records, size_t rec_bytes, const float *Lbuf,
                                                 const float *ckpt, const float *lam_end, const bf16 *v,
                                                 const bf16 *d_o, int lane) {
    constexpr int C = 64, D = 128;
    const size_t mbase = ((size_t)slot * H + h) * (size_t)D * D;
    const F32Record rec = f32_record(records, rec_bytes, slot, H, h, C, D, D);
    if (lane == 0) {
        prefetch_l2(ckpt + mbase, D * D * 4);
        prefetch_l2(lam_end + mbase, D * D * 4);
        prefetch_l2(rec.W, 2 * C * D * 4);         // W, U
        prefetch_l2(rec.K, (C * D + C * C) * 4);   // K~, A
        prefetch_l2(Lbuf + ((size_t)slot * H + h) * (size_t)C * C, C * C * 4);
    }
    for (int r = lane; r < len; r += 32) {
        const int64_t idx = ((t0 + r) * H + h) * (int64_t)D;
        prefetch_l2(d_o + idx, D * 2);
        prefetch_l2(v + idx, D * 2);
    }
}

// Persistent: CTA b takes the items (slot, head) w = b, b + gridDim.x, ... (slot = w / H), and asks L2
// for its next item while it works on the current one.
__global__ void __launch_bounds__(256, 1)
chunk_bwd_value_tc_kernel(int64_t T, int N, const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_start,
                          int H, const char *__restrict__ records, size_t rec_bytes,
                          const float *__restrict__ Lbuf, const float *__restrict__ ckpt,
                          const float *__restrict__ lam_end, float scale, const bf16 *__restrict__ v,
                          const bf16 *__restrict__ beta, const bf16 *__restrict__ d_o, bf16 *__restrict__ grad_v,
                          float *__restrict__ part, int *err) {
    using namespace tc;
    constexpr int C = 64, D = 128;
    extern __shared__ unsigned char vt_raw[];
    unsigned char *sm = vt_align1024(vt_raw);
    const int64_t items = (int64_t)chunk_start[N] * H;
    if ((int64_t)blockIdx.x >= items) return;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = (warp & 3) * 32, row = lq + lane;  // TMEM lane quarter of this warp; this thread's lane
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + vt::BAR);
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + vt::TSLOT);
    float *Lf = reinterpret_cast<float *>(sm + vt::LF), *bet = reinterpret_cast<float *>(sm + vt::BET);
    float *red = reinterpret_cast<float *>(sm + vt::RED), *dgam = reinterpret_cast<float *>(sm + vt::DGAM);
    const Part P{C, D};
    if (tid == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        mbar_init(&bar[2], 1);
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    fence_proxy_async();
    vt_sync();
    const uint32_t tb = *tslot;
    const uint32_t s0 = smem_u32(sm);
    auto where = [&](int64_t w, int64_t &slot, int &h, int64_t &t0, int &len) {
        slot = w / H;
        h = (int)(w - slot * H);
        int n;
        locate_chunk(chunk_start, cu, T, N, C, slot, n, t0, len);
    };
    bool ok = true;
    uint32_t ph = 0;
    {
        int64_t slot, t0;
        int h, len;
        where(blockIdx.x, slot, h, t0, len);
        if (warp == 0) vt_prefetch_item(slot, h, t0, len, H, records, rec_bytes, Lbuf, ckpt, lam_end, v, d_o, lane);
    }
    for (int64_t w = blockIdx.x; w < items && ok; w += gridDim.x, ph ^= 1u) {
        int64_t slot, t0;
        int h, len;
        where(w, slot, h, t0, len);
        if (warp == 0 && w + gridDim.x < items) {
            int64_t s2, t2;
            int h2, l2;
            where(w + gridDim.x, s2, h2, t2, l2);
            vt_prefetch_item(s2, h2, t2, l2, H, records, rec_bytes, Lbuf, ckpt, lam_end, v, d_o, lane);
        }
        float *pp = part + ((size_t)slot * H + h) * (size_t)P.size();
        const F32Record rec = f32_record(records, rec_bytes, slot, H, h, C, D, D);
        const size_t mbase = ((size_t)slot * H + h) * (size_t)D * D;

        // operand images; each loop's loads are issued before its stores
        tile_async(Lf, C, Lbuf + ((size_t)slot * H + h) * (size_t)C * C, C, C, C, tid, 256);
#pragma unroll 1
        for (int bq = 0; bq < 2; ++bq) {  // S and Lambda; d gamma = row sums of S o Lambda
            float sv[4][8], lv[4][8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = tid + 256 * (4 * bq + q), c = e >> 4, jc = e & 15;
                vt_load8(ckpt + mbase + (size_t)c * D + 8 * jc, sv[q]);
                vt_load8(lam_end + mbase + (size_t)c * D + 8 * jc, lv[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = tid + 256 * (4 * bq + q), c = e >> 4, jc = e & 15;
                const uint32_t off = img_chunk_off(128, c, jc);
                *reinterpret_cast<uint4 *>(sm + vt::SIMG + off) = vt_pack8(sv[q]);
                *reinterpret_cast<uint4 *>(sm + vt::LIMG + off) = vt_pack8(lv[q]);
                float dot = 0.f;
#pragma unroll
                for (int u = 0; u < 8; ++u) dot += sv[q][u] * lv[q][u];
#pragma unroll
                for (int o = 8; o > 0; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
                if ((lane & 15) == 0) dgam[c] = dot;
            }
        }
        {  // K~ (rows 0..63) and W (rows 64..127)
            float x[8][8];
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = tid + 256 * q, r = e >> 4, jc = e & 15;
                vt_load8((r < C ? rec.K + (size_t)r * D : rec.W + (size_t)(r - C) * D) + 8 * jc, x[q]);
            }
#pragma unroll
            for (int q = 0; q < 8; ++q) {
                const int e = tid + 256 * q, r = e >> 4, jc = e & 15;
                *reinterpret_cast<uint4 *>(sm + vt::KWIMG + img_chunk_off(128, r, jc)) = vt_pack8(x[q]);
            }
        }
        {  // dO (zero past the sequence), scale A (rows i), U transposed (row j holds U[0..63][j])
            uint4 uo[4];
            float xa[2][8], xu[4][8];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = tid + 256 * q, r = e >> 4, jc = e & 15;
                uo[q] = make_uint4(0u, 0u, 0u, 0u);
                if (r < len) uo[q] = *reinterpret_cast<const uint4 *>(d_o + ((t0 + r) * H + h) * (int64_t)D + 8 * jc);
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int e = tid + 256 * q, i = e >> 3, rc = e & 7;
                vt_load8(rec.A + (size_t)i * C + 8 * rc, xa[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = tid + 256 * q, j = e & 127, ic = e >> 7;
#pragma unroll
                for (int u = 0; u < 8; ++u) xu[q][u] = rec.U[(size_t)(8 * ic + u) * D + j];
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = tid + 256 * q, r = e >> 4, jc = e & 15;
                *reinterpret_cast<uint4 *>(sm + vt::DOIMG + img_chunk_off(64, r, jc)) = uo[q];
            }
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int e = tid + 256 * q, i = e >> 3, rc = e & 7;
#pragma unroll
                for (int u = 0; u < 8; ++u) xa[q][u] *= scale;
                *reinterpret_cast<uint4 *>(sm + vt::AIMG + img_chunk_off(64, i, rc)) = vt_pack8(xa[q]);
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int e = tid + 256 * q, j = e & 127, ic = e >> 7;
                *reinterpret_cast<uint4 *>(sm + vt::VUIMG + 16384 + img_chunk_off(128, j, ic)) = vt_pack8(xu[q]);
            }
        }
        if (tid < C) bet[tid] = tid < len ? ld(beta + (t0 + tid) * H + h) : 0.f;
        cp_async_wait_all();
        fence_proxy_async();
        vt_sync();

        if (tid == 0) {
            mma_bf16_mnk(tb + 0, s0 + vt::SIMG, 16384, s0 + vt::KWIMG + 8192, 128, 8, idesc_bf16(128, 64, true, false),
                         false);
            mma_bf16_mnk(tb + 64, s0 + vt::LIMG, 16384, s0 + vt::KWIMG, 128, 8, idesc_bf16(128, 64, true, false),
                         false);
            mma_bf16_mnmn(tb + 64, s0 + vt::DOIMG, 8192, s0 + vt::AIMG, 8192, 4, idesc_bf16(128, 64, true, true),
                          true);
            mma_bf16_k(tb + 128, s0 + vt::SIMG, 128, s0 + vt::DOIMG, 64, 8, idesc_bf16(128, 64), false);
            mma_commit(&bar[0]);
        }
        ok = vt_wait(&bar[0], ph);
        if (!ok) break;
        if (warp < 4) {  // value channel j = row
            const int j = row;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {  // V~ = U - W S, column j -> row j of the V~ group
                float d[32];
                tmem_ld32(tmem_addr(tb + 0, lq, 32 * hf), d);
#pragma unroll
                for (int u = 0; u < 32; ++u) d[u] = rec.U[(size_t)(32 * hf + u) * D + j] - d[u];
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    *reinterpret_cast<uint4 *>(sm + vt::VUIMG + img_chunk_off(128, j, 4 * hf + q)) =
                        vt_pack8(d + 8 * q);
            }
            float x[64];
            tmem_ld32(tmem_addr(tb + 64, lq, 0), x);
            tmem_ld32(tmem_addr(tb + 64, lq, 32), x + 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4 *>(sm + vt::DVIMG + img_chunk_off(128, j, q)) = vt_pack8(x + 8 * q);
            vt_solve_ut_tmem(tmem_addr(tb + 64, lq, 0), Lf);  // dX_U = T^T dV~
            tmem_ld32(tmem_addr(tb + 64, lq, 0), x);
            tmem_ld32(tmem_addr(tb + 64, lq, 32), x + 32);
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4 *>(sm + vt::DXUIMG + img_chunk_off(128, j, q)) = vt_pack8(x + 8 * q);
#pragma unroll
            for (int r0 = 0; r0 < C; r0 += 16) {  // dv = beta dX_U; the X_U part of d beta, sum_j dX_U v
                float vv[16];
#pragma unroll
                for (int u = 0; u < 16; ++u)
                    vv[u] = r0 + u < len ? ld(v + ((t0 + r0 + u) * H + h) * (int64_t)D + j) : 0.f;
#pragma unroll
                for (int u = 0; u < 16; ++u) {
                    const int r = r0 + u;
                    if (r < len) st(grad_v + ((t0 + r) * H + h) * (int64_t)D + j, bet[r] * x[r]);
                    x[r] *= vv[u];
                }
            }
            const int b = vt_reduce_scatter64(x, lane);
            red[warp * 64 + b] = x[0];
            red[warp * 64 + b + 1] = x[1];
        } else {  // key channel c = row: dQ^ = scale dO S^T
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float d[32];
                tmem_ld32(tmem_addr(tb + 128, lq, 32 * hf), d);
#pragma unroll
                for (int u = 0; u < 32; ++u) pp[P.dQ() + (32 * hf + u) * D + row] = scale * d[u];
            }
        }
        fence_proxy_async();
        vt_sync();
        if (tid == 0) {
            mma_bf16_kmn(tb + 0, s0 + vt::SIMG, 128, s0 + vt::DVIMG, 16384, 8, idesc_bf16(128, 64, false, true),
                         false);
            mma_bf16_kmn(tb + 64, s0 + vt::LIMG, 128, s0 + vt::VUIMG, 16384, 8, idesc_bf16(128, 64, false, true),
                         false);
            mma_bf16_mnk(tb + 128, s0 + vt::VUIMG, 16384, s0 + vt::DOIMG, 64, 8, idesc_bf16(128, 64, true, false),
                         false);
            mma_bf16_mnmn(tb + 192, s0 + vt::VUIMG, 16384, s0 + vt::DXUIMG, 16384, 8,
                          idesc_bf16(128, 64, true, true), false);
            mma_commit(&bar[1]);
        }
        ok = vt_wait(&bar[1], ph);
        if (!ok) break;
        if (warp < 4) {  // key channel c = row: dX_W = T^T dW, dW = -(S dV~^T)^T
            float x[64];
            vt_solve_ut_tmem(tmem_addr(tb + 0, lq, 0), Lf);  // linear: solve S dV~^T, then negate
            tmem_ld32(tmem_addr(tb + 0, lq, 0), x);
            tmem_ld32(tmem_addr(tb + 0, lq, 32), x + 32);
#pragma unroll
            for (int r = 0; r < C; ++r) x[r] = -x[r];
#pragma unroll
            for (int q = 0; q < 8; ++q)
                *reinterpret_cast<uint4 *>(sm + vt::DXWIMG + img_chunk_off(128, row, q)) = vt_pack8(x + 8 * q);
#pragma unroll
            for (int r = 0; r < C; ++r) pp[P.dW() + r * D + row] = x[r];
        } else {  // dK~ = V~ Lambda^T; the rows of V~ in [V~; U] dO^T give dA
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float d[32];
                tmem_ld32(tmem_addr(tb + 64, lq, 32 * hf), d);
#pragma unroll
                for (int u = 0; u < 32; ++u) pp[P.dK() + (32 * hf + u) * D + row] = d[u];
            }
            if (warp < 6) {  // i = row < 64: dA[r][i] = scale (dO V~^T)[r][i] for i <= r
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    float d[32];
                    tmem_ld32(tmem_addr(tb + 128, lq, 32 * hf), d);
#pragma unroll
                    for (int u = 0; u < 32; ++u) {
                        const int r = 32 * hf + u;
                        pp[P.dA() + r * C + row] = row <= r ? scale * d[u] : 0.f;
                    }
                }
            }
        }
        fence_proxy_async();
        vt_sync();
        if (tid == 0) {
            mma_bf16_kmn(tb + 192, s0 + vt::KWIMG, 128, s0 + vt::DXWIMG, 16384, 8, idesc_bf16(128, 64, false, true),
                         true);
            mma_commit(&bar[2]);
        }
        ok = vt_wait(&bar[2], ph);
        if (!ok) break;
        if (warp >= 6) {  // i = row - 64: dL[r][i] = -(dX_U U^T + dX_W W^T)[r][i] for i < r
            const int i = row - 64;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                float d[32];
                tmem_ld32(tmem_addr(tb + 192, lq, 32 * hf), d);
#pragma unroll
                for (int u = 0; u < 32; ++u) {
                    const int r = 32 * hf + u;
                    pp[P.dLu() + r * C + i] = i < r ? -d[u] : 0.f;
                }
            }
        }
        if (tid < D) pp[P.dgam() + tid] = dgam[tid];
        if (tid < C) pp[P.dbu() + tid] = red[tid] + red[64 + tid] + red[128 + tid] + red[192 + tid];
        vt_sync();  // every read of this item's images and tensor memory is done
    }
    if (!ok && tid == 0) set_error(err, KDA_ERR_DEVICE_TIMEOUT);
    vt_sync();
    if (warp == 0) tmem_dealloc(tb, 256);
}

// ------------------------------------------------------------------ reverse chain on the tensor cores
// bf16 I/O with d_k = d_v = 128: one 256-thread CTA per (sequence, head) keeps Lambda^T (rows = value
// channels j = TMEM lanes, columns = key channels c) in tensor memory, fp32, and per chunk, last to first:
//   writes Lambda (leaving the chunk) to lam_end and as a bf16 image, scales it by gamma in place, then
//   dV~^T = Lambda^T K~^T + dO^T (scale A)          (into TMEM columns 128..191)
//   Lambda^T += dO^T (scale Q^) + (-dV~^T) W          (two accumulating products)
// Warps 4-7 turn the fp32 records of the chunks ahead into bf16 operand images (two buffers: the
// chunk after next is filled while this one runs; a buffer is released by the commit that follows
// the last product reading it); warps 0-3 move Lambda and dV~ between TMEM and shared memory, and
// their first thread issues the products.
namespace rc {
constexpr uint32_t KI = 0, QI = 16384, WI = 32768, DI = 49152, AI = 65536, GM = 73728;  // within a buffer
constexpr uint32_t BUF = 74752;            // one chunk's images: K~, scale Q^, W, dO (rows r, 16 KB each),
                                           // scale A (rows i, 8 KB), gamma (fp32 [128])
constexpr uint32_t LIMG = 2 * BUF;         // Lambda^T, bf16, K-major: rows j (128), two blocks of 64 c
constexpr uint32_t DVIMG = LIMG + 32768;   // -dV~^T, bf16, K-major: rows j (128), 64 tokens
constexpr uint32_t BAR = DVIMG + 16384;    // full[2], empty[2], mma1, mma2
constexpr uint32_t TSLOT = BAR + 64;       // TMEM base
constexpr uint32_t FAIL = TSLOT + 8;       // a bounded wait gave up
constexpr uint32_t TOTAL = FAIL + 8 + 1024;
}  // namespace rc

// And-reduction of v over the n threads of named barrier id (also a barrier among them).
__device__ __forceinline__ bool rc_all(int id, int n, bool v) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.and.pred q, %2, %3, p;\n\t"
                 "selp.u32 %0, 1, 0, q;\n\t}\n"
                 : "=r"(r) : "r"((uint32_t)v), "r"(id), "r"(n) : "memory");
    return r != 0;
}
__device__ __forceinline__ void rc_bar(int id, int n) { asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(n) : "memory"); }
// Bounded wait on an mbarrier phase that also gives up once the other role has failed.
__device__ __forceinline__ bool rc_wait(uint64_t *bar, uint32_t parity, volatile int *fail) {
    if (tc::mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = tc::globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (tc::mbar_try_wait(bar, parity)) return true;
        if (*fail) return false;
        if (tc::globaltimer_ns() - t0 > 1000000000ull) {
            *fail = 1;
            return false;
        }
    }
}

__global__ void __launch_bounds__(256, 1)
chunk_rev_chain_tc_kernel(int64_t T, int N, const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_start,
                          int H, const char *__restrict__ records, size_t rec_bytes, float scale,
                          const bf16 *__restrict__ d_o, const float *__restrict__ d_final,
                          float *__restrict__ lam_end, float *__restrict__ d_init, int *err) {
    using namespace tc;
    constexpr int C = 64, D = 128;
    extern __shared__ unsigned char rc_raw[];
    unsigned char *sm = vt_align1024(rc_raw);
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = (warp & 3) * 32, row = lq + lane;  // TMEM lane quarter of this warp; this thread's lane
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + rc::BAR), *empty = full + 2, *bmma1 = full + 4,
             *bmma2 = full + 5;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + rc::TSLOT);
    volatile int *fail = reinterpret_cast<volatile int *>(sm + rc::FAIL);
    const int64_t s_tok = cu ? (int64_t)cu[n] : (T / N) * n;
    const int64_t e_tok = cu ? (int64_t)cu[n + 1] : s_tok + T / N;
    const int c0 = chunk_start[n], c1 = chunk_start[n + 1];
    const int nst = c1 - c0;
    const size_t sbase = ((size_t)n * H + h) * (size_t)D * D;
    if (tid == 0) {
        mbar_init(&full[0], 128);
        mbar_init(&full[1], 128);
        mbar_init(&empty[0], 1);
        mbar_init(&empty[1], 1);
        mbar_init(bmma1, 1);
        mbar_init(bmma2, 1);
        *fail = 0;
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    fence_proxy_async();
    vt_sync();
    const uint32_t tb = *tslot;  // Lambda^T: columns [0, 128); dV~^T: [128, 192)

    if (warp < 4) {
        // Lambda^T <- d final_state^T (or 0)
#pragma unroll 1
        for (int cb = 0; cb < D; cb += 16) {
            float x[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) x[u] = d_final ? d_final[sbase + (size_t)(cb + u) * D + row] : 0.f;
            tmem_st16(tmem_addr(tb, lq, cb), x);
        }
        tmem_st_wait();
        bool ok = true;
        for (int s = 0; s < nst; ++s) {
            const int cix = c1 - 1 - s, b = s & 1;
            unsigned char *B = sm + b * rc::BUF;
            ok = rc_all(1, 128, rc_wait(&full[b], (s >> 1) & 1, fail));
            if (!ok) break;
            // Lambda leaving this chunk: to lam_end and the image; then Diag(gamma) Lambda in place
            const float *gam = reinterpret_cast<const float *>(B + rc::GM);
            float *lg = lam_end + ((size_t)cix * H + h) * (size_t)D * D;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                float x[32];
                tmem_ld32(tmem_addr(tb, lq, 32 * q), x);
#pragma unroll
                for (int u = 0; u < 32; ++u) lg[(size_t)(32 * q + u) * D + row] = x[u];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint4 *>(sm + rc::LIMG + img_chunk_off(128, row, 4 * q + k)) = vt_pack8(x + 8 * k);
#pragma unroll
                for (int u = 0; u < 32; ++u) x[u] *= gam[32 * q + u];
                tmem_st32(tmem_addr(tb, lq, 32 * q), x);
            }
            tmem_st_wait();
            fence_proxy_async();
            fence_before_sync();
            rc_bar(1, 128);
            fence_after_sync();
            const uint32_t sb = smem_u32(B), s0 = smem_u32(sm);
            if (tid == 0) {
                mma_bf16_k(tb + 128, s0 + rc::LIMG, 128, sb + rc::KI, 64, 8, idesc_bf16(128, 64), false);
                mma_bf16_mnmn(tb + 128, sb + rc::DI, 8192, sb + rc::AI, 8192, 4, idesc_bf16(128, 64, true, true), true);
                mma_bf16_mnmn(tb + 0, sb + rc::DI, 8192, sb + rc::QI, 8192, 4, idesc_bf16(128, 128, true, true), true);
                mma_commit(bmma1);
            }
            ok = rc_all(1, 128, rc_wait(bmma1, s & 1, fail));
            if (!ok) break;
            fence_after_sync();
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {  // -dV~^T, row j of the image
                float x[32];
                tmem_ld32(tmem_addr(tb + 128, lq, 32 * hf), x);
#pragma unroll
                for (int u = 0; u < 32; ++u) x[u] = -x[u];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint4 *>(sm + rc::DVIMG + img_chunk_off(128, row, 4 * hf + k)) = vt_pack8(x + 8 * k);
            }
            fence_proxy_async();
            fence_before_sync();
            rc_bar(1, 128);
            fence_after_sync();
            if (tid == 0) {
                mma_bf16_kmn(tb + 0, s0 + rc::DVIMG, 128, sb + rc::WI, 8192, 4, idesc_bf16(128, 128, false, true), true);
                mma_commit(&empty[b]);  // this chunk's images are read by nothing after these products
                mma_commit(bmma2);
            }
            ok = rc_all(1, 128, rc_wait(bmma2, s & 1, fail));
            if (!ok) break;
            fence_after_sync();
        }
        if (ok && d_init) {  // d S0 = Lambda entering the sequence
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                float x[32];
                tmem_ld32(tmem_addr(tb, lq, 32 * q), x);
#pragma unroll
                for (int u = 0; u < 32; ++u) d_init[sbase + (size_t)(32 * q + u) * D + row] = x[u];
            }
        }
    } else {  // fill warps
        const int ft = tid - 128;
        for (int s = 0; s < nst; ++s) {
            const int cix = c1 - 1 - s, b = s & 1;
            if (s >= 2 && !rc_all(2, 128, rc_wait(&empty[b], ((s >> 1) - 1) & 1, fail))) break;
            if (ft == 0 && cix - 2 >= c0)  // the record two chunks on, into L2
                prefetch_l2(records + ((size_t)(cix - 2) * H + h) * rec_bytes, (uint32_t)rec_bytes);
            unsigned char *B = sm + b * rc::BUF;
            const F32Record rec = f32_record(records, rec_bytes, cix, H, h, C, D, D);
            const int64_t t0 = s_tok + (int64_t)(cix - c0) * C;
            const int len = (int)min((int64_t)C, e_tok - t0);
#pragma unroll 2
            for (int q = 0; q < 8; ++q) {  // K~, scale Q^, W: rows r, 8 channels per piece
                const int e = ft + 128 * q, r = e >> 4, jc = e & 15;
                float xk[8], xq[8], xw[8];
                vt_load8(rec.K + (size_t)r * D + 8 * jc, xk);
                vt_load8(rec.Q + (size_t)r * D + 8 * jc, xq);
                vt_load8(rec.W + (size_t)r * D + 8 * jc, xw);
#pragma unroll
                for (int u = 0; u < 8; ++u) xq[u] *= scale;
                const uint32_t off = img_chunk_off(64, r, jc);
                *reinterpret_cast<uint4 *>(B + rc::KI + off) = vt_pack8(xk);
                *reinterpret_cast<uint4 *>(B + rc::QI + off) = vt_pack8(xq);
                *reinterpret_cast<uint4 *>(B + rc::WI + off) = vt_pack8(xw);
            }
            {
                uint4 uo[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {  // dO, zero past the sequence
                    const int e = ft + 128 * q, r = e >> 4, jc = e & 15;
                    uo[q] = make_uint4(0u, 0u, 0u, 0u);
                    if (r < len) uo[q] = *reinterpret_cast<const uint4 *>(d_o + ((t0 + r) * H + h) * (int64_t)D + 8 * jc);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int e = ft + 128 * q, r = e >> 4, jc = e & 15;
                    *reinterpret_cast<uint4 *>(B + rc::DI + img_chunk_off(64, r, jc)) = uo[q];
                }
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {  // scale A, rows i
                const int e = ft + 128 * q, i = e >> 3, rcn = e & 7;
                float x[8];
                vt_load8(rec.A + (size_t)i * C + 8 * rcn, x);
#pragma unroll
                for (int u = 0; u < 8; ++u) x[u] *= scale;
                *reinterpret_cast<uint4 *>(B + rc::AI + img_chunk_off(64, i, rcn)) = vt_pack8(x);
            }
            reinterpret_cast<float *>(B + rc::GM)[ft] = rec.gam[ft];
            fence_proxy_async();
            mbar_arrive(&full[b]);
        }
    }
    __syncthreads();
    if (tid == 0 && *fail) set_error(err, KDA_ERR_DEVICE_TIMEOUT);
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tb, 256);
}

// ------------------------------------------------------------------ forward chain with checkpoints on the tensor cores
// The backward pass's recomputation of the state entering every chunk (no outputs), bf16 I/O with
// d_k = d_v = 128: one 256-thread CTA per (sequence, head) keeps S^T (rows = value channels j = TMEM
// lanes, columns = key channels c) in tensor memory, fp32, and per chunk writes S (entering it) to
// the checkpoints and as a bf16 image, scales it by gamma in place, then
//   V~^T = U^T - S^T W^T         (S^T W^T into TMEM columns 128..191; U from the fp32 record)
//   S^T += V~^T K~               (accumulating product)
// Warps 4-7 fill two buffers of the chunks ahead (W and K~ as bf16 images, U fp32, gamma); warps 0-3
// move S and V~ between TMEM and shared memory, and their first thread issues the products.
namespace fc {
constexpr uint32_t WI = 0, KI = 16384, UF = 32768, GM = 65536;  // within a buffer
constexpr uint32_t BUF = 67584;           // W, K~ (rows r, bf16, 16 KB each), U fp32 [64][128], gamma [128]
constexpr uint32_t SIMG = 2 * BUF;        // S^T, bf16, K-major: rows j (128), two blocks of 64 c
constexpr uint32_t VIMG = SIMG + 32768;   // V~^T, bf16, K-major: rows j (128), 64 tokens
constexpr uint32_t BAR = VIMG + 16384;    // full[2], empty[2], mma1, mma2
constexpr uint32_t TSLOT = BAR + 64;
constexpr uint32_t FAIL = TSLOT + 8;
constexpr uint32_t TOTAL = FAIL + 8 + 1024;
}  // namespace fc

__global__ void __launch_bounds__(256, 1)
chunk_chain_ckpt_tc_kernel(int64_t T, int N, const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_start,
                           int H, const char *__restrict__ records, size_t rec_bytes,
                           const float *__restrict__ initial_state, float *__restrict__ final_state,
                           float *__restrict__ ckpt, int *err) {
    using namespace tc;
    constexpr int C = 64, D = 128;
    extern __shared__ unsigned char fc_raw[];
    unsigned char *sm = vt_align1024(fc_raw);
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = (warp & 3) * 32, row = lq + lane;
    uint64_t *full = reinterpret_cast<uint64_t *>(sm + fc::BAR), *empty = full + 2, *bmma1 = full + 4,
             *bmma2 = full + 5;
    uint32_t *tslot = reinterpret_cast<uint32_t *>(sm + fc::TSLOT);
    volatile int *fail = reinterpret_cast<volatile int *>(sm + fc::FAIL);
    const int c0 = chunk_start[n], c1 = chunk_start[n + 1];
    const int nst = c1 - c0;
    const size_t sbase = ((size_t)n * H + h) * (size_t)D * D;
    if (tid == 0) {
        mbar_init(&full[0], 128);
        mbar_init(&full[1], 128);
        mbar_init(&empty[0], 1);
        mbar_init(&empty[1], 1);
        mbar_init(bmma1, 1);
        mbar_init(bmma2, 1);
        *fail = 0;
    }
    if (warp == 0) tmem_alloc(tslot, 256);
    fence_proxy_async();
    vt_sync();
    const uint32_t tb = *tslot;  // S^T: columns [0, 128); S^T W^T: [128, 192)

    if (warp < 4) {
#pragma unroll 1
        for (int cb = 0; cb < D; cb += 16) {  // S^T <- S0^T (or 0)
            float x[16];
#pragma unroll
            for (int u = 0; u < 16; ++u) x[u] = initial_state ? initial_state[sbase + (size_t)(cb + u) * D + row] : 0.f;
            tmem_st16(tmem_addr(tb, lq, cb), x);
        }
        tmem_st_wait();
        bool ok = true;
        for (int s = 0; s < nst; ++s) {
            const int cix = c0 + s, b = s & 1;
            unsigned char *B = sm + b * fc::BUF;
            ok = rc_all(1, 128, rc_wait(&full[b], (s >> 1) & 1, fail));
            if (!ok) break;
            const float *gam = reinterpret_cast<const float *>(B + fc::GM);
            float *cg = ckpt + ((size_t)cix * H + h) * (size_t)D * D;
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {  // S entering the chunk: checkpoint, image, then Diag(gamma) S
                float x[32];
                tmem_ld32(tmem_addr(tb, lq, 32 * q), x);
#pragma unroll
                for (int u = 0; u < 32; ++u) cg[(size_t)(32 * q + u) * D + row] = x[u];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint4 *>(sm + fc::SIMG + img_chunk_off(128, row, 4 * q + k)) = vt_pack8(x + 8 * k);
#pragma unroll
                for (int u = 0; u < 32; ++u) x[u] *= gam[32 * q + u];
                tmem_st32(tmem_addr(tb, lq, 32 * q), x);
            }
            tmem_st_wait();
            fence_proxy_async();
            fence_before_sync();
            rc_bar(1, 128);
            fence_after_sync();
            const uint32_t sb = smem_u32(B), s0 = smem_u32(sm);
            if (tid == 0) {
                mma_bf16_k(tb + 128, s0 + fc::SIMG, 128, sb + fc::WI, 64, 8, idesc_bf16(128, 64), false);
                mma_commit(bmma1);
            }
            ok = rc_all(1, 128, rc_wait(bmma1, s & 1, fail));
            if (!ok) break;
            fence_after_sync();
            const float *Uf = reinterpret_cast<const float *>(B + fc::UF);
#pragma unroll 1
            for (int hf = 0; hf < 2; ++hf) {  // V~^T = U^T - S^T W^T, row j of the image
                float x[32];
                tmem_ld32(tmem_addr(tb + 128, lq, 32 * hf), x);
#pragma unroll
                for (int u = 0; u < 32; ++u) x[u] = Uf[(32 * hf + u) * D + row] - x[u];
#pragma unroll
                for (int k = 0; k < 4; ++k)
                    *reinterpret_cast<uint4 *>(sm + fc::VIMG + img_chunk_off(128, row, 4 * hf + k)) = vt_pack8(x + 8 * k);
            }
            fence_proxy_async();
            fence_before_sync();
            rc_bar(1, 128);
            fence_after_sync();
            if (tid == 0) {
                mma_bf16_kmn(tb + 0, s0 + fc::VIMG, 128, sb + fc::KI, 8192, 4, idesc_bf16(128, 128, false, true), true);
                mma_commit(&empty[b]);
                mma_commit(bmma2);
            }
            ok = rc_all(1, 128, rc_wait(bmma2, s & 1, fail));
            if (!ok) break;
            fence_after_sync();
        }
        if (ok && final_state) {
#pragma unroll 1
            for (int q = 0; q < 4; ++q) {
                float x[32];
                tmem_ld32(tmem_addr(tb, lq, 32 * q), x);
#pragma unroll
                for (int u = 0; u < 32; ++u) final_state[sbase + (size_t)(32 * q + u) * D + row] = x[u];
            }
        }
    } else {  // fill warps
        const int ft = tid - 128;
        for (int s = 0; s < nst; ++s) {
            const int cix = c0 + s, b = s & 1;
            if (s >= 2 && !rc_all(2, 128, rc_wait(&empty[b], ((s >> 1) - 1) & 1, fail))) break;
            if (ft == 0 && cix + 2 < c1)
                prefetch_l2(records + ((size_t)(cix + 2) * H + h) * rec_bytes, (uint32_t)rec_bytes);
            unsigned char *B = sm + b * fc::BUF;
            const F32Record rec = f32_record(records, rec_bytes, cix, H, h, C, D, D);
            tile_async(reinterpret_cast<float *>(B + fc::UF), D, rec.U, D, C, D, ft, 128);
#pragma unroll
            for (int m = 0; m < 2; ++m) {  // W, then K~: rows r, pieces of 8 channels, loads before stores
                const float *src = m == 0 ? rec.W : rec.K;
                float x[8][8];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int e = ft + 128 * q, r = e >> 4, jc = e & 15;
                    vt_load8(src + (size_t)r * D + 8 * jc, x[q]);
                }
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int e = ft + 128 * q, r = e >> 4, jc = e & 15;
                    *reinterpret_cast<uint4 *>(B + (m == 0 ? fc::WI : fc::KI) + img_chunk_off(64, r, jc)) =
                        vt_pack8(x[q]);
                }
            }
            reinterpret_cast<float *>(B + fc::GM)[ft] = rec.gam[ft];
            cp_async_wait_all();
            fence_proxy_async();
            mbar_arrive(&full[b]);
        }
    }
    __syncthreads();
    if (tid == 0 && *fail) set_error(err, KDA_ERR_DEVICE_TIMEOUT);
    fence_after_sync();
    if (warp == 0) tmem_dealloc(tb, 256);
}

// ------------------------------------------------------------------ key side, per (chunk, head)
// Thread t owns channel c = t % DK of the RPT = C DK / NT consecutive rows (t / DK) RPT + [0, RPT):
// their in-chunk log-decay (a prefix sum within the rows, then the earlier row groups' totals), their
// pairwise A and L terms, dq, dk and dG (kept in registers), and afterwards the gate's derivative of
// the same rows, the reverse cumulative sum of dG reaching them through the later row groups'
// totals.  q and k sit in shared memory in the I/O type (exact), so that with bf16 I/O two CTAs
// share an SM.
template <typename Tio, int DK>
__global__ void __launch_bounds__(NT, 2)
chunk_bwd_key_kernel(int64_t T, int N, const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_start,
                     int H, int dv, const char *__restrict__ records, size_t rec_bytes,
                     const float *__restrict__ part, const Tio *__restrict__ q,
                     const Tio *__restrict__ k, const Tio *__restrict__ z, const Tio *__restrict__ beta,
                     const float *__restrict__ bias, const float *__restrict__ A_log, float g_min, int kind,
                     Tio *__restrict__ grad_q, Tio *__restrict__ grad_k, Tio *__restrict__ grad_z,
                     Tio *__restrict__ grad_beta, float *__restrict__ gate_part) {
    constexpr int C = 64, dk = DK;
    constexpr int NR = NT / DK;   // row groups
    constexpr int RPT = C / NR;   // rows per thread
    constexpr int NWC = DK / 32;  // warps per row group (a warp's lanes share their rows)
    extern __shared__ float sm[];
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    int n, len;
    int64_t t0;
    if (!locate_chunk(chunk_start, cu, T, N, C, slot, n, t0, len)) return;
    const int tid = threadIdx.x, lane = tid & 31;
    const int c = tid % DK, rg = tid / DK, r0 = rg * RPT;
    float *Gs = sm;                  // [C][dk]  in-chunk cumulative log-decay (base 2 after the prefix pass)
    float *dAs = Gs + C * dk;        // [C][C]
    float *dLs = dAs + C * C;        // [C][C]
    float *bet = dLs + C * C;        // [C]
    float *red = bet + C;            // [2][NR][dk] per-row-group channel sums
    float *dbp = red + 2 * NR * dk;  // [C][NWC] the warps' shares of d beta
    Tio *qs = reinterpret_cast<Tio *>(dbp + C * NWC);  // [C][dk]
    Tio *ks = qs + C * dk;                             // [C][dk]

    const Part P{C, dk};
    const float *pp = part + ((size_t)slot * H + h) * (size_t)P.size();
    tile_async(dAs, C, pp + P.dA(), C, C, C, tid, NT);
    tile_async(dLs, C, pp + P.dLu(), C, C, C, tid, NT);  // the whole dL (strictly lower)
    const float eA = A_log ? expf(A_log[h]) : 1.f;
    const float bc = bias ? bias[h * dk + c] : 0.f;
    float gsum = 0.f;
#pragma unroll 4
    for (int m = 0; m < RPT; ++m) {
        const int r = r0 + m;
        const bool ok = r < len;
        const int64_t idx = ((t0 + r) * H + h) * (int64_t)dk + c;
        st(qs + r * dk + c, ok ? ld(q + idx) : 0.f);
        st(ks + r * dk + c, ok ? ld(k + idx) : 0.f);
        gsum += ok ? gate_log(kind, ld(z + idx), bc, eA, g_min) : 0.f;
        Gs[r * dk + c] = gsum;
    }
    red[rg * dk + c] = gsum;
    for (int r = tid; r < C; r += NT) bet[r] = r < len ? ld(beta + (t0 + r) * H + h) : 0.f;
    cp_async_wait_all();
    __syncthreads();
    {  // cumulative log-decay within the chunk (Eq. 3), base 2
        float off = 0.f;
        for (int g = 0; g < rg; ++g) off += red[g * dk + c];
#pragma unroll 4
        for (int m = 0; m < RPT; ++m) {
            const int r = r0 + m;
            Gs[r * dk + c] = (Gs[r * dk + c] + off) * 1.4426950408889634f;
        }
    }
    __syncthreads();
    // per (row, channel): dq, dk, dG and the d beta terms
    const float Gl = Gs[(C - 1) * dk + c];
    float dGr[RPT];
    float xk_sum = 0.f, gtot = 0.f;  // sums over this thread's rows of dK~ * K~ (flows to G_last) and of dG
#pragma unroll
    for (int m = 0; m < RPT; ++m) {
        const int r = r0 + m;
        float dg = 0.f, dbt = 0.f;
        if (r < len) {
            const float Gr = Gs[r * dk + c];
            const float eG = exp2f(Gr), eL = exp2f(Gl - Gr);
            const float qr = ld(qs + r * dk + c), kr = ld(ks + r * dk + c), br = bet[r];
            const float dqh = pp[P.dQ() + r * dk + c], dkt = pp[P.dK() + r * dk + c];
            const float dxw = pp[P.dW() + r * dk + c];  // dX_W = T^T dW (solved by the value side)
            float ra = 0.f, rl = 0.f;  // sum_{i <= r} dA_ri k_ic E_ric,  sum_{i < r} dL_ri k_ic E_ric
            for (int i = 0; i < r; ++i) {
                const float kE = ld(ks + i * dk + c) * exp2f(Gr - Gs[i * dk + c]);
                ra += dAs[r * C + i] * kE;
                rl += dLs[r * C + i] * kE;
            }
            ra += dAs[r * C + r] * kr;
            // sum_{r' >= r} dA_r'r q_r'c E,  sum_{r' > r} dL_r'r b_r' k_r'c E
            float ca = dAs[r * C + r] * qr, cl = 0.f;
            for (int i = r + 1; i < len; ++i) {
                const float E = exp2f(Gs[i * dk + c] - Gr);
                ca += dAs[i * C + r] * ld(qs + i * dk + c) * E;
                cl += dLs[i * C + r] * bet[i] * ld(ks + i * dk + c) * E;
            }
            const float ktil = kr * eL;
            const float dq = dqh * eG + ra;
            const float dkk = br * dxw * eG + dkt * eL + ca + br * rl + cl;
            dg = dxw * br * kr * eG + dqh * qr * eG - dkt * ktil + qr * ra - kr * ca + br * kr * rl - kr * cl;
            dbt = kr * (eG * dxw + rl);  // this element's share of d beta_r
            xk_sum += dkt * ktil;
            const int64_t idx = ((t0 + r) * H + h) * (int64_t)dk + c;
            st(grad_q + idx, dq);
            st(grad_k + idx, dkk);
        }
        dGr[m] = dg;
        gtot += dg;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) dbt += __shfl_xor_sync(0xffffffffu, dbt, off);
        if (lane == 0) dbp[r * NWC + (c >> 5)] = dbt;
    }
    red[rg * dk + c] = xk_sum;
    red[(NR + rg) * dk + c] = gtot;
    __syncthreads();
    // G_last collects d gamma * gamma and the K~ terms of every row; dg of row r = that plus the sum of
    // dG over the rows r' >= r; then the gate's derivative
    float run;
    {
        const F32Record rec = f32_record(records, rec_bytes, slot, H, h, C, dk, dv);
        run = pp[P.dgam() + c] * rec.gam[c];
        for (int g = 0; g < NR; ++g) run += red[g * dk + c];
        for (int g = rg + 1; g < NR; ++g) run += red[(NR + g) * dk + c];
    }
    float db = 0.f, da = 0.f;
#pragma unroll
    for (int m = RPT - 1; m >= 0; --m) {
        const int r = r0 + m;
        run += dGr[m];
        if (r < len) {
            const int64_t idx = ((t0 + r) * H + h) * (int64_t)dk + c;
            const float zz = ld(z + idx);
            float dz, dA;
            if (kind == KDA_GATE_SOFTPLUS) {
                const float x = zz + bc;
                const float sg = 1.f / (1.f + expf(-x));
                const float g = gate_log(kind, zz, bc, eA, g_min);
                dz = run * (-eA * sg);
                dA = run * g;
            } else {
                const float x = eA * (zz + bc);
                const float sg = 1.f / (1.f + expf(-x));
                dz = run * g_min * sg * (1.f - sg) * eA;
                dA = dz * (zz + bc);
            }
            st(grad_z + idx, dz);
            db += dz;
            da += dA;
        }
    }
    __syncthreads();  // every thread has read red
    red[rg * dk + c] = db;
    red[(NR + rg) * dk + c] = da;
    __syncthreads();
    float *gp = gate_part + ((size_t)slot * H + h) * (size_t)(dk + 1);
    if (tid < dk) {
        float s = 0.f;
        for (int g = 0; g < NR; ++g) s += red[g * dk + tid];
        gp[tid] = s;
    } else if (tid < dk + 32) {
        float s = 0.f;
        for (int e = lane; e < NR * dk; e += 32) s += red[NR * dk + e];
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (lane == 0) gp[dk] = s;
    }
    for (int r = tid; r < len; r += NT) {  // d beta: X_W and L terms per channel, plus the X_U part
        float s = pp[P.dbu() + r];
#pragma unroll
        for (int w = 0; w < NWC; ++w) s += dbp[r * NWC + w];
        st(grad_beta + (t0 + r) * H + h, s);
    }
}

// d dt_bias[h][c] = sum over the chunk slots in use (chunk_start[N] of them; the launch's bound `slots`
// may be larger, and slots past the last chunk hold no partials); d A_log[h] likewise
__global__ void bwd_gate_param_kernel(const float *__restrict__ gate_part, int64_t slots,
                                      const int32_t *__restrict__ chunk_start, int N, int H, int dk,
                                      float *__restrict__ grad_bias, float *__restrict__ grad_alog) {
    const int h = blockIdx.x;
    const int64_t used = chunk_start ? min(slots, (int64_t)chunk_start[N]) : slots;
    for (int c = threadIdx.x; c <= dk; c += blockDim.x) {
        float acc = 0.f;
        for (int64_t s = 0; s < used; ++s) acc += gate_part[((size_t)s * H + h) * (size_t)(dk + 1) + c];
        if (c < dk) {
            if (grad_bias) grad_bias[h * dk + c] = acc;
        } else if (grad_alog) {
            grad_alog[h] = acc;
        }
    }
}

}  // namespace bw
}  // namespace kda

using namespace kda;

// The backward pass's forward chain (checkpoints, final state, no outputs) on the tensor cores when the
// problem allows it (bf16, d_k = d_v = 128); false otherwise (the caller then runs the CUDA-core chain).
bool kda_launch_chain_ckpt_tc(const kda_chunk_args *a, const int32_t *chunk_start, const char *records,
                              size_t rec_bytes, float *ckpt, cudaStream_t stream) {
    if (!ckpt || a->dtype != KDA_BF16 || a->dk != 128 || a->dv != 128 || a->o) return false;
    cudaFuncSetAttribute(bw::chunk_chain_ckpt_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                         (int)bw::fc::TOTAL);
    bw::chunk_chain_ckpt_tc_kernel<<<(unsigned)(a->N * a->H), 256, bw::fc::TOTAL, stream>>>(
        a->T, (int)a->N, a->cu_seqlens, chunk_start, a->H, records, rec_bytes, a->initial_state, a->final_state,
        ckpt, kda_device_error_ptr());
    return true;
}

namespace {

struct BwdLayout {
    kda_chunk_plan p;  // chunk table and fp32 records of the forward recomputation
    int64_t slots;
    size_t off_L, off_ckpt, off_lam, off_part, off_gate, total;
};

size_t align256(size_t x) { return (x + 255) & ~(size_t)255; }

bool bwd_layout(int64_t T, int64_t N, int H, int dk, int dv, int C, BwdLayout *L) {
    if (!kda_make_chunk_plan(T, N, H, dk, dv, KDA_F32, C, &L->p, nullptr, 0, true)) return false;
    const size_t s = (size_t)L->p.max_chunks * H;
    L->slots = L->p.max_chunks;
    L->off_L = align256(L->p.total_bytes);
    L->off_ckpt = align256(L->off_L + s * C * C * sizeof(float));
    L->off_lam = align256(L->off_ckpt + s * dk * dv * sizeof(float));
    L->off_part = align256(L->off_lam + s * dk * dv * sizeof(float));
    const bw::Part P{C, dk};
    L->off_gate = align256(L->off_part + s * (size_t)P.size() * sizeof(float));
    L->total = align256(L->off_gate + s * (size_t)(dk + 1) * sizeof(float));
    return true;
}

template <typename Tio>
kda_status_t launch_bwd(const kda_chunk_bwd_args *a, const BwdLayout &Ly, void *ws, cudaStream_t stream) {
    const int C = 64, dk = a->dk, dv = a->dv, H = a->H;
    char *base = (char *)ws;
    float *Lbuf = (float *)(base + Ly.off_L), *ckpt = (float *)(base + Ly.off_ckpt);
    float *lam = (float *)(base + Ly.off_lam), *part = (float *)(base + Ly.off_part);
    float *gpart = (float *)(base + Ly.off_gate);
    // 1. the forward again on the fp32 path: records, L and the state entering every chunk
    kda_chunk_args f{};
    f.T = a->T; f.N = a->N; f.H = H; f.dk = dk; f.dv = dv; f.dtype = a->dtype;
    f.q = a->q; f.k = a->k; f.z = a->z; f.v = a->v; f.beta = a->beta;
    f.dt_bias = a->dt_bias; f.A_log = a->A_log; f.g_min = a->g_min; f.scale = a->scale;
    f.cu_seqlens = a->cu_seqlens; f.initial_state = a->initial_state; f.chunk_size = 64;
    f.gate_kind = a->gate_kind;
    kda_status_t st = kda_launch_chunk_simt_recompute(&f, Ly.p, ws, Lbuf, ckpt, stream);
    if (st != KDA_OK) return st;
    const int32_t *chunk_start = (const int32_t *)(base + Ly.p.off_chunk_start);
    const char *records = base + Ly.p.off_records;
    const size_t rb = Ly.p.record_bytes;
    // 2. Lambda over the chunks in reverse; d initial_state
    // Ws, Qs, Kt [C][dk + 4]; As [C][C + 4]; dOs, dVt [C][TILE + 4]; Lm [dk][TILE + 4]; gam [dk]
    // + the staging buffer of the next chunk's dO slice [C][TILE] in the I/O type
    const size_t smem_rev = sizeof(float) * ((size_t)3 * C * (dk + 4) + (size_t)C * (C + 4) +
                                             (2 * (size_t)C + dk) * (bw::TILE + 4) + dk) +
                            sizeof(Tio) * (size_t)C * bw::TILE;
    const int staged = ((uintptr_t)a->grad_o & 15) == 0 ? 1 : 0;  // dO rows copied in 16-byte pieces
    {
        auto rev = [&](auto kern) {
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_rev);
            kern<<<dim3((unsigned)(a->N * H), (unsigned)(dv / bw::TILE)), bw::NT, smem_rev, stream>>>(
                a->T, (int)a->N, a->cu_seqlens, chunk_start, H, dv, records, rb, a->scale, (const Tio *)a->grad_o,
                a->grad_final_state, lam, a->grad_initial_state, staged);
        };
        if (a->dtype == KDA_BF16 && dk == 128 && dv == 128 && staged) {  // on the tensor cores
            cudaFuncSetAttribute(bw::chunk_rev_chain_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)bw::rc::TOTAL);
            bw::chunk_rev_chain_tc_kernel<<<(unsigned)(a->N * H), 256, bw::rc::TOTAL, stream>>>(
                a->T, (int)a->N, a->cu_seqlens, chunk_start, H, records, rb, a->scale, (const bf16 *)a->grad_o,
                a->grad_final_state, lam, a->grad_initial_state, kda_device_error_ptr());
        } else if (dk == 128) {
            rev(bw::chunk_rev_chain_kernel<Tio, 128>);
        } else {
            rev(bw::chunk_rev_chain_kernel<Tio, 64>);
        }
    }
    kda_profile_mark(4, stream);
    st = kda_cuda_status(cudaGetLastError());
    if (st != KDA_OK) return st;
    if (Ly.slots == 0 || a->T == 0) {  // no tokens: the parameter gradients are zero
        if (a->grad_dt_bias || a->grad_A_log) {
            bw::bwd_gate_param_kernel<<<(unsigned)H, 128, 0, stream>>>(gpart, 0, nullptr, 0, H, dk, a->grad_dt_bias,
                                                                       a->grad_A_log);
            st = kda_cuda_status(cudaGetLastError());
        }
        return st;
    }
    // 3. value side per (chunk, head): on the tensor cores for bf16 I/O at d_k = d_v = 128 (dO read, and the
    // rows of dO and v prefetched, in 16-byte pieces), else on CUDA cores, the value channels 32 at a time
    if (a->dtype == KDA_BF16 && dk == 128 && dv == 128 && ((uintptr_t)a->grad_o & 15) == 0 &&
        ((uintptr_t)a->v & 15) == 0) {
        cudaFuncSetAttribute(bw::chunk_bwd_value_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             (int)bw::vt::TOTAL);
        int dev = 0, sms = 148;
        if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        const int64_t items = Ly.slots * H;
        bw::chunk_bwd_value_tc_kernel<<<(unsigned)std::min<int64_t>(sms, items), 256, bw::vt::TOTAL, stream>>>(
            a->T, (int)a->N, a->cu_seqlens, chunk_start, H, records, rb, Lbuf, ckpt, lam, a->scale,
            (const bf16 *)a->v, (const bf16 *)a->beta, (const bf16 *)a->grad_o, (bf16 *)a->grad_v, part,
            kda_device_error_ptr());
    } else {
        const size_t smem_val = sizeof(float) * (2 * (size_t)C * (dk + 4) + 2 * (size_t)C * (C + 4) +
                                                 2 * (size_t)dk * (bw::TILE + 1) + 5 * (size_t)C * (bw::TILE + 1) + C);
        const void *kern = dk == 128 ? (const void *)bw::chunk_bwd_value_kernel_t<128>
                                     : (const void *)bw::chunk_bwd_value_kernel_t<64>;
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_val);
        const dim3 grid((unsigned)Ly.slots, (unsigned)H);
        const int b16 = a->dtype == KDA_BF16 ? 1 : 0;
        if (dk == 128)
            bw::chunk_bwd_value_kernel_t<128><<<grid, bw::NTV, smem_val, stream>>>(
                a->T, (int)a->N, a->cu_seqlens, chunk_start, H, dv, records, rb, Lbuf, ckpt, lam, a->scale, a->v,
                a->beta, a->grad_o, a->grad_v, b16, part);
        else
            bw::chunk_bwd_value_kernel_t<64><<<grid, bw::NTV, smem_val, stream>>>(
                a->T, (int)a->N, a->cu_seqlens, chunk_start, H, dv, records, rb, Lbuf, ckpt, lam, a->scale, a->v,
                a->beta, a->grad_o, a->grad_v, b16, part);
    }
    kda_profile_mark(5, stream);
    st = kda_cuda_status(cudaGetLastError());
    if (st != KDA_OK) return st;
    // 4. key side per (chunk, head): Gs [C][dk], dA and dL [C][C], bet [C], red [2][NT / dk][dk],
    // dbp [C][dk / 32] fp32; q and k [C][dk] in the I/O type
    const size_t smem_key = sizeof(float) * ((size_t)C * dk + 2 * (size_t)C * C + C + 2 * (size_t)bw::NT +
                                             (size_t)C * (dk / 32)) + 2 * sizeof(Tio) * (size_t)C * dk;
    {
        auto key = [&](auto kern) {
            cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_key);
            kern<<<dim3((unsigned)Ly.slots, (unsigned)H), bw::NT, smem_key, stream>>>(
                a->T, (int)a->N, a->cu_seqlens, chunk_start, H, dv, records, rb, part, (const Tio *)a->q,
                (const Tio *)a->k, (const Tio *)a->z, (const Tio *)a->beta, a->dt_bias, a->A_log, a->g_min,
                a->gate_kind, (Tio *)a->grad_q, (Tio *)a->grad_k, (Tio *)a->grad_z, (Tio *)a->grad_beta, gpart);
        };
        if (dk == 128) key(bw::chunk_bwd_key_kernel<Tio, 128>);
        else key(bw::chunk_bwd_key_kernel<Tio, 64>);
    }
    kda_profile_mark(6, stream);
    st = kda_cuda_status(cudaGetLastError());
    if (st != KDA_OK) return st;
    // 5. gate parameters
    if (a->grad_dt_bias || a->grad_A_log) {
        bw::bwd_gate_param_kernel<<<(unsigned)H, 128, 0, stream>>>(gpart, Ly.slots, chunk_start, (int)a->N, H, dk,
                                                                   a->grad_dt_bias, a->grad_A_log);
        st = kda_cuda_status(cudaGetLastError());
    }
    kda_profile_mark(7, stream);
    return st;
}

// One long sequence in segments of S chunks, when the whole pass's scratch does not fit: a forward sweep
// stores the state entering each segment; then the segments run last to first, each a full backward pass
// over its tokens from its entering state, the gradient of its final state being the gradient of the next
// segment's initial state (the state's adjoint crosses the boundary exactly as it crosses a chunk boundary
// inside one pass), and the dt_bias and A_log gradients summed over the segments.  Workspace: one
// segment's scratch, the entering states [K][H][dk][dv], two adjoint buffers [H][dk][dv] and the gate
// parameters' per-segment sums.
struct SegLayout {
    BwdLayout seg;
    int64_t S, K;  // chunks per segment, segments
    size_t off_states, off_carry, off_gpart, total;
};

bool seg_layout(int64_t T, int H, int dk, int dv, int64_t S, SegLayout *L) {
    const int64_t seg_tokens = S * 64;
    if (!bwd_layout(std::min(T, seg_tokens), 1, H, dk, dv, 64, &L->seg)) return false;
    L->S = S;
    L->K = (T + seg_tokens - 1) / seg_tokens;
    const size_t st = (size_t)H * dk * dv * sizeof(float);
    L->off_states = align256(L->seg.total);
    L->off_carry = align256(L->off_states + (size_t)L->K * st);
    L->off_gpart = align256(L->off_carry + 2 * st);
    L->total = align256(L->off_gpart + (size_t)H * (dk + 1) * sizeof(float));
    return true;
}

__global__ void bwd_accumulate_kernel(float *dst, const float *src, int n, int first) {
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += gridDim.x * blockDim.x)
        dst[i] = first ? src[i] : dst[i] + src[i];
}

template <typename Tio>
kda_status_t launch_bwd_segmented(const kda_chunk_bwd_args *a, const SegLayout &Ls, void *ws, cudaStream_t stream) {
    const int H = a->H, dk = a->dk, dv = a->dv;
    const size_t es = sizeof(Tio), stz = (size_t)H * dk * dv;
    char *base = (char *)ws;
    float *states = (float *)(base + Ls.off_states), *carry = (float *)(base + Ls.off_carry);
    float *gp_bias = (float *)(base + Ls.off_gpart), *gp_alog = gp_bias + (size_t)H * dk;
    const int64_t seg_tokens = Ls.S * 64;
    auto seg_len = [&](int64_t k) { return std::min(seg_tokens, a->T - k * seg_tokens); };
    auto off = [&](const void *p, int64_t k, int width) -> const char * {
        return p ? (const char *)p + (size_t)(k * seg_tokens) * H * width * es : nullptr;
    };
    // forward sweep: the state entering segments 1 .. K - 1 (fp32 path, as the backward recomputes)
    float *Lbuf = (float *)(base + Ls.seg.off_L), *ckpt = (float *)(base + Ls.seg.off_ckpt);
    for (int64_t k = 0; k + 1 < Ls.K; ++k) {
        kda_chunk_args f{};
        f.T = seg_len(k); f.N = 1; f.H = H; f.dk = dk; f.dv = dv; f.dtype = a->dtype;
        f.q = off(a->q, k, dk); f.k = off(a->k, k, dk); f.z = off(a->z, k, dk); f.v = off(a->v, k, dv);
        f.beta = off(a->beta, k, 1);
        f.dt_bias = a->dt_bias; f.A_log = a->A_log; f.g_min = a->g_min; f.scale = a->scale;
        f.initial_state = k == 0 ? a->initial_state : states + (size_t)k * stz;
        f.final_state = states + (size_t)(k + 1) * stz;
        f.chunk_size = 64; f.gate_kind = a->gate_kind;
        const kda_status_t st = kda_launch_chunk_simt_recompute(&f, Ls.seg.p, ws, Lbuf, ckpt, stream);
        if (st != KDA_OK) return st;
    }
    // the segments last to first
    for (int64_t k = Ls.K - 1; k >= 0; --k) {
        kda_chunk_bwd_args b = *a;
        b.T = seg_len(k); b.N = 1; b.cu_seqlens = nullptr;
        b.q = off(a->q, k, dk); b.k = off(a->k, k, dk); b.z = off(a->z, k, dk); b.v = off(a->v, k, dv);
        b.beta = off(a->beta, k, 1); b.grad_o = off(a->grad_o, k, dv);
        b.grad_q = (void *)off(a->grad_q, k, dk); b.grad_k = (void *)off(a->grad_k, k, dk);
        b.grad_z = (void *)off(a->grad_z, k, dk); b.grad_v = (void *)off(a->grad_v, k, dv);
        b.grad_beta = (void *)off(a->grad_beta, k, 1);
        b.initial_state = k == 0 ? a->initial_state : states + (size_t)k * stz;
        b.grad_final_state = k == Ls.K - 1 ? a->grad_final_state : carry + (size_t)((k + 1) & 1) * stz;
        b.grad_initial_state = k == 0 ? a->grad_initial_state : carry + (size_t)(k & 1) * stz;
        b.grad_dt_bias = a->grad_dt_bias ? gp_bias : nullptr;
        b.grad_A_log = a->grad_A_log ? gp_alog : nullptr;
        kda_status_t st = launch_bwd<Tio>(&b, Ls.seg, ws, stream);
        if (st != KDA_OK) return st;
        const int first = k == Ls.K - 1 ? 1 : 0;
        if (a->grad_dt_bias)
            bwd_accumulate_kernel<<<(H * dk + 255) / 256, 256, 0, stream>>>(a->grad_dt_bias, gp_bias, H * dk, first);
        if (a->grad_A_log) bwd_accumulate_kernel<<<1, 256, 0, stream>>>(a->grad_A_log, gp_alog, H, first);
        st = kda_cuda_status(cudaGetLastError());
        if (st != KDA_OK) return st;
    }
    return KDA_OK;
}

// Chunks per segment of the segmented pass for this workspace (0: it does not fit, or the pass
// cannot be segmented): the largest power of two, at least 16, whose layout fits.
int64_t seg_chunks_for(int64_t T, int64_t N, int H, int dk, int dv, size_t ws_bytes) {
    if (N != 1 || T <= 16 * 64) return 0;
    const int64_t chunks = (T + 63) / 64;
    for (int64_t S = (int64_t)1 << 40; S >= 16; S >>= 1) {
        if (S >= chunks) continue;
        SegLayout L;
        if (seg_layout(T, H, dk, dv, S, &L) && L.total <= ws_bytes) return S;
    }
    return 0;
}

}  // namespace

size_t kda_chunk_bwd_layout_bytes(int64_t T, int64_t N, int H, int dk, int dv) {
    BwdLayout L;
    return bwd_layout(T, N, H, dk, dv, 64, &L) ? L.total : 0;
}

size_t kda_chunk_bwd_min_layout_bytes(int64_t T, int64_t N, int H, int dk, int dv) {
    const size_t full = kda_chunk_bwd_layout_bytes(T, N, H, dk, dv);
    if (N != 1 || T <= 16 * 64) return full;
    SegLayout L;
    return seg_layout(T, H, dk, dv, 16, &L) ? std::min(full, L.total) : full;
}

kda_status_t kda_launch_chunk_bwd(const kda_chunk_bwd_args *a, void *ws, size_t ws_bytes, cudaStream_t stream) {
    BwdLayout L;
    if (!bwd_layout(a->T, a->N, a->H, a->dk, a->dv, 64, &L)) return KDA_ERR_INVALID_ARG;
    if (!ws) return KDA_ERR_WORKSPACE;
    if (ws_bytes >= L.total)
        return a->dtype == KDA_BF16 ? launch_bwd<bf16>(a, L, ws, stream) : launch_bwd<float>(a, L, ws, stream);
    const int64_t S = seg_chunks_for(a->T, a->N, a->H, a->dk, a->dv, ws_bytes);
    if (S == 0) return KDA_ERR_WORKSPACE;
    SegLayout Ls;
    if (!seg_layout(a->T, a->H, a->dk, a->dv, S, &Ls)) return KDA_ERR_INVALID_ARG;
    return a->dtype == KDA_BF16 ? launch_bwd_segmented<bf16>(a, Ls, ws, stream)
                                : launch_bwd_segmented<float>(a, Ls, ws, stream);
}
