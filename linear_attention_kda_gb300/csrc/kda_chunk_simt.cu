// fp32 CUDA-core path of kda_chunk_fwd (any supported head size, fp32 or bf16
// I/O).  It is the full-precision path: fp32 operands and fp32 accumulation
// everywhere, so that fp32 I/O meets a 1e-4 relative error bound.
//
// Two kernels, following Eq. 3 and Eq. 4 of the Kimi K3 report (section 2.1.1):
//
// 1. intra (one CTA per (chunk, head), all chunks in parallel):
//    g from Eq. 5 (or the unbounded softplus gate: this path is the one that gate
//    takes, see below), G = in-chunk cumulative log-decay (Eq. 3 in log space),
//    L[r,i] = beta_r sum_c k_rc k_ic e^{G_rc - G_ic}  (i < r),
//    A[r,i] =        sum_c q_rc k_ic e^{G_rc - G_ic}  (i <= r, diagonal kept),
//    [W | U] = (I + L)^{-1} [diag(beta)(Gamma * K) | diag(beta) V]   (UT transform,
//    by forward substitution, one column per thread),
//    Q^ = Gamma * Q,  K~ = K * e^{G_last - G},  gamma^C = e^{G_last}.
//    The relative decays are formed as e^{G_r - G_i} directly, never as a
//    product of Gamma and 1/Gamma, so nothing overflows at any chunk length or
//    for any gate value: every factor is <= 1 and a deep decay underflows to 0.
// 2. chain (one CTA per (sequence, head, 32 value columns), chunks in order):
//    V~ = U - W S;  O = scale (Q^ S + A V~);  S <- Diag(gamma^C) S + K~^T V~.
//    Columns of S evolve independently (Eq. 1 acts on S from the left), so the
//    value dimension is split across CTAs.
// Tokens past the end of a sequence inside its last chunk are loaded as zeros
// with g = 0 and beta = 0, which leaves every valid row and the state unchanged.
#include "kda_common.cuh"
#include <algorithm>
#include "kda_internal.h"
#include "kda_f32_records.cuh"

namespace kda {

constexpr int SIMT_THREADS = 256;
constexpr int SLICE = 32;  // value columns per chain CTA

// One CTA per (chunk, head).  Shared memory holds k, G and q (then v, in q's place, once the records
// that need q are written) and L, ~113 KB at d = 128, so that two CTAs share an SM; A goes straight to
// the record.
template <typename Tio>
__global__ void __launch_bounds__(SIMT_THREADS, 2)
chunk_intra_simt_kernel(const Tio *__restrict__ q, const Tio *__restrict__ k, const Tio *__restrict__ v,
                        const Tio *__restrict__ z, const Tio *__restrict__ beta,
                        const float *__restrict__ bias, const float *__restrict__ A_log, float g_min,
                        int kind, int64_t T, int N, const int32_t *__restrict__ cu,
                        const int32_t *__restrict__ chunk_start, int H, int dk, int dv, int C,
                        char *__restrict__ records, size_t rec_bytes, float *__restrict__ Lout) {
    extern __shared__ float sm[];
    const int64_t slot = blockIdx.x;
    const int h = blockIdx.y;
    int n, len;
    int64_t t0;
    if (!locate_chunk(chunk_start, cu, T, N, C, slot, n, t0, len)) return;
    const int tid = threadIdx.x;
    const int PK = dk + 1, PV = dv + 1, PC = C;
    float *Ks = sm;               // [C][PK]
    float *Gs = Ks + C * PK;      // [C][PK]
    float *Qs = Gs + C * PK;      // [C][PK]  q, then v ([C][PV]) in the same place
    float *Vs = Qs;
    float *Ls = Qs + C * max(PK, PV);  // [C][PC]
    auto bet = [&](int r) { return r < len ? ld(beta + (t0 + r) * H + h) : 0.f; };

    for (int r = tid; r < len; r += SIMT_THREADS) {  // v is read after A and L: ask L2 for it now
        const char *row = reinterpret_cast<const char *>(v + ((t0 + r) * H + h) * (int64_t)dv);
        for (int o = 0; o < dv * (int)sizeof(Tio); o += 128) asm volatile("prefetch.global.L2 [%0];" :: "l"(row + o));
    }
    const float eA = A_log ? expf(A_log[h]) : 1.f;
#pragma unroll 4
    for (int e = tid; e < C * dk; e += SIMT_THREADS) {
        const int r = e / dk, c = e % dk;
        const bool ok = r < len;
        const int64_t idx = ((t0 + r) * H + h) * (int64_t)dk + c;
        Ks[r * PK + c] = ok ? ld(k + idx) : 0.f;
        Qs[r * PK + c] = ok ? ld(q + idx) : 0.f;
        Gs[r * PK + c] = ok ? gate_log(kind, ld(z + idx), bias ? bias[h * dk + c] : 0.f, eA, g_min) : 0.f;
    }
    __syncthreads();
    // in-chunk cumulative log-decay (Eq. 3), kept in base 2 (G log2 e) so that every decay below is
    // one exp2 of a difference
    for (int c = tid; c < dk; c += SIMT_THREADS) {
        float acc = 0.f;
        for (int r = 0; r < C; ++r) {
            acc += Gs[r * PK + c];
            Gs[r * PK + c] = acc * 1.4426950408889634f;
        }
    }
    __syncthreads();
    F32Record rec = f32_record(records, rec_bytes, slot, H, h, C, dk, dv);
    // A and L, four key rows i per thread sharing the query row r's values; the exponent is clamped at
    // 0 only so that the block's entries above the diagonal (discarded) cannot overflow
    for (int it = tid; it < C * (C / 4); it += SIMT_THREADS) {
        const int r = it / (C / 4), ib = (it % (C / 4)) * 4;
        float4 a4 = make_float4(0.f, 0.f, 0.f, 0.f), l4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (ib <= r) {
            float sl[4] = {0.f, 0.f, 0.f, 0.f}, sa[4] = {0.f, 0.f, 0.f, 0.f};
            for (int c = 0; c < dk; ++c) {
                const float Gr = Gs[r * PK + c], kr = Ks[r * PK + c], qr = Qs[r * PK + c];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                    const float ki = Ks[(ib + u) * PK + c] * exp2f(fminf(Gr - Gs[(ib + u) * PK + c], 0.f));
                    sl[u] += kr * ki;
                    sa[u] += qr * ki;
                }
            }
            const float br = bet(r);
            l4 = make_float4(ib < r ? br * sl[0] : 0.f, ib + 1 < r ? br * sl[1] : 0.f,
                             ib + 2 < r ? br * sl[2] : 0.f, ib + 3 < r ? br * sl[3] : 0.f);
            a4 = make_float4(sa[0], ib + 1 <= r ? sa[1] : 0.f, ib + 2 <= r ? sa[2] : 0.f, ib + 3 <= r ? sa[3] : 0.f);
        }
        *reinterpret_cast<float4 *>(Ls + r * PC + ib) = l4;
        *reinterpret_cast<float4 *>(rec.A + r * C + ib) = a4;
    }
    __syncthreads();
    if (Lout) {  // the backward pass reuses L (strictly lower, zeros elsewhere)
        float *Lg = Lout + ((size_t)slot * H + h) * (size_t)C * C;
        for (int e = tid; e < C * C; e += SIMT_THREADS) Lg[e] = Ls[e];
    }
    for (int e = tid; e < C * dk; e += SIMT_THREADS) {
        const int r = e / dk, c = e % dk;
        const float G = Gs[r * PK + c], Gl = Gs[(C - 1) * PK + c];  // base 2; flat past len
        rec.Q[e] = Qs[r * PK + c] * exp2f(G);
        rec.K[e] = Ks[r * PK + c] * exp2f(Gl - G);
        if (r == 0) rec.gam[c] = exp2f(Gl);
    }
    __syncthreads();  // q is no longer needed: v takes its place
    // right-hand sides of the UT transform, in place
    for (int e = tid; e < C * dk; e += SIMT_THREADS) {
        const int r = e / dk, c = e % dk;
        Ks[r * PK + c] = bet(r) * Ks[r * PK + c] * exp2f(Gs[r * PK + c]);
    }
#pragma unroll 8
    for (int e = tid; e < C * dv; e += SIMT_THREADS) {
        const int r = e / dv, c = e % dv;
        Vs[r * PV + c] = r < len ? bet(r) * ld(v + ((t0 + r) * H + h) * (int64_t)dv + c) : 0.f;
    }
    __syncthreads();
    // forward substitution (I + L) X = RHS, one column per thread
    for (int j = tid; j < dk + dv; j += SIMT_THREADS) {
        float *X = j < dk ? Ks + j : Vs + (j - dk);
        const int P = j < dk ? PK : PV;
        for (int r = 1; r < C; ++r) {
            float x = X[r * P];
            for (int i = 0; i < r; ++i) x -= Ls[r * PC + i] * X[i * P];
            X[r * P] = x;
        }
    }
    __syncthreads();
    for (int e = tid; e < C * dk; e += SIMT_THREADS) rec.W[e] = Ks[(e / dk) * PK + e % dk];
    for (int e = tid; e < C * dv; e += SIMT_THREADS) rec.U[e] = Vs[(e / dv) * PV + e % dv];
}

template <typename Tio, int DK>
__global__ void __launch_bounds__(SIMT_THREADS)
chunk_chain_simt_kernel(int64_t T, int N, const int32_t *__restrict__ cu,
                        const int32_t *__restrict__ chunk_start, int H, int dv, int C_,
                        const char *__restrict__ records, size_t rec_bytes, float scale,
                        const float *initial_state, float *final_state, Tio *__restrict__ o,
                        float *__restrict__ ckpt) {
    extern __shared__ float sm[];
    constexpr int C = 64, dk = DK;
    const int n = blockIdx.x / H, h = blockIdx.x % H;
    const int j0 = blockIdx.y * SLICE;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    constexpr int NWARP = SIMT_THREADS / 32;
    constexpr int RW = C / NWARP, CW = DK / NWARP;  // rows of V~ / O and rows of S per warp
    // row pitches padded to 16 bytes (tiles arrive by 16-byte asynchronous copies, row operands are
    // read as 16-byte broadcasts); the lane-indexed operands are lane-contiguous: no bank conflicts
    constexpr int PK = dk + 4, PC = C + 4, PS = SLICE + 4;
    float *Ws = sm;               // [C][PK]
    float *Qs = Ws + C * PK;      // [C][PK]
    float *Kt = Qs + C * PK;      // [C][PK]
    float *As = Kt + C * PK;      // [C][PC]
    float *Us = As + C * PC;      // [C][PS]
    float *Vt = Us + C * PS;      // [C][PS]
    float *Ss = Vt + C * PS;      // [dk][PS]
    float *gam = Ss + dk * PS;    // [dk]

    const size_t sbase = ((size_t)n * H + h) * (size_t)dk * dv;
    const int64_t s_tok = cu ? (int64_t)cu[n] : (T / N) * n;
    const int64_t e_tok = cu ? (int64_t)cu[n + 1] : s_tok + T / N;
    const int c0 = chunk_start[n], c1 = chunk_start[n + 1];
    // A chunk's tiles come in two groups of asynchronous copies, each issued as soon as the phase that
    // last read the previous chunk's copy is done: W, U (and Q^, A with outputs) after the V~ / O phase,
    // K~ and gamma after the state update.
    auto issue_vo = [&](int cix) {
        const F32Record rec = f32_record(records, rec_bytes, cix, H, h, C, dk, dv);
        tile_async(Ws, PK, rec.W, dk, C, dk, tid, SIMT_THREADS);
        tile_async(Us, PS, rec.U + j0, dv, C, SLICE, tid, SIMT_THREADS);
        if (o) {
            tile_async(Qs, PK, rec.Q, dk, C, dk, tid, SIMT_THREADS);
            tile_async(As, PC, rec.A, C, C, C, tid, SIMT_THREADS);
        }
    };
    auto issue_s = [&](int cix) {
        const F32Record rec = f32_record(records, rec_bytes, cix, H, h, C, dk, dv);
        tile_async(Kt, PK, rec.K, dk, C, dk, tid, SIMT_THREADS);
        tile_async(gam, dk, rec.gam, dk, 1, dk, tid, SIMT_THREADS);
    };
    if (initial_state) {
        tile_async(Ss, PS, initial_state + sbase + j0, dv, dk, SLICE, tid, SIMT_THREADS);
    } else {
        for (int e = tid; e < dk * SLICE; e += SIMT_THREADS) Ss[(e / SLICE) * PS + e % SLICE] = 0.f;
    }
    if (c0 < c1) issue_vo(c0);
    cp_async_commit();
    if (c0 < c1) issue_s(c0);
    cp_async_commit();
    for (int cix = c0; cix < c1; ++cix) {
        const int64_t t0 = s_tok + (int64_t)(cix - c0) * C;
        const int len = (int)min((int64_t)C, e_tok - t0);
        if (tid == 0 && cix + 1 < c1)  // the next chunk's record, into L2 while this one runs
            prefetch_l2(records + ((size_t)(cix + 1) * H + h) * rec_bytes, (uint32_t)rec_bytes);
        cp_async_wait_group1();  // this chunk's W, U (, Q^, A) and, the first time, the entering state
        __syncthreads();
        if (ckpt) {  // the state entering this chunk, for the backward pass
            float *cg = ckpt + ((size_t)cix * H + h) * (size_t)dk * dv;
            for (int e = tid; e < dk * SLICE; e += SIMT_THREADS) {
                const int c = e / SLICE, j = e % SLICE;
                cg[(size_t)c * dv + j0 + j] = Ss[c * PS + j];
            }
        }
        // Register-blocked products: warp w owns rows [RW w, RW w + RW) of V~ and O and rows
        // [CW w, CW w + CW) of S; a lane-indexed operand is read once per reduction index for all
        // of the warp's rows, row operands four at a time as 16-byte broadcasts.
        const int r0 = warp * RW, cb = warp * CW;
        {  // V~ = U - W S and the Q^ S part of O
            float vt[RW], oq[RW];
#pragma unroll
            for (int i = 0; i < RW; ++i) {
                vt[i] = Us[(r0 + i) * PS + lane];
                oq[i] = 0.f;
            }
            for (int c = 0; c < dk; c += 4) {
                const float s0 = Ss[c * PS + lane], s1 = Ss[(c + 1) * PS + lane];
                const float s2 = Ss[(c + 2) * PS + lane], s3 = Ss[(c + 3) * PS + lane];
#pragma unroll
                for (int i = 0; i < RW; ++i) {
                    const float4 w = *reinterpret_cast<const float4 *>(&Ws[(r0 + i) * PK + c]);
                    vt[i] -= w.x * s0 + w.y * s1 + w.z * s2 + w.w * s3;
                    if (o) {
                        const float4 q4 = *reinterpret_cast<const float4 *>(&Qs[(r0 + i) * PK + c]);
                        oq[i] += q4.x * s0 + q4.y * s1 + q4.z * s2 + q4.w * s3;
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < RW; ++i) Vt[(r0 + i) * PS + lane] = vt[i];
            __syncthreads();
            if (o) {  // O = scale (Q^ S + A V~); A is zero above its diagonal
                for (int i0 = 0; i0 < r0 + RW; i0 += 4) {
                    const float v0 = Vt[i0 * PS + lane], v1 = Vt[(i0 + 1) * PS + lane];
                    const float v2 = Vt[(i0 + 2) * PS + lane], v3 = Vt[(i0 + 3) * PS + lane];
#pragma unroll
                    for (int i = 0; i < RW; ++i) {
                        const float4 a4 = *reinterpret_cast<const float4 *>(&As[(r0 + i) * PC + i0]);
                        oq[i] += a4.x * v0 + a4.y * v1 + a4.z * v2 + a4.w * v3;
                    }
                }
#pragma unroll
                for (int i = 0; i < RW; ++i)
                    if (r0 + i < len) st(o + ((t0 + r0 + i) * H + h) * (int64_t)dv + j0 + lane, scale * oq[i]);
            }
        }
        __syncthreads();  // every read of S, W, U, Q^ and A in this chunk is done
        if (cix + 1 < c1) issue_vo(cix + 1);
        cp_async_commit();
        cp_async_wait_group1();  // this chunk's K~ and gamma
        __syncthreads();
        {  // S <- Diag(gamma^C) S + K~^T V~
            float sn[CW];
#pragma unroll
            for (int i = 0; i < CW; ++i) sn[i] = gam[cb + i] * Ss[(cb + i) * PS + lane];
            for (int r = 0; r < len; ++r) {
                const float v = Vt[r * PS + lane];
#pragma unroll
                for (int j = 0; j < CW; j += 4) {
                    const float4 k4 = *reinterpret_cast<const float4 *>(&Kt[r * PK + cb + j]);
                    sn[j] += k4.x * v;
                    sn[j + 1] += k4.y * v;
                    sn[j + 2] += k4.z * v;
                    sn[j + 3] += k4.w * v;
                }
            }
#pragma unroll
            for (int i = 0; i < CW; ++i) Ss[(cb + i) * PS + lane] = sn[i];
        }
        __syncthreads();  // K~ and gamma are free
        if (cix + 1 < c1) issue_s(cix + 1);
        cp_async_commit();
    }
    cp_async_wait_all();  // a sequence without chunks: the initial state's copy
    __syncthreads();
    if (final_state) {
        for (int e = tid; e < dk * SLICE; e += SIMT_THREADS) {
            const int c = e / SLICE, j = e % SLICE;
            final_state[sbase + (size_t)c * dv + j0 + j] = Ss[c * PS + j];
        }
    }
}

}  // namespace kda

using namespace kda;

kda_status_t kda_launch_chunk_plan(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                   cudaStream_t stream);

// The fp32 path; with Lout / ckpt (the backward pass's recomputation) the intra kernel also writes
// L per (chunk slot, head) and the chain writes the state entering every chunk slot.
static kda_status_t launch_simt(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws, cudaStream_t stream,
                                float *Lout, float *ckpt) {
    kda_profile_mark(0, stream);
    kda_status_t st = kda_launch_chunk_plan(a, p, ws, stream);
    if (st != KDA_OK) return st;
    kda_profile_mark(1, stream);
    const int C = p.C, dk = p.dk, dv = p.dv, H = p.H;
    const int32_t *chunk_start = (const int32_t *)((char *)ws + p.off_chunk_start);
    char *records = (char *)ws + p.off_records;
    const size_t smem_intra =
        sizeof(float) * ((size_t)2 * C * (dk + 1) + (size_t)C * (std::max(dk, dv) + 1) + (size_t)C * C);
    const size_t smem_chain = sizeof(float) * ((size_t)3 * C * (dk + 4) + (size_t)C * (C + 4) +
                                               2 * (size_t)C * (SLICE + 4) + (size_t)dk * (SLICE + 4) + dk);
    const bool b16 = a->dtype == KDA_BF16;
    if (p.max_chunks > 0 && a->T > 0) {
        dim3 grid((unsigned)p.max_chunks, (unsigned)H);
        if (b16) {
            cudaFuncSetAttribute(chunk_intra_simt_kernel<bf16>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_intra);
            chunk_intra_simt_kernel<bf16><<<grid, SIMT_THREADS, smem_intra, stream>>>(
                (const bf16 *)a->q, (const bf16 *)a->k, (const bf16 *)a->v, (const bf16 *)a->z,
                (const bf16 *)a->beta, a->dt_bias, a->A_log, a->g_min, a->gate_kind, a->T, (int)a->N, a->cu_seqlens,
                chunk_start, H, dk, dv, C, records, p.record_bytes, Lout);
        } else {
            cudaFuncSetAttribute(chunk_intra_simt_kernel<float>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_intra);
            chunk_intra_simt_kernel<float><<<grid, SIMT_THREADS, smem_intra, stream>>>(
                (const float *)a->q, (const float *)a->k, (const float *)a->v, (const float *)a->z,
                (const float *)a->beta, a->dt_bias, a->A_log, a->g_min, a->gate_kind, a->T, (int)a->N, a->cu_seqlens,
                chunk_start, H, dk, dv, C, records, p.record_bytes, Lout);
        }
        {
            const kda_status_t cst = kda_cuda_status(cudaGetLastError());
            if (cst != KDA_OK) return cst;
        }
    }
    kda_profile_mark(2, stream);
    if (kda_launch_chain_ckpt_tc(a, chunk_start, records, p.record_bytes, ckpt, stream)) {
        kda_profile_mark(3, stream);
        return kda_cuda_status(cudaGetLastError());
    }
    dim3 grid2((unsigned)(a->N * H), (unsigned)(dv / SLICE));
    auto chain = [&](auto kern, auto *out) {
        cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem_chain);
        kern<<<grid2, SIMT_THREADS, smem_chain, stream>>>(a->T, (int)a->N, a->cu_seqlens, chunk_start, H, dv, C,
                                                          records, p.record_bytes, a->scale, a->initial_state,
                                                          a->final_state, out, ckpt);
    };
    if (b16) {
        if (dk == 128) chain(chunk_chain_simt_kernel<bf16, 128>, (bf16 *)a->o);
        else chain(chunk_chain_simt_kernel<bf16, 64>, (bf16 *)a->o);
    } else {
        if (dk == 128) chain(chunk_chain_simt_kernel<float, 128>, (float *)a->o);
        else chain(chunk_chain_simt_kernel<float, 64>, (float *)a->o);
    }
    kda_profile_mark(3, stream);
    return kda_cuda_status(cudaGetLastError());
}

kda_status_t kda_launch_chunk_simt(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                   cudaStream_t stream) {
    return launch_simt(a, p, ws, stream, nullptr, nullptr);
}

kda_status_t kda_launch_chunk_simt_recompute(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                             float *Lout, float *ckpt, cudaStream_t stream) {
    return launch_simt(a, p, ws, stream, Lout, ckpt);
}
