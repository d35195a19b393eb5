// The fp32 path's per-(chunk slot, head) intra-chunk record and chunk-slot lookup, shared by the
// fp32 forward (kda_chunk_simt.cu) and the backward pass (kda_chunk_bwd.cu).
#pragma once
#include <stdint.h>

namespace kda {

// Record of one (chunk slot, head), fp32, rows token-major: W, Q^, K~ [C][dk]; U [C][dv]; A [C][C]
// (lower triangle, diagonal kept); gamma^C [dk].
struct F32Record {
    float *W, *U, *Q, *K, *A, *gam;
};
__device__ __forceinline__ F32Record f32_record(const char *base, size_t rec_bytes, int64_t slot, int H, int h,
                                                int C, int dk, int dv) {
    float *r = (float *)(base + ((size_t)slot * H + h) * rec_bytes);
    F32Record v;
    v.W = r;
    v.U = v.W + C * dk;
    v.Q = v.U + C * dv;
    v.K = v.Q + C * dk;
    v.A = v.K + C * dk;
    v.gam = v.A + C * C;
    return v;
}

// Chunk slot -> (sequence n, first token t0, valid length len); false past the last chunk.  Chunks
// start at every sequence's first token (cu_seqlens, or N equal lengths T / N without it).
__device__ __forceinline__ bool locate_chunk(const int32_t *chunk_start, const int32_t *cu, int64_t T, int N,
                                             int C, int64_t slot, int &n, int64_t &t0, int &len) {
    if (slot >= chunk_start[N]) return false;
    int lo = 0, hi = N;  // largest n with chunk_start[n] <= slot
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (chunk_start[mid] <= slot) lo = mid; else hi = mid;
    }
    n = lo;
    const int64_t s = cu ? (int64_t)cu[n] : (T / N) * n;
    const int64_t e = cu ? (int64_t)cu[n + 1] : s + T / N;
    t0 = s + (slot - chunk_start[n]) * (int64_t)C;
    len = (int)min((int64_t)C, e - t0);
    return true;
}

}  // namespace kda
