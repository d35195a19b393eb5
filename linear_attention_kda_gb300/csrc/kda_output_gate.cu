// Output epilogue of Eq. 6 (Kimi K3 technical report, section 2.1.1) without the projections:
//     y[t,h,c] = Sigmoid(g[t,h,c]) * w[h,c] * o[t,h,c] / sqrt(mean_c' o[t,h,c']^2 + eps),
// the per-head RMSNorm of the recurrent output followed by the data-dependent output gate.
//
// One warp per RPW (token, head) rows; each lane holds VPL = dv / 32 consecutive channels of a row (one
// vector load per tensor), the sum of squares is a warp-shuffle reduction.  All of a warp's loads are
// issued before the first is used, so that enough bytes are in flight to cover HBM latency.  HBM-bound: o and g are read
// once, y written once (y may alias o: every element is read before it is written, by the same
// thread).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace og {

template <int BYTES>
__device__ __forceinline__ void ld_bytes(const void *p, uint32_t *w) {
    if constexpr (BYTES == 2) {
        w[0] = *reinterpret_cast<const unsigned short *>(p);
    } else if constexpr (BYTES == 4) {
        w[0] = *reinterpret_cast<const uint32_t *>(p);
    } else if constexpr (BYTES == 8) {
        const uint2 v = *reinterpret_cast<const uint2 *>(p);
        w[0] = v.x; w[1] = v.y;
    } else {
#pragma unroll
        for (int i = 0; i < BYTES / 16; ++i) {
            const uint4 v = reinterpret_cast<const uint4 *>(p)[i];
            w[4 * i] = v.x; w[4 * i + 1] = v.y; w[4 * i + 2] = v.z; w[4 * i + 3] = v.w;
        }
    }
}
template <int BYTES>
__device__ __forceinline__ void st_bytes(void *p, const uint32_t *w) {
    if constexpr (BYTES == 2) {
        *reinterpret_cast<unsigned short *>(p) = (unsigned short)w[0];
    } else if constexpr (BYTES == 4) {
        *reinterpret_cast<uint32_t *>(p) = w[0];
    } else if constexpr (BYTES == 8) {
        *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
    } else {
#pragma unroll
        for (int i = 0; i < BYTES / 16; ++i)
            reinterpret_cast<uint4 *>(p)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
    }
}

// VPL values of type T (bf16 or fp32) as fp32, from / to 32-bit words
template <typename T, int VPL>
__device__ __forceinline__ void unpack(const uint32_t *w, float *f) {
#pragma unroll
    for (int e = 0; e < VPL; ++e) {
        if constexpr (sizeof(T) == 4) {
            f[e] = __uint_as_float(w[e]);
        } else {
            const uint32_t x = w[e >> 1];
            f[e] = __uint_as_float(((e & 1) ? (x & 0xFFFF0000u) : (x << 16)));
        }
    }
}
template <typename T, int VPL>
__device__ __forceinline__ void pack(const float *f, uint32_t *w) {
#pragma unroll
    for (int e = 0; e < VPL; ++e) {
        if constexpr (sizeof(T) == 4) {
            w[e] = __float_as_uint(f[e]);
        } else {
            const uint32_t b = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f[e]));
            if (e & 1) w[e >> 1] |= b << 16; else w[e >> 1] = b;
        }
    }
}

constexpr int RPW = 4;  // rows per warp: their loads are all issued before any is used

template <typename T, int VPL>
__global__ void __launch_bounds__(256) output_gate_kernel(const T *__restrict__ o, const T *__restrict__ g,
                                                          const float *__restrict__ w, float eps, int64_t rows,
                                                          int H, T *y) {
    constexpr int DV = 32 * VPL, BYTES = VPL * (int)sizeof(T), WORDS = (BYTES + 3) / 4;
    const int lane = threadIdx.x & 31;
    const int64_t row0 = ((int64_t)blockIdx.x * 8 + (threadIdx.x >> 5)) * RPW;
    uint32_t ow[RPW][WORDS], gw[RPW][WORDS];
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        if (row0 + i < rows) {
            const size_t base = (size_t)(row0 + i) * DV + (size_t)VPL * lane;
            ld_bytes<BYTES>(o + base, ow[i]);
            ld_bytes<BYTES>(g + base, gw[i]);
        }
    }
#pragma unroll
    for (int i = 0; i < RPW; ++i) {
        const int64_t row = row0 + i;
        if (row >= rows) break;  // warp-uniform
        const int h = (int)(row % H);
        float ov[VPL], gv[VPL];
        unpack<T, VPL>(ow[i], ov);
        unpack<T, VPL>(gw[i], gv);
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < VPL; ++e) ss = fmaf(ov[e], ov[e], ss);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
        const float r = rsqrtf(ss * (1.0f / DV) + eps);
        float yv[VPL];
#pragma unroll
        for (int e = 0; e < VPL; ++e) {
            const float wv = w ? __ldg(w + (size_t)h * DV + VPL * lane + e) : 1.f;
            yv[e] = __fdividef(ov[e] * r * wv, 1.0f + __expf(-gv[e]));  // 1 + e^{-g} >= 1; inf gives 0
        }
        uint32_t yw[WORDS];
        pack<T, VPL>(yv, yw);
        st_bytes<BYTES>(y + (size_t)row * DV + (size_t)VPL * lane, yw);
    }
}

template <typename T>
static kda_status_t launch_t(const kda_output_gate_args *a, cudaStream_t stream) {
    const int64_t rows = a->T * (int64_t)a->H;
    const unsigned grid = (unsigned)((rows + 8 * RPW - 1) / (8 * RPW));
    const T *o = (const T *)a->o, *g = (const T *)a->g;
    T *y = (T *)a->y;
    switch (a->dv) {
        case 32: output_gate_kernel<T, 1><<<grid, 256, 0, stream>>>(o, g, a->norm_weight, a->eps, rows, a->H, y); break;
        case 64: output_gate_kernel<T, 2><<<grid, 256, 0, stream>>>(o, g, a->norm_weight, a->eps, rows, a->H, y); break;
        case 128: output_gate_kernel<T, 4><<<grid, 256, 0, stream>>>(o, g, a->norm_weight, a->eps, rows, a->H, y); break;
        case 256: output_gate_kernel<T, 8><<<grid, 256, 0, stream>>>(o, g, a->norm_weight, a->eps, rows, a->H, y); break;
        default: return KDA_ERR_UNSUPPORTED_SHAPE;
    }
    return kda_cuda_status(cudaGetLastError());
}

}  // namespace og
}  // namespace kda

kda_status_t kda_launch_output_gate(const kda_output_gate_args *a, cudaStream_t stream) {
    if (a->T == 0) return KDA_OK;
    return a->dtype == KDA_BF16 ? kda::og::launch_t<__nv_bfloat16>(a, stream) : kda::og::launch_t<float>(a, stream);
}
