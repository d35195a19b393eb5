// Output epilogue of Eq. 6 (Kimi K3 technical report, section 2.1.1) without the projections:
//     y[t,h,c] = Sigmoid(g[t,h,c]) * w[h,c] * o[t,h,c] / sqrt(mean_c' o[t,h,c']^2 + eps),
// the per-head RMSNorm of the recurrent output followed by the data-dependent output gate.
//
// Every lane moves whole 16-byte vectors: a row (one token, one head) is split over the fewest lanes
// that hold it in 16-byte pieces (4 to 32 lanes), the sum of squares is a shuffle reduction over those
// lanes, and a warp keeps the loads of two groups of four passes (8 to 32 rows each) in flight, so that
// enough bytes are outstanding to cover HBM latency.  HBM-bound: o and g are read once, y written once
// (y may alias o: every element is read before it is written, by the same thread).
#include "kda_common.cuh"
#include "kda_internal.h"

namespace kda {
namespace og {

// 8 bf16 or 4 fp32 values of one 16-byte vector, as fp32
template <typename T>
__device__ __forceinline__ void unpack16(const uint4 &u, float *f) {
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
    if constexpr (sizeof(T) == 4) {
#pragma unroll
        for (int e = 0; e < 4; ++e) f[e] = __uint_as_float(w[e]);
    } else {
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            f[2 * e] = __uint_as_float(w[e] << 16);
            f[2 * e + 1] = __uint_as_float(w[e] & 0xFFFF0000u);
        }
    }
}
template <typename T>
__device__ __forceinline__ uint4 pack16(const float *f) {
    if constexpr (sizeof(T) == 4) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3]));
    } else {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e)
            w[e] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f[2 * e])) |
                   ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f[2 * e + 1])) << 16);
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
}

// A row (one token, one head: DV values) is split over LPR lanes, each holding VPL 16-byte vectors;
// a warp pass covers 32 / LPR rows and a warp's unit of work is PASSES passes (a "row group").
constexpr int PASSES = 4;

template <typename T, int DV>
struct RowSplit {
    static constexpr int VEC = 16 / (int)sizeof(T);       // values per 16-byte vector
    static constexpr int NV = DV / VEC;                   // vectors per row
    static constexpr int LPR = NV < 32 ? NV : 32;         // lanes per row
    static constexpr int VPL = NV / LPR;                  // vectors per lane
    static constexpr int RPP = 32 / LPR;                  // rows per warp pass
    static constexpr int ROWS_PER_GROUP = RPP * PASSES;
    static_assert(NV % LPR == 0 && 32 % LPR == 0, "row split");
};

// Persistent: a grid that fills the GPU once; warp q of the grid takes row groups q, q + Q, ... and
// issues the loads of its next group before it computes the current one, so that every warp keeps
// two groups of o and g in flight (no tail wave, no gap between groups).
template <typename T, int DV>
__global__ void __launch_bounds__(256) output_gate_kernel(const T *__restrict__ o, const T *__restrict__ g,
                                                          const float *__restrict__ w, float eps, int64_t rows,
                                                          int H, T *y) {
    using RS = RowSplit<T, DV>;
    constexpr int VEC = RS::VEC, LPR = RS::LPR, VPL = RS::VPL, RPP = RS::RPP, RG = RS::ROWS_PER_GROUP;
    const int lane = threadIdx.x & 31, sub = lane / LPR, li = lane % LPR;
    const int64_t groups = (rows + RG - 1) / RG;
    const int64_t q0 = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int64_t Q = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int c0 = li * VPL * VEC;  // first channel of this lane
    uint4 ov[2][PASSES][VPL], gv[2][PASSES][VPL];
    auto load = [&](int64_t grp, int buf) {
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            const int64_t row = grp * RG + p * RPP + sub;
#pragma unroll
            for (int j = 0; j < VPL; ++j) {
                if (row < rows) {
                    const size_t off = (size_t)row * DV + c0 + j * VEC;
                    ov[buf][p][j] = __ldcs(reinterpret_cast<const uint4 *>(o + off));  // read once: streaming
                    gv[buf][p][j] = __ldcs(reinterpret_cast<const uint4 *>(g + off));
                } else {
                    ov[buf][p][j] = gv[buf][p][j] = make_uint4(0, 0, 0, 0);
                }
            }
        }
    };
    auto compute = [&](int64_t grp, int buf) {
#pragma unroll
        for (int p = 0; p < PASSES; ++p) {
            const int64_t row = grp * RG + p * RPP + sub;
            float of[VPL * VEC];
#pragma unroll
            for (int j = 0; j < VPL; ++j) unpack16<T>(ov[buf][p][j], of + j * VEC);
            float ss = 0.f;
#pragma unroll
            for (int e = 0; e < VPL * VEC; ++e) ss = fmaf(of[e], of[e], ss);
#pragma unroll
            for (int off = LPR / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);  // the row's lanes
            if (row >= rows) continue;  // after the shuffles, which every lane joins
            const float r = rsqrtf(ss * (1.0f / DV) + eps);
            const int h = (int)(row % H);
#pragma unroll
            for (int j = 0; j < VPL; ++j) {
                float gf[VEC], yf[VEC], wf[VEC];
                unpack16<T>(gv[buf][p][j], gf);
#pragma unroll
                for (int e = 0; e < VEC; e += 4) {
                    const float4 w4 = w ? __ldg(reinterpret_cast<const float4 *>(w + (size_t)h * DV + c0 + j * VEC + e))
                                        : make_float4(1.f, 1.f, 1.f, 1.f);
                    wf[e] = w4.x; wf[e + 1] = w4.y; wf[e + 2] = w4.z; wf[e + 3] = w4.w;
                }
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    yf[e] = __fdividef(of[j * VEC + e] * r * wf[e], 1.0f + __expf(-gf[e]));  // 1 + e^{-g} >= 1; inf gives 0
                __stcs(reinterpret_cast<uint4 *>(y + (size_t)row * DV + c0 + j * VEC), pack16<T>(yf));
            }
        }
    };
    if (q0 >= groups) return;
    // two register buffers in turn (y may alias o: the next group's rows are other rows, and every row
    // is read before it is written)
    load(q0, 0);
    for (int64_t grp = q0; grp < groups; grp += 2 * Q) {
        if (grp + Q < groups) load(grp + Q, 1);
        compute(grp, 0);
        if (grp + Q >= groups) break;
        if (grp + 2 * Q < groups) load(grp + 2 * Q, 0);
        compute(grp + Q, 1);
    }
}

template <typename T, int DV>
static void launch_dv(const kda_output_gate_args *a, int64_t rows, cudaStream_t stream) {
    constexpr int RG = RowSplit<T, DV>::ROWS_PER_GROUP;
    static int per_sm = 0, sms = 0;  // occupancy of this instantiation and the device's SMs (looked up once)
    if (per_sm == 0) {
        int dev = 0;
        cudaGetDevice(&dev);
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
        if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, output_gate_kernel<T, DV>, 256, 0) != cudaSuccess ||
            per_sm < 1)
            per_sm = 1;
    }
    const int64_t groups = (rows + RG - 1) / RG, need = (groups + 7) / 8;  // 8 warps per block
    const int64_t full = (int64_t)sms * per_sm;
    const unsigned grid = (unsigned)(need < full ? need : full);
    output_gate_kernel<T, DV><<<grid, 256, 0, stream>>>((const T *)a->o, (const T *)a->g, a->norm_weight, a->eps,
                                                        rows, a->H, (T *)a->y);
}

template <typename T>
static kda_status_t launch_t(const kda_output_gate_args *a, cudaStream_t stream) {
    const int64_t rows = a->T * (int64_t)a->H;
    switch (a->dv) {
        case 32: launch_dv<T, 32>(a, rows, stream); break;
        case 64: launch_dv<T, 64>(a, rows, stream); break;
        case 128: launch_dv<T, 128>(a, rows, stream); break;
        case 256: launch_dv<T, 256>(a, rows, stream); break;
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
