// Tensor-core path of kda_chunk_fwd: bf16 I/O, d_k = d_v = 128, C = 64.
//
// The kernels below (plus the chunk plan) evaluate Eq. 3 and Eq. 4 of the Kimi K3
// report (section 2.1.1).  Every dense contraction runs on tcgen05.mma
// (kind::f16, bf16 operands in shared memory, fp32 accumulators in tensor
// memory); the scan-like and exponential work runs on the CUDA cores in fp32.
//
// 1. chunk_intra_tc (persistent, one CTA per SM over the (chunk, head) items)
//    computes the gate, the decays, A, the UT transform T = (I + L)^{-1}, W and U
//    of each chunk and writes a per-(chunk, head) packet of ready-to-use operand
//    images: W^T [128 x 64], Q^ = Q Gamma [64 x 128], K~ = K e^{G_last - G}
//    [64 x 128], A [64 x 64], U^T [128 x 64], gamma^C [128] fp32.
// 2. chunk_inter_tc (one CTA per (segment, head); chunks in order)
//    The state is kept transposed in tensor memory, S^T [d_v lanes x d_k
//    columns] fp32, and as a bf16 operand image in shared memory.  Per chunk:
//      V~^T = U^T - S^T W^T                      (MMA, M = 128, N = 64, K = 128)
//      O^T  = S^T Q^^T + V~^T A^T                (MMA, K = 128 then K = 64)
//      S^T <- S^T Diag(gamma^C) + V~^T K~        (scale in fp32, MMA N = 128, K = 64)
//    Packets are streamed by 1-D bulk copies, double buffered.
// 3. chunk_segsum_tc / chunk_fold_tc: the split-sequence state pass (section 5.1.2).
// Waits on mbarriers give up after about a second, set KDA_ERR_DEVICE_TIMEOUT,
// and the kernel still releases its tensor memory before it returns.
#include "kda_common.cuh"
#include "kda_internal.h"
#include "tc_util.cuh"

#include <cuda.h>

#include <atomic>
#include <chrono>

namespace kda {
namespace tcp {

using namespace kda::tc;

constexpr int C = 64;   // chunk
constexpr int D = 128;  // d_k = d_v

// packet layout (bytes)
// Operands are token-major ([token][channel] rows of 128 bytes, 128-byte swizzle), except U, kept
// as U^T (rows are value channels).  Part 1
// ([W; Q^], U, gamma) is what a chunk's first MMAs and the decay of the state before it read; part 2
// (K~, A) is read last, so the output pass loads and releases the two parts separately.
constexpr uint32_t PK_WQ = 0;         // [W; Q^]: one K-major 128-row image (rows 0-63 W, rows 64-127 Q^),
                                      // 16 KB per 64-channel block
constexpr uint32_t PK_U = 32768;      // U^T [128 channels][64 tokens]: K-major image, rows d_v
constexpr uint32_t PK_G = 49152;      // gamma^C fp32 [128]
constexpr uint32_t PK_K = 50176;      // K~ [64 tokens][128 channels] (two halves)
constexpr uint32_t PK_A = 66560;      // A [64 query rows][64 keys]
constexpr uint32_t PK_STRIDE = 74752; // multiple of 1024
constexpr uint32_t PK_P1 = PK_G + 512;        // bytes of part 1 (at 0)
constexpr uint32_t PK_P2 = PK_STRIDE - PK_K;  // bytes of part 2 (at PK_K)

// inter kernel shared memory
// Output pass: two stages hold whole packets (two bulk copies each, one per part); without flags
// the packet after them is prefetched into L2.
constexpr uint32_t CS_ST_BYTES = PK_STRIDE;            // stage stride (multiple of 1024)
constexpr uint32_t CS_OIMG = 2 * CS_ST_BYTES;          // o staging, 2 buffers x (64 tokens x 128, 2 x 8 KB)
constexpr uint32_t CS_GIMG = CS_OIMG + 32768;          // output epilogue: gate tiles, 2 buffers (same layout)
constexpr uint32_t CS_W = CS_GIMG + 32768;             // output epilogue: RMSNorm weight of the head, fp32 [128]
constexpr uint32_t CS_BAR = CS_W + 512;                // 15 mbarriers
constexpr uint32_t CS_TSLOT = CS_BAR + 128;            // TMEM base, failure flag
constexpr uint32_t CS_TOTAL = CS_BAR + 192 + 1024;
static_assert(PK_P1 <= PK_K && PK_P1 % 16 == 0 && PK_P2 % 16 == 0, "packet parts");

__device__ __forceinline__ unsigned char *align1024(unsigned char *p) {
    const uint32_t s = smem_u32(p);
    return p + ((1024u - (s & 1023u)) & 1023u);
}

// Float offset of element (i, c) of a 128 x 128 fp32 matrix kept in the workspace in "lane-major"
// order: float4 (c / 4) of row i at ((c / 4) * 128 + i) * 4, so that the 32 rows of a warp (one row per
// thread) read or write 512 contiguous bytes per float4 column.
__device__ __forceinline__ size_t ll_off(int i, int c) { return ((size_t)(c >> 2) * 128 + i) * 4 + (c & 3); }

__device__ __forceinline__ void named_sync(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(nthreads) : "memory");
}

// bar.red.popc over the n threads of named barrier id: the number of them with pred set.
__device__ __forceinline__ int bar_red_popc(int id, int n, bool pred) {
    int r;
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.popc.u32 %0, %2, %3, p;\n\t}\n"
                 : "=r"(r) : "r"((unsigned)pred), "r"(id), "r"(n) : "memory");
    return r;
}

// bar.red.popc over the 256 threads of named barrier 1.
__device__ __forceinline__ int __syncthreads_count_named1(bool pred) {
    int r;
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.u32 p, %1, 0;\n\tbar.red.popc.u32 %0, 1, 256, p;\n\t}\n"
                 : "=r"(r) : "r"((unsigned)pred) : "memory");
    return r;
}

__device__ __forceinline__ void sync_all() {
    fence_before_sync();
    __syncthreads();
    fence_after_sync();
}

// 8 bf16 <-> fp32
__device__ __forceinline__ void unpack8(const uint4 &u, float *f) {
    const __nv_bfloat162 *h = reinterpret_cast<const __nv_bfloat162 *>(&u);
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const float2 x = __bfloat1622float2(h[i]);
        f[2 * i] = x.x;
        f[2 * i + 1] = x.y;
    }
}
__device__ __forceinline__ uint4 pack8(const float *f) {
    uint4 u;
    u.x = pack_bf16(f[0], f[1]);
    u.y = pack_bf16(f[2], f[3]);
    u.z = pack_bf16(f[4], f[5]);
    u.w = pack_bf16(f[6], f[7]);
    return u;
}

// Waits on an mbarrier from every thread; returns a CTA-uniform "all ok".
__device__ __forceinline__ bool wait_all(uint64_t *bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return __syncthreads_and(ok ? 1 : 0) != 0;
}

// =====================================================================================
// Persistent intra-chunk kernel: one CTA per SM works through the (chunk, head) items
// w = slot * H + h, taking them two at a time from a launch-wide counter.  Its sixteen warps form two
// groups of eight; group g takes the second (g = 1) or first (g = 0) item of each pair and owns a full
// set of buffers (a ~100 KB region of shared memory and 256 tensor-memory columns), so that the two
// groups run out of phase: while one inverts (I + L) (a latency-bound step), the other runs the gate
// and element pass of its next item (MUFU and shared-memory bound).  The group's warp 0 moves its
// data: the q, z, k, v tiles (128-byte-swizzled TMA boxes of 64 tokens x 64 channels) and the item's
// beta, bias and A_log in (cp.async), the packet out by bulk copies.
//
// Tiles stay token-major ([token][channel], the TMA layout) from load to packet: tcgen05 reads a
// token-major tile as a K-major operand when the contraction runs over channels and, through an
// MN-major descriptor, as its transpose when it runs over tokens.  Per item:
//   GATE gate (Eq. 5) and in-chunk cumulative log-decay G (Eq. 3), in base-2 units; thread = (16-byte
//        chunk of 8 channels, 4 tokens), G kept in registers.
//   ELEM element pass, same threads: every decay factor and operand image, 16 bytes per access.  The q and z boxes are
//        loaded as one 128-row image [q; z]; it becomes the row image [q E; k E] in place.  Keys
//        scaled to the second reference overwrite k; X = Gamma K goes to its own tile.  Q^ = Q Gamma
//        and K~ = K e^{G_63 - G} go straight from registers to the packet in global memory.
//   MMA  A = Tril[(Q Gamma)(K / Gamma)^T] and L = StrictTril[diag(beta)(K Gamma)(K / Gamma)^T]:
//        M = 128 (64 query rows over 64 key rows), N = 32 + 64 (keys scaled to either
//        reference), K = 128 channels.
//   INV  T = (I + L)^{-1} in fp32: 16 x 16 diagonal blocks by substitution, then one 16-row and
//        one 32-row block merge, T21 = -T22 L21 T11.
//   MMA  W = (T diag beta) X and U^T = V^T (T diag beta)^T, X and V read MN-major.
//   OUT  packet: [W; Q^], U^T, gamma, K~, A.
//
// Exponent safety.  Each log-decay step lies in (g_min, 0) = (-5, 0), so 16 tokens span less than
// 80 in the exponent, inside the fp32 / bf16 range of e^{+-88}.  The chunk is cut into two
// 32-token halves with references p0 = 15 and p1 = 47, 16 tokens from either end of their half.
// Rows r of half b are scaled by E_r = e^{G_r - G_pb} (|exponent| <= 80).  Keys of half 0 are
// scaled by e^{G_p0 - G_i} for the products with rows of half 0 (<= e^{80}), and every key by
// e^{G_p1 - G_i} for the products with rows of half 1 (<= 1 for keys of half 0).  Each factor is
// the exponential of its own exponent, never a product of two large and small factors, so a key
// factor that underflows loses at most e^{75 - 87} of a term.  Entries above the diagonal may
// overflow to inf; they are discarded by selects and never multiplied.
constexpr int NT2 = 512;      // 2 consumer groups x 8 warps
constexpr int NCG = 256;      // threads of a consumer group
// Per-group shared-memory region (offsets from the group's base, multiple of 1024)
constexpr uint32_t GR_QZ = 0;          // 32 KB: TMA boxes q h0 | z h0 | q h1 | z h1 = a K-major 128-row image
                                       // [q; z]; then the row image [q E; k E]; after the A / L product the
                                       // fp32 L, T and P of the inverse (which spill into GR_K)
constexpr uint32_t GR_K = 32768;       // 16 KB: k tile -> keys scaled to p1 (64-row K-major image)
constexpr uint32_t GR_V = 49152;       // 16 KB: v tile -> U^T image [128 channels][64 tokens]
constexpr uint32_t GR_X = 65536;       // 16 KB: X = Gamma K (token-major) -> W rows
constexpr uint32_t GR_K0 = 81920;      // 8 KB: keys 0-31 scaled to p0 (32 rows); then the (T diag beta) image
constexpr uint32_t GR_A = 90112;       // 8 KB: A image (rows 64-127 of the W product's A operand)
constexpr uint32_t GR_GAM = 98304;     // gamma^C fp32 [128]
constexpr uint32_t GR_TOT = GR_GAM + 512;    // quarter sums of the log-decays, fp32 [4][128]
constexpr uint32_t GR_BETA = GR_TOT + 2048;  // 2 slots x fp32 [64]
constexpr uint32_t GR_BIAS = GR_BETA + 512;  // 2 slots x fp32 [128]
constexpr uint32_t GR_INFO = GR_BIAS + 1024; // 2 slots x {int64 t0, len, h, w; float e^{A_log}} (64 B)
constexpr uint32_t GR_BAR = GR_INFO + 128;   // mbarriers: ld_qzk, ld_v, mma
constexpr uint32_t GR_BYTES = 103424;        // 101 KB
static_assert(GR_BAR + 64 <= GR_BYTES && GR_BYTES % 1024 == 0, "group region");
// The fp32 L and T of the inverse are kept as SW128 images (fimg below): the tf32 products of its
// last merge read them in place.
constexpr uint32_t GR_L = GR_QZ;             // fp32 L image (16 KB)
constexpr uint32_t GR_T = GR_QZ + 16384;     // fp32 T image (16 KB)
constexpr uint32_t GR_P = GR_K + 8192;       // P^T (P = L_21 T_11) as a K-major tf32 image, 32 rows (4 KB)
constexpr uint32_t GR_TT = GR_K + 12288;     // T_11^T as a K-major tf32 image, 32 rows (4 KB)
constexpr uint32_t J_SH = 2 * GR_BYTES;       // shared by both groups
constexpr uint32_t J_TSLOT = J_SH;            // TMEM base
constexpr uint32_t J_TOK = J_SH + 16;         // mbarriers tok[2]: group g may start its gate and element pass
constexpr uint32_t J_PAIR = J_SH + 32;        // int64 [4]: items taken from the launch's counter
// Tables a CTA keeps while it runs both roles (fused and team launches): past the shared memory of either
constexpr uint32_t J_TAB0 = (J_SH + 64 > CS_BAR + 256 ? J_SH + 64 : CS_BAR + 256);
constexpr uint32_t J_TBL = (J_TAB0 + 63) / 64 * 64;  // int32 [J_TBL_N + 1]: producer chunks before each sequence
constexpr int J_TBL_N = KDA_FUSED_MAX_SEQS;   // sequences the table holds
constexpr uint32_t J_CS = J_TBL + 4 * (J_TBL_N + 1);  // fused launch: chunk_start [N + 1]
constexpr uint32_t J_SS = J_CS + 4 * (J_TBL_N + 1);   //               seg_start [N + 1], then a flag
constexpr uint32_t J_CU = J_SS + 4 * (J_TBL_N + 2);   // cu_seqlens [N + 1] (and chunk_start in J_CS), so that
                                                      // the producers locate their items without global loads
constexpr uint32_t J_TOTAL = J_CU + 4 * (J_TBL_N + 1) + 1024;
// TMEM columns of a group (base + 256 g): the A / L product in [0, 96); later W in [0, 128) (lanes
// 0-63) and U^T in [128, 192)
constexpr uint32_t TM_DA = 0, TM_DW = 0, TM_DUT = 128;

constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ float ex2_approx(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

struct TileMaps {
    CUtensorMap q, k, v, z;
};

// Named barrier of consumer group g (ids 1, 2), with tcgen05 ordering.
__device__ __forceinline__ void gsync(int g) {
    fence_before_sync();
    named_sync(1 + g, NCG);
    fence_after_sync();
}
// All threads of group g: true iff pred held in every one of them.
__device__ __forceinline__ bool gsync_and(int g, bool pred) {
    return bar_red_popc(1 + g, NCG, pred) == NCG;
}
// Waits on an mbarrier from every thread of group g; group-uniform result.
__device__ __forceinline__ bool gwait(int g, uint64_t *bar, uint32_t parity) {
    const bool ok = mbar_wait(bar, parity);
    return gsync_and(g, ok);
}

// Float index of element (r, c) of a 64 x 64 fp32 matrix kept as a K-major SW128 image: two column
// blocks of 32 values (8 KB each), rows of 128 bytes, 16-byte chunk j of row r at position j ^ (r % 8).
// Read by tf32 MMAs as an A operand (rows M, columns K) or, rows being K, as an MN-major B operand.
__device__ __forceinline__ int fimg(int r, int c) {
    return ((c >> 5) << 11) + (r << 5) + ((((c & 31) >> 2) ^ (r & 7)) << 2) + (c & 3);
}

// Partial products of the level-1 block merges of the UT-transform inverse: P[q + 4 a][jc] =
// L[ro + q + 4 a][co .. co + 15] . T[co .. co + 15][co + jc], starting at column K0 <= jc (T is zero
// above the diagonal).
template <int K0>
__device__ __forceinline__ void inv_l1_partial(const float *Lm, const float *Tm, int ro, int co, int q, int jc,
                                               float *p) {
    float tc[16];
#pragma unroll
    for (int k = K0; k < 16; ++k) tc[k] = Tm[fimg(co + k, co + jc)];
#pragma unroll
    for (int a = 0; a < 4; ++a) {
        float acc = 0.f;
#pragma unroll
        for (int k = K0; k < 16; k += 4) {
            const float4 l4 = *reinterpret_cast<const float4 *>(Lm + fimg(ro + q + 4 * a, co + k));
            acc += l4.x * tc[k] + l4.y * tc[k + 1] + l4.z * tc[k + 2] + l4.w * tc[k + 3];
        }
        p[a] = acc;
    }
}

__device__ __forceinline__ float bf_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

// Packed fp32 pairs: one instruction computes both lanes (round to nearest even, as the scalar forms).
__device__ __forceinline__ unsigned long long f2u(float2 a) {
    return (unsigned long long)__float_as_uint(a.x) | ((unsigned long long)__float_as_uint(a.y) << 32);
}
__device__ __forceinline__ float2 u2f(unsigned long long u) {
    return make_float2(__uint_as_float((uint32_t)u), __uint_as_float((uint32_t)(u >> 32)));
}
__device__ __forceinline__ float2 fmul2(float2 a, float2 b) {
    unsigned long long r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(r);
}
__device__ __forceinline__ float2 fsub2(float2 a, float2 b) {
    unsigned long long r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(f2u(a)), "l"(f2u(b)));
    return u2f(r);
}
__device__ __forceinline__ uint32_t pack2(float2 a) { return pack_bf16(a.x, a.y); }

// Packet publication between CTAs of one (cooperative) launch: the producer releases a flag once the
// packet's writes have completed; the consumer acquires it before its bulk reads.
__device__ __forceinline__ void fence_proxy_async_global() { asm volatile("fence.proxy.async.global;" ::: "memory"); }
// Drops one 128-byte line from L2 without writing it back (its contents become undefined).
__device__ __forceinline__ void discard_l2(const void *p) {
    asm volatile("discard.global.L2 [%0], 128;" :: "l"(p) : "memory");
}

// Flags hold the epoch of the launch that published them (a per-process counter that never repeats),
// so a workspace needs no clearing between launches.
__device__ __forceinline__ void flag_release(uint64_t *f, uint64_t epoch) {
    asm volatile("st.release.gpu.global.b64 [%0], %1;" :: "l"(f), "l"(epoch) : "memory");
}
__device__ __forceinline__ uint64_t flag_acquire(const uint64_t *f) {
    uint64_t v;
    asm volatile("ld.acquire.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}
__device__ __forceinline__ uint64_t flag_relaxed(const uint64_t *f) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}
// Bounded wait (~1 s) for a packet flag to reach this launch's epoch.  The flag is polled with relaxed
// loads (an acquiring load per poll would order, and slow, the SM's other memory traffic); the read that
// sees the epoch is followed by an acquire fence, which orders the caller's later reads after it.
__device__ __forceinline__ bool flag_wait(const uint64_t *f, uint64_t epoch) {
    if (flag_acquire(f) == epoch) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 16; ++i) {
            if (flag_relaxed(f) == epoch) {
                asm volatile("fence.acq_rel.gpu;" ::: "memory");
                return true;
            }
            __nanosleep(32);
        }
        if (globaltimer_ns() - t0 > 1000000000ull) return false;
    }
}

// Team mode of the intra-chunk role (a producer CTA of a chain team): the team's chains in the order
// its chain CTA runs them, and the number of the team's items (chunks) before each chain.  Producer q of
// K takes the team's items q, q + K, ...; it starts an item only once the chain has started on the item
// `window` of its own items earlier, so that packets are read from L2 soon after they are written.
struct TeamItems {
    const int32_t *chain;  // [count] n * H + h
    const int32_t *pre;    // [count + 1]
    int count, K, q, window;
    const uint64_t *consumed;  // per item: the launch's epoch once the chain has started on it
};

// The intra-chunk work of one CTA.  Items (chunk slot, head) are numbered w = slot * H + h.
//  - own_n < 0, kpre == 0: worker `worker` of `nworkers` takes items worker, worker + nworkers, ...
//  - own_n < 0, kpre > 0: the same over the items left once the first kpre chunks of every
//    sequence are taken away (in the same order);
//  - own_n >= 0: the first kpre chunks of sequence own_n for head own_h;
//  - team != nullptr: the items of a chain team (see TeamItems).
// Each mode orders its items (k = 0, 1, ...).  Without `ctr` the CTA takes items k = worker,
// worker + nworkers, ... (a team producer q of K: q, q + K, ...), its it-th item going to consumer group
// it & 1.  With `ctr` (not for own_n >= 0), the CTA takes pairs of consecutive items, one per group, from
// a counter shared by the launch, so that CTAs on slower SMs take fewer items; the counter holds
// (low 32 bits of the epoch) << 32 | items taken, and the first CTA to see a stale tag installs this
// launch's.  With `flags`, each item's packet is published (flags[item] = epoch) once its writes have
// completed.  With own_n >= 0 the CTA keeps its right to allocate tensor memory (its chain runs next).
__device__ __forceinline__ void intra_role(unsigned char *sm, const TileMaps &tm, const bf16 *__restrict__ beta,
                                           const float *__restrict__ bias, const float *__restrict__ A_log,
                                           float g_min, int64_t T, int N, const int32_t *__restrict__ cu,
                                           const int32_t *__restrict__ chunk_start, int H,
                                           unsigned char *__restrict__ packets, int *err, int worker, int nworkers,
                                           uint64_t *flags, uint64_t epoch, int kpre, int own_n, int own_h,
                                           const TeamItems *team = nullptr, uint64_t *ctr = nullptr) {
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *tbl = (int32_t *)(sm + J_TBL);  // kpre > 0: tbl[n] = producer chunks of sequences before n
    int64_t n_all = 0;                       // items of the mode
    if (team) {
        n_all = team->pre[team->count];
    } else if (own_n >= 0) {
        n_all = min(kpre, chunk_start[own_n + 1] - chunk_start[own_n]);
    } else if (kpre > 0) {
        if (warp == 0) {
            int carry = 0;
            if (lane == 0) tbl[0] = 0;
            for (int base = 0; base < N; base += 32) {
                const int m = base + lane;
                int x = m < N ? max(0, chunk_start[m + 1] - chunk_start[m] - kpre) : 0;
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const int y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                if (m < N) tbl[m + 1] = carry + x;
                carry += __shfl_sync(0xffffffffu, x, 31);
            }
        }
        __syncthreads();
        n_all = (int64_t)tbl[N] * H;
    } else {
        n_all = (int64_t)chunk_start[N] * H;
    }
    const bool dyn = ctr != nullptr && own_n < 0;
    const int64_t k_first = team ? team->q : (own_n >= 0 ? 0 : worker);
    const int64_t k_step = team ? team->K : (own_n >= 0 ? 1 : nworkers);
    const int team_window = team ? team->window * team->K : 0;  // in team items
    int64_t *pk = (int64_t *)(sm + J_PAIR);  // dynamic: the first item of the CTA's pair j in pk[j & 3]
    bool ctr_live = false;                   // thread 0: the counter holds this launch's tag
    auto grab = [&]() -> uint64_t {          // thread 0: the counter before this CTA's next pair (low 32 bits:
                                             // its first item)
        const uint64_t tag = (uint64_t)(uint32_t)epoch << 32, hi = 0xffffffff00000000ull;
        unsigned long long *c = reinterpret_cast<unsigned long long *>(ctr);
        if (!ctr_live) {
            uint64_t cur = atomicAdd(c, 0ull);
            for (int i = 0; i < 1024 && (cur & hi) != tag; ++i) {
                const uint64_t prev = atomicCAS(c, cur, tag | 2ull);
                if (prev == cur) {
                    ctr_live = true;
                    return tag;
                }
                cur = prev;
            }
            if ((cur & hi) != tag) {
                set_error(err, KDA_ERR_DEVICE_TIMEOUT);
                return tag | (uint64_t)n_all;
            }
            ctr_live = true;
        }
        return atomicAdd(c, 2ull);
    };
    if (dyn) {
        if (tid == 0) {
            pk[0] = (int64_t)(grab() & 0xffffffffull);
            pk[1] = (int64_t)(grab() & 0xffffffffull);
        }
        __syncthreads();
        if (pk[0] >= n_all) return;
    } else if (k_first >= n_all) {
        return;
    }
    auto k_of = [&](int j, int gg) -> int64_t {  // mode item of group gg's j-th item
        return dyn ? pk[j & 3] + gg : k_first + (int64_t)(2 * j + gg) * k_step;
    };
    auto has = [&](int j, int gg) -> bool { return k_of(j, gg) < n_all; };
    auto w_of = [&](int64_t k64) -> int64_t {  // global item index of the mode's item k
        if (team) {
            const int k = (int)k64;
            int lo = 0, hi = team->count;  // the chain holding team item k: largest m with pre[m] <= k
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (team->pre[mid] <= k) lo = mid; else hi = mid;
            }
            const int id = team->chain[lo];
            return (int64_t)(chunk_start[id / H] + (k - team->pre[lo])) * H + (id % H);
        }
        if (own_n >= 0) return (int64_t)(chunk_start[own_n] + k64) * H + own_h;
        const int64_t k = k64;
        if (kpre <= 0) return k;
        const int64_t kk = k / H;
        int lo = 0, hi = N;  // the sequence holding producer chunk kk: largest n with tbl[n] <= kk
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (tbl[mid] <= kk) lo = mid; else hi = mid;
        }
        return (int64_t)(chunk_start[lo] + kpre + (kk - tbl[lo])) * H + (int)(k % H);
    };
    uint32_t *tslot = (uint32_t *)(sm + J_TSLOT);
    if (tid < 2) {
        uint64_t *b = (uint64_t *)(sm + tid * GR_BYTES + GR_BAR);
        mbar_init(&b[0], 1 + 32);  // ld_qzk: the TMA arrival and one per lane of warp 0 (the item's slot)
        for (int i = 1; i < 3; ++i) mbar_init(&b[i], 1);
        mbar_init((uint64_t *)(sm + J_TOK) + tid, 1);
    }
    if (warp == 0) tmem_alloc(tslot, 512, own_n < 0);
    fence_proxy_async();
    sync_all();
    const uint32_t tb = *tslot;

    // ------------------------------------------------ consumer group g (warps 8 g .. 8 g + 7).  Its thread 0
    // also moves the data: the next item's q, z and k tiles are loaded once the inverse has freed their
    // buffers, its v tile once the packet copies of the previous item have read the U^T image; the
    // packet's A image, W, U^T and gamma leave by bulk copies, and an item is published (flags) during the
    // A / L product of the group's next item, when its copies have long completed (in a chain team, at
    // the start of the next item, which may wait for the chain).
    const int g = warp >> 3, gt = tid & (NCG - 1), gw = gt >> 5;
    unsigned char *R = sm + g * GR_BYTES;
    uint64_t *bar = (uint64_t *)(R + GR_BAR);
    uint64_t *ld_qzk = bar, *ld_v = bar + 1, *bar_mma = bar + 2;
    const uint32_t tbg = tb + 256u * (uint32_t)g;
    // The two groups take turns at the gate and element pass (MUFU and shared-memory bound), each
    // starting it once the other has finished its own, so that one group's element pass overlaps the
    // other's inverse and products.  Group 0 starts.
    uint64_t *tok = (uint64_t *)(sm + J_TOK);
    uint32_t mph = 0;
    auto mwait = [&]() -> bool {  // the group's last MMA commit: thread 0 waits, the others sleep at the barrier
        bool o = true;
        if (gt == 0) o = mbar_wait(bar_mma, mph & 1);
        ++mph;
        return gsync_and(g, o);
    };
    // Item j's slot (warp 0 of the group): its location (from the chunk layout), and by asynchronous copies
    // that complete on the mbarrier of the item's tiles (each lane arrives once its copies have landed): the
    // 32-bit words holding its beta values (bf16; the gate pass widens them in place), its bias row and
    // A_log.  Nothing waits on these loads until the item starts; the slot (j & 1) was last used by item j - 2.
    // The slot's plain stores are ordered before their readers by the group barriers in between.
    int n_hint = 0;  // warp 0: the sequence of the group's last item
    auto fill_slot = [&](int j) {
        const int s = j & 1;
        const bool take = dyn && g == 0 && lane == 0 && j >= 1;  // group 0 takes pair j + 1 (the
        uint64_t nxt = 0;                                        // atomic's result is used at the end)
        if (take) nxt = grab();
        const int64_t w = w_of(k_of(j, g));
        int n = 0, len = 0, h;
        int64_t t0 = 0, slot;
        if (w <= 0xffffffffll) {  // 32-bit division where it suffices
            slot = (int64_t)((uint32_t)w / (uint32_t)H);
            h = (int)((uint32_t)w - (uint32_t)slot * (uint32_t)H);
        } else {
            slot = w / H;
            h = (int)(w % H);
        }
        // the sequence holding the slot: a group's slots mostly grow, so search forward from the last
        // one's sequence for a few steps, else bisect
        n = n_hint;
        if (slot < chunk_start[n]) n = 0;
        for (int step = 0; step < 4 && chunk_start[n + 1] <= slot; ++step) ++n;
        if (chunk_start[n + 1] <= slot) {
            int lo = n, hi = N;  // largest lo with chunk_start[lo] <= slot
            while (hi - lo > 1) {
                const int mid = (lo + hi) >> 1;
                if (chunk_start[mid] <= slot) lo = mid; else hi = mid;
            }
            n = lo;
        }
        n_hint = n;
        {
            const int64_t sb = cu ? (int64_t)cu[n] : (T / N) * n;
            const int64_t se = cu ? (int64_t)cu[n + 1] : sb + T / N;
            t0 = sb + (slot - chunk_start[n]) * (int64_t)C;
            len = (int)min((int64_t)C, se - t0);
        }
        uint32_t *bw = (uint32_t *)(R + GR_BETA) + 64 * s;
        float *bia = (float *)(R + GR_BIAS) + 128 * s;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const int t = lane + 32 * i;
            if (t < len)  // the aligned word holding the value: inside the tensor's pages
                cp_async4(bw + t, (const void *)((uintptr_t)(beta + (t0 + t) * H + h) & ~(uintptr_t)3));
            else
                bw[t] = 0u;
        }
        if (bias) cp_async16(bia + 4 * lane, bias + (size_t)h * D + 4 * lane);
        else reinterpret_cast<float4 *>(bia)[lane] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (lane == 0) {
            int64_t *info = (int64_t *)(R + GR_INFO + 64 * s);
            info[0] = t0;
            info[1] = len;
            info[2] = h;
            info[3] = w;
            float *al = reinterpret_cast<float *>(info + 4);  // A_log (0 without: e^0 = 1)
            if (A_log) cp_async4(al, A_log + h);
            else *al = 0.f;
        }
        cp_async_arrive_noinc(ld_qzk);
        if (take) pk[(j + 1) & 3] = (int64_t)(nxt & 0xffffffffull);
    };
    // Item j's q, z, k (and v) tiles by TMA (thread 0, which filled the slot)
    auto issue_tma = [&](int j, bool with_v) {
        const int64_t *info = (const int64_t *)(R + GR_INFO + 64 * (j & 1));
        const int t0 = (int)info[0], h = (int)info[2];
        mbar_arrive_expect_tx(ld_qzk, 6 * 8192);
        tma_load_3d(R + GR_QZ, &tm.q, 0, h, t0, ld_qzk);
        tma_load_3d(R + GR_QZ + 8192, &tm.z, 0, h, t0, ld_qzk);
        tma_load_3d(R + GR_QZ + 16384, &tm.q, 64, h, t0, ld_qzk);
        tma_load_3d(R + GR_QZ + 24576, &tm.z, 64, h, t0, ld_qzk);
        tma_load_3d(R + GR_K, &tm.k, 0, h, t0, ld_qzk);
        tma_load_3d(R + GR_K + 8192, &tm.k, 64, h, t0, ld_qzk);
        if (with_v) {
            mbar_arrive_expect_tx(ld_v, 2 * 8192);
            tma_load_3d(R + GR_V, &tm.v, 0, h, t0, ld_v);
            tma_load_3d(R + GR_V + 8192, &tm.v, 64, h, t0, ld_v);
        }
    };
    auto publish = [&](int64_t w) {  // thread 0: the item's packet copies have completed
        bulk_wait0();
        if (flags) {
            fence_proxy_async_global();
            flag_release(flags + w, epoch);
        }
    };
    bool ok = true;
    if (gw == 0 && has(0, g)) {
        fill_slot(0);
        if (lane == 0) issue_tma(0, true);
    }
    ok = gsync_and(g, ok);
    int64_t w_prev = -1;  // the group's previous item, published during the next one
    // element mapping: 8 channels (one 16-byte chunk cg of 64-channel block hb) x 4 tokens 16 tq + 4 tl + i
    const int hb = gw & 1, tq = gw >> 1, cg = lane & 7, tl = lane >> 3;
    const int c0 = 64 * hb + 8 * cg;
    for (int j = 0; has(j, g) && ok; ++j) {
        const uint32_t par = j & 1;
        const int s = j & 1;
        if (gt == 0 && j > 0) {
            // the previous item's copies have read X, A, gamma and the U^T image, so this item's v tile can
            // take the V buffer (their writes complete later: the packet is published after this item's
            // A / L product is issued)
            bulk_wait_read0();
            const int64_t *ip = (const int64_t *)(R + GR_INFO + 64 * s);
            mbar_arrive_expect_tx(ld_v, 2 * 8192);
            tma_load_3d(R + GR_V, &tm.v, 0, (int)ip[2], (int)ip[0], ld_v);
            tma_load_3d(R + GR_V + 8192, &tm.v, 64, (int)ip[2], (int)ip[0], ld_v);
        }
        {
            bool okt = true;
            if (gt == 0) {
                // a chain team's producer publishes its previous item before it may wait for the chain
                // (the chain may be waiting for that very packet)
                if (team && j > 0) publish(w_prev);
                const int64_t kb = k_of(j, g) - (int64_t)team_window;
                if (team && kb >= 0)  // start at most `window` items of each producer ahead of the chain
                    okt = flag_wait(team->consumed + w_of(kb), epoch);
                if (!okt) {
                } else if (g == 1) okt = mbar_wait(&tok[1], j & 1);       // group 0 has done its item j
                else if (j > 0) okt = mbar_wait(&tok[0], (j - 1) & 1);      // group 1 has done its item j - 1
            }
            ok = gsync_and(g, okt);
            if (!ok) break;
        }
        ok = gwait(g, ld_qzk, par);
        if (!ok) break;
        const int64_t *info = (const int64_t *)(R + GR_INFO + 64 * s);
        const int len = (int)info[1];
        const int64_t w = info[3];
        const float eA = __expf(*reinterpret_cast<const float *>(info + 4));
        const float *bet = (const float *)(R + GR_BETA) + 64 * s;
        const float *bia = (const float *)(R + GR_BIAS) + 128 * s;
        unsigned char *pk = packets + (size_t)w * PK_STRIDE;

        // ---- GATE: g = g_min Sigmoid(e^A (z + b)) (Eq. 5) in base-2 units (times log2 e), prefix sums over
        //      the thread's 4 tokens, then over the 4 threads of its 16-token quarter (shuffles), then (shared
        //      memory) over the quarters
        float G[4][8];
        {
            const float cz = -eA * LOG2E, gm = g_min * LOG2E;
            float cb[8];
            {
                const float4 b0 = *reinterpret_cast<const float4 *>(bia + c0);
                const float4 b1 = *reinterpret_cast<const float4 *>(bia + c0 + 4);
                const float bb[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
                for (int e = 0; e < 8; ++e) cb[e] = cz * bb[e];
            }
            const unsigned char *zb = R + GR_QZ + hb * 16384;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 16 * tq + 4 * tl + i;
                const uint4 zz = *reinterpret_cast<const uint4 *>(zb + (64 + t) * 128 + ((cg ^ (t & 7)) << 4));
                const uint32_t zw[4] = {zz.x, zz.y, zz.z, zz.w};
                const bool live = t < len;  // tokens past the end of the sequence: g = 0 (an exact no-op)
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float g0 = __fdividef(gm, 1.0f + ex2_approx(fmaf(bf_lo(zw[e]), cz, cb[2 * e])));
                    const float g1 = __fdividef(gm, 1.0f + ex2_approx(fmaf(bf_hi(zw[e]), cz, cb[2 * e + 1])));
                    G[i][2 * e] = live ? g0 : 0.f;
                    G[i][2 * e + 1] = live ? g1 : 0.f;
                }
            }
#pragma unroll
            for (int i = 1; i < 4; ++i)
#pragma unroll
                for (int e = 0; e < 8; ++e) G[i][e] += G[i - 1][e];
#pragma unroll
            for (int e = 0; e < 8; ++e) {  // inclusive scan of the thread sums over tl (lanes 8 apart)
                float x = G[3][e];
#pragma unroll
                for (int off = 8; off < 32; off <<= 1) {
                    const float y = __shfl_up_sync(0xffffffffu, x, off);
                    if (lane >= off) x += y;
                }
                const float base = x - G[3][e];
#pragma unroll
                for (int i = 0; i < 4; ++i) G[i][e] += base;
            }
            if (tl == 3) {  // the quarter's sums
                float *tot = (float *)(R + GR_TOT) + 128 * tq + c0;
                *reinterpret_cast<float4 *>(tot) = make_float4(G[3][0], G[3][1], G[3][2], G[3][3]);
                *reinterpret_cast<float4 *>(tot + 4) = make_float4(G[3][4], G[3][5], G[3][6], G[3][7]);
            }
        }
        if (gt < 64) {  // beta of token gt: the bf16 half of its word (0 past the end), widened in place
            uint32_t *bw = (uint32_t *)(R + GR_BETA) + 64 * s;
            const uint32_t x = bw[gt];
            const uintptr_t ad = (uintptr_t)(beta + (info[0] + gt) * H + info[2]);
            reinterpret_cast<float *>(bw)[gt] = __uint_as_float((ad & 2) ? (x & 0xffff0000u) : (x << 16));
        }
        ok = gsync_and(g, true);  // quarter sums written; z read by every thread (its rows are rewritten below)
        float Gr[8], G47[8], eGr[8], f63[8];  // (base 2) reference G (p0 or p1), G_47; e^{G_ref}, e^{G_63 - G_47}
        {
            const float *tot = (const float *)(R + GR_TOT);
            float q4[4][8];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const float4 a4 = *reinterpret_cast<const float4 *>(tot + 128 * u + c0);
                const float4 b4 = *reinterpret_cast<const float4 *>(tot + 128 * u + c0 + 4);
                q4[u][0] = a4.x; q4[u][1] = a4.y; q4[u][2] = a4.z; q4[u][3] = a4.w;
                q4[u][4] = b4.x; q4[u][5] = b4.y; q4[u][6] = b4.z; q4[u][7] = b4.w;
            }
            float g63[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                float base = 0.f;
#pragma unroll
                for (int u = 0; u < 3; ++u)
                    if (u < tq) base += q4[u][e];
#pragma unroll
                for (int i = 0; i < 4; ++i) G[i][e] += base;
                G47[e] = q4[0][e] + q4[1][e] + q4[2][e];
                g63[e] = G47[e] + q4[3][e];
                Gr[e] = tq < 2 ? q4[0][e] : G47[e];
                eGr[e] = ex2_approx(Gr[e]);
                f63[e] = ex2_approx(g63[e] - G47[e]);
            }
            if (tq == 3 && tl == 3) {
                float *gam = (float *)(R + GR_GAM) + c0;
                *reinterpret_cast<float4 *>(gam) =
                    make_float4(ex2_approx(g63[0]), ex2_approx(g63[1]), ex2_approx(g63[2]), ex2_approx(g63[3]));
                *reinterpret_cast<float4 *>(gam + 4) =
                    make_float4(ex2_approx(g63[4]), ex2_approx(g63[5]), ex2_approx(g63[6]), ex2_approx(g63[7]));
            }
        }
        // ---- ELEM: per token t and channel: E = e^{G_t - G_ref}, f1 = e^{G_47 - G_t} (keys against the
        //      second reference), k0 = e^{G_15 - G_t} (first half only); 16-byte rows of 8 channels
        {
            unsigned char *qz = R + GR_QZ + hb * 16384;
            unsigned char *kb = R + GR_K + hb * 8192;
            unsigned char *k0b = R + GR_K0 + hb * 4096;
            unsigned char *xb = R + GR_X + hb * 8192;
            unsigned char *qhat = pk + PK_WQ + hb * 16384;
            unsigned char *ktil = pk + PK_K + hb * 8192;
            // two passes over the thread's tokens (fewer values live at once): the outputs scaled by E, then
            // those scaled by f1 (k is read again)
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 16 * tq + 4 * tl + i;
                const uint32_t o = (uint32_t)(t * 128 + ((cg ^ (t & 7)) << 4));
                const uint4 qq = *reinterpret_cast<const uint4 *>(qz + o);
                const uint4 kk = *reinterpret_cast<const uint4 *>(kb + o);
                const uint32_t qw[4] = {qq.x, qq.y, qq.z, qq.w}, kw[4] = {kk.x, kk.y, kk.z, kk.w};
                uint32_t rq[4], rk[4], qh[4], xk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 qf = make_float2(bf_lo(qw[e]), bf_hi(qw[e]));
                    const float2 kf = make_float2(bf_lo(kw[e]), bf_hi(kw[e]));
                    const float2 dd = fsub2(make_float2(G[i][2 * e], G[i][2 * e + 1]), make_float2(Gr[2 * e], Gr[2 * e + 1]));
                    const float2 E = make_float2(ex2_approx(dd.x), ex2_approx(dd.y));  // e^{G_t - G_ref}
                    const float2 eg = fmul2(E, make_float2(eGr[2 * e], eGr[2 * e + 1]));  // e^{G_t}
                    rq[e] = pack2(fmul2(qf, E));
                    rk[e] = pack2(fmul2(kf, E));
                    qh[e] = pack2(fmul2(qf, eg));
                    xk[e] = pack2(fmul2(kf, eg));
                }
                *reinterpret_cast<uint4 *>(qz + o) = make_uint4(rq[0], rq[1], rq[2], rq[3]);
                *reinterpret_cast<uint4 *>(qz + 64 * 128 + o) = make_uint4(rk[0], rk[1], rk[2], rk[3]);
                *reinterpret_cast<uint4 *>(xb + o) = make_uint4(xk[0], xk[1], xk[2], xk[3]);
                *reinterpret_cast<uint4 *>(qhat + 64 * 128 + o) = make_uint4(qh[0], qh[1], qh[2], qh[3]);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int t = 16 * tq + 4 * tl + i;
                const uint32_t o = (uint32_t)(t * 128 + ((cg ^ (t & 7)) << 4));
                const uint4 kk = *reinterpret_cast<const uint4 *>(kb + o);
                const uint32_t kw[4] = {kk.x, kk.y, kk.z, kk.w};
                uint32_t k1[4], k0[4], kt[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 kf = make_float2(bf_lo(kw[e]), bf_hi(kw[e]));
                    const float2 gt2 = make_float2(G[i][2 * e], G[i][2 * e + 1]);
                    const float2 fa = fsub2(make_float2(G47[2 * e], G47[2 * e + 1]), gt2);
                    const float2 f1 = make_float2(ex2_approx(fa.x), ex2_approx(fa.y));  // e^{G_47 - G_t}
                    const float2 kf1 = fmul2(kf, f1);
                    k1[e] = pack2(kf1);
                    kt[e] = pack2(fmul2(kf1, make_float2(f63[2 * e], f63[2 * e + 1])));  // e^{G_63 - G_t}
                    if (tq < 2) {  // e^{G_15 - G_t}
                        const float2 dn = fsub2(make_float2(Gr[2 * e], Gr[2 * e + 1]), gt2);
                        k0[e] = pack2(fmul2(kf, make_float2(ex2_approx(dn.x), ex2_approx(dn.y))));
                    }
                }
                *reinterpret_cast<uint4 *>(kb + o) = make_uint4(k1[0], k1[1], k1[2], k1[3]);
                if (tq < 2) *reinterpret_cast<uint4 *>(k0b + o) = make_uint4(k0[0], k0[1], k0[2], k0[3]);
                *reinterpret_cast<uint4 *>(ktil + o) = make_uint4(kt[0], kt[1], kt[2], kt[3]);
            }
        }
        fence_proxy_async();
        gsync(g);
        if (gt == 0) {
            // rows over keys 0-31 scaled to p0 (N = 32), then over keys 0-63 scaled to p1 (N = 64)
            mma_bf16_k(tbg + TM_DA, smem_u32(R + GR_QZ), 128, smem_u32(R + GR_K0), 32, 8, idesc_bf16(128, 32), false);
            mma_bf16_k(tbg + TM_DA + 32, smem_u32(R + GR_QZ), 128, smem_u32(R + GR_K), 64, 8, idesc_bf16(128, 64),
                       false);
            mma_commit(bar_mma);
            // the other group's turn, while it has an item left that waits for this one: group 1's item j
            // waits for group 0's item j, group 0's item j + 1 for group 1's item j
            if (g == 0 ? has(j, 1) : has(j + 1, 0)) mbar_arrive(&tok[1 - g]);
            if (flags && !team && j > 0) publish(w_prev);  // while the product runs
        }
        ok = mwait();
        if (!ok) break;
        fence_after_sync();
        // ---- A rows -> A image (causal, diagonal kept); L rows -> fp32 (strictly lower, times beta).
        //      Rows of the first half take keys 0-31 from columns 0-31, rows of the second half keys
        //      0-63 from columns 32-95; the two warps of a TMEM lane quarter split the columns.
        float *Lm = (float *)(R + GR_L);
        float *Tm = (float *)(R + GR_T);
        {
            const int lq = gw & 3, cp = gw >> 2;
            const int r = (32 * lq + lane) & 63;  // token row
            if ((lq & 1) == 0) {                  // rows of the first half: columns [16 cp, 16 cp + 16)
                float d[16];
                tmem_ld16(tmem_addr(tbg + TM_DA, 32 * lq, 16 * cp), d);
                if (lq == 0) {
#pragma unroll
                    for (int jj = 0; jj < 2; ++jj) {
                        const int cj = 2 * cp + jj;
                        float o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = (8 * cj + e <= r) ? d[8 * jj + e] : 0.f;
                        *reinterpret_cast<uint4 *>(R + GR_A + img_chunk_off(64, r, cj)) = pack8(o);
                        *reinterpret_cast<uint4 *>(R + GR_A + img_chunk_off(64, r, 4 + cj)) = make_uint4(0, 0, 0, 0);
                    }
                } else {
                    const float br = bet[r];
#pragma unroll
                    for (int e = 0; e < 16; e += 4) {
                        const int i = 16 * cp + e;
                        *reinterpret_cast<float4 *>(&Lm[fimg(r, i)]) =
                            make_float4((i < r) ? br * d[e] : 0.f, (i + 1 < r) ? br * d[e + 1] : 0.f,
                                        (i + 2 < r) ? br * d[e + 2] : 0.f, (i + 3 < r) ? br * d[e + 3] : 0.f);
                    }
                }
            } else {  // rows of the second half: columns 32 + [32 cp, 32 cp + 32) = keys [32 cp, 32 cp + 32)
                float d[32];
                tmem_ld32(tmem_addr(tbg + TM_DA + 32, 32 * lq, 32 * cp), d);
                if (lq == 1) {
#pragma unroll
                    for (int jj = 0; jj < 4; ++jj) {
                        const int cj = 4 * cp + jj;
                        float o[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e) o[e] = (8 * cj + e <= r) ? d[8 * jj + e] : 0.f;
                        *reinterpret_cast<uint4 *>(R + GR_A + img_chunk_off(64, r, cj)) = pack8(o);
                    }
                } else {
                    const float br = bet[r];
#pragma unroll
                    for (int e = 0; e < 32; e += 4) {
                        const int i = 32 * cp + e;
                        *reinterpret_cast<float4 *>(&Lm[fimg(r, i)]) =
                            make_float4((i < r) ? br * d[e] : 0.f, (i + 1 < r) ? br * d[e + 1] : 0.f,
                                        (i + 2 < r) ? br * d[e + 2] : 0.f, (i + 3 < r) ? br * d[e + 3] : 0.f);
                    }
                }
            }
        }
        fence_proxy_async();
        gsync(g);
        if (gt == 0) {  // the A image leaves for the packet
            bulk_s2g(pk + PK_A, R + GR_A, 8192);
            bulk_commit();
        }
        // ---- T = (I + L)^{-1}.  Level 0: the four 16 x 16 diagonal blocks, one column per thread,
        //      by forward substitution; the blocks above the diagonal inside each 32-row half are
        //      zeroed so that the merges below can run full-length dot products.
        if (gt < 64) {
            const int b = gt >> 4, jc = gt & 15, o0 = 16 * b;
            float x[16];
#pragma unroll
            for (int r = 0; r < 16; ++r) x[r] = (r == jc) ? 1.f : 0.f;
#pragma unroll
            for (int i = 0; i < 15; ++i) {
                const float xi = x[i];
#pragma unroll
                for (int r = i + 1; r < 16; ++r) x[r] -= Lm[fimg(o0 + r, o0 + i)] * xi;
            }
#pragma unroll
            for (int r = 0; r < 16; ++r) Tm[fimg(o0 + r, o0 + jc)] = x[r];
            if ((b & 1) == 0) {
#pragma unroll
                for (int r = 0; r < 16; ++r) Tm[fimg(o0 + r, o0 + 16 + jc)] = 0.f;
            }
            if (b < 2) {  // T_11 = T[0:32][0:32] also transposed (the B operand of the level-2 merge)
                float *Tt = (float *)(R + GR_TT);
#pragma unroll
                for (int r = 0; r < 16; r += 4) {
                    *reinterpret_cast<float4 *>(Tt + fimg(o0 + jc, o0 + r)) = make_float4(x[r], x[r + 1], x[r + 2], x[r + 3]);
                    if (b == 0) *reinterpret_cast<float4 *>(Tt + fimg(16 + jc, r)) = make_float4(0.f, 0.f, 0.f, 0.f);
                }
            }
        }
        gsync(g);
        // Level 1: T_10 = -T_11 L_10 T_00 inside each 32-row half.  Thread = (half mg, column jc,
        // rows q + 4 a); the four threads of a column share their partial products by shuffles.
        if (gt < 128) {
            const int mg = gt >> 6, q = lane & 3;
            const int jc = ((gt >> 5) & 1) * 8 + (lane >> 2);
            const int ro = 32 * mg + 16, co = 32 * mg;
            float p[4];
            if (gw & 1) inv_l1_partial<8>(Lm, Tm, ro, co, q, jc, p);
            else inv_l1_partial<0>(Lm, Tm, ro, co, q, jc, p);
            float pc[16];  // P[:, jc], row q2 + 4 a from lane q2
#pragma unroll
            for (int q2 = 0; q2 < 4; ++q2)
#pragma unroll
                for (int a = 0; a < 4; ++a) pc[q2 + 4 * a] = __shfl_sync(0xffffffffu, p[a], (lane & ~3) | q2);
#pragma unroll
            for (int a = 0; a < 4; ++a) {
                float acc = 0.f;
#pragma unroll
                for (int k = 0; k < 4 * (a + 1); k += 4) {
                    const float4 t4 = *reinterpret_cast<const float4 *>(Tm + fimg(ro + q + 4 * a, ro + k));
                    acc += t4.x * pc[k] + t4.y * pc[k + 1] + t4.z * pc[k + 2] + t4.w * pc[k + 3];
                }
                Tm[fimg(ro + q + 4 * a, co + jc)] = -acc;
                if (mg == 0) reinterpret_cast<float *>(R + GR_TT)[fimg(co + jc, ro + q + 4 * a)] = -acc;
            }
        }
        // Level 2: T_[23][01] = -T_[23][23] (L_[23][01] T_[01][01]) on 32 x 32 blocks, as two tf32
        // products on the tensor cores (M = 128, the 32 rows of interest in TMEM lanes 32-63; the other
        // lanes hold products of rows that are not needed), both operands K-major.  P = L_[23][01] T_[01][01]:
        // A = L's first column block read as 128 rows (L rows 32-63 are rows 32-63), B = T_[01][01]^T.
        // Then T_[23][23] P: A = T's second column block read as 128 rows, B = P^T.
        // Meanwhile the T image is written where it does not depend on this merge.
        fence_proxy_async();
        gsync(g);
        if (gt == 0) {
            mma_tf32_k32(tbg + 0, smem_u32(R + GR_L), smem_u32(R + GR_TT), idesc_tf32(128, 32), false);
            mma_commit(bar_mma);
        }
        // (T diag beta) image into the dead key-0 image, rows 0-31 and the columns 32-63 of rows 32-63:
        // item e -> (row r, 8-key chunk jj); entries above the diagonal are zero
        for (int e = gt; e < 384; e += NCG) {
            const int r = e < 256 ? (e >> 3) : 32 + ((e - 256) >> 2);
            const int jj = e < 256 ? (e & 7) : 4 + ((e - 256) & 3);
            const float4 t0v = *reinterpret_cast<const float4 *>(Tm + fimg(r, 8 * jj));
            const float4 t1v = *reinterpret_cast<const float4 *>(Tm + fimg(r, 8 * jj + 4));
            const float tv[8] = {t0v.x, t0v.y, t0v.z, t0v.w, t1v.x, t1v.y, t1v.z, t1v.w};
            float o[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) o[q] = (8 * jj + q <= r) ? tv[q] * bet[8 * jj + q] : 0.f;
            *reinterpret_cast<uint4 *>(R + GR_K0 + img_chunk_off(64, r, jj)) = pack8(o);
        }
        ok = mwait();
        if (!ok) break;
        fence_after_sync();
        const bool mid = (gw & 3) == 1;  // the warps of TMEM lanes 32-63 (rows 32-63), 16 columns each
        const int c16 = 16 * (gw >> 2);
        if (mid) {  // P row `lane` (TMEM lane 32 + lane), columns c16 .. c16 + 15 -> column `lane` of P^T
            float d[16];
            tmem_ld16(tmem_addr(tbg + c16, 32, 0), d);
            float *Pt = (float *)(R + GR_P);
#pragma unroll
            for (int e = 0; e < 16; ++e) Pt[fimg(c16 + e, lane)] = d[e];
        }
        fence_proxy_async();
        gsync(g);
        if (gt == 0) {
            mma_tf32_k32(tbg + 32, smem_u32(R + GR_T + 8192), smem_u32(R + GR_P), idesc_tf32(128, 32), false);
            mma_commit(bar_mma);
        }
        ok = mwait();
        if (!ok) break;
        fence_after_sync();
        if (mid) {  // T_[23][01] = -(T_[23][23] P): row 32 + lane, keys c16 .. c16 + 15, times beta, into the T image
            float d[16];
            tmem_ld16(tmem_addr(tbg + 32 + c16, 32, 0), d);
            const int r = 32 + lane;
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                float o[8];
#pragma unroll
                for (int q = 0; q < 8; ++q) o[q] = -d[8 * h2 + q] * bet[c16 + 8 * h2 + q];
                *reinterpret_cast<uint4 *>(R + GR_K0 + img_chunk_off(64, r, (c16 >> 3) + h2)) = pack8(o);
            }
        } else if (gw == 0 && has(j + 1, g)) {
            fill_slot(j + 1);  // while warps 1 and 5 read the merge out
        }
        fence_proxy_async();
        gsync(g);
        bool okm = true;
        if (gt == 0) {
            okm = mbar_wait(ld_v, par);
            if (okm) {
                // W = (T diag beta) X: A = the T image read as 128 rows (rows 64-127 are the A image behind it
                // and land in unused TMEM lanes), B = X (MN-major).  U^T = V^T (T diag beta)^T: A = V (MN-major,
                // M = d_v), B = the T image (K-major, 64 rows).
                mma_bf16_kmn(tbg + TM_DW, smem_u32(R + GR_K0), 128, smem_u32(R + GR_X), 8192, 4,
                             idesc_bf16(128, 128, false, true), false);
                mma_bf16_mnk(tbg + TM_DUT, smem_u32(R + GR_V), 8192, smem_u32(R + GR_K0), 64, 4,
                             idesc_bf16(128, 64, true, false), false);
                mma_commit(bar_mma);
            }
        }
        // L and T are dead: while the products run, the next item's q, z and k tiles come in
        if (gt == 0 && has(j + 1, g) && okm) issue_tma(j + 1, false);
        ok = gsync_and(g, ok && okm);
        if (!ok) break;
        ok = mwait();
        if (!ok) break;
        fence_after_sync();
        // ---- W rows (token-major, TMEM lanes 0-63) into the dead X tile, U^T rows (value channels, all
        //      lanes) into the dead V tile
        if ((gw & 3) < 2) {
            const int r = 32 * (gw & 3) + lane, cq = gw >> 2;  // columns [64 cq, 64 cq + 64)
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                float d[32];
                tmem_ld32(tmem_addr(tbg + TM_DW, 32 * (gw & 3), 64 * cq + 32 * h2), d);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj)
                    *reinterpret_cast<uint4 *>(R + GR_X + img_chunk_off(64, r, 8 * cq + 4 * h2 + jj)) = pack8(d + 8 * jj);
            }
        }
        {
            const int vr = 32 * (gw & 3) + lane, tq2 = gw >> 2;  // tokens [32 tq2, 32 tq2 + 32)
            float d[32];
            tmem_ld32(tmem_addr(tbg + TM_DUT, 32 * (gw & 3), 32 * tq2), d);
#pragma unroll
            for (int jj = 0; jj < 4; ++jj)
                *reinterpret_cast<uint4 *>(R + GR_V + img_chunk_off(128, vr, 4 * tq2 + jj)) = pack8(d + 8 * jj);
        }
        // Q^ and K~ went to the packet by plain stores: the group barriers order them before thread 0's flag
        // store (release, GPU scope), which publishes them with the rest of the packet
        fence_proxy_async();
        gsync(g);
        if (gt == 0) {  // the rest of the packet: W rows of the [W; Q^] image, U^T, gamma
            bulk_s2g(pk + PK_WQ, R + GR_X, 8192);
            bulk_s2g(pk + PK_WQ + 16384, R + GR_X + 8192, 8192);
            bulk_s2g(pk + PK_U, R + GR_V, 16384);
            bulk_s2g(pk + PK_G, R + GR_GAM, 512);
            bulk_commit();
        }
        w_prev = w;
    }
    if (gt == 0) {
        if (ok && w_prev >= 0) publish(w_prev);
        if (!ok) set_error(err, KDA_ERR_DEVICE_TIMEOUT);
        bulk_wait0();
    }
    __syncthreads();
    if (tid < 2) {  // the group regions are reused as plain memory after this role
        uint64_t *b = (uint64_t *)(sm + tid * GR_BYTES + GR_BAR);
        for (int i = 0; i < 3; ++i) mbar_inval(&b[i]);
        mbar_inval((uint64_t *)(sm + J_TOK) + tid);
    }
    if (warp == 0) tmem_dealloc(tb, 512);
    __syncthreads();
}

__global__ void __launch_bounds__(NT2, 1)
chunk_intra_tc_kernel(const __grid_constant__ TileMaps tm, const bf16 *__restrict__ beta,
                      const float *__restrict__ bias, const float *__restrict__ A_log, float g_min,
                      int64_t T, int N, const int32_t *__restrict__ cu,
                      const int32_t *__restrict__ chunk_start, int H, unsigned char *__restrict__ packets,
                      int *err, uint64_t *ctr, uint64_t epoch) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = align1024(smem_raw);
    const int32_t *cs = chunk_start, *cu_l = cu;
    if (N <= J_TBL_N) {  // the chunk layout in shared memory: items are located without global loads
        int32_t *a = (int32_t *)(sm + J_CS), *c = (int32_t *)(sm + J_CU);
        for (int n = threadIdx.x; n <= N; n += blockDim.x) {
            a[n] = chunk_start[n];
            if (cu) c[n] = cu[n];
        }
        __syncthreads();
        cs = a;
        if (cu) cu_l = c;
    }
    intra_role(sm, tm, beta, bias, A_log, g_min, T, N, cu_l, cs, H, packets, err, (int)blockIdx.x, (int)gridDim.x,
               nullptr, epoch, 0, -1, 0, nullptr, ctr);
}

constexpr int NT3 = 512;  // warps 0-7: recurrence; 8: MMA issue; 9: packet loads; 12-15: output; 10, 11 idle
// The state is kept transposed: S^T [d_v lanes x d_k columns] fp32 in tensor memory.  Its bf16 copy
// and V~^T (bf16 pairs per 32-bit column) are the A operands of the MMAs, read from tensor memory, so
// that the recurrence moves no operand through shared memory.  Per chunk k (one thread of warp 8
// issues every MMA, in order; D is one of two 128-column buffers):
//   MMA1   D = S^T [W; Q^]^T           D[:, 0:64] = (W S)^T, D[:, 64:128] = (Q^ S)^T
//   V~     V~^T = U^T - D[:, 0:64] (U^T from the packet) as bf16 pairs into tensor memory
//   MMA3   S^T += V~^T K~              the decay Diag(gamma) was applied to S^T by the CUDA cores
//   S      bf16 copy of S_{k+1}^T, then S^T scaled by gamma_{k+1} (per column)
//   MMA2   D[:, 64:128] += V~^T A^T    O^T = (Q^ S + A V~)^T, issued after MMA1 of chunk k + 1 so that
//                                      the in-order tensor pipe runs it during the next V~ phase (its
//                                      completion frees the packet stage for the loader, two chunks ahead)
// The output warps read O^T of chunk k once its MMAs are done, release the D buffer, and store o
// through a staging tile and TMA.
// Tensor memory columns: S^T fp32 [0, 128), D buffers [128, 384), bf16 S^T [384, 448), bf16 V~^T
// buffers [448, 512).
constexpr uint32_t TM_S = 0, TM_D0 = 128, TM_SB = 384, TM_VT = 448;

// The output pass of segment g, head h in one CTA (threads 0-511).  With `flags`, a packet is loaded
// only after its producer has published it.
__device__ __forceinline__ void chain_role(unsigned char *sm, const CUtensorMap &omap, int64_t T, int N,
                                           const int32_t *__restrict__ cu, const int32_t *__restrict__ chunk_start,
                                           const int32_t *__restrict__ seg_start, int64_t seg_len,
                                           const float *__restrict__ seg_in, int H,
                                           const unsigned char *__restrict__ packets, float scale,
                                           const float *initial_state, float *final_state, bf16 *__restrict__ o,
                                           int *err, int g, int h, const uint64_t *flags, uint64_t epoch,
                                           uint64_t *consumed = nullptr, bool relinquish = true,
                                           const CUtensorMap *gmap = nullptr, const float *epi_w = nullptr,
                                           float epi_eps = 0.f) {
    // segment g of sequence n, head h: chunks [kk0, kk0 + nc) of the sequence (without seg_start, one
    // segment per sequence: g = n)
    if (seg_start ? g >= seg_start[N] : g >= N) return;
    int n = g;
    if (seg_start) {
        int lo = 0, hi = N;  // largest n with seg_start[n] <= g
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (seg_start[mid] <= g) lo = mid; else hi = mid;
        }
        n = lo;
    }
    const int seg_i = seg_start ? g - seg_start[n] : 0, nseg = seg_start ? seg_start[n + 1] - seg_start[n] : 1;
    const bool last_seg = (seg_i == nseg - 1);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = warp & 3;           // TMEM lane quarter
    const int v = 32 * lq + lane;      // TMEM lane: d_v channel
    uint64_t *bar_ld1 = (uint64_t *)(sm + CS_BAR);  // [2] part 1 of a packet stage loaded
    uint64_t *bar_ld2 = bar_ld1 + 2;                // [2] part 2 loaded
    uint64_t *bar_o = bar_ld1 + 4;                  // [2] all MMAs of a chunk done
    uint64_t *bar_free = bar_ld1 + 6;               // [2] O^T of a D buffer read by the output warps
    uint64_t *bar_v = bar_ld1 + 8;                  // MMA1 done
    uint64_t *bar_s = bar_ld1 + 9;                  // MMA3 done
    uint64_t *bar_sb = bar_ld1 + 10;                // bf16 S^T written (one arrival per recurrence warp)
    uint64_t *bar_vt = bar_ld1 + 11;                // [2] V~^T of chunk kk written (one arrival per
                                                    // recurrence warp); double-buffered so that the
                                                    // loader, which also waits on it, can never see a
                                                    // phase two ahead
    uint64_t *bar_g = bar_ld1 + 13;                 // [2] output epilogue: gate tile of chunk kk loaded
    uint32_t *tslot = (uint32_t *)(sm + CS_TSLOT);
    int *s_fail = (int *)(sm + CS_TSLOT + 8);
    const int64_t kk0 = (int64_t)seg_i * seg_len;
    const int nc_seq = chunk_start[n + 1] - chunk_start[n];
    const int c_begin = chunk_start[n] + (int)kk0;
    const int nc = (int)max((int64_t)0, min(seg_len, (int64_t)nc_seq - kk0));
    const int64_t s_tok = (cu ? (int64_t)cu[n] : (T / N) * n) + kk0 * C;
    const int64_t e_tok = cu ? (int64_t)cu[n + 1] : (T / N) * (n + 1);
    const size_t st_off = ((size_t)n * H + h) * D * D;
    // entering state: the sequence's initial state for a lone segment; otherwise the fold's output
    // (segment 0 included, lane-major, see ll_off), so that final_state may alias initial_state
    const bool s_in_ll = (nseg > 1);
    const float *s_in = s_in_ll ? seg_in + ((size_t)g * H + h) * D * D
                                : (initial_state ? initial_state + st_off : nullptr);

    if (tid == 0) {
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_ld1[i], 1);
            mbar_init(&bar_ld2[i], 1);
            mbar_init(&bar_o[i], 1);
            mbar_init(&bar_free[i], 128);
        }
        mbar_init(bar_v, 1);
        mbar_init(bar_s, 1);
        mbar_init(bar_sb, 8);
        mbar_init(&bar_vt[0], 8);
        mbar_init(&bar_vt[1], 8);
        mbar_init(&bar_g[0], 1);
        mbar_init(&bar_g[1], 1);
        *s_fail = 0;
    }
    // a CTA that runs several chains keeps its right to allocate tensor memory
    if (warp == 0) tmem_alloc(tslot, 512, relinquish);
    fence_proxy_async();  // barrier init visible to the async proxy
    sync_all();
    const uint32_t tb = *tslot;
    auto tDbuf = [&](int kk) { return tb + TM_D0 + 128 * (uint32_t)(kk & 1); };
    auto packet = [&](int kk) { return packets + ((size_t)(c_begin + kk) * H + h) * PK_STRIDE; };
    auto stage = [&](int kk) { return sm + (kk & 1) * CS_ST_BYTES; };
    auto acquire = [&](int kk) {  // the packet of chunk kk is published (false: it never was)
        if (flags) {
            const size_t item = (size_t)(c_begin + kk) * H + h;
            if (!flag_wait(flags + item, epoch)) return false;
            fence_proxy_async_global();
            // its producer may now run further ahead (the mark only paces production; packets are never
            // reused within a launch)
            if (consumed) asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(consumed + item), "l"(epoch) : "memory");
        }
        return true;
    };
    auto load_part1 = [&](int kk) {
        uint64_t *b = &bar_ld1[kk & 1];
        mbar_arrive_expect_tx(b, PK_P1);
        bulk_g2s(stage(kk), packet(kk), PK_P1, b);
    };
    auto load_part2 = [&](int kk) {
        uint64_t *b = &bar_ld2[kk & 1];
        mbar_arrive_expect_tx(b, PK_P2);
        bulk_g2s(stage(kk) + PK_K, packet(kk) + PK_K, PK_P2, b);
    };

    if (warp == 8) {
        // ------------------------------------------------ MMA issue (one thread)
        if (lane == 0) {
            const uint32_t id1 = idesc_bf16(128, 128, false, false);  // A = bf16 S^T, B = [W; Q^] (K-major)
            const uint32_t id3 = idesc_bf16(128, 128, false, true);   // A = V~^T, B = K~ (MN-major)
            const uint32_t id2 = idesc_bf16(128, 64, false, false);   // A = V~^T, B = A (K-major)
            bool ok = true;
            auto mma2 = [&](int kk) {  // O^T of chunk kk += V~^T A^T
                mma_ts_k(tDbuf(kk) + 64, tb + TM_VT + 32 * (kk & 1), smem_u32(stage(kk) + PK_A), 64, 4, id2, true);
                mma_commit(&bar_o[kk & 1]);
            };
            for (int kk = 0; kk < nc && ok; ++kk) {
                unsigned char *P = stage(kk);
                if (kk >= 2) ok = mbar_wait_spin(&bar_free[kk & 1], ((kk >> 1) - 1) & 1);  // O of chunk kk - 2 read
                ok = ok && mbar_wait_spin(&bar_ld1[kk & 1], (kk >> 1) & 1);               // part 1 of packet kk
                ok = ok && mbar_wait_spin(bar_sb, kk & 1);                                  // bf16 S_kk^T written
                if (!ok) break;
                fence_after_sync();
                mma_ts_k(tDbuf(kk), tb + TM_SB, smem_u32(P + PK_WQ), 128, 8, id1, false);
                mma_commit(bar_v);
                if (kk > 0) mma2(kk - 1);
                ok = mbar_wait_spin(&bar_vt[kk & 1], (kk >> 1) & 1);  // V~^T written, S^T scaled by gamma_kk
                ok = ok && mbar_wait_spin(&bar_ld2[kk & 1], (kk >> 1) & 1);  // part 2 of packet kk
                if (!ok) break;
                fence_after_sync();
                mma_ts_mn(tb + TM_S, tb + TM_VT + 32 * (kk & 1), smem_u32(P + PK_K), 8192, 4, id3, true);
                mma_commit(bar_s);
            }
            if (ok && nc > 0) mma2(nc - 1);
            if (!ok) atomicExch(s_fail, 1);
        }
    } else if (warp == 9) {
        // ------------------------------------------------ packet loads (lane 0); once a packet part has
        // been consumed from its stage, the whole warp drops that part's lines from L2 (this role is its
        // last reader: the lines are never read again and need no write-back to DRAM)
        bool ok = true;
        if (lane == 0) {
            for (int kk = 0; kk < 2 && kk < nc && ok; ++kk) {
                ok = acquire(kk);
                if (ok) {
                    load_part1(kk);
                    load_part2(kk);
                }
            }
            if (ok && nc > 2 && !flags) bulk_prefetch_l2(packet(2), PK_STRIDE);
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        for (int kk = 0; kk + 2 < nc && ok; ++kk) {
            if (lane == 0) {
                // MMA_U and MMA1 of chunk kk done and gamma_kk read (V~^T of chunk kk written): part 1 of
                // its stage takes chunk kk + 2
                ok = mbar_wait_spin(&bar_vt[kk & 1], (kk >> 1) & 1) && acquire(kk + 2);
                if (ok) load_part1(kk + 2);
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            for (int l = lane; l < PK_K / 128; l += 32) discard_l2(packet(kk) + l * 128);  // part 1 (+ pad)
            if (lane == 0) {
                ok = mbar_wait_spin(&bar_o[kk & 1], (kk >> 1) & 1);  // all MMAs of chunk kk done: part 2
                if (ok) {
                    load_part2(kk + 2);
                    if (kk + 3 < nc && !flags) bulk_prefetch_l2(packet(kk + 3), PK_STRIDE);
                }
            }
            ok = __shfl_sync(0xffffffffu, ok, 0);
            if (!ok) break;
            for (int l = PK_K / 128 + lane; l < PK_STRIDE / 128; l += 32) discard_l2(packet(kk) + l * 128);
        }
        if (!ok && lane == 0) atomicExch(s_fail, 1);
    } else if (warp >= 12 && warp < 16) {
        // ------------------------------------------------ output warps 12-15 (128 threads, one d_v lane each).
        // With the output epilogue (Eq. 6 without its projections: y = Sigmoid(g) w o~ / sqrt(mean o~^2 + eps)
        // per token over the head's d_v channels), o~ goes through the staging tile as bf16, as it would be
        // stored, and a second pass over the tile (thread = token, 8-channel chunk; the row's 16 chunks
        // in 16 lanes) normalises and gates it before the store; the gate tiles come in by TMA, two chunks
        // ahead.  o~ then never leaves the chip.
        const int ot = tid - 384;
        const bool epi = gmap != nullptr;
        // byte offset of (token t, channel v) in the staging tile (two 64-channel SW128 halves): row part
        const uint32_t vh = (uint32_t)(v >> 6) * 8192 + ((uint32_t)(v & 7) << 1);
        const int vc = (v & 63) >> 3;
        bool ok = true;
        auto load_g = [&](int kk) {  // gate tile of chunk kk (ot == 0)
            unsigned char *gt = sm + CS_GIMG + 16384 * (kk & 1);
            const int64_t tp = s_tok + (int64_t)kk * C;
            mbar_arrive_expect_tx(&bar_g[kk & 1], 16384);
            tma_load_3d(gt, gmap, 0, h, (int)tp, &bar_g[kk & 1]);
            tma_load_3d(gt + 8192, gmap, 64, h, (int)tp, &bar_g[kk & 1]);
        };
        if (epi) {
            float *wv = reinterpret_cast<float *>(sm + CS_W);
            wv[ot] = epi_w ? epi_w[(size_t)h * D + ot] : 1.f;
            if (ot == 0) {
                for (int kk = 0; kk < 2 && kk < nc; ++kk) load_g(kk);
            }
        }
        for (int kk = 0; kk < nc && ok; ++kk) {
            ok = mbar_wait(&bar_o[kk & 1], (kk >> 1) & 1);
            if (!ok) break;
            fence_after_sync();
            uint32_t ob[32];  // O^T[v][2i], O^T[v][2i + 1] as bf16 pairs
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                float d[32];
                tmem_ld32(tDbuf(kk) + ((uint32_t)(32 * lq) << 16) + 64 + 32 * h2, d);
#pragma unroll
                for (int i = 0; i < 16; ++i) ob[16 * h2 + i] = pack_bf16(scale * d[2 * i], scale * d[2 * i + 1]);
            }
            fence_before_sync();
            mbar_arrive(&bar_free[kk & 1]);  // TMEM buffer read
            const int64_t tp = s_tok + (int64_t)kk * C;
            const int lenp = (int)min((int64_t)C, e_tok - tp);
            if (lenp == C || epi) {  // through the staging tile (double-buffered)
                unsigned char *stg = sm + CS_OIMG + 16384 * (kk & 1);
                if (ot == 0 && kk >= 2) {
                    if (lenp == C) bulk_wait_read1();  // the store of chunk kk - 2 has left this buffer
                    else bulk_wait_read0();
                }
                named_sync(2, 128);
#pragma unroll
                for (int t = 0; t < 64; ++t) {
                    const uint32_t w = ob[t >> 1];
                    *reinterpret_cast<uint16_t *>(stg + vh + t * 128 + ((vc ^ (t & 7)) << 4)) =
                        (uint16_t)((t & 1) ? (w >> 16) : (w & 0xFFFFu));
                }
                if (epi) {
                    ok = bar_red_popc(2, 128, mbar_wait(&bar_g[kk & 1], (kk >> 1) & 1)) == 128;
                    const unsigned char *gtile = sm + CS_GIMG + 16384 * (kk & 1);
                    const float *wv = reinterpret_cast<const float *>(sm + CS_W);
                    const int cc = ot & 15;                      // 8-channel chunk of the row
                    const uint32_t half = (uint32_t)(cc >> 3) * 8192;
                    float w8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) w8[e] = wv[8 * cc + e];
#pragma unroll 2
                    for (int i = 0; i < 8; ++i) {
                        const int t = (ot >> 4) + 8 * i;         // the 16 lanes of a row share t
                        const uint32_t off = half + (uint32_t)t * 128 + ((((uint32_t)cc & 7) ^ (uint32_t)(t & 7)) << 4);
                        const uint4 ov = *reinterpret_cast<const uint4 *>(stg + off);
                        const uint4 gv = *reinterpret_cast<const uint4 *>(gtile + off);
                        const uint32_t ow[4] = {ov.x, ov.y, ov.z, ov.w}, gw4[4] = {gv.x, gv.y, gv.z, gv.w};
                        float of[8], gf[8];
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            of[2 * e] = bf_lo(ow[e]);
                            of[2 * e + 1] = bf_hi(ow[e]);
                            gf[2 * e] = bf_lo(gw4[e]);
                            gf[2 * e + 1] = bf_hi(gw4[e]);
                        }
                        float ss = 0.f;
#pragma unroll
                        for (int e = 0; e < 8; ++e) ss = fmaf(of[e], of[e], ss);
#pragma unroll
                        for (int off2 = 8; off2 > 0; off2 >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off2);
                        const float r = rsqrtf(ss * (1.0f / D) + epi_eps);
                        float y[8];
#pragma unroll
                        for (int e = 0; e < 8; ++e)
                            y[e] = __fdividef(of[e] * r * w8[e], 1.0f + __expf(-gf[e]));  // inf gives 0
                        *reinterpret_cast<uint4 *>(stg + off) = pack8(y);
                    }
                    fence_proxy_async();
                    named_sync(2, 128);  // the gate tile has been read: chunk kk + 2 takes its buffer
                    if (ot == 0 && kk + 2 < nc) load_g(kk + 2);
                } else {
                    fence_proxy_async();
                    named_sync(2, 128);
                }
                if (lenp == C) {
                    if (ot == 0) {
                        tma_store_3d(&omap, stg, 0, h, (int)tp);
                        tma_store_3d(&omap, stg + 8192, 64, h, (int)tp);
                        bulk_commit();
                    }
                } else {  // the ragged last chunk of a sequence: rows past its end stay untouched
                    const int cc = ot & 15;
                    const uint32_t half = (uint32_t)(cc >> 3) * 8192;
                    for (int i = 0; i < 8; ++i) {
                        const int t = (ot >> 4) + 8 * i;
                        if (t < lenp)
                            *reinterpret_cast<uint4 *>(o + ((tp + t) * H + h) * D + 8 * cc) = *reinterpret_cast<const uint4 *>(
                                stg + half + (uint32_t)t * 128 + ((((uint32_t)cc & 7) ^ (uint32_t)(t & 7)) << 4));
                    }
                }
            } else {  // the ragged last chunk of a sequence: rows past its end stay untouched
                bf16 *dst = o + (tp * H + h) * D + v;
#pragma unroll
                for (int t = 0; t < 64; ++t) {
                    const uint32_t w = ob[t >> 1];
                    if (t < lenp)
                        *reinterpret_cast<uint16_t *>(dst + (size_t)t * H * D) =
                            (uint16_t)((t & 1) ? (w >> 16) : (w & 0xFFFFu));
                }
            }
        }
        if (ot == 0) bulk_wait0();
        if (!ok) atomicExch(s_fail, 1);
    } else if (warp < 8) {
        // ------------------------------------------------ recurrence warps 0-7: lanes of quarter lq,
        // d_k columns [64 j, 64 j + 64) of S^T and tokens [32 j, 32 j + 32) of V~^T
        const int j = warp >> 2;
        bool ok = true;
        if (nc > 0) ok = mbar_wait_spin(&bar_ld1[0], 0);
        // S_0^T, 32 columns at a time: bf16 copy, and the fp32 state scaled by gamma_0
#pragma unroll 1
        for (int h2 = 0; h2 < 2 && ok; ++h2) {
            const int c0 = 64 * j + 32 * h2;
            float x[32];
#pragma unroll
            for (int e = 0; e < 32; ++e)
                x[e] = s_in ? s_in[s_in_ll ? ll_off(c0 + e, v) : (size_t)(c0 + e) * D + v] : 0.f;
            if (nc == 0) {
                if (final_state && last_seg) {
#pragma unroll
                    for (int e = 0; e < 32; ++e) final_state[st_off + (size_t)(c0 + e) * D + v] = x[e];
                }
                continue;
            }
            uint32_t pk[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(x[2 * i], x[2 * i + 1]);
            tmem_st16u(tmem_addr(tb + TM_SB, 32 * lq, c0 / 2), pk);
            const float *gam = reinterpret_cast<const float *>(stage(0) + PK_G) + c0;
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] *= gam[e];
            tmem_st32(tmem_addr(tb + TM_S, 32 * lq, c0), x);
        }
        tmem_st_wait();
        fence_before_sync();
        __syncwarp();
        if (lane == 0 && nc > 0 && ok) mbar_arrive(bar_sb);
        for (int kk = 0; kk < nc && ok; ++kk) {
            // invariant: part 1 of packet kk resident; bf16 S_kk^T written; TMEM S^T = (Diag(gamma_kk) S_kk)^T
            uint4 ua[4];  // U^T row v, tokens [32 j, 32 j + 32), read before MMA1 is done
            {
                const unsigned char *ut = stage(kk) + PK_U + v * 128;
#pragma unroll
                for (int q = 0; q < 4; ++q) ua[q] = *reinterpret_cast<const uint4 *>(ut + (((4 * j + q) ^ (v & 7)) << 4));
            }
            ok = mbar_wait_spin(bar_v, kk & 1) && (*(volatile int *)s_fail == 0);
            if (!ok) break;
            fence_after_sync();
            {  // V~^T row v, tokens [32 j, 32 j + 32) = U^T - (W S)^T
                float d[32];
                tmem_ld32(tmem_addr(tDbuf(kk), 32 * lq, 32 * j), d);
                uint32_t pk[16];
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    float u[8];
                    unpack8(ua[q], u);
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        pk[4 * q + e] = pack_bf16(u[2 * e] - d[8 * q + 2 * e], u[2 * e + 1] - d[8 * q + 2 * e + 1]);
                }
                tmem_st16u(tmem_addr(tb + TM_VT + 32 * (kk & 1), 32 * lq, 16 * j), pk);
                tmem_st_wait();
            }
            fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bar_vt[kk & 1]);
            const bool last = (kk == nc - 1);
            ok = mbar_wait_spin(bar_s, kk & 1);
            if (!ok) break;
            fence_after_sync();
            if (!last) {
                // bf16 S_{kk+1}^T first (MMA1 of the next chunk waits for it), then the fp32 copy scaled
                // by gamma_{kk+1} from packet kk + 1 (MMA3 of the next chunk, issued after this warp's next
                // V~, needs it)
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int c0 = 64 * j + 32 * h2;
                    float x[32];
                    tmem_ld32(tmem_addr(tb + TM_S, 32 * lq, c0), x);
                    uint32_t pk[16];
#pragma unroll
                    for (int i = 0; i < 16; ++i) pk[i] = pack_bf16(x[2 * i], x[2 * i + 1]);
                    tmem_st16u(tmem_addr(tb + TM_SB, 32 * lq, c0 / 2), pk);
                }
                tmem_st_wait();
                fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(bar_sb);
                ok = mbar_wait_spin(&bar_ld1[(kk + 1) & 1], ((kk + 1) >> 1) & 1);
                if (!ok) break;
                const float *gam = reinterpret_cast<const float *>(stage(kk + 1) + PK_G);
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int c0 = 64 * j + 32 * h2;
                    float x[32];
                    tmem_ld32(tmem_addr(tb + TM_S, 32 * lq, c0), x);
#pragma unroll
                    for (int e = 0; e < 32; ++e) x[e] *= gam[c0 + e];
                    tmem_st32(tmem_addr(tb + TM_S, 32 * lq, c0), x);
                }
                tmem_st_wait();
            } else if (final_state && last_seg) {
#pragma unroll
                for (int h2 = 0; h2 < 2; ++h2) {
                    const int c0 = 64 * j + 32 * h2;
                    float x[32];
                    tmem_ld32(tmem_addr(tb + TM_S, 32 * lq, c0), x);
#pragma unroll
                    for (int e = 0; e < 32; ++e) final_state[st_off + (size_t)(c0 + e) * D + v] = x[e];
                }
            }
        }
        if (!ok) atomicExch(s_fail, 1);
    }
    __syncthreads();
    if (tid == 0 && *(volatile int *)s_fail) set_error(err, KDA_ERR_DEVICE_TIMEOUT);
    sync_all();
    if (tid == 0) {  // the CTA may run another chain over the same shared memory
        for (int i = 0; i < 15; ++i) mbar_inval(bar_ld1 + i);
    }
    if (warp == 0) tmem_dealloc(tb, 512);
    __syncthreads();
}

__global__ void __launch_bounds__(NT3, 1)
chunk_inter_tc_kernel(const __grid_constant__ CUtensorMap omap, int64_t T, int N, const int32_t *__restrict__ cu,
                      const int32_t *__restrict__ chunk_start, const int32_t *__restrict__ seg_start,
                      int64_t seg_len, const float *__restrict__ seg_in, int H,
                      const unsigned char *__restrict__ packets, float scale, const float *initial_state,
                      float *final_state, bf16 *__restrict__ o, int *err, const __grid_constant__ CUtensorMap gmap,
                      int epi, const float *epi_w, float epi_eps, const int32_t *__restrict__ unit_seg,
                      int *unit_ctr) {
    // persistent: each CTA takes (segment, head) units from the counter, segments longest first
    // (unit u = segment unit_seg[u / H], head u % H), and keeps its right to allocate tensor memory
    extern __shared__ unsigned char smem_raw[];
    __shared__ int s_u;
    const int64_t n_units = (int64_t)seg_start[N] * H;
    for (;;) {
        if (threadIdx.x == 0) s_u = atomicAdd(unit_ctr, 1);
        __syncthreads();
        const int64_t u = s_u;
        __syncthreads();  // read before thread 0 takes the next unit
        if (u >= n_units) break;
        chain_role(align1024(smem_raw), omap, T, N, cu, chunk_start, seg_start, seg_len, seg_in, H, packets, scale,
                   initial_state, final_state, o, err, unit_seg[u / H], (int)(u % H), nullptr, 0, nullptr, false,
                   epi ? &gmap : nullptr, epi_w, epi_eps);
        if (*(volatile int *)err == KDA_ERR_DEVICE_TIMEOUT) break;  // a wait gave up: stop taking work
    }
}

// =====================================================================================
// Intra-chunk work and the output pass in one launch, for inputs whose chains (one per sequence and
// head) are few: CTAs [0, n_chain) run the chains (no segment split), each first producing the first
// kpre chunks of its own sequence and head; the others produce the remaining packets in chunk order
// and publish them through `flags`; a chain waits for each packet before loading it.  Every CTA
// derives the chunk layout from cu_seqlens itself (at most KDA_FUSED_MAX_SEQS sequences), so the launch
// needs no planning kernel.  Launched cooperatively, so every CTA is resident and the producers always
// make progress; every wait is bounded.
__global__ void __launch_bounds__(NT2, 1)
chunk_fused_tc_kernel(const __grid_constant__ TileMaps tm, const __grid_constant__ CUtensorMap omap,
                      const bf16 *__restrict__ beta, const float *__restrict__ bias, const float *__restrict__ A_log,
                      float g_min, int64_t T, int N, const int32_t *__restrict__ cu, int H,
                      unsigned char *__restrict__ packets, float scale, const float *initial_state,
                      float *final_state, bf16 *__restrict__ o, int *err, int n_chain, uint64_t *flags,
                      uint64_t epoch, int kpre, const __grid_constant__ CUtensorMap gmap, int epi,
                      const float *epi_w, float epi_eps, uint64_t *ctr) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = align1024(smem_raw);
    const int b = (int)blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *cs = (int32_t *)(sm + J_CS);  // chunk_start [N + 1]
    int32_t *ss = (int32_t *)(sm + J_SS);  // seg_start [N + 1]: one segment per sequence
    int32_t *cus = (int32_t *)(sm + J_CU);  // cu_seqlens [N + 1]
    const int32_t *cu_l = cu ? cus : nullptr;
    int *s_bad = (int *)(sm + J_SS + 4 * (J_TBL_N + 1));
    if (warp == 0) {  // validate cu_seqlens (0 = c_0 <= ... <= c_N = T) and count chunks per sequence
        bool bad = false;
        if (cu) {
            for (int n = lane; n <= N; n += 32) {
                const int64_t x = cu[n];
                cus[n] = (int32_t)x;
                bad = bad || (n == 0 && x != 0) || (n == N && x != T) || (n > 0 && x < (int64_t)cu[n - 1]);
            }
        }
        bad = __any_sync(0xffffffffu, bad);
        int carry = 0;
        for (int base = 0; base < N; base += 32) {
            const int m = base + lane;
            int x = 0;
            if (m < N && !bad) {
                const int64_t len = cu ? (int64_t)cu[m + 1] - cu[m] : T / N;
                x = (int)((len + C - 1) / C);
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            if (m < N) cs[m + 1] = carry + x;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        for (int n = lane; n <= N; n += 32) ss[n] = n;
        if (lane == 0) {
            cs[0] = 0;
            *s_bad = bad ? 1 : 0;
        }
    }
    __syncthreads();
    if (*(volatile int *)s_bad) {
        if (b == 0 && tid == 0) set_error(err, KDA_ERR_BAD_SEQLENS);
        return;
    }
    if (b < n_chain) {
        if (kpre > 0) {
            intra_role(sm, tm, beta, bias, A_log, g_min, T, N, cu_l, cs, H, packets, err, 0, 1, flags, epoch, kpre,
                       b / H, b % H);
            __syncthreads();
        }
        chain_role(sm, omap, T, N, cu, cs, ss, (int64_t)1 << 30, nullptr, H, packets, scale, initial_state,
                   final_state, o, err, b / H, b % H, flags, epoch, nullptr, true, epi ? &gmap : nullptr, epi_w,
                   epi_eps);
    } else {
        intra_role(sm, tm, beta, bias, A_log, g_min, T, N, cu_l, cs, H, packets, err, b - n_chain,
                   (int)gridDim.x - n_chain, flags, epoch, kpre, -1, 0, nullptr, ctr);
    }
}

// =====================================================================================
// Intra-chunk work and the output pass in one launch, for inputs with many chains: the grid is cut into
// `teams` teams of one chain CTA and K producer CTAs.  The chains (one per sequence and head) are dealt
// to the teams longest first, in snake order (team 0, 1, ..., T - 1, T - 1, ..., 0, ...), which balances
// their lengths; a team's chain CTA runs its chains one after another, and its producers produce their
// chunks in that order, at most `window` of their own items ahead of the chain.  Packets are published
// through `flags` as in the fused launch and are consumed soon after they are written, so they are read
// from L2 and dropped from it unwritten.  Launched cooperatively (every CTA resident); every wait is
// bounded.
constexpr int TEAM_MAX_CHAINS = 512;  // chains per team the producers' table holds
constexpr uint32_t J_TCH = J_CU + 4 * (J_TBL_N + 1);   // team mode: chain table [TEAM_MAX_CHAINS]
constexpr uint32_t J_TPRE = J_TCH + 4 * TEAM_MAX_CHAINS;  //            item prefix [TEAM_MAX_CHAINS + 1]
constexpr uint32_t J_TEAM_TOTAL = J_TPRE + 4 * (TEAM_MAX_CHAINS + 1) + 1024;

__global__ void __launch_bounds__(NT2, 1)
chunk_team_tc_kernel(const __grid_constant__ TileMaps tm, const __grid_constant__ CUtensorMap omap,
                     const bf16 *__restrict__ beta, const float *__restrict__ bias, const float *__restrict__ A_log,
                     float g_min, int64_t T, int N, const int32_t *__restrict__ cu, int H,
                     unsigned char *__restrict__ packets, float scale, const float *initial_state,
                     float *final_state, bf16 *__restrict__ o, int *err, int teams, int K, int window,
                     uint64_t *flags, uint64_t *consumed, uint64_t epoch, const __grid_constant__ CUtensorMap gmap,
                     int epi, const float *epi_w, float epi_eps, uint64_t *ctr) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = align1024(smem_raw);
    const int b = (int)blockIdx.x, tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    int32_t *cs = (int32_t *)(sm + J_CS);    // chunk_start [N + 1]
    int32_t *perm = (int32_t *)(sm + J_SS);  // sequences by decreasing chunk count
    int32_t *cus = (int32_t *)(sm + J_CU);   // cu_seqlens [N + 1]
    const int32_t *cu_l = cu ? cus : nullptr;
    int *s_bad = (int *)(sm + J_SS + 4 * (J_TBL_N + 1));
    if (warp == 0) {  // validate cu_seqlens (0 = c_0 <= ... <= c_N = T) and count chunks per sequence
        bool bad = false;
        if (cu) {
            for (int n = lane; n <= N; n += 32) {
                const int64_t x = cu[n];
                cus[n] = (int32_t)x;
                bad = bad || (n == 0 && x != 0) || (n == N && x != T) || (n > 0 && x < (int64_t)cu[n - 1]);
            }
        }
        bad = __any_sync(0xffffffffu, bad);
        int carry = 0;
        for (int base = 0; base < N; base += 32) {
            const int m = base + lane;
            int x = 0;
            if (m < N && !bad) {
                const int64_t len = cu ? (int64_t)cu[m + 1] - cu[m] : T / N;
                x = (int)((len + C - 1) / C);
            }
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, off);
                if (lane >= off) x += y;
            }
            if (m < N) cs[m + 1] = carry + x;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) {
            cs[0] = 0;
            *s_bad = bad ? 1 : 0;
        }
    }
    __syncthreads();
    if (*(volatile int *)s_bad) {
        if (b == 0 && tid == 0) set_error(err, KDA_ERR_BAD_SEQLENS);
        return;
    }
    for (int n = tid; n < N; n += blockDim.x) {  // rank by (chunks descending, index ascending)
        const int cn = cs[n + 1] - cs[n];
        int r = 0;
        for (int m = 0; m < N; ++m) {
            const int cm = cs[m + 1] - cs[m];
            r += (cm > cn || (cm == cn && m < n)) ? 1 : 0;
        }
        perm[r] = n;
    }
    __syncthreads();
    const int t = b / (K + 1), role = b % (K + 1);
    if (t >= teams) return;
    const int chains = N * H;
    auto chain_of = [&](int blk) -> int {  // rank of the team's blk-th chain, or -1
        const int r = blk * teams + ((blk & 1) ? teams - 1 - t : t);
        return r < chains ? r : -1;
    };
    if (role == 0) {
        for (int blk = 0;; ++blk) {
            const int r = chain_of(blk);
            if (r < 0) break;
            chain_role(sm, omap, T, N, cu, cs, nullptr, (int64_t)1 << 30, nullptr, H, packets, scale, initial_state,
                       final_state, o, err, perm[r / H], r % H, flags, epoch, consumed, false,
                       epi ? &gmap : nullptr, epi_w, epi_eps);
        }
    } else {
        int32_t *tch = (int32_t *)(sm + J_TCH), *tpre = (int32_t *)(sm + J_TPRE);
        __shared__ int s_count;
        if (tid == 0) {
            int c = 0;
            tpre[0] = 0;
            for (int blk = 0; c < TEAM_MAX_CHAINS; ++blk) {
                const int r = chain_of(blk);
                if (r < 0) break;
                const int n = perm[r / H];
                tch[c] = n * H + r % H;
                tpre[c + 1] = tpre[c] + (cs[n + 1] - cs[n]);
                ++c;
            }
            s_count = c;
        }
        __syncthreads();
        const TeamItems ti{tch, tpre, s_count, K, role - 1, window, consumed};
        intra_role(sm, tm, beta, bias, A_log, g_min, T, N, cu_l, cs, H, packets, err, 0, 1, flags, epoch, 0, -1, 0,
                   &ti, ctr ? ctr + KDA_CTR_STRIDE * t : nullptr);
    }
}

// =====================================================================================
// Segment summaries (section 5.1.2, Eq. 17, used inside one device): for every segment but
// the last of its sequence, run the state recurrence over the segment's chunks on the pair
// [S~ | M] from [0 | I]: S~ with the segment's values, M with values zero.  Then for any
// entering state, S_out = M S_in + S~.  [S~ | M] is kept like the state of the output pass
// (d_k lanes; 256 columns), so per chunk:
//   MMA1  D = W [S~ | M]                       (M = 128 with rows 64-127 unused, K = 128)
//   V~    = [U - W S~ | -W M]                  (TMEM lanes 0-63), token-major images
//   MMA2  [S~ | M] <- Diag(gamma) [S~ | M] + K~^T [V~_S | V~_M]   (K = 64)
// S~ and M are independent chains (N = 128 each) run by separate warp groups.
// A stage holds [W half 0 | K~ half 0 | W half 1 | K~ half 1 | gamma]: read as a 128-row K-major image
// it is W (rows 64-127 are K~ and land in unused lanes); K~ is read MN-major with its halves 16 KB
// apart.  U (kept as U^T in the packet) goes from global memory to registers one chunk ahead.
constexpr uint32_t SS_NST = 3;
constexpr uint32_t SS_STAGE_BYTES = 33792;
constexpr uint32_t SS_G = 32768;
constexpr uint32_t SS_SIMG = SS_NST * SS_STAGE_BYTES;  // [S~ | M] image: rows d_k, 4 x 64 columns (16 KB each)
constexpr uint32_t SS_VIMG = SS_SIMG + 65536;          // [V~_S | V~_M] token-major image, 4 x 8 KB
constexpr uint32_t SS_BAR = SS_VIMG + 32768;
constexpr uint32_t SS_TSLOT = SS_BAR + 64;
constexpr uint32_t SS_TOTAL = SS_BAR + 128 + 1024;
constexpr uint32_t SS_TX = 4 * 8192 + 512;
// Summary record per (segment, head): S~ fp32 (lane-major, see ll_off), then M as bf16 high and low
// K-major images.
constexpr size_t SUM_M_HI = 65536, SUM_M_LO = 98304;

__global__ void __launch_bounds__(512, 1)
chunk_segsum_tc_kernel(int N, const int32_t *__restrict__ chunk_start, const int32_t *__restrict__ seg_start,
                       int64_t seg_len, int H, const unsigned char *__restrict__ packets,
                       float *__restrict__ seg_sum, int *err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = align1024(smem_raw);
    const int g = blockIdx.x, h = blockIdx.y;
    if (g >= seg_start[N]) return;
    int n = 0;
    {
        int lo = 0, hi = N;
        while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (seg_start[mid] <= g) lo = mid; else hi = mid;
        }
        n = lo;
    }
    const int seg_i = g - seg_start[n], nseg = seg_start[n + 1] - seg_start[n];
    if (seg_i == nseg - 1) return;  // the last segment of a sequence needs no summary
    const int64_t kk0 = (int64_t)seg_i * seg_len;
    const int c_begin = chunk_start[n] + (int)kk0;
    const int nc = (int)min(seg_len, (int64_t)(chunk_start[n + 1] - chunk_start[n]) - kk0);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = warp & 3, cg = warp >> 2;  // TMEM lane quarter; 64-column group of 256
    const int row = 32 * lq + lane;
    uint64_t *bar_ld = (uint64_t *)(sm + SS_BAR);  // [3]
    uint64_t *bar_v = bar_ld + 3, *bar_s = bar_ld + 5;  // [2 chains] each
    uint32_t *tslot = (uint32_t *)(sm + SS_TSLOT);
    if (tid == 0) {
        for (int i = 0; i < 3; ++i) mbar_init(&bar_ld[i], 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(&bar_v[i], 1);
            mbar_init(&bar_s[i], 1);
        }
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    fence_proxy_async();
    sync_all();
    const uint32_t tb = *tslot;
    const uint32_t tSM = tb, tDV = tb + 256;  // [S~ | M] (256 columns); D (256 columns, lanes 0-63)
    auto packet = [&](int kk) { return packets + ((size_t)(c_begin + kk) * H + h) * PK_STRIDE; };
    auto issue = [&](int kk) {
        unsigned char *dst = sm + (kk % SS_NST) * SS_STAGE_BYTES;
        uint64_t *b = &bar_ld[kk % SS_NST];
        const unsigned char *pk = packet(kk);
        mbar_arrive_expect_tx(b, SS_TX);
        bulk_g2s(dst, pk + PK_WQ, 8192, b);
        bulk_g2s(dst + 8192, pk + PK_K, 8192, b);
        bulk_g2s(dst + 16384, pk + PK_WQ + 16384, 8192, b);
        bulk_g2s(dst + 24576, pk + PK_K + 8192, 8192, b);
        bulk_g2s(dst + SS_G, pk + PK_G, 512, b);
    };
    if (tid == 0) {
        for (int kk = 0; kk < (int)SS_NST && kk < nc; ++kk) issue(kk);
    }
    bool ok = wait_all(&bar_ld[0], 0);
    fence_after_sync();
    if (ok) {  // [S~ | M] = [0 | I]: image, and TMEM scaled by gamma_0 (a per-row scale)
        const float gr = reinterpret_cast<const float *>(sm + SS_G)[row];
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
            float x[16], xs[16];
#pragma unroll
            for (int e = 0; e < 16; ++e) {
                const int c = 64 * cg + c0 + e;
                x[e] = (c >= 128 && c - 128 == row) ? 1.f : 0.f;
                xs[e] = x[e] * gr;
            }
            tmem_st16(tmem_addr(tSM, 32 * lq, 64 * cg + c0), xs);
            *reinterpret_cast<uint4 *>(sm + SS_SIMG + img_chunk_off(128, row, (64 * cg + c0) / 8)) = pack8(x);
            *reinterpret_cast<uint4 *>(sm + SS_SIMG + img_chunk_off(128, row, (64 * cg + c0) / 8 + 1)) = pack8(x + 8);
        }
        tmem_st_wait();
    }
    fence_proxy_async();
    sync_all();
    // Two independent chains: warps 0-7 carry S~ (columns 0-127 of [S~ | M]), warps 8-15 carry M
    // (columns 128-255); each issues its own MMAs and synchronises on its own barriers, so one chain's
    // CUDA-core phases overlap the other's products.
    const int ch = warp >> 3, nb = 1 + ch, ct = tid & 255;
    // U row `row` (a token), columns [64 cg, 64 cg + 64) for warps with lq < 2 and cg < 2
    const bool vrow = (lq < 2), uneed = vrow && (cg < 2);
    uint4 ua[8];
    auto load_u = [&](int kk) {  // from the U^T image (rows are channels): one bf16 per load, coalesced
        const unsigned char *src = packet(kk) + PK_U;
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int c = 64 * cg + 8 * jj + 2 * e;
                const uint32_t lo = __ldg(reinterpret_cast<const unsigned short *>(src + img_off(128, c, row)));
                const uint32_t hi = __ldg(reinterpret_cast<const unsigned short *>(src + img_off(128, c + 1, row)));
                w[e] = lo | (hi << 16);
            }
            ua[jj] = make_uint4(w[0], w[1], w[2], w[3]);
        }
    };
    if (uneed && nc > 0) load_u(0);
    const uint32_t id1 = idesc_bf16(128, 128, false, true), id2 = idesc_bf16(128, 128, true, true);
    for (int kk = 0; kk < nc && ok; ++kk) {
        unsigned char *P = sm + (kk % SS_NST) * SS_STAGE_BYTES;
        if (ct == 0) {  // D[:, chain] = W [S~ | M][:, chain]
            fence_after_sync();
            mma_bf16_kmn(tDV + 128 * ch, smem_u32(P), 128, smem_u32(sm + SS_SIMG + 32768 * ch), 16384, 8, id1, false);
            mma_commit(&bar_v[ch]);
            ok = mbar_wait_spin(&bar_v[ch], kk & 1);
        }
        ok = bar_red_popc(nb, 256, ok) == 256;
        if (!ok) break;
        fence_after_sync();
        if (vrow) {  // V~ row `row`: columns [64 cg, 64 cg + 64) of [U - W S~ | -W M]
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
                float d[32], u[8], vo[8];
                tmem_ld32(tmem_addr(tDV, 32 * lq, 64 * cg + 32 * h2), d);
#pragma unroll
                for (int jj = 0; jj < 4; ++jj) {
                    if (uneed) {
                        unpack8(ua[4 * h2 + jj], u);
#pragma unroll
                        for (int e = 0; e < 8; ++e) vo[e] = u[e] - d[8 * jj + e];
                    } else {
#pragma unroll
                        for (int e = 0; e < 8; ++e) vo[e] = -d[8 * jj + e];
                    }
                    *reinterpret_cast<uint4 *>(sm + SS_VIMG + img_chunk_off(64, row, 8 * cg + 4 * h2 + jj)) = pack8(vo);
                }
            }
            if (uneed && kk + 1 < nc) load_u(kk + 1);
        }
        fence_proxy_async();
        fence_before_sync();
        named_sync(nb, 256);
        const bool last = (kk == nc - 1);
        if (ct == 0) {  // [S~ | M][:, chain] += K~^T V~[:, chain]
            fence_after_sync();
            mma_bf16_mnmn(tSM + 128 * ch, smem_u32(P + 8192), 16384, smem_u32(sm + SS_VIMG + 16384 * ch), 8192, 4, id2,
                          true);
            mma_commit(&bar_s[ch]);
            const bool okl = last || mbar_wait_spin(&bar_ld[(kk + 1) % SS_NST], ((kk + 1) / SS_NST) & 1);
            ok = mbar_wait_spin(&bar_s[ch], kk & 1) && okl;
        }
        ok = bar_red_popc(nb, 256, ok) == 256;
        if (!ok) break;
        fence_after_sync();
        const float gr = reinterpret_cast<const float *>(sm + ((kk + 1) % SS_NST) * SS_STAGE_BYTES + SS_G)[row];
        float *out = seg_sum + ((size_t)g * H + h) * 2 * D * D;
#pragma unroll
        for (int h2 = 0; h2 < 2; ++h2) {
            const int c0 = 64 * cg + 32 * h2;  // column in [S~ | M]
            float x[32];
            tmem_ld32(tmem_addr(tSM, 32 * lq, c0), x);
            if (!last) {
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8)
                    *reinterpret_cast<uint4 *>(sm + SS_SIMG + img_chunk_off(128, row, c0 / 8 + q8)) = pack8(x + 8 * q8);
#pragma unroll
                for (int e = 0; e < 32; ++e) x[e] *= gr;
                tmem_st32(tmem_addr(tSM, 32 * lq, c0), x);
            } else if (c0 < 128) {  // S~ row `row`, fp32
#pragma unroll
                for (int e = 0; e < 32; e += 4)
                    *reinterpret_cast<float4 *>(out + ll_off(row, c0 + e)) =
                        make_float4(x[e], x[e + 1], x[e + 2], x[e + 3]);
            } else {  // M row `row` as bf16 high / low parts of a K-major image (the fold's A operand)
                unsigned char *mimg = reinterpret_cast<unsigned char *>(out);
#pragma unroll
                for (int q8 = 0; q8 < 4; ++q8) {
                    float hi[8], lo[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        hi[e] = __bfloat162float(__float2bfloat16_rn(x[8 * q8 + e]));
                        lo[e] = x[8 * q8 + e] - hi[e];
                    }
                    const uint32_t off = img_chunk_off(128, row, (c0 - 128) / 8 + q8);
                    *reinterpret_cast<uint4 *>(mimg + SUM_M_HI + off) = pack8(hi);
                    *reinterpret_cast<uint4 *>(mimg + SUM_M_LO + off) = pack8(lo);
                }
            }
        }
        if (!last) tmem_st_wait();
        fence_proxy_async();
        fence_before_sync();
        named_sync(nb, 256);
        // stage kk is free once both chains' products of chunk kk are done
        if (ch == 1 && ct == 0 && kk + (int)SS_NST < nc) {
            if (mbar_wait_spin(&bar_s[0], kk & 1)) issue(kk + SS_NST);
            else ok = false;
        }
    }
    if (!ok && tid == 0) set_error(err, KDA_ERR_DEVICE_TIMEOUT);
    sync_all();
    if (warp == 0) tmem_dealloc(tb, 512);
}

// =====================================================================================
// Fold of the segment summaries of each (sequence, head) in order (section 5.1.2: the
// rank-level updates compose associatively): S_in(i+1) = M_i S_in(i) + S~_i, starting from
// the sequence's initial state.  An MMA with A = M (K-major high / low images written by the summary
// pass) and B = S_in (rows d_k, read MN-major); both factors are split into bf16 high and low parts
// and hi*hi + hi*lo + lo*hi is accumulated (near-fp32 accuracy): one N = 256 product
// M_hi [S_hi | S_lo] and one N = 128 product M_lo S_hi.  The M images of step i + 2 are bulk-copied
// while step i runs; S~ of step i + 1 is read into registers during step i and placed in tensor
// memory, where the readout adds it.
constexpr uint32_t FD_STG = 0;                 // 2 stages x [M hi | M lo] (64 KB each)
constexpr uint32_t FD_B = 131072;              // [S_in hi | S_in lo] image: rows d_k, 4 x 64 columns (64 KB)
constexpr uint32_t FD_BAR = FD_B + 65536;      // ld[2], mma
constexpr uint32_t FD_TSLOT = FD_BAR + 32;
constexpr uint32_t FD_TOTAL = FD_BAR + 64 + 1024;
constexpr uint32_t TF_D = 0, TF_ST = 256;      // TMEM: products (256 columns), S~ (128 columns)

__global__ void __launch_bounds__(256, 1)
chunk_fold_tc_kernel(int N, const int32_t *__restrict__ seg_start, int H, const float *initial_state,
                     const float *__restrict__ seg_sum, float *__restrict__ seg_in, int *err) {
    extern __shared__ unsigned char smem_raw[];
    unsigned char *sm = align1024(smem_raw);
    const int n = blockIdx.x, h = blockIdx.y;
    const int g0 = seg_start[n], nseg = seg_start[n + 1] - g0;
    if (nseg <= 1) return;
    const int steps = nseg - 1;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int lq = warp & 3, hf = warp >> 2;
    const int row = lq * 32 + lane;  // d_k row of S = TMEM lane
    uint64_t *bar_ld = (uint64_t *)(sm + FD_BAR);
    uint64_t *bar_mma = bar_ld + 2;
    uint32_t *tslot = (uint32_t *)(sm + FD_TSLOT);
    auto summary = [&](int i) { return seg_sum + ((size_t)(g0 + i) * H + h) * 2 * D * D; };
    auto issue = [&](int i) {  // M hi / lo images of step i into stage i & 1
        mbar_arrive_expect_tx(&bar_ld[i & 1], 65536);
        bulk_g2s(sm + FD_STG + (i & 1) * 65536, reinterpret_cast<const unsigned char *>(summary(i)) + SUM_M_HI,
                 65536, &bar_ld[i & 1]);
    };
    if (tid == 0) {
        mbar_init(&bar_ld[0], 1);
        mbar_init(&bar_ld[1], 1);
        mbar_init(bar_mma, 1);
    }
    if (warp == 0) tmem_alloc(tslot, 512);
    fence_proxy_async();
    sync_all();
    const uint32_t tb = *tslot;
    if (tid == 0) {
        issue(0);
        if (steps > 1) issue(1);
    }
    const size_t st_off = ((size_t)n * H + h) * D * D;
    float sreg[64];  // S row `row`, columns [64 hf, 64 hf + 64)
#pragma unroll
    for (int e = 0; e < 64; e += 4) {
        float4 v4 = make_float4(0.f, 0.f, 0.f, 0.f);
        if (initial_state) v4 = *reinterpret_cast<const float4 *>(initial_state + st_off + (size_t)row * D + 64 * hf + e);
        sreg[e] = v4.x; sreg[e + 1] = v4.y; sreg[e + 2] = v4.z; sreg[e + 3] = v4.w;
    }
    {
        float *dst0 = seg_in + ((size_t)g0 * H + h) * D * D;  // segment 0 enters with S0
#pragma unroll
        for (int e = 0; e < 64; e += 4)
            *reinterpret_cast<float4 *>(dst0 + ll_off(row, 64 * hf + e)) =
                make_float4(sreg[e], sreg[e + 1], sreg[e + 2], sreg[e + 3]);
    }
    float nxt[64];  // S~ row `row` of the current step
#pragma unroll
    for (int e = 0; e < 64; e += 4) {
        const float4 v4 = *reinterpret_cast<const float4 *>(summary(0) + ll_off(row, 64 * hf + e));
        nxt[e] = v4.x; nxt[e + 1] = v4.y; nxt[e + 2] = v4.z; nxt[e + 3] = v4.w;
    }
    bool ok = true;
    const uint32_t id256 = idesc_bf16(128, 256, false, true), id128 = idesc_bf16(128, 128, false, true);
    for (int i = 0; i < steps && ok; ++i) {
        // S~ into TMEM; S_in hi / lo images (rows d_k)
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) tmem_st16(tmem_addr(tb + TF_ST, lq * 32, 64 * hf + c0), nxt + c0);
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 8) {
            float hi[8], lo[8];
#pragma unroll
            for (int e = 0; e < 8; ++e) {
                hi[e] = __bfloat162float(__float2bfloat16_rn(sreg[c0 + e]));
                lo[e] = sreg[c0 + e] - hi[e];
            }
            const uint32_t off = img_chunk_off(128, row, (64 * hf + c0) / 8);
            *reinterpret_cast<uint4 *>(sm + FD_B + off) = pack8(hi);
            *reinterpret_cast<uint4 *>(sm + FD_B + 32768 + off) = pack8(lo);
        }
        tmem_st_wait();
        fence_proxy_async();
        ok = wait_all(&bar_ld[i & 1], (i >> 1) & 1);
        if (!ok) break;
        fence_after_sync();
        if (tid == 0) {
            const uint32_t A = smem_u32(sm + FD_STG + (i & 1) * 65536);
            mma_bf16_kmn(tb + TF_D, A, 128, smem_u32(sm + FD_B), 16384, 8, id256, false);
            mma_bf16_kmn(tb + TF_D, A + 32768, 128, smem_u32(sm + FD_B), 16384, 8, id128, true);
            mma_commit(bar_mma);
        }
        if (i + 1 < steps) {
#pragma unroll
            for (int e = 0; e < 64; e += 4) {
                const float4 v4 = *reinterpret_cast<const float4 *>(summary(i + 1) + ll_off(row, 64 * hf + e));
                nxt[e] = v4.x; nxt[e + 1] = v4.y; nxt[e + 2] = v4.z; nxt[e + 3] = v4.w;
            }
        }
        ok = wait_all(bar_mma, i & 1);
        if (!ok) break;
        fence_after_sync();
        if (tid == 0 && i + 2 < steps) issue(i + 2);  // stage i & 1 has been read
        float *dst = seg_in + ((size_t)(g0 + i + 1) * H + h) * D * D;
#pragma unroll
        for (int c0 = 0; c0 < 64; c0 += 16) {
            float a[16], b[16], c[16];
            tmem_ld16(tmem_addr(tb + TF_D, lq * 32, 64 * hf + c0), a);
            tmem_ld16(tmem_addr(tb + TF_D, lq * 32, 128 + 64 * hf + c0), b);
            tmem_ld16(tmem_addr(tb + TF_ST, lq * 32, 64 * hf + c0), c);
#pragma unroll
            for (int e = 0; e < 16; ++e) sreg[c0 + e] = a[e] + b[e] + c[e];
#pragma unroll
            for (int e = 0; e < 16; e += 4)
                *reinterpret_cast<float4 *>(dst + ll_off(row, 64 * hf + c0 + e)) =
                    make_float4(sreg[c0 + e], sreg[c0 + e + 1], sreg[c0 + e + 2], sreg[c0 + e + 3]);
        }
        fence_before_sync();
        __syncthreads();
        fence_after_sync();
    }
    if (!ok && tid == 0) set_error(err, KDA_ERR_DEVICE_TIMEOUT);
    sync_all();
    if (warp == 0) tmem_dealloc(tb, 512);
}

}  // namespace tcp
}  // namespace kda

using namespace kda;

size_t kda_tc_packet_stride() { return tcp::PK_STRIDE; }

kda_status_t kda_launch_chunk_plan(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                   cudaStream_t stream);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no link-time libcuda dependency).
typedef CUresult (*encode_tiled_fn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                    const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                    CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                    CUtensorMapFloatOOBfill);

static encode_tiled_fn get_encode_tiled() {
    static encode_tiled_fn fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (encode_tiled_fn)p;
    }
    return fn;
}

// [T, H, 128] bf16 as a 3-D map (channel, head, token) with 64 x 1 x 64 boxes (128 bytes per
// token row) and 128-byte swizzle: a box lands as the [64 tokens][64 channels] half of an operand
// tile.  Tokens past T read as zeros.
static bool make_tile_map(CUtensorMap *m, const void *base, int64_t T, int H) {
    encode_tiled_fn enc = get_encode_tiled();
    if (!enc) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)T};
    const cuuint64_t strides[2] = {256, (cuuint64_t)H * 256};
    const cuuint32_t box[3] = {64, 1, 64};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

static kda_status_t set_smem(const void *kernel, uint32_t bytes) {
    return kda_cuda_status(cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes));
}

// The fused schedule: one cooperative launch of chains + producers.  Returns false (and clears the
// launch error) when the device refuses to make every CTA resident; the caller then runs the
// separate kernels, which need the same workspace.
// A launch epoch for the packet flags: a per-process counter that never repeats (and is never 0).
static uint64_t next_launch_epoch() {
    static std::atomic<uint64_t> next_epoch{0};
    uint64_t expected = 0;  // first use: start the epochs at a value unlikely to sit in fresh memory
    if (next_epoch.load() == 0)
        next_epoch.compare_exchange_strong(
            expected, ((uint64_t)std::chrono::steady_clock::now().time_since_epoch().count() << 20) | 1u);
    uint64_t epoch = next_epoch.fetch_add(1);
    if (epoch == 0) epoch = next_epoch.fetch_add(1);
    return epoch;
}

static bool launch_fused(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws, cudaStream_t stream,
                         const tcp::TileMaps &tm, const CUtensorMap &omap, int sms, int *err,
                         const CUtensorMap &gmap, int epi) {
    const uint32_t smem = tcp::J_TOTAL > tcp::CS_TOTAL ? tcp::J_TOTAL : tcp::CS_TOTAL;
    if (set_smem((const void *)tcp::chunk_fused_tc_kernel, smem) != KDA_OK) return false;
    int per_sm = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tcp::chunk_fused_tc_kernel, tcp::NT2, smem) !=
            cudaSuccess ||
        per_sm < 1)
        return false;
    uint64_t epoch = next_launch_epoch();
    uint64_t *flags = (uint64_t *)((char *)ws + p.off_flags);
    unsigned char *packets = (unsigned char *)ws + p.off_records;
    const bf16 *beta = (const bf16 *)a->beta;
    const float *bias = a->dt_bias, *A_log = a->A_log, *init = a->initial_state;
    float g_min = a->g_min, scale = a->scale;
    int64_t T = a->T;
    int N = (int)a->N, H = p.H, n_chain = (int)(a->N * p.H), kpre = p.kpre;
    const int32_t *cu = a->cu_seqlens;
    float *fin = a->final_state;
    bf16 *o = (bf16 *)a->o;
    const float *epi_w = a->out_norm_weight;
    float epi_eps = a->out_norm_eps;
    uint64_t *ctr = (uint64_t *)((char *)ws + p.off_ctr);
    void *args[] = {(void *)&tm, (void *)&omap, &beta, &bias, &A_log, &g_min, &T, &N, &cu, &H, &packets,
                    &scale, &init, &fin, &o, &err, &n_chain, &flags, &epoch, &kpre, (void *)&gmap, &epi, &epi_w,
                    &epi_eps, &ctr};
    if (cudaLaunchCooperativeKernel((const void *)tcp::chunk_fused_tc_kernel, dim3((unsigned)sms), dim3(tcp::NT2),
                                    args, smem, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return true;
}

// The chain-team schedule (see chunk_team_tc_kernel).  Returns false (and clears the launch error)
// when the device refuses to make every CTA resident; the caller then runs the separate kernels.
static bool launch_team(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws, cudaStream_t stream,
                        const tcp::TileMaps &tm, const CUtensorMap &omap, int sms, int *err, uint64_t epoch,
                        const CUtensorMap &gmap, int epi) {
    const uint32_t smem = tcp::J_TEAM_TOTAL > tcp::CS_TOTAL ? tcp::J_TEAM_TOTAL : tcp::CS_TOTAL;
    if (set_smem((const void *)tcp::chunk_team_tc_kernel, smem) != KDA_OK) return false;
    int per_sm = 0;
    const int grid = p.teams * (p.team_k + 1);
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, tcp::chunk_team_tc_kernel, tcp::NT2, smem) !=
            cudaSuccess ||
        per_sm < 1 || grid > sms * per_sm)
        return false;
    uint64_t *flags = (uint64_t *)((char *)ws + p.off_flags);
    uint64_t *consumed = (uint64_t *)((char *)ws + p.off_consumed);
    unsigned char *packets = (unsigned char *)ws + p.off_records;
    const bf16 *beta = (const bf16 *)a->beta;
    const float *bias = a->dt_bias, *A_log = a->A_log, *init = a->initial_state;
    float g_min = a->g_min, scale = a->scale;
    int64_t T = a->T;
    int N = (int)a->N, H = p.H, teams = p.teams, K = p.team_k, window = p.team_window;
    const int32_t *cu = a->cu_seqlens;
    float *fin = a->final_state;
    bf16 *o = (bf16 *)a->o;
    const float *epi_w = a->out_norm_weight;
    float epi_eps = a->out_norm_eps;
    uint64_t *ctr = (uint64_t *)((char *)ws + p.off_ctr);
    void *args[] = {(void *)&tm, (void *)&omap, &beta, &bias, &A_log, &g_min, &T, &N, &cu, &H, &packets, &scale,
                    &init, &fin, &o, &err, &teams, &K, &window, &flags, &consumed, &epoch, (void *)&gmap, &epi, &epi_w,
                    &epi_eps, &ctr};
    if (cudaLaunchCooperativeKernel((const void *)tcp::chunk_team_tc_kernel, dim3((unsigned)grid), dim3(tcp::NT2), args,
                                    smem, stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return false;
    }
    return true;
}

kda_status_t kda_launch_chunk_tc(const kda_chunk_args *a, const kda_chunk_plan &p, void *ws,
                                 cudaStream_t stream) {
    int *err = kda_device_error_ptr();
    if (!err) return KDA_ERR_CUDA;
    const int32_t *chunk_start = (const int32_t *)((char *)ws + p.off_chunk_start);
    unsigned char *packets = (unsigned char *)ws + p.off_records;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    tcp::TileMaps tm;
    CUtensorMap omap, gmap;
    const int epi = (a->out_gate && p.epi_fused) ? 1 : 0;  // the output epilogue runs in the output pass
    if (!make_tile_map(&tm.q, a->q, a->T, p.H) || !make_tile_map(&tm.k, a->k, a->T, p.H) ||
        !make_tile_map(&tm.v, a->v, a->T, p.H) || !make_tile_map(&tm.z, a->z, a->T, p.H) ||
        !make_tile_map(&omap, a->o, a->T, p.H) || !make_tile_map(&gmap, epi ? a->out_gate : a->o, a->T, p.H))
        return KDA_ERR_CUDA;
    kda_profile_mark(0, stream);
    // The fused launch publishes packets through flags tagged with a host-side epoch.  A captured
    // graph would replay one fixed epoch against flags its previous replay left in the same
    // workspace, so under stream capture (or when the capture state cannot be read) the flag-free
    // separate kernels run instead.
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(stream, &cap) != cudaSuccess) {
        (void)cudaGetLastError();
        cap = cudaStreamCaptureStatusActive;
    }
    const bool capturing = cap != cudaStreamCaptureStatusNone;
    if (p.fused && !capturing && p.max_chunks > 0 && a->T > 0 &&
        launch_fused(a, p, ws, stream, tm, omap, sms, err, gmap, epi)) {
        kda_profile_mark(1, stream);
        return kda_cuda_status(cudaGetLastError());
    }
    if (p.team && !capturing && p.max_chunks > 0 && a->T > 0 &&
        launch_team(a, p, ws, stream, tm, omap, sms, err, next_launch_epoch(), gmap, epi)) {
        kda_profile_mark(1, stream);
        return kda_cuda_status(cudaGetLastError());
    }
    // separate kernels (also the fallback when the fused launch cannot make every CTA resident)
    kda_status_t st = kda_launch_chunk_plan(a, p, ws, stream);
    if (st != KDA_OK) return st;
    kda_profile_mark(1, stream);
    if (p.max_chunks > 0 && a->T > 0) {
        st = set_smem((const void *)tcp::chunk_intra_tc_kernel, tcp::J_TOTAL);
        if (st != KDA_OK) return st;
        const int64_t items = p.max_chunks * (int64_t)p.H;
        const unsigned grid = (unsigned)(items < sms ? items : sms);
        // items are handed out through a launch-tagged counter; a captured graph would replay one tag,
        // so under capture every CTA takes a fixed share instead
        uint64_t *ctr = capturing ? nullptr : (uint64_t *)((char *)ws + p.off_ctr);
        tcp::chunk_intra_tc_kernel<<<grid, tcp::NT2, tcp::J_TOTAL, stream>>>(
            tm, (const bf16 *)a->beta, a->dt_bias, a->A_log, a->g_min, a->T, (int)a->N, a->cu_seqlens,
            chunk_start, p.H, packets, err, ctr, next_launch_epoch());
        st = kda_cuda_status(cudaGetLastError());
        if (st != KDA_OK) return st;
    }
    kda_profile_mark(2, stream);
    const int32_t *seg_start = (const int32_t *)((char *)ws + p.off_seg_start);
    float *seg_sum = (float *)((char *)ws + p.off_seg_sum);
    float *seg_in = (float *)((char *)ws + p.off_seg_in);
    int mark = 3;
    if (p.split) {
        st = set_smem((const void *)tcp::chunk_segsum_tc_kernel, tcp::SS_TOTAL);
        if (st != KDA_OK) return st;
        tcp::chunk_segsum_tc_kernel<<<dim3((unsigned)p.max_segs, (unsigned)p.H), 512, tcp::SS_TOTAL, stream>>>(
            (int)a->N, chunk_start, seg_start, p.seg_len, p.H, packets, seg_sum, err);
        st = kda_cuda_status(cudaGetLastError());
        if (st != KDA_OK) return st;
        kda_profile_mark(mark++, stream);
        st = set_smem((const void *)tcp::chunk_fold_tc_kernel, tcp::FD_TOTAL);
        if (st != KDA_OK) return st;
        tcp::chunk_fold_tc_kernel<<<dim3((unsigned)a->N, (unsigned)p.H), 256, tcp::FD_TOTAL, stream>>>(
            (int)a->N, seg_start, p.H, a->initial_state, seg_sum, seg_in, err);
        st = kda_cuda_status(cudaGetLastError());
        if (st != KDA_OK) return st;
        kda_profile_mark(mark++, stream);
    }
    st = set_smem((const void *)tcp::chunk_inter_tc_kernel, tcp::CS_TOTAL);
    if (st != KDA_OK) return st;
    {
        // one persistent CTA per SM (at most one per unit); the planning kernel reset the unit counter
        const int64_t units = p.max_segs * (int64_t)p.H;
        const unsigned grid = (unsigned)(units < sms ? units : sms);
        const int32_t *unit_seg = (const int32_t *)((char *)ws + p.off_unit);
        int *unit_ctr = (int *)((char *)ws + p.off_ctr + sizeof(uint64_t) * KDA_CTR_STRIDE);
        tcp::chunk_inter_tc_kernel<<<grid, tcp::NT3, tcp::CS_TOTAL, stream>>>(
            omap, a->T, (int)a->N, a->cu_seqlens, chunk_start, seg_start, p.seg_len, seg_in, p.H, packets, a->scale,
            a->initial_state, a->final_state, (bf16 *)a->o, err, gmap, epi, a->out_norm_weight, a->out_norm_eps,
            unit_seg, unit_ctr);
    }
    kda_profile_mark(mark, stream);
    return kda_cuda_status(cudaGetLastError());
}
