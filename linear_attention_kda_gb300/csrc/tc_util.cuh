// Blackwell (sm_103a) building blocks written as inline PTX: shared-memory
// operand images and descriptors for tcgen05.mma (kind::f16, bf16 inputs, fp32
// accumulators in tensor memory), TMEM allocation and access, mbarriers with
// bounded waits, and 1-D bulk async copies.
//
// Operand images use the canonical K-major, 128-byte-swizzled layout: an
// R x K bf16 tile (R a multiple of 8, K a multiple of 64) is stored as K / 64
// blocks of R rows x 128 bytes; inside a block, the 16-byte chunk j of row r
// sits at chunk position j ^ (r % 8).  Every block starts on a 1024-byte
// boundary, so each group of 8 rows is one swizzle atom (SBO = 1024 bytes).
#pragma once
#include <cuda_bf16.h>
#include <stdint.h>

namespace kda {
namespace tc {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Byte offset of element (r, k) in a K-major SW128 image with R rows.
__device__ __forceinline__ uint32_t img_off(int R, int r, int k) {
    return (uint32_t)((k >> 6) * (R * 128) + r * 128 + ((((k & 63) >> 3) ^ (r & 7)) << 4) + ((k & 7) << 1));
}
// Byte offset of the 16-byte chunk holding elements (r, 8 j .. 8 j + 7), j in [0, K / 8).
__device__ __forceinline__ uint32_t img_chunk_off(int R, int r, int j) {
    return (uint32_t)((j >> 3) * (R * 128) + r * 128 + (((j & 7) ^ (r & 7)) << 4));
}

// Shared-memory matrix descriptor (tcgen05 format): start address >> 4, LBO >> 4
// (unused for swizzled K-major), SBO >> 4 = 1024 B between 8-row atoms, version 1,
// swizzle mode 2 (128-byte).
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Descriptor of K-step s (16 bf16 = 32 bytes each) of an image with R rows.
__device__ __forceinline__ uint64_t desc_kstep(uint32_t base, int R, int s) {
    return desc_sw128(base + (uint32_t)((s >> 2) * (R * 128) + (s & 3) * 32));
}

// Descriptor of an MN-major ("transposed") SW128 operand kept token-major: rows of 128 bytes hold
// 64 consecutive elements along M (or N), consecutive rows are consecutive K, 8-row atoms are
// 1024 bytes apart (SBO) and further 64-element groups along M (or N) lbo bytes apart (LBO).  A
// [rows][128] tile stored as two [rows][64] halves is read this way with lbo = rows * 128.
__device__ __forceinline__ uint64_t desc_sw128_mn(uint32_t saddr, uint32_t lbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

// Instruction descriptor, kind::f16: D fp32, A and B bf16, dense; A / B K-major unless a_mn / b_mn.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, bool a_mn = false, bool b_mn = false) {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Instruction descriptor, kind::tf32: D fp32, A and B tf32 (fp32 in memory, 10-bit mantissa used), dense.
__host__ __device__ constexpr uint32_t idesc_tf32(int M, int N, bool a_mn = false, bool b_mn = false) {
    return (1u << 4) | (2u << 7) | (2u << 10) | ((a_mn ? 1u : 0u) << 15) | ((b_mn ? 1u : 0u) << 16) |
           ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A(smem desc) * B(smem desc)^T, issued by one thread.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                         uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n"
        :: "r"(d_tmem), "l"(a), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// kind::tf32 product of one K-block (K = 32 fp32 values, four K-steps of 8), both operands K-major SW128
// images (rows of 128 bytes = 32 values along K; each K-step starts 32 bytes further along the rows).
__device__ __forceinline__ void mma_tf32_k32(uint32_t d_tmem, uint32_t a_base, uint32_t b_base, uint32_t idesc,
                                             bool accumulate) {
    const uint64_t da = desc_sw128(a_base), db = desc_sw128(b_base);
#pragma unroll
    for (int s = 0; s < 4; ++s) {
        asm volatile(
            "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
            "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}\n"
            :: "r"(d_tmem), "l"(da + (uint64_t)((32 * s) >> 4)), "l"(db + (uint64_t)((32 * s) >> 4)), "r"(idesc),
               "r"((accumulate || s > 0) ? 1u : 0u)
            : "memory");
    }
}

// Full product over K = 16 * ksteps: A image with RA rows, B image with RB rows.  The descriptors
// of later K-steps differ from the first only in the start-address field (address >> 4, no carry
// out of its 14 bits for shared-memory addresses), so they are formed by integer adds.
__device__ __forceinline__ void mma_bf16_k(uint32_t d_tmem, uint32_t a_base, int RA, uint32_t b_base,
                                           int RB, int ksteps, uint32_t idesc, bool accumulate) {
    const uint64_t da = desc_sw128(a_base), db = desc_sw128(b_base);
#pragma unroll
    for (int s = 0; s < ksteps; ++s)
        mma_bf16(d_tmem, da + (uint64_t)((((s >> 2) * RA * 128) + (s & 3) * 32) >> 4),
                 db + (uint64_t)((((s >> 2) * RB * 128) + (s & 3) * 32) >> 4), idesc,
                 (accumulate || s > 0) ? 1u : 0u);
}

// Full product over K = 16 * ksteps with A K-major (image with RA rows) and B MN-major (K-step s
// starts 16 rows = 2048 bytes further; N-groups b_lbo bytes apart).
__device__ __forceinline__ void mma_bf16_kmn(uint32_t d_tmem, uint32_t a_base, int RA, uint32_t b_base,
                                             uint32_t b_lbo, int ksteps, uint32_t idesc, bool accumulate) {
    const uint64_t da = desc_sw128(a_base), db = desc_sw128_mn(b_base, b_lbo);
#pragma unroll
    for (int s = 0; s < ksteps; ++s)
        mma_bf16(d_tmem, da + (uint64_t)((((s >> 2) * RA * 128) + (s & 3) * 32) >> 4),
                 db + (uint64_t)((2048 * s) >> 4), idesc, (accumulate || s > 0) ? 1u : 0u);
}
// Full product over K = 16 * ksteps with A MN-major (groups along M a_lbo bytes apart) and B K-major
// (image with RB rows).
__device__ __forceinline__ void mma_bf16_mnk(uint32_t d_tmem, uint32_t a_base, uint32_t a_lbo, uint32_t b_base,
                                             int RB, int ksteps, uint32_t idesc, bool accumulate) {
    const uint64_t da = desc_sw128_mn(a_base, a_lbo), db = desc_sw128(b_base);
#pragma unroll
    for (int s = 0; s < ksteps; ++s)
        mma_bf16(d_tmem, da + (uint64_t)((2048 * s) >> 4),
                 db + (uint64_t)((((s >> 2) * RB * 128) + (s & 3) * 32) >> 4), idesc,
                 (accumulate || s > 0) ? 1u : 0u);
}

// Full product over K = 16 * ksteps with both operands MN-major (K-step s starts 2048 bytes further in
// each; groups along M / N a_lbo / b_lbo bytes apart).
__device__ __forceinline__ void mma_bf16_mnmn(uint32_t d_tmem, uint32_t a_base, uint32_t a_lbo, uint32_t b_base,
                                              uint32_t b_lbo, int ksteps, uint32_t idesc, bool accumulate) {
    const uint64_t da = desc_sw128_mn(a_base, a_lbo), db = desc_sw128_mn(b_base, b_lbo);
#pragma unroll
    for (int s = 0; s < ksteps; ++s)
        mma_bf16(d_tmem, da + (uint64_t)((2048 * s) >> 4), db + (uint64_t)((2048 * s) >> 4), idesc,
                 (accumulate || s > 0) ? 1u : 0u);
}
// 32 consecutive fp32 columns into TMEM.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v);

// D[tmem] (+)= A(tmem) * B(smem desc)^T, issued by one thread.  A sits in tensor memory with row m in
// lane m and bf16 pairs packed per 32-bit column (element 2j in the low half of column j), so that
// one K-step of 16 elements is 8 columns.
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                       uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n"
        :: "r"(d_tmem), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate) : "memory");
}
// Full product over K = 16 * ksteps, A in tensor memory, B a K-major image with RB rows.
__device__ __forceinline__ void mma_ts_k(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, int RB, int ksteps,
                                         uint32_t idesc, bool accumulate) {
    const uint64_t db = desc_sw128(b_base);
#pragma unroll
    for (int s = 0; s < ksteps; ++s)
        mma_ts(d_tmem, a_tmem + 8 * s, db + (uint64_t)((((s >> 2) * RB * 128) + (s & 3) * 32) >> 4), idesc,
               (accumulate || s > 0) ? 1u : 0u);
}
// Full product over K = 16 * ksteps, A in tensor memory, B MN-major (groups along N b_lbo bytes apart).
__device__ __forceinline__ void mma_ts_mn(uint32_t d_tmem, uint32_t a_tmem, uint32_t b_base, uint32_t b_lbo,
                                          int ksteps, uint32_t idesc, bool accumulate) {
    const uint64_t db = desc_sw128_mn(b_base, b_lbo);
#pragma unroll
    for (int s = 0; s < ksteps; ++s)
        mma_ts(d_tmem, a_tmem + 8 * s, db + (uint64_t)((2048 * s) >> 4), idesc, (accumulate || s > 0) ? 1u : 0u);
}

// 32 / 64 consecutive fp32 columns of this thread's TMEM lane in one load.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float *v) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void fence_before_sync() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_after_sync() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
// Makes generic-proxy shared-memory writes visible to the async proxy (MMA, bulk copies).
__device__ __forceinline__ void fence_proxy_async() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }

// TMEM allocation: executed by one full warp.  With `relinquish`, the CTA then gives up the right
// to allocate again (other CTAs on the SM need not wait for it).
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols, bool relinquish = true) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(smem_u32(dst_smem)), "r"(ncols) : "memory");
    if (relinquish) asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}

// 16 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float *v) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
// 8 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float *v) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
           "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
           "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
           "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
           "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
           "r"(__float_as_uint(v[15]))
        : "memory");
}
// 16 consecutive 32-bit columns (e.g. bf16 pairs) into TMEM.
__device__ __forceinline__ void tmem_st16u(uint32_t taddr, const uint32_t *v) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
        :: "r"(taddr), "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]),
           "r"(v[8]), "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float *v) {
    tmem_st16(taddr, v);
    tmem_st16(taddr + 16, v + 16);
}
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// TMEM address of (lane, column) relative to an allocation base.
__device__ __forceinline__ uint32_t tmem_addr(uint32_t base, int lane, int col) {
    return base + ((uint32_t)lane << 16) + (uint32_t)col;
}

// ---------------------------------------------------------------- mbarriers
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(smem_u32(bar)), "r"(count) : "memory");
}
// Invalidates an mbarrier so that its shared memory can be used for something else.
__device__ __forceinline__ void mbar_inval(uint64_t *bar) {
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;"
                 :: "r"(smem_u32(bar)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Waits for the phase with the given parity to complete; gives up after ~1 s
// (returns false) so that a lost arrival can never hang the GPU.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 64; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > 1000000000ull) return false;
    }
}

// Non-blocking test of a phase; mbar_wait_spin polls it (no suspension between polls), for waits on
// the critical path of a recurrence where the wake-up delay of a suspended try_wait would show.  Also
// gives up after ~1 s.
__device__ __forceinline__ bool mbar_test_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\tmbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\tselp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ bool mbar_wait_spin(uint64_t *bar, uint32_t parity) {
    if (mbar_test_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    while (true) {
        for (int i = 0; i < 256; ++i)
            if (mbar_test_wait(bar, parity)) return true;
        if (globaltimer_ns() - t0 > 1000000000ull) return false;
    }
}

// ---------------------------------------------------------------- bulk copies (1-D, 16-byte granules)
__device__ __forceinline__ void bulk_g2s(void *smem_dst, const void *gsrc, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(smem_u32(smem_dst)), "l"(gsrc), "r"(bytes), "r"(smem_u32(bar)) : "memory");
}
// Tiled TMA load of one box of a 3-D tensor map (coordinates innermost first).
__device__ __forceinline__ void tma_load_3d(void *smem_dst, const void *tmap, int c0, int c1, int c2,
                                            uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        :: "r"(smem_u32(smem_dst)), "l"(reinterpret_cast<uint64_t>(tmap)), "r"(c0), "r"(c1), "r"(c2),
           "r"(smem_u32(bar)) : "memory");
}
// Tiled TMA store of one box of a 3-D tensor map from shared memory (bulk-group completion).
__device__ __forceinline__ void tma_store_3d(const void *tmap, const void *smem_src, int c0, int c1, int c2) {
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];"
                 :: "l"(reinterpret_cast<uint64_t>(tmap)), "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2)
                 : "memory");
}
// Prefetch of a global range into L2 (size a multiple of 16 bytes).
__device__ __forceinline__ void bulk_prefetch_l2(const void *gsrc, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" :: "l"(gsrc), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_s2g(void *gdst, const void *smem_src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;"
                 :: "l"(gdst), "r"(smem_u32(smem_src)), "r"(bytes) : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read0() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_read1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait0() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t *>(&h);
}

}  // namespace tc
}  // namespace kda
