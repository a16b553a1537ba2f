// pkv_tcgen05.cuh -- 5th-generation tensor core (tcgen05) building blocks for
// sm_100-family GPUs: tensor-memory (TMEM) allocation, shared-memory matrix
// descriptors, the kind::f16 instruction descriptor, MMA issue/commit and the
// TMEM <-> register moves of the 32x32b shape.
#pragma once

#include <stdint.h>

namespace pkv {
namespace tc {

// ---------------------------------------------------------------------------
// TMEM allocation (one full warp executes these)
// ---------------------------------------------------------------------------
__device__ __forceinline__ void tmem_alloc(uint32_t smem_dst, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                     smem_dst),
                 "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}

__device__ __forceinline__ void fence_before_sync() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}

__device__ __forceinline__ void fence_after_sync() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// ---------------------------------------------------------------------------
// descriptors
// ---------------------------------------------------------------------------
// Shared-memory matrix descriptor, 128-byte swizzle (layout type 2), version 1.
//   lbo: leading-dimension byte offset, sbo: stride-dimension byte offset.
// K-major operand (rows of 128 B along K): sbo = distance between 8-row
// groups (1024 for packed rows); lbo unused.  MN-major operand (rows of 128 B
// along MN = 64 bf16, one row per K index): lbo = distance between 64-element
// column blocks along MN, sbo = distance between 8-row groups along K.
__device__ __forceinline__ uint64_t smem_desc_sw128(uint32_t smem_addr, uint32_t lbo,
                                                    uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05
    d |= (uint64_t)2 << 61;  // 128-byte swizzle
    return d;
}

// Shared-memory descriptor of a K-major operand without swizzle, made of 8x8
// core matrices (8 rows of 16 bytes, 128 bytes each): lbo = bytes between the
// core matrices adjacent along K, sbo = bytes between 8-row groups.
__device__ __forceinline__ uint64_t smem_desc_noswz(uint32_t smem_addr, uint32_t lbo,
                                                    uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((smem_addr >> 4) & 0x3FFFu);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;  // descriptor version for tcgen05; layout type 0: no swizzle
    return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: bf16 A and B, fp32 D.
//   a_mn_major / b_mn_major: 0 = K-major, 1 = MN-major.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, int a_mn_major,
                                                      int b_mn_major) {
    return (1u << 4)                                  // D format: f32
           | (1u << 7)                                // A format: bf16
           | (1u << 10)                               // B format: bf16
           | ((uint32_t)a_mn_major << 15) | ((uint32_t)b_mn_major << 16) |
           ((uint32_t)(N >> 3) << 17)                 // N / 8
           | ((uint32_t)(M >> 4) << 24);              // M / 16
}

// ---------------------------------------------------------------------------
// MMA issue (a single thread issues; completion is tracked by commit)
// ---------------------------------------------------------------------------
// D[tmem] (+)= A[smem] * B[smem]
__device__ __forceinline__ void mma_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]
__device__ __forceinline__ void mma_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                       uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Eight back-to-back MMAs into one accumulator, issued from one asm block so
// that the issuing thread spends as few instructions per MMA as it can: the
// accumulate predicate is set once (the first MMA takes `accumulate`, the rest
// accumulate), and per MMA only the low word of a descriptor moves.  A start
// address (bytes / 16) stays below 2^14 in shared memory, so the low word
// never carries into the high one.
//
// mma_ss8: k-steps of a 128-byte-swizzled K-major pair of operands (A and B
// alike): 16 elements = 32 bytes per step inside a 64-element block, the
// second block one `half_bytes` further.
template <int HALF_BYTES>
__device__ __forceinline__ void mma_ss8(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
    constexpr int H = HALF_BYTES >> 4;
    static_assert(H > 6, "half block");
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 al, ah, bl, bh, t0, t1;\n\t.reg .b64 a, b;\n\t"
        "mov.b64 {al, ah}, %1;\n\tmov.b64 {bl, bh}, %2;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t"
        "setp.eq.b32 p, %4, %4;\n\t"
        "add.s32 t0, al, 2;\n\tadd.s32 t1, bl, 2;\n\tmov.b64 a, {t0, ah};\n\tmov.b64 b, {t1, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p;\n\t"
        "add.s32 t0, al, 4;\n\tadd.s32 t1, bl, 4;\n\tmov.b64 a, {t0, ah};\n\tmov.b64 b, {t1, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p;\n\t"
        "add.s32 t0, al, 6;\n\tadd.s32 t1, bl, 6;\n\tmov.b64 a, {t0, ah};\n\tmov.b64 b, {t1, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p;\n\t"
        "add.s32 t0, al, %5;\n\tadd.s32 t1, bl, %5;\n\tmov.b64 a, {t0, ah};\n\tmov.b64 b, {t1, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p;\n\t"
        "add.s32 t0, al, %6;\n\tadd.s32 t1, bl, %6;\n\tmov.b64 a, {t0, ah};\n\tmov.b64 b, {t1, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p;\n\t"
        "add.s32 t0, al, %7;\n\tadd.s32 t1, bl, %7;\n\tmov.b64 a, {t0, ah};\n\tmov.b64 b, {t1, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p;\n\t"
        "add.s32 t0, al, %8;\n\tadd.s32 t1, bl, %8;\n\tmov.b64 a, {t0, ah};\n\tmov.b64 b, {t1, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], a, b, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate), "n"(H), "n"(H + 2), "n"(H + 4),
        "n"(H + 6)
        : "memory");
}

// mma_ts8: A from tensor memory (8 columns = 16 bf16 elements per step), B an
// MN-major 128-byte-swizzled operand whose K index advances 16 rows of 128
// bytes (2 KB) per step.
__device__ __forceinline__ void mma_ts8(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                        uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t.reg .b32 bl, bh, t, ta;\n\t.reg .b64 b;\n\t"
        "mov.b64 {bl, bh}, %2;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t"
        "setp.eq.b32 p, %4, %4;\n\t"
        "add.s32 ta, %1, 8;\n\tadd.s32 t, bl, 128;\n\tmov.b64 b, {t, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, p;\n\t"
        "add.s32 ta, %1, 16;\n\tadd.s32 t, bl, 256;\n\tmov.b64 b, {t, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, p;\n\t"
        "add.s32 ta, %1, 24;\n\tadd.s32 t, bl, 384;\n\tmov.b64 b, {t, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, p;\n\t"
        "add.s32 ta, %1, 32;\n\tadd.s32 t, bl, 512;\n\tmov.b64 b, {t, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, p;\n\t"
        "add.s32 ta, %1, 40;\n\tadd.s32 t, bl, 640;\n\tmov.b64 b, {t, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, p;\n\t"
        "add.s32 ta, %1, 48;\n\tadd.s32 t, bl, 768;\n\tmov.b64 b, {t, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, p;\n\t"
        "add.s32 ta, %1, 56;\n\tadd.s32 t, bl, 896;\n\tmov.b64 b, {t, bh};\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [ta], b, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}

// Arrive once on the mbarrier when every MMA this thread issued so far is done.
__device__ __forceinline__ void commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}

// ---------------------------------------------------------------------------
// TMEM <-> registers, 32x32b shape: thread i of the warp moves lane
// (warp quarter * 32 + i), 32 consecutive 32-bit columns.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),
          "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]),
          "=r"(r[31])
        : "r"(taddr));
}

__device__ __forceinline__ void ld_32x32b_x16(uint32_t taddr, uint32_t *r) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}

__device__ __forceinline__ void st_32x32b_x32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
        "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
        "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
        "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void st_32x32b_x16(uint32_t taddr, const uint32_t *r) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
        "r"(r[15])
        : "memory");
}

__device__ __forceinline__ void wait_ld() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void wait_st() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

}  // namespace tc
}  // namespace pkv
