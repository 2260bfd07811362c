// Fifth-generation tensor core (tcgen05) building blocks for sm_103a, written
// from the PTX ISA's description of the tcgen05 instructions:
//   - tensor memory (TMEM): 128 lanes x 512 columns of 32-bit cells per SM,
//     allocated by one warp of a block (a power of two >= 32 columns) and
//     freed by it before the block exits; a warp reaches only its own quarter
//     of the lanes (lanes 32 (w % 4) .. 32 (w % 4) + 31);
//   - tcgen05.mma, issued by one thread: D (in TMEM) = A B^T (+ D), A and B
//     read from shared memory through 64-bit matrix descriptors (or A from
//     TMEM), the shape and types in a 32-bit instruction descriptor; its
//     completion is signalled on an mbarrier by tcgen05.commit;
//   - tcgen05.ld / tcgen05.st move TMEM cells to and from registers
//     (shape 32x32b: thread i of the warp holds lane 32 (w % 4) + i, one
//     register per column).
// For an M = 128 product with cta_group::1, row m of D sits in TMEM lane m and
// its 32-bit column n in column base + n.
//
// Shared-memory operands use the 128-byte-swizzled K-major layout: a "panel"
// holds R rows of 32 floats (128 bytes per row) for 32 consecutive k, rows
// contiguous, the 16-byte chunk c of row r stored at chunk position c ^ (r % 8)
// (the pattern a tiled TMA load with 128-byte swizzle writes into a 1024-byte
// aligned destination).  Eight rows make one 1024-byte swizzle atom; the
// descriptor's stride byte offset is the distance between atoms along the rows
// (1024), and a K = 8 step of a tf32 product starts 32 bytes further into the
// same rows.
#pragma once

#include <cstdint>

#include "mgs_device.cuh"

namespace mgs {

// ---- TMEM allocation (called by every lane of one warp) ----
__device__ __forceinline__ void tmem_alloc(uint32_t *slot, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(slot)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

// Ordering of tcgen05 operations across a thread barrier: "before" ahead of
// the barrier in the thread whose tcgen05 work must be ordered first, "after"
// behind it in the thread that continues.
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Instruction descriptor of a dense kind::tf32 product with f32 accumulation:
// bits 4-5 D format (1 = f32), 7-9 / 10-12 A / B format (2 = tf32), 15 / 16
// A / B major (0 = K-major), 17-22 N / 8, 24-28 M / 16.
__host__ __device__ constexpr uint32_t umma_idesc_tf32(int M, int N, bool a_mn_major = false,
                                                       bool b_mn_major = false) {
    return (1u << 4) | (2u << 7) | (2u << 10) | (uint32_t(a_mn_major) << 15) | (uint32_t(b_mn_major) << 16) |
           (uint32_t(N >> 3) << 17) | (uint32_t(M >> 4) << 24);
}

// Shared-memory matrix descriptor with 128-byte swizzle: bits 0-13 start
// address / 16, 16-29 leading byte offset / 16, 32-45 stride byte offset / 16,
// 46-47 descriptor version (1), 61-63 layout (2 = 128-byte swizzle).
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    return uint64_t((saddr >> 4) & 0x3FFFu) | (uint64_t((lbo >> 4) & 0x3FFFu) << 16) |
           (uint64_t((sbo >> 4) & 0x3FFFu) << 32) | (uint64_t(1) << 46) | (uint64_t(2) << 61);
}

// Byte offset of element (row, k) of a K-major panel (k within the panel's
// 32 columns).
__host__ __device__ __forceinline__ uint32_t sw128_off(int row, int k) {
    return uint32_t(row) * 128u + ((uint32_t((k >> 2) & 7) ^ uint32_t(row & 7)) << 4) + uint32_t(k & 3) * 4u;
}

// D[tmem] (+)= A B^T, A and B from shared memory.
__device__ __forceinline__ void umma_tf32_ss(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
        : "memory");
}

// D[tmem] (+)= A B^T, A from TMEM (row m in lane m, one column per k), B from
// shared memory.
__device__ __forceinline__ void umma_tf32_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                             bool accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
        "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(uint32_t(accumulate))
        : "memory");
}

// Arrives once on `bar` when every tcgen05.mma this thread issued before has
// completed (its shared-memory reads and TMEM writes done).
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_addr(bar))
                 : "memory");
}

// 16 consecutive columns of the warp's 32 lanes into registers (thread i: lane
// 32 (w % 4) + i), waiting for the load inside the same statement so that the
// registers are defined when it returns.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&r)[16]) {
    uint32_t u[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
        "[%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) r[i] = __uint_as_float(u[i]);
}

// As tmem_ld16, 8 columns.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&r)[8]) {
    uint32_t u[8];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) r[i] = __uint_as_float(u[i]);
}

// As tmem_ld16, 32 columns in one load.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&r)[32]) {
    uint32_t u[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(u[0]), "=r"(u[1]), "=r"(u[2]), "=r"(u[3]), "=r"(u[4]), "=r"(u[5]), "=r"(u[6]), "=r"(u[7]),
          "=r"(u[8]), "=r"(u[9]), "=r"(u[10]), "=r"(u[11]), "=r"(u[12]), "=r"(u[13]), "=r"(u[14]), "=r"(u[15]),
          "=r"(u[16]), "=r"(u[17]), "=r"(u[18]), "=r"(u[19]), "=r"(u[20]), "=r"(u[21]), "=r"(u[22]), "=r"(u[23]),
          "=r"(u[24]), "=r"(u[25]), "=r"(u[26]), "=r"(u[27]), "=r"(u[28]), "=r"(u[29]), "=r"(u[30]), "=r"(u[31])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = __uint_as_float(u[i]);
}

// NC (8, 16 or 32) consecutive columns.
template <int NC>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&r)[NC]) {
    static_assert(NC == 8 || NC == 16 || NC == 32, "8, 16 or 32 columns");
    if constexpr (NC == 8) tmem_ld8(taddr, r);
    else if constexpr (NC == 16) tmem_ld16(taddr, r);
    else tmem_ld32(taddr, r);
}

// Two loads of NC (8, 16 or 32) consecutive columns each (at a and b), both
// in flight together, one wait.
#define MGS_O8(x, o)                                                                                            \
    "=r"(x[o + 0]), "=r"(x[o + 1]), "=r"(x[o + 2]), "=r"(x[o + 3]), "=r"(x[o + 4]), "=r"(x[o + 5]),             \
        "=r"(x[o + 6]), "=r"(x[o + 7])
template <int NC>
__device__ __forceinline__ void tmem_ld_pair(uint32_t a, float (&va)[NC], uint32_t b, float (&vb)[NC]) {
    static_assert(NC == 8 || NC == 16 || NC == 32, "8, 16 or 32 columns");
    uint32_t u[NC], w[NC];
    if constexpr (NC == 8) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%16];\n\t"
            "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%8,%9,%10,%11,%12,%13,%14,%15}, [%17];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : MGS_O8(u, 0), MGS_O8(w, 0)
            : "r"(a), "r"(b)
            : "memory");
    } else if constexpr (NC == 16) {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
            "[%32];\n\t"
            "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,"
            "%31}, [%33];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : MGS_O8(u, 0), MGS_O8(u, 8), MGS_O8(w, 0), MGS_O8(w, 8)
            : "r"(a), "r"(b)
            : "memory");
    } else {
        asm volatile(
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
            "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
            "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,"
            "%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
            "tcgen05.wait::ld.sync.aligned;"
            : MGS_O8(u, 0), MGS_O8(u, 8), MGS_O8(u, 16), MGS_O8(u, 24), MGS_O8(w, 0), MGS_O8(w, 8),
              MGS_O8(w, 16), MGS_O8(w, 24)
            : "r"(a), "r"(b)
            : "memory");
    }
#pragma unroll
    for (int i = 0; i < NC; ++i) {
        va[i] = __uint_as_float(u[i]);
        vb[i] = __uint_as_float(w[i]);
    }
}
#undef MGS_O8

// 16 consecutive columns of the warp's 32 lanes from registers; waits for the
// store to complete.
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const float (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
        "r"(__float_as_uint(r[0])), "r"(__float_as_uint(r[1])), "r"(__float_as_uint(r[2])),
        "r"(__float_as_uint(r[3])), "r"(__float_as_uint(r[4])), "r"(__float_as_uint(r[5])),
        "r"(__float_as_uint(r[6])), "r"(__float_as_uint(r[7])), "r"(__float_as_uint(r[8])),
        "r"(__float_as_uint(r[9])), "r"(__float_as_uint(r[10])), "r"(__float_as_uint(r[11])),
        "r"(__float_as_uint(r[12])), "r"(__float_as_uint(r[13])), "r"(__float_as_uint(r[14])),
        "r"(__float_as_uint(r[15]))
        : "memory");
}

// Two runs of 32 consecutive columns (at ca and cb) of the warp's 32 lanes
// from registers, then one wait for both stores.
__device__ __forceinline__ void tmem_st32x2(uint32_t ca, const float (&a)[32], uint32_t cb, const float (&b)[32]) {
#define MGS_R32(x)                                                                                              \
    "r"(__float_as_uint(x[0])), "r"(__float_as_uint(x[1])), "r"(__float_as_uint(x[2])),                         \
        "r"(__float_as_uint(x[3])), "r"(__float_as_uint(x[4])), "r"(__float_as_uint(x[5])),                     \
        "r"(__float_as_uint(x[6])), "r"(__float_as_uint(x[7])), "r"(__float_as_uint(x[8])),                     \
        "r"(__float_as_uint(x[9])), "r"(__float_as_uint(x[10])), "r"(__float_as_uint(x[11])),                   \
        "r"(__float_as_uint(x[12])), "r"(__float_as_uint(x[13])), "r"(__float_as_uint(x[14])),                  \
        "r"(__float_as_uint(x[15])), "r"(__float_as_uint(x[16])), "r"(__float_as_uint(x[17])),                  \
        "r"(__float_as_uint(x[18])), "r"(__float_as_uint(x[19])), "r"(__float_as_uint(x[20])),                  \
        "r"(__float_as_uint(x[21])), "r"(__float_as_uint(x[22])), "r"(__float_as_uint(x[23])),                  \
        "r"(__float_as_uint(x[24])), "r"(__float_as_uint(x[25])), "r"(__float_as_uint(x[26])),                  \
        "r"(__float_as_uint(x[27])), "r"(__float_as_uint(x[28])), "r"(__float_as_uint(x[29])),                  \
        "r"(__float_as_uint(x[30])), "r"(__float_as_uint(x[31]))
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,"
        "%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33};\n\t"
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%1], {%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
        "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63,%64,%65};\n\t"
        "tcgen05.wait::st.sync.aligned;" ::"r"(ca),
        "r"(cb), MGS_R32(a), MGS_R32(b)
        : "memory");
#undef MGS_R32
}

// TMEM address of lane `lane0`, column `col` relative to an allocation base.
__device__ __forceinline__ uint32_t tmem_at(uint32_t base, int lane0, int col) {
    return base + (uint32_t(lane0) << 16) + uint32_t(col);
}

}  // namespace mgs
