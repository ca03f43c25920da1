// w4_tc.cuh -- tcgen05 helpers shared by the tensor-core kernels (w4_gemm.cu,
// w4_tcdec.cu): the shared-memory descriptor of a 128-byte-swizzled K-major
// operand, the UMMA with its A operand in tensor memory, tensor-memory stores,
// the 4-bit dequantization of eight codes, and shared-memory loads.
#pragma once

#include "w4_device.cuh"

namespace w4 {

// Shared-memory matrix descriptor for a K-major operand stored as rows of
// 64 bf16 (128 bytes) with the 128-byte swizzle, 8-row atoms 1024 bytes
// apart: start address >> 4 (bits 0-13), leading-byte offset 16 B (unused
// for swizzled K-major, bits 16-29), stride-byte offset 1024 B (bits 32-45),
// descriptor version 1 (bits 46-47), swizzle mode 2 = 128 B (bits 61-63).
__device__ __forceinline__ uint64_t sw128_kmajor_desc(uint32_t saddr) {
    return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(16 >> 4) << 16) | ((uint64_t)(1024 >> 4) << 32) |
           (1ull << 46) | (2ull << 61);
}

// D[tmem] (+)= A[tmem] . B[smem desc]^T, kind::f16: the A operand (M=128 rows
// x K=16) is read from tensor memory, two bf16 of consecutive k a column.
__device__ __forceinline__ void umma_bf16_tmem_a(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc, uint32_t idesc,
                                                 uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "r"(a_tmem), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// 16 consecutive 32-bit columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_st_16cols(uint32_t taddr, const uint4& a, const uint4& b, const uint4& c,
                                               const uint4& d) {
    asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                 :: "r"(taddr), "r"(a.x), "r"(a.y), "r"(a.z), "r"(a.w), "r"(b.x), "r"(b.y), "r"(b.z), "r"(b.w),
                    "r"(c.x), "r"(c.y), "r"(c.z), "r"(c.w), "r"(d.x), "r"(d.y), "r"(d.z), "r"(d.w)
                 : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}

// Eight codes of one 32-bit word (k0..k7, k0 in the low nibble) -> eight bf16
// w' = q*s + o in k order: LOP3 gives the pairs (128+q_i, 128+q_{i+4}), an exact
// subtract of 128 and one bf16 FMA with the (s,s) and (o,o) pairs dequantize
// them, four PRMTs restore the order.
__device__ __forceinline__ uint4 dequant8(uint32_t w, uint32_t s2, uint32_t o2, uint32_t cm, uint32_t cg) {
    uint4 r;
    asm("{\n\t.reg .b32 t, p0, p1, p2, p3;\n\t"
        "lop3.b32 p0, %4, %7, %8, 0xEA;\n\t"
        "shr.b32 t, %4, 4;\n\t"
        "lop3.b32 p1, t, %7, %8, 0xEA;\n\t"
        "shr.b32 t, %4, 8;\n\t"
        "lop3.b32 p2, t, %7, %8, 0xEA;\n\t"
        "shr.b32 t, %4, 12;\n\t"
        "lop3.b32 p3, t, %7, %8, 0xEA;\n\t"
        "sub.rn.bf16x2 p0, p0, %8;\n\t"
        "sub.rn.bf16x2 p1, p1, %8;\n\t"
        "sub.rn.bf16x2 p2, p2, %8;\n\t"
        "sub.rn.bf16x2 p3, p3, %8;\n\t"
        "fma.rn.bf16x2 p0, p0, %5, %6;\n\t"
        "fma.rn.bf16x2 p1, p1, %5, %6;\n\t"
        "fma.rn.bf16x2 p2, p2, %5, %6;\n\t"
        "fma.rn.bf16x2 p3, p3, %5, %6;\n\t"
        "prmt.b32 %0, p0, p1, 0x5410;\n\t"
        "prmt.b32 %1, p2, p3, 0x5410;\n\t"
        "prmt.b32 %2, p0, p1, 0x7632;\n\t"
        "prmt.b32 %3, p2, p3, 0x7632;\n\t}"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
        : "r"(w), "r"(s2), "r"(o2), "r"(cm), "r"(cg));
    return r;
}
__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint32_t pick_word(const uint4& v, int i) {
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

}  // namespace w4
