// w4_mma.cuh -- mma.sync helpers of the stream-K decode kernel (w4_stream.cu):
// the dequantize-and-multiply step on packed codes, the raw-code step of the
// one-token slice-sum path, shared-memory loads, the X-slot swizzle and bf16
// unpacking.
#pragma once

#include "w4_device.cuh"

namespace w4 {

__device__ __forceinline__ void mma_bf16_16816_st(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                                  uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}
__device__ __forceinline__ uint4 lds128_st(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds_u16_st(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
// (w & mask) | magic with both constants in registers (one LOP3, no constant rematerialization)
__device__ __forceinline__ uint32_t lop_and_or(uint32_t w, uint32_t mask, uint32_t magic) {
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0xEA;" : "=r"(r) : "r"(w), "r"(mask), "r"(magic));
    return r;
}
__device__ __forceinline__ void cp_async_4(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ int st_x_slot(int c) { return c ^ (((c >> 3) & 1) << 1); }

// One MMA step from packed codes: nibble pairs (SH, SH+4) and (SH+1... ) of the
// 32-bit code words of rows a and b become the four A-fragment registers
// (128+q via LOP3, exact -128, one bf16 FMA with scale and offset) inside the
// same asm block as the mma.sync, so they are born in the operand registers.
// SH = 0 takes nibbles (0,4) and (1,5); SH = 8 takes (2,6) and (3,7).
template <int SH>
__device__ __forceinline__ void dq_mma(float (&c)[4], uint32_t wa, uint32_t wb, uint32_t sa2, uint32_t oa2,
                                       uint32_t sb2, uint32_t ob2, uint32_t x0, uint32_t x1, uint32_t cm,
                                       uint32_t cg, uint32_t c128) {
    asm volatile(
        "{\n\t.reg .b32 a0, a1, b0, b1, t;\n\t"
        "shr.b32 t, %4, %15;\n\t"
        "lop3.b32 a0, t, %12, %13, 0xEA;\n\t"
        "shr.b32 t, %4, %16;\n\t"
        "lop3.b32 a1, t, %12, %13, 0xEA;\n\t"
        "shr.b32 t, %5, %15;\n\t"
        "lop3.b32 b0, t, %12, %13, 0xEA;\n\t"
        "shr.b32 t, %5, %16;\n\t"
        "lop3.b32 b1, t, %12, %13, 0xEA;\n\t"
        "sub.rn.bf16x2 a0, a0, %14;\n\t"
        "sub.rn.bf16x2 a1, a1, %14;\n\t"
        "sub.rn.bf16x2 b0, b0, %14;\n\t"
        "sub.rn.bf16x2 b1, b1, %14;\n\t"
        "fma.rn.bf16x2 a0, a0, %6, %7;\n\t"
        "fma.rn.bf16x2 a1, a1, %6, %7;\n\t"
        "fma.rn.bf16x2 b0, b0, %8, %9;\n\t"
        "fma.rn.bf16x2 b1, b1, %8, %9;\n\t"
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {a0,b0,a1,b1}, {%10,%11}, "
        "{%0,%1,%2,%3};\n\t}"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(wa), "r"(wb), "r"(sa2), "r"(oa2), "r"(sb2), "r"(ob2), "r"(x0), "r"(x1), "r"(cm), "r"(cg),
          "r"(c128), "n"(SH), "n"(SH + 4));
}

// One MMA step on raw codes (the one-token path): A = 128 + q straight from
// LOP3, B = X or zero per lane.  ZC starts from a zero accumulator.
template <int SH, bool ZC>
__device__ __forceinline__ void raw_mma(float (&c)[4], uint32_t wa, uint32_t wb, uint32_t x0, uint32_t x1,
                                        uint32_t cm, uint32_t cg) {
    if constexpr (ZC) {
        asm volatile(
            "{\n\t.reg .b32 a0, a1, b0, b1, t;\n\t"
            "shr.b32 t, %4, %11;\n\t"
            "lop3.b32 a0, t, %8, %9, 0xEA;\n\t"
            "shr.b32 t, %4, %12;\n\t"
            "lop3.b32 a1, t, %8, %9, 0xEA;\n\t"
            "shr.b32 t, %5, %11;\n\t"
            "lop3.b32 b0, t, %8, %9, 0xEA;\n\t"
            "shr.b32 t, %5, %12;\n\t"
            "lop3.b32 b1, t, %8, %9, 0xEA;\n\t"
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {a0,b0,a1,b1}, {%6,%7}, "
            "{%10,%10,%10,%10};\n\t}"
            : "=f"(c[0]), "=f"(c[1]), "=f"(c[2]), "=f"(c[3])
            : "r"(wa), "r"(wb), "r"(x0), "r"(x1), "r"(cm), "r"(cg), "f"(0.0f), "n"(SH), "n"(SH + 4));
    } else {
        asm volatile(
            "{\n\t.reg .b32 a0, a1, b0, b1, t;\n\t"
            "shr.b32 t, %4, %10;\n\t"
            "lop3.b32 a0, t, %8, %9, 0xEA;\n\t"
            "shr.b32 t, %4, %11;\n\t"
            "lop3.b32 a1, t, %8, %9, 0xEA;\n\t"
            "shr.b32 t, %5, %10;\n\t"
            "lop3.b32 b0, t, %8, %9, 0xEA;\n\t"
            "shr.b32 t, %5, %11;\n\t"
            "lop3.b32 b1, t, %8, %9, 0xEA;\n\t"
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {a0,b0,a1,b1}, {%6,%7}, "
            "{%0,%1,%2,%3};\n\t}"
            : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
            : "r"(wa), "r"(wb), "r"(x0), "r"(x1), "r"(cm), "r"(cg), "n"(SH), "n"(SH + 4));
    }
}
__device__ __forceinline__ uint32_t lds_u32_st(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
// sum of eight bf16 values in fp32
__device__ __forceinline__ float bf16x8_sum(uint4 v) {
    const float a = bf16_lo(v.x) + bf16_hi(v.x), b = bf16_lo(v.y) + bf16_hi(v.y);
    const float c = bf16_lo(v.z) + bf16_hi(v.z), d = bf16_lo(v.w) + bf16_hi(v.w);
    return (a + b) + (c + d);
}
// MX: token capacity (1, 2, 4; X staged in shared memory).
// RT: 16-row tiles per unit, 1, or 2 for one token on large problems (the X
// staging, slice sums and ring work of a unit then serve 32 weight rows).
}  // namespace w4
