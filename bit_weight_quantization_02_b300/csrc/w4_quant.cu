// w4_quant.cu -- group-wise int4 quantize and dequantize kernels (and the
// same affine path with 2- and 8-bit codes).
//
// Method: affine group projection with an offset and torch.round (half to
// even) integer mapping, Optimum Quanto "Design overview / Tensors"; groups
// of g = 32/64/128 consecutive k of one output row (same page, "Design
// overview / Modules"; torchao README "Quick start").  Per group:
//   s32 = (max - min)/15, clamped below at 1e-6;  s = bf16(s32);  o = min;
//   q = clamp(rne((w - o)/s), 0, 15);  w' = bf16(q*s + o).
// Every floating-point step is one IEEE fp32 operation with round-to-nearest
// (__fsub_rn / __fdiv_rn / __fmul_rn / __fadd_rn: no contraction, no
// approximate division), so the results are bit-exact and independent of the
// launch shape.  The per-weight quotient (w - o)/s takes a fast route that
// gives the same code: t' = (w - o) * r, with r the hardware reciprocal of s
// (relative error below 2^-22), differs from the correctly rounded quotient t
// by less than 2^-18 (|t| < 16: 2^-22 + 2^-24 relative, plus half an ulp of
// t), so rint(t') == rint(t) unless t' lies within 2^-16 of a half-integer;
// those chunks (exact ties included) are divided exactly.  The scale's
// division by 15 is a correctly rounded multiply-and-correct (div15_rn).
//
// At b = 2 or 8 bits (Optimum Quanto's int2 / int8 weights; torchao's int8
// weight-only per group of 128) the same steps run with L = 2^b - 1 levels:
// s32 = (max - min)/L by IEEE division, q = clamp(rne((w - o)/s), 0, L), and
// 8/b codes a byte, the lowest k in the lowest bits.  The quotient bound grows
// with L (|t| < 257 at 8 bits: |t' - t| < 2^-13 + 2^-15 + 2^-16), so 8-bit
// codes take the exact division within 2^-12 of a half-integer.  At 8 bits
// the bf16 rounding of the scale (up to 2^-8 relative) can put the group
// maximum as high as L + 1, so the clamp there is real.
//
// Both kernels are HBM-bound streams: a thread owns chunks of 8 consecutive
// weights (one 16-byte load of bf16, one b-byte store of codes each), four at a
// time with all loads issued first; the g/8 threads of a group reduce min and
// max with xor shuffles.  Groups never straddle a warp (g/8 divides 32 and rows
// hold whole groups).
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {

constexpr float QUANT_EPS = 1e-6f;
constexpr int QUANT_THREADS = 256;

// packed fp32 pairs (element 0 in the low half); each element is one IEEE fp32
// operation with round-to-nearest
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float f32x2_lo(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float f32x2_hi(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }
__device__ __forceinline__ uint64_t f32x2_sub(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_mul(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ uint64_t f32x2_add(uint64_t a, uint64_t b) {
    uint64_t r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}

// Order-preserving signed key of two packed bf16 values: negative values get
// their magnitude bits flipped so that the signed 16-bit order of the keys is
// the numeric order, with -0.0 (key -1) below +0.0 (key 0).  The map is its
// own inverse.
__device__ __forceinline__ uint32_t bf16x2_order_key(uint32_t x) {
    uint32_t neg;  // 0xFFFF in each lane whose sign bit is set (prmt selectors 9 / 11: byte 1 / 3, sign replicated)
    asm("prmt.b32 %0, %1, 0, 0xBB99;" : "=r"(neg) : "r"(x));
    return x ^ (neg & 0x7FFF7FFFu);
}
// (mx - mn) / 15 correctly rounded, for 0 <= x < 2^128: q0 = x * RN(1/15), then
// one correction from the exact residual x - 15 q0 (Markstein's method for
// division by a constant).  Checked against IEEE division for every finite
// non-negative fp32 x: identical.
__device__ __forceinline__ float div15_rn(float x) {
    constexpr float c = 1.0f / 15.0f;
    const float q0 = __fmul_rn(x, c);
    return __fmaf_rn(__fmaf_rn(-q0, 15.0f, x), c, q0);
}
__device__ __forceinline__ float rcp_approx(float x) {
    float r;
    asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}

// The 8 codes of one chunk as stored: B = 2: 16 bits, 4: 32 bits, 8: 64 bits.
template <int B>
struct ChunkCodes;
template <>
struct ChunkCodes<2> {
    using type = uint16_t;
};
template <>
struct ChunkCodes<4> {
    using type = uint32_t;
};
template <>
struct ChunkCodes<8> {
    using type = uint2;
};

// Quantize one 8-weight chunk (chunk index c; `valid` false past the end, where
// the lanes still take part in the group's shuffles) into B-bit codes.
template <int G, int B>
__device__ __forceinline__ void quantize_chunk(const uint4 raw, int64_t c, bool valid, int lane,
                                               typename ChunkCodes<B>::type* __restrict__ Wq,
                                               uint16_t* __restrict__ scales, uint16_t* __restrict__ offsets) {
    constexpr int LV = (1 << B) - 1;  // levels
    constexpr int L = G / 8;  // threads per group
    // min / max of the 8 values, on order keys, two lanes per 32-bit word
    const uint32_t k0 = bf16x2_order_key(raw.x), k1 = bf16x2_order_key(raw.y);
    const uint32_t k2 = bf16x2_order_key(raw.z), k3 = bf16x2_order_key(raw.w);
    uint32_t kmin = __vmins2(__vmins2(k0, k1), __vmins2(k2, k3));
    uint32_t kmax = __vmaxs2(__vmaxs2(k0, k1), __vmaxs2(k2, k3));
#pragma unroll
    for (int off = 1; off < L; off <<= 1) {
        kmin = __vmins2(kmin, __shfl_xor_sync(0xffffffffu, kmin, off));
        kmax = __vmaxs2(kmax, __shfl_xor_sync(0xffffffffu, kmax, off));
    }
    // fold the two 16-bit lanes
    kmin = __vmins2(kmin, kmin >> 16) & 0xFFFFu;
    kmax = __vmaxs2(kmax, kmax >> 16) & 0xFFFFu;
    const uint32_t mn_bits = bf16x2_order_key(kmin) & 0xFFFFu;
    const uint32_t mx_bits = bf16x2_order_key(kmax) & 0xFFFFu;

    const float mn = bf16_bits_to_float(mn_bits);
    const float mx = bf16_bits_to_float(mx_bits);
    float s32 = B == 4 ? div15_rn(__fsub_rn(mx, mn)) : __fdiv_rn(__fsub_rn(mx, mn), (float)LV);
    s32 = (s32 < QUANT_EPS) ? QUANT_EPS : s32;
    const uint32_t s_bits = float_to_bf16_bits(s32);
    const float s = bf16_bits_to_float(s_bits);
    const float o = mn;

    const float rs = rcp_approx(s);  // 1/s within 2^-22 relative (s >= 1e-6, a normal bf16 value)
    // Two weights per instruction (packed fp32 pairs, each element one IEEE fp32 operation with
    // round-to-nearest, as the scalar ops): d = w - o (>= 0: o is the group minimum), t = d * rs,
    // m = t + 2^23 (its mantissa is rint(t), half to even, for 0 <= t < 2^22), r = m - 2^23,
    // and t - r exactly.
    const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
    const uint64_t o2 = pack_f32x2(o, o), rs2 = pack_f32x2(rs, rs), mg2 = pack_f32x2(8388608.0f, 8388608.0f);
    // |t' - rint(t')| above this: within 2^-16 (8 bits: 2^-12) of a half-integer
    constexpr float NEAR = B == 8 ? 0.499755859375f : 0.4999847412109375f;
    uint32_t bytes[4], qv[8];
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        // (w[2j], w[2j+1]) as fp32: the low bf16 shifted up, the high one masked in place
        const uint64_t w2 = pack_f32x2(__uint_as_float(words[j] << 16), __uint_as_float(words[j] & 0xFFFF0000u));
        const uint64_t d2 = f32x2_sub(w2, o2);
        const uint64_t t2 = f32x2_mul(d2, rs2);
        const uint64_t m2 = f32x2_add(t2, mg2);
        const uint64_t e2 = f32x2_sub(t2, f32x2_sub(m2, mg2));  // t' - rint(t'), exact
        float mlo = f32x2_lo(m2), mhi = f32x2_hi(m2);
        // near a half-integer t' may round differently from the correctly rounded quotient:
        // divide exactly (only the lanes and weights that need it)
        if (fabsf(f32x2_lo(e2)) > NEAR) mlo = __fadd_rn(__fdiv_rn(f32x2_lo(d2), s), 8388608.0f);
        if (fabsf(f32x2_hi(e2)) > NEAR) mhi = __fadd_rn(__fdiv_rn(f32x2_hi(d2), s), 8388608.0f);
        // the low mantissa bits of m are the code (rint(t) <= L at 2 and 4 bits: t <= L / (1 - 2^-8)
        // < L + 1/2 because s rounds Delta/L to bf16, so the clamp to [0, L] never changes it);
        // 4 bits: byte j = q[2j] | q[2j+1] << 4
        if constexpr (B == 4) {
            bytes[j] = __float_as_uint(mlo) + (__float_as_uint(mhi) << 4);
        } else if constexpr (B == 2) {
            qv[2 * j] = __float_as_uint(mlo) & 3u;
            qv[2 * j + 1] = __float_as_uint(mhi) & 3u;
        } else {  // 8 bits: rint(t) can reach 256 (clamped to 255)
            qv[2 * j] = min(__float_as_uint(mlo) & 0x1FFu, 255u);
            qv[2 * j + 1] = min(__float_as_uint(mhi) & 0x1FFu, 255u);
        }
    }
    typename ChunkCodes<B>::type packed;
    if constexpr (B == 4) {
        packed = __byte_perm(__byte_perm(bytes[0], bytes[1], 0x0040), __byte_perm(bytes[2], bytes[3], 0x0040), 0x5410);
    } else if constexpr (B == 2) {
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) v |= qv[i] << (2 * i);
        packed = (uint16_t)v;
    } else {
        packed.x = __byte_perm(__byte_perm(qv[0], qv[1], 0x0040), __byte_perm(qv[2], qv[3], 0x0040), 0x5410);
        packed.y = __byte_perm(__byte_perm(qv[4], qv[5], 0x0040), __byte_perm(qv[6], qv[7], 0x0040), 0x5410);
    }
    if (valid) {
        Wq[c] = packed;
        if ((lane & (L - 1)) == 0) {
            const int64_t grp = c / L;
            scales[grp] = (uint16_t)s_bits;
            offsets[grp] = (uint16_t)mn_bits;
        }
    }
}

// A warp takes QUANT_UNROLL rows of 32 consecutive chunks at a time and issues
// all their loads before any arithmetic (more bytes in flight per thread); a
// persistent grid strides over warps.
constexpr int QUANT_UNROLL = 4;
constexpr int QUANT_WARPS = QUANT_THREADS / 32;

template <int G, int B>
__global__ void __launch_bounds__(QUANT_THREADS)
quantize_kernel(const uint4* __restrict__ W, int64_t n_chunks, typename ChunkCodes<B>::type* __restrict__ Wq,
                uint16_t* __restrict__ scales, uint16_t* __restrict__ offsets) {
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * QUANT_WARPS;
    for (int64_t w = (int64_t)blockIdx.x * QUANT_WARPS + (threadIdx.x >> 5); w * (32 * QUANT_UNROLL) < n_chunks;
         w += nwarps) {
        const int64_t c0 = w * (32 * QUANT_UNROLL) + lane;
        uint4 raw[QUANT_UNROLL];
#pragma unroll
        for (int u = 0; u < QUANT_UNROLL; ++u) {
            const int64_t c = c0 + 32 * u;
            raw[u] = c < n_chunks ? ldg_stream_v4(W + c) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < QUANT_UNROLL; ++u)
            quantize_chunk<G, B>(raw[u], c0 + 32 * u, c0 + 32 * u < n_chunks, lane, Wq, scales, offsets);
    }
}

__device__ __forceinline__ uint64_t chunk_bits(uint16_t v) { return v; }
__device__ __forceinline__ uint64_t chunk_bits(uint32_t v) { return v; }
__device__ __forceinline__ uint64_t chunk_bits(uint2 v) { return (uint64_t)v.x | ((uint64_t)v.y << 32); }

template <int G, int B>
__global__ void __launch_bounds__(QUANT_THREADS)
dequantize_kernel(const typename ChunkCodes<B>::type* __restrict__ Wq, const uint16_t* __restrict__ scales,
                  const uint16_t* __restrict__ offsets, int64_t n_chunks, uint4* __restrict__ W_out) {
    constexpr int L = G / 8;
    constexpr uint32_t MASK = (1u << B) - 1u;
    const int lane = threadIdx.x & 31;
    const int64_t nwarps = (int64_t)gridDim.x * QUANT_WARPS;
    for (int64_t w = (int64_t)blockIdx.x * QUANT_WARPS + (threadIdx.x >> 5); w * (32 * QUANT_UNROLL) < n_chunks;
         w += nwarps) {
        const int64_t c0 = w * (32 * QUANT_UNROLL) + lane;
        uint64_t packed[QUANT_UNROLL];
        uint32_t sb[QUANT_UNROLL], ob[QUANT_UNROLL];
#pragma unroll
        for (int u = 0; u < QUANT_UNROLL; ++u) {
            const int64_t c = c0 + 32 * u;
            const bool in = c < n_chunks;
            packed[u] = in ? chunk_bits(__ldg(Wq + c)) : 0u;
            sb[u] = in ? ldg_nc_u16(scales + c / L) : 0u;
            ob[u] = in ? ldg_nc_u16(offsets + c / L) : 0u;
        }
#pragma unroll
        for (int u = 0; u < QUANT_UNROLL; ++u) {
            const int64_t c = c0 + 32 * u;
            if (c >= n_chunks) continue;
            const float s = bf16_bits_to_float(sb[u]), o = bf16_bits_to_float(ob[u]);
            uint32_t out[4];
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const float q0 = (float)((uint32_t)(packed[u] >> (B * e)) & MASK);
                const float q1 = (float)((uint32_t)(packed[u] >> (B * e + B)) & MASK);
                const uint32_t lo = float_to_bf16_bits(__fadd_rn(__fmul_rn(q0, s), o));
                const uint32_t hi = float_to_bf16_bits(__fadd_rn(__fmul_rn(q1, s), o));
                out[e >> 1] = lo | (hi << 16);
            }
            W_out[c] = make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
}

// one wave of resident blocks at most (a second, partial wave would run alone
// at the end), and no more warps than rows of chunks
static cudaError_t quant_grid(const void* kernel, int64_t n_chunks, unsigned* grid) {
    int sms = 0, per_sm = 0;
    const cudaError_t e = resident_blocks(kernel, QUANT_THREADS, 0, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t want = (n_chunks + 32 * QUANT_UNROLL * QUANT_WARPS - 1) / (32 * QUANT_UNROLL * QUANT_WARPS);
    const int64_t cap = (int64_t)sms * per_sm;
    *grid = (unsigned)(want < cap ? want : cap);
    return cudaSuccess;
}

template <int B>
static cudaError_t launch_quantize_b(const uint16_t* W, int64_t N, int64_t K, int g, uint8_t* Wq, uint16_t* scales,
                                     uint16_t* offsets, cudaStream_t stream) {
    using CT = typename ChunkCodes<B>::type;
    const int64_t n_chunks = N * K / 8;
    const uint4* w = reinterpret_cast<const uint4*>(W);
    CT* q = reinterpret_cast<CT*>(Wq);
    auto kern = g == 32 ? quantize_kernel<32, B> : g == 64 ? quantize_kernel<64, B> : quantize_kernel<128, B>;
    unsigned grid = 0;
    const cudaError_t e = quant_grid(reinterpret_cast<const void*>(kern), n_chunks, &grid);
    if (e != cudaSuccess) return e;
    kern<<<grid, QUANT_THREADS, 0, stream>>>(w, n_chunks, q, scales, offsets);
    return cudaGetLastError();
}

template <int B>
static cudaError_t launch_dequantize_b(const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N,
                                       int64_t K, int g, uint16_t* W_out, cudaStream_t stream) {
    using CT = typename ChunkCodes<B>::type;
    const int64_t n_chunks = N * K / 8;
    const CT* q = reinterpret_cast<const CT*>(Wq);
    uint4* out = reinterpret_cast<uint4*>(W_out);
    auto kern = g == 32 ? dequantize_kernel<32, B> : g == 64 ? dequantize_kernel<64, B> : dequantize_kernel<128, B>;
    unsigned grid = 0;
    const cudaError_t e = quant_grid(reinterpret_cast<const void*>(kern), n_chunks, &grid);
    if (e != cudaSuccess) return e;
    kern<<<grid, QUANT_THREADS, 0, stream>>>(q, scales, offsets, n_chunks, out);
    return cudaGetLastError();
}

cudaError_t launch_quantize(const uint16_t* W, int64_t N, int64_t K, int g, int bits, uint8_t* Wq, uint16_t* scales,
                            uint16_t* offsets, cudaStream_t stream) {
    if (bits == 2) return launch_quantize_b<2>(W, N, K, g, Wq, scales, offsets, stream);
    if (bits == 8) return launch_quantize_b<8>(W, N, K, g, Wq, scales, offsets, stream);
    return launch_quantize_b<4>(W, N, K, g, Wq, scales, offsets, stream);
}

cudaError_t launch_dequantize(const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N,
                              int64_t K, int g, int bits, uint16_t* W_out, cudaStream_t stream) {
    if (bits == 2) return launch_dequantize_b<2>(Wq, scales, offsets, N, K, g, W_out, stream);
    if (bits == 8) return launch_dequantize_b<8>(Wq, scales, offsets, N, K, g, W_out, stream);
    return launch_dequantize_b<4>(Wq, scales, offsets, N, K, g, W_out, stream);
}

}  // namespace w4
