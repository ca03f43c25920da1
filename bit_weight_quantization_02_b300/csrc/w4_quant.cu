// w4_quant.cu -- group-wise int4 quantize and dequantize kernels.
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
// gives the same code: t' = (w - o) * rcp_rn(s) differs from the correctly
// rounded quotient t by less than 2^-18 (|t| < 16: two roundings of 2^-24
// relative plus half an ulp of t), so rint(t') == rint(t) unless t' lies
// within 2^-16 of a half-integer; those weights (exact ties included) are
// divided exactly.
//
// Both kernels are HBM-bound streams: one thread owns 8 consecutive weights
// (one 16-byte load of bf16, one 4-byte store of codes); the g/8 threads of a
// group reduce min and max with xor shuffles.  Groups never straddle a warp
// (g/8 divides 32 and rows hold whole groups).
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {

constexpr float QUANT_EPS = 1e-6f;
constexpr int QUANT_THREADS = 256;

// Order-preserving signed key of two packed bf16 values: negative values get
// their magnitude bits flipped so that the signed 16-bit order of the keys is
// the numeric order, with -0.0 (key -1) below +0.0 (key 0).  The map is its
// own inverse.
__device__ __forceinline__ uint32_t bf16x2_order_key(uint32_t x) {
    const uint32_t sign = (x >> 15) & 0x00010001u;
    return x ^ (sign * 0x7FFFu);
}

template <int G>
__global__ void __launch_bounds__(QUANT_THREADS)
quantize_kernel(const uint4* __restrict__ W, int64_t n_chunks, uint32_t* __restrict__ Wq,
                uint16_t* __restrict__ scales, uint16_t* __restrict__ offsets) {
    constexpr int L = G / 8;  // threads per group
    const int64_t c = (int64_t)blockIdx.x * QUANT_THREADS + threadIdx.x;
    const bool active = c < n_chunks;
    const uint4 raw = active ? ldg_stream_v4(W + c) : make_uint4(0u, 0u, 0u, 0u);

    // min / max of the 8 values, on order keys, two lanes per 32-bit word
    uint32_t k0 = bf16x2_order_key(raw.x), k1 = bf16x2_order_key(raw.y);
    uint32_t k2 = bf16x2_order_key(raw.z), k3 = bf16x2_order_key(raw.w);
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
    float s32 = __fdiv_rn(__fsub_rn(mx, mn), 15.0f);
    s32 = (s32 < QUANT_EPS) ? QUANT_EPS : s32;
    const uint32_t s_bits = float_to_bf16_bits(s32);
    const float s = bf16_bits_to_float(s_bits);
    const float o = mn;

    const float rs = __frcp_rn(s);  // correctly rounded 1/s (s >= 1e-6, a normal bf16 value)
    const uint32_t words[4] = {raw.x, raw.y, raw.z, raw.w};
    uint32_t packed = 0;
#pragma unroll
    for (int e = 0; e < 8; ++e) {
        const uint32_t b = (e & 1) ? (words[e >> 1] >> 16) : (words[e >> 1] & 0xFFFFu);
        const float v = bf16_bits_to_float(b);
        const float d = __fsub_rn(v, o);
        float t = __fmul_rn(d, rs);
        if (fabsf(__fsub_rn(t - floorf(t), 0.5f)) < 1.52587890625e-05f)  // within 2^-16 of x.5
            t = __fdiv_rn(d, s);
        int q = __float2int_rn(t);
        q = min(max(q, 0), 15);
        packed |= (uint32_t)q << (4 * e);
    }
    if (active) {
        Wq[c] = packed;
        if ((threadIdx.x & (L - 1)) == 0) {
            const int64_t grp = c / L;
            scales[grp] = (uint16_t)s_bits;
            offsets[grp] = (uint16_t)mn_bits;
        }
    }
}

template <int G>
__global__ void __launch_bounds__(QUANT_THREADS)
dequantize_kernel(const uint32_t* __restrict__ Wq, const uint16_t* __restrict__ scales,
                  const uint16_t* __restrict__ offsets, int64_t n_chunks, uint4* __restrict__ W_out) {
    constexpr int L = G / 8;
    const int64_t c = (int64_t)blockIdx.x * QUANT_THREADS + threadIdx.x;
    if (c >= n_chunks) return;
    const uint32_t packed = ldg_nc_u32(Wq + c);
    const int64_t grp = c / L;
    const float s = bf16_bits_to_float(ldg_nc_u16(scales + grp));
    const float o = bf16_bits_to_float(ldg_nc_u16(offsets + grp));
    uint32_t out[4];
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const float q0 = (float)((packed >> (4 * e)) & 15u);
        const float q1 = (float)((packed >> (4 * e + 4)) & 15u);
        const uint32_t lo = float_to_bf16_bits(__fadd_rn(__fmul_rn(q0, s), o));
        const uint32_t hi = float_to_bf16_bits(__fadd_rn(__fmul_rn(q1, s), o));
        out[e >> 1] = lo | (hi << 16);
    }
    W_out[c] = make_uint4(out[0], out[1], out[2], out[3]);
}

cudaError_t launch_quantize(const uint16_t* W, int64_t N, int64_t K, int g, uint8_t* Wq, uint16_t* scales,
                            uint16_t* offsets, cudaStream_t stream) {
    const int64_t n_chunks = N * K / 8;
    const int64_t blocks = (n_chunks + QUANT_THREADS - 1) / QUANT_THREADS;
    const dim3 grid((unsigned)blocks);
    const uint4* w = reinterpret_cast<const uint4*>(W);
    uint32_t* q = reinterpret_cast<uint32_t*>(Wq);
    switch (g) {
        case 32: quantize_kernel<32><<<grid, QUANT_THREADS, 0, stream>>>(w, n_chunks, q, scales, offsets); break;
        case 64: quantize_kernel<64><<<grid, QUANT_THREADS, 0, stream>>>(w, n_chunks, q, scales, offsets); break;
        default: quantize_kernel<128><<<grid, QUANT_THREADS, 0, stream>>>(w, n_chunks, q, scales, offsets); break;
    }
    return cudaGetLastError();
}

cudaError_t launch_dequantize(const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N,
                              int64_t K, int g, uint16_t* W_out, cudaStream_t stream) {
    const int64_t n_chunks = N * K / 8;
    const int64_t blocks = (n_chunks + QUANT_THREADS - 1) / QUANT_THREADS;
    const dim3 grid((unsigned)blocks);
    const uint32_t* q = reinterpret_cast<const uint32_t*>(Wq);
    uint4* out = reinterpret_cast<uint4*>(W_out);
    switch (g) {
        case 32: dequantize_kernel<32><<<grid, QUANT_THREADS, 0, stream>>>(q, scales, offsets, n_chunks, out); break;
        case 64: dequantize_kernel<64><<<grid, QUANT_THREADS, 0, stream>>>(q, scales, offsets, n_chunks, out); break;
        default: dequantize_kernel<128><<<grid, QUANT_THREADS, 0, stream>>>(q, scales, offsets, n_chunks, out); break;
    }
    return cudaGetLastError();
}

}  // namespace w4
