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
// gives the same code: the exact product p = (w - o) * r (inside one fused
// multiply-add with 2^23, which rounds it to an integer), with r the hardware
// reciprocal of s (relative error below 2^-22), differs from the correctly
// rounded quotient t by less than 2^-18 + 2^-21 (|t| < 16: 2^-22 relative,
// plus half an ulp of t), so rint(p) == rint(t) unless p lies within 2^-16 of
// a half-integer; those weights (exact ties included) are divided exactly.
// The scale's division by 15 is a correctly rounded multiply-and-correct
// (div15_rn).
//
// At b = 2 or 8 bits (Optimum Quanto's int2 / int8 weights; torchao's int8
// weight-only per group of 128) the same steps run with L = 2^b - 1 levels:
// s32 = (max - min)/L by IEEE division, q = clamp(rne((w - o)/s), 0, L), and
// 8/b codes a byte, the lowest k in the lowest bits.  The quotient bound grows
// with L (|t| < 257 at 8 bits: |p - t| < 257 * 2^-22 + 2^-16 < 2^-12), so
// 8-bit codes take the exact division within 2^-12 of a half-integer.  At 8 bits
// the bf16 rounding of the scale (up to 2^-8 relative) can put the group
// maximum as high as L + 1, so the clamp there is real.
//
// Both kernels are HBM-bound streams.  Quantize: a lane owns 64 consecutive
// weights (two groups at g = 32, one at 64, half of one at 128), staged through
// shared memory by asynchronous copies; the group min / max is a native bf16x2
// min / max, redone on order keys (-0.0 below +0.0) when it lands on a zero.
// Dequantize: a thread owns chunks of 8 weights (one b-byte load of codes, one
// 16-byte store of bf16), four at a time with all loads issued first.
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

__device__ __forceinline__ uint64_t f32x2_fma(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ uint4 lds_v4(uint32_t a) {
    uint4 r;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "r"(a));
    return r;
}
// 16 bytes global -> shared, asynchronous, L2 only; src_bytes = 0 fills the 16 bytes with zeros
__device__ __forceinline__ void cp_async_16(uint32_t dst, const void* src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() {
    asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

__device__ __forceinline__ uint32_t bf16x2_min(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("min.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}
__device__ __forceinline__ uint32_t bf16x2_max(uint32_t a, uint32_t b) {
    uint32_t r;
    asm("max.bf16x2 %0, %1, %2;" : "=r"(r) : "r"(a), "r"(b));
    return r;
}

// One warp's tile: 32 segments of 64 consecutive weights (128 bytes of bf16), one per lane.  A
// segment holds two groups at g = 32, one at g = 64 and half of one at g = 128 (lanes 2i and
// 2i + 1 share it and swap their min / max once), so a group's min / max, scale and reciprocal
// are computed by the lanes that hold it, not by every lane of a chunk-per-lane mapping.  The
// warp copies the tile from HBM with coalesced 16-byte asynchronous copies (lane l takes pieces
// l, l + 32, ...) into one of its two shared-memory buffers, with a 16-byte gap after each
// segment, and each lane reads its segment back from there: with that gap, the 8 lanes of a
// 16-byte access phase hit distinct banks on both sides.  The next tile's copies are in flight
// while a tile is quantized.
constexpr int QSEG_W = 64;                          // weights per segment
constexpr int QSEG_PIECES = QSEG_W / 8;             // 16-byte pieces per segment
constexpr int QSEG_PITCH = 2 * QSEG_W + 16;         // bytes per segment in shared memory
constexpr int QTILE_PIECES = 32 * QSEG_PIECES;      // per warp tile
constexpr int QUANT_WARPS = QUANT_THREADS / 32;
constexpr int QBUF = 32 * QSEG_PITCH;                     // one tile buffer
constexpr int QSTAGES = 2;                                // tile buffers per warp
constexpr int QUANT_SMEM = QUANT_WARPS * QSTAGES * QBUF;
constexpr int QUANT_MIN_BLOCKS = QSTAGES == 2 ? 3 : 2;    // blocks per SM the registers are capped for

// The codes of 8 weights from the bits of m = rint(t) + 2^23 (the code is in the low mantissa
// bits: rint(t) <= L at 2 and 4 bits, as t <= L / (1 - 2^-8) < L + 1/2 because s rounds Delta/L
// to bf16, so the clamp to [0, L] never binds there), packed as stored: 4 bits: byte k = q[2k] |
// q[2k+1] << 4 in x; 2 bits: 16 bits in x; 8 bits: x and y.
template <int B>
__device__ __forceinline__ uint2 pack_piece(const uint32_t (&m)[8]) {
    if constexpr (B == 4) {
        uint32_t bytes[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) bytes[k] = m[2 * k] + (m[2 * k + 1] << 4);
        return make_uint2(
            __byte_perm(__byte_perm(bytes[0], bytes[1], 0x0040), __byte_perm(bytes[2], bytes[3], 0x0040), 0x5410), 0u);
    } else if constexpr (B == 2) {
        uint32_t v = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) v |= (m[i] & 3u) << (2 * i);
        return make_uint2(v, 0u);
    } else {  // 8 bits: rint(t) can reach 256 (clamped to 255)
        uint32_t qv[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) qv[i] = min(m[i] & 0x1FFu, 255u);
        return make_uint2(__byte_perm(__byte_perm(qv[0], qv[1], 0x0040), __byte_perm(qv[2], qv[3], 0x0040), 0x5410),
                          __byte_perm(__byte_perm(qv[4], qv[5], 0x0040), __byte_perm(qv[6], qv[7], 0x0040), 0x5410));
    }
}


// Exact min / max keys of n pieces at `ga` (order keys: -0.0 below +0.0), folded to 16 bits and
// sign-extended in the low halves.  Used when the fast bf16x2 min / max landed on a zero, whose
// sign they do not order.
__device__ __forceinline__ void minmax_keys(uint32_t ga, int n, uint32_t& kmin, uint32_t& kmax) {
    kmin = 0x7FFF7FFFu;
    kmax = 0x80008000u;
    for (int c = 0; c < n; ++c) {
        const uint4 r = lds_v4(ga + 16 * c);
        const uint32_t k0 = bf16x2_order_key(r.x), k1 = bf16x2_order_key(r.y);
        const uint32_t k2 = bf16x2_order_key(r.z), k3 = bf16x2_order_key(r.w);
        kmin = __vmins2(kmin, __vmins2(__vmins2(k0, k1), __vmins2(k2, k3)));
        kmax = __vmaxs2(kmax, __vmaxs2(__vmaxs2(k0, k1), __vmaxs2(k2, k3)));
    }
    kmin = __vmins2(kmin, kmin >> 16) & 0xFFFFu;
    kmax = __vmaxs2(kmax, kmax >> 16) & 0xFFFFu;
}

// Quantize one segment (QSEG_PIECES pieces at `ga` in shared memory) of tile-local segment index
// `seg`: its groups' codes to `codes` (64 * B / 8 bytes), scales and offsets to `scales` /
// `offsets` (the segment's first group).  `nvalid` = the segment's groups that exist (past the
// last group nothing is stored; at g = 32 the last segment may hold one).
template <int G, int B>
__device__ __forceinline__ void quantize_segment(uint32_t ga, int lane, int nvalid, uint8_t* __restrict__ codes,
                                                 uint16_t* __restrict__ scales, uint16_t* __restrict__ offsets) {
    constexpr int LV = (1 << B) - 1;                 // levels
    constexpr int GPS = G <= QSEG_W ? QSEG_W / G : 1;  // groups per segment (g = 128: half a group)
    constexpr int PPG = G <= QSEG_W ? G / 8 : QSEG_PIECES;  // pieces of a group in this segment
    // pass 1: min / max of each group, packed (min in the low half, max in the high half)
    uint32_t mm[GPS];
#pragma unroll
    for (int j = 0; j < GPS; ++j) {
        uint32_t lo = 0, hi = 0;
#pragma unroll
        for (int c = 0; c < PPG; ++c) {
            const uint4 r = lds_v4(ga + 16 * (j * PPG + c));
            const uint32_t a = bf16x2_min(bf16x2_min(r.x, r.y), bf16x2_min(r.z, r.w));
            const uint32_t b = bf16x2_max(bf16x2_max(r.x, r.y), bf16x2_max(r.z, r.w));
            lo = c == 0 ? a : bf16x2_min(lo, a);
            hi = c == 0 ? b : bf16x2_max(hi, b);
        }
        // fold the two halves: (min, max) of the group in the low / high half
        const uint32_t x = __byte_perm(lo, hi, 0x5410), y = __byte_perm(lo, hi, 0x7632);
        mm[j] = __byte_perm(bf16x2_min(x, y), bf16x2_max(x, y), 0x7610);
        if constexpr (G > QSEG_W) {  // the other half of the group is on the partner lane
            const uint32_t p = __shfl_xor_sync(0xffffffffu, mm[j], 1);
            mm[j] = __byte_perm(bf16x2_min(mm[j], p), bf16x2_max(mm[j], p), 0x7610);
        }
    }
    // a zero min or max may carry either sign: redo those groups on order keys (rare)
    bool zero = false;
#pragma unroll
    for (int j = 0; j < GPS; ++j) zero |= (mm[j] & 0x7FFFu) == 0 || (mm[j] & 0x7FFF0000u) == 0;
    if (__any_sync(0xffffffffu, zero)) {
#pragma unroll
        for (int j = 0; j < GPS; ++j) {
            uint32_t kmin, kmax;
            minmax_keys(ga + 16 * j * PPG, PPG, kmin, kmax);
            if constexpr (G > QSEG_W) {
                kmin = __vmins2(kmin, __shfl_xor_sync(0xffffffffu, kmin, 1)) & 0xFFFFu;
                kmax = __vmaxs2(kmax, __shfl_xor_sync(0xffffffffu, kmax, 1)) & 0xFFFFu;
            }
            mm[j] = (bf16x2_order_key(kmin) & 0xFFFFu) | (bf16x2_order_key(kmax) << 16);
        }
    }

    constexpr int WORDS = QSEG_W * B / 32;  // 32-bit code words of the segment
    uint32_t outw[WORDS];
    uint32_t sbits[GPS];
#pragma unroll
    for (int j = 0; j < GPS; ++j) {
        const uint32_t mn_bits = mm[j] & 0xFFFFu, mx_bits = mm[j] >> 16;
        const float mn = bf16_bits_to_float(mn_bits);
        const float mx = bf16_bits_to_float(mx_bits);
        float s32 = B == 4 ? div15_rn(__fsub_rn(mx, mn)) : __fdiv_rn(__fsub_rn(mx, mn), (float)LV);
        s32 = (s32 < QUANT_EPS) ? QUANT_EPS : s32;
        sbits[j] = float_to_bf16_bits(s32);
        const float s = bf16_bits_to_float(sbits[j]);
        const float o = mn;
        const float rs = rcp_approx(s);  // 1/s within 2^-22 relative (s >= 1e-6, a normal bf16 value)
        // Two weights per instruction (packed fp32 pairs, each element one IEEE fp32 operation
        // with round-to-nearest): d = w - o (>= 0: o is the group minimum), m = d * rs + 2^23 with
        // one rounding (its mantissa is rint(d * rs), half to even, as 0 <= d * rs < 2^22), and
        // e = d * rs - (m - 2^23), the distance of the exact product from that integer.
        const uint64_t o2 = pack_f32x2(o, o), rs2 = pack_f32x2(rs, rs), mg2 = pack_f32x2(8388608.0f, 8388608.0f);
        // |e| above this: within 2^-16 (8 bits: 2^-12) of a half-integer
        constexpr float NEAR = B == 8 ? 0.499755859375f : 0.4999847412109375f;
#pragma unroll
        for (int c = 0; c < PPG; ++c) {
            const int pc = j * PPG + c;  // piece of the segment
            const uint4 r = lds_v4(ga + 16 * pc);
            const uint32_t words[4] = {r.x, r.y, r.z, r.w};
            uint32_t m[8];
            float e[8], d[8];
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                // (w[2k], w[2k+1]) as fp32: the low bf16 shifted up, the high one masked in place
                const uint64_t w2 =
                    pack_f32x2(__uint_as_float(words[k] << 16), __uint_as_float(words[k] & 0xFFFF0000u));
                const uint64_t d2 = f32x2_sub(w2, o2);
                const uint64_t m2 = f32x2_fma(d2, rs2, mg2);
                const uint64_t e2 = f32x2_fma(d2, rs2, f32x2_sub(mg2, m2));
                m[2 * k] = __float_as_uint(f32x2_lo(m2));
                m[2 * k + 1] = __float_as_uint(f32x2_hi(m2));
                e[2 * k] = f32x2_lo(e2), e[2 * k + 1] = f32x2_hi(e2);
                d[2 * k] = f32x2_lo(d2), d[2 * k + 1] = f32x2_hi(d2);
            }
            // near a half-integer the product may round differently from the correctly rounded
            // quotient: divide exactly (only the weights that need it; rare)
            bool near = false;
#pragma unroll
            for (int i = 0; i < 8; ++i) near |= fabsf(e[i]) > NEAR;
            if (near) {
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    if (fabsf(e[i]) > NEAR) m[i] = __float_as_uint(__fadd_rn(__fdiv_rn(d[i], s), 8388608.0f));
            }
            const uint2 pk = pack_piece<B>(m);
            if constexpr (B == 4) {
                outw[pc] = pk.x;
            } else if constexpr (B == 2) {
                if (pc % 2 == 0)
                    outw[pc / 2] = pk.x;
                else
                    outw[pc / 2] |= pk.x << 16;
            } else {
                outw[2 * pc] = pk.x;
                outw[2 * pc + 1] = pk.y;
            }
        }
    }
    if (nvalid <= 0) return;
    constexpr int GROUP_CODE_BYTES = G * B / 8 < QSEG_W * B / 8 ? G * B / 8 : QSEG_W * B / 8;
    if (nvalid == GPS) {
#pragma unroll
        for (int k = 0; k < WORDS / 4; ++k)
            *reinterpret_cast<uint4*>(codes + 16 * k) = make_uint4(outw[4 * k], outw[4 * k + 1], outw[4 * k + 2], outw[4 * k + 3]);
    } else if constexpr (GPS > 1) {  // g = 32: only the first group of the last segment exists
        if constexpr (GROUP_CODE_BYTES >= 16) {
#pragma unroll
            for (int k = 0; k < GROUP_CODE_BYTES / 16; ++k)
                *reinterpret_cast<uint4*>(codes + 16 * k) = make_uint4(outw[4 * k], outw[4 * k + 1], outw[4 * k + 2], outw[4 * k + 3]);
        } else {
            *reinterpret_cast<uint2*>(codes) = make_uint2(outw[0], outw[1]);
        }
    }
    if constexpr (G > QSEG_W) {  // one scale per pair of lanes: the even lane stores it
        if ((lane & 1) == 0) {
            *scales = (uint16_t)sbits[0];
            *offsets = (uint16_t)(mm[0] & 0xFFFFu);
        }
    } else if constexpr (GPS == 2) {
        if (nvalid == 2) {  // two neighbouring groups: one 4-byte store each
            *reinterpret_cast<uint32_t*>(scales) = sbits[0] | (sbits[1] << 16);
            *reinterpret_cast<uint32_t*>(offsets) = __byte_perm(mm[0], mm[1], 0x5410);
        } else {
            *scales = (uint16_t)sbits[0];
            *offsets = (uint16_t)(mm[0] & 0xFFFFu);
        }
    } else {
        *scales = (uint16_t)sbits[0];
        *offsets = (uint16_t)(mm[0] & 0xFFFFu);
    }
}

// A persistent grid of one wave strides over warp tiles; each warp keeps its next tile's copies in
// flight (QSTAGES - 1 tiles ahead) while it quantizes the current one.
template <int G, int B>
__global__ void __launch_bounds__(QUANT_THREADS, QUANT_MIN_BLOCKS)
quantize_kernel(const uint4* __restrict__ W, int64_t n_groups, uint8_t* __restrict__ Wq,
                uint16_t* __restrict__ scales, uint16_t* __restrict__ offsets) {
    constexpr int GPS = G <= QSEG_W ? QSEG_W / G : 1;
    extern __shared__ __align__(16) unsigned char q_smem[];
    const int lane = threadIdx.x & 31;
    const uint32_t area = smem_u32(q_smem) + (threadIdx.x >> 5) * (QSTAGES * QBUF);
    // piece lane + 32u of the tile is piece (lane % 8) of segment 4u + lane / 8
    const uint32_t cp_off = (lane >> 3) * QSEG_PITCH + 16 * (lane & 7);
    const int64_t n_pieces = n_groups * (G / 8);
    const int64_t n_segs = (n_pieces + QSEG_PIECES - 1) / QSEG_PIECES;
    const int64_t nwarps = (int64_t)gridDim.x * QUANT_WARPS;
    int64_t t = (int64_t)blockIdx.x * QUANT_WARPS + (threadIdx.x >> 5);
    auto copy_tile = [&](int64_t tile, uint32_t buf) {
        if (tile * 32 < n_segs) {
#pragma unroll
            for (int u = 0; u < QSEG_PIECES; ++u) {
                const int64_t p = tile * QTILE_PIECES + lane + 32 * u;
                cp_async_16(buf + cp_off + u * (4 * QSEG_PITCH), W + (p < n_pieces ? p : 0), p < n_pieces ? 16u : 0u);
            }
        }
        cp_async_commit();  // possibly empty: one group per tile slot keeps the wait count uniform
    };
#pragma unroll
    for (int k = 0; k < QSTAGES - 1; ++k) copy_tile(t + k * nwarps, area + k * QBUF);
    for (int i = 0; t * 32 < n_segs; t += nwarps, ++i) {
        const uint32_t buf = area + (i % QSTAGES) * QBUF;
        copy_tile(t + (QSTAGES - 1) * nwarps, area + ((i + QSTAGES - 1) % QSTAGES) * QBUF);
        cp_async_wait<QSTAGES - 1>();  // this lane's copies of tile t are done
        __syncwarp();       // and every lane's
        const int64_t seg = t * 32 + lane;
        const int64_t first = seg * QSEG_W / G;  // the segment's first group
        int nvalid = 0;
        if (seg < n_segs) nvalid = (int)(n_groups - first < GPS ? n_groups - first : GPS);
        quantize_segment<G, B>(buf + lane * QSEG_PITCH, lane, nvalid, Wq + seg * (QSEG_W * B / 8), scales + first,
                               offsets + first);
        __syncwarp();  // every lane is done reading buf before its next refill
    }
}

// The dequantize kernel: a warp takes QUANT_UNROLL rows of 32 consecutive chunks at a time and
// issues all their loads before any arithmetic.
constexpr int QUANT_UNROLL = 4;

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
// at the end), and no more warps than work units (warp tiles or rows of chunks)
static cudaError_t quant_grid(const void* kernel, size_t smem, int64_t units, unsigned* grid) {
    int sms = 0, per_sm = 0;
    const cudaError_t e = resident_blocks(kernel, QUANT_THREADS, smem, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t want = (units + QUANT_WARPS - 1) / QUANT_WARPS;
    const int64_t cap = (int64_t)sms * per_sm;
    *grid = (unsigned)(want < cap ? want : cap);
    return cudaSuccess;
}

template <int G, int B>
static cudaError_t launch_quantize_gb(const uint16_t* W, int64_t N, int64_t K, uint8_t* Wq, uint16_t* scales,
                                      uint16_t* offsets, cudaStream_t stream) {
    const int64_t n_groups = N * K / G;
    if (n_groups == 0) return cudaSuccess;
    const void* kern = reinterpret_cast<const void*>(quantize_kernel<G, B>);
    constexpr int SMEM = QUANT_SMEM;
    cudaError_t e = ensure_kernel_attrs(kern, SMEM, false);
    if (e != cudaSuccess) return e;
    unsigned grid = 0;
    const int64_t n_segs = (n_groups * G + QSEG_W - 1) / QSEG_W;
    if ((e = quant_grid(kern, SMEM, (n_segs + 31) / 32, &grid)) != cudaSuccess) return e;
    quantize_kernel<G, B><<<grid, QUANT_THREADS, SMEM, stream>>>(reinterpret_cast<const uint4*>(W), n_groups, Wq,
                                                                 scales, offsets);
    return cudaGetLastError();
}

template <int B>
static cudaError_t launch_quantize_b(const uint16_t* W, int64_t N, int64_t K, int g, uint8_t* Wq, uint16_t* scales,
                                     uint16_t* offsets, cudaStream_t stream) {
    if (g == 32) return launch_quantize_gb<32, B>(W, N, K, Wq, scales, offsets, stream);
    if (g == 64) return launch_quantize_gb<64, B>(W, N, K, Wq, scales, offsets, stream);
    return launch_quantize_gb<128, B>(W, N, K, Wq, scales, offsets, stream);
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
    const cudaError_t e =
        quant_grid(reinterpret_cast<const void*>(kern), 0, (n_chunks + 32 * QUANT_UNROLL - 1) / (32 * QUANT_UNROLL), &grid);
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
