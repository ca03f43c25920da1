// w4_batch.cu -- persistent stream-K bf16 x int4 linear for batched decode
// (5 <= M <= 32 tokens) on the canonical layout; also the decode linear
// (1 <= M <= 32) of 2- and 8-bit codes.
//
// Y[m,n] = sum_k X[m,k] * w'[n,k], w' = bf16(q*s + o), fp32 accumulation
// (Optimum Quanto: bf16 x int4 matmul, result accumulated at higher precision,
// "Pitfalls when quantizing activations").
//
// With 16 or 32 tokens the tokens' activations are as many bytes per unit as
// the codes, and every 16-row tile of weights needs all of them.  So a unit
// here is 64 weight rows x 256 k, one 16-row tile per warp of a 4-warp block,
// and the block stages the unit's X slice once, by TMA, for its four warps:
//  * Ring of 2-3 stages per block; a stage holds the unit's codes (one
//    64 x 128-byte TMA box, 128-byte swizzle), its X slice (four 64-k boxes of
//    the padded token rows, 128-byte swizzle, rows past M zero) and its scales
//    and offsets (two TMA boxes, or 4-byte cp.async by every thread).  Codes
//    and qparams of the first units are requested before the
//    programmatic-dependent-launch wait, their X after it.
//  * B fragments come from the staged X with ldmatrix (one x4 load = two
//    token groups' fragments of one 16-k step).  A fragment k index i is the
//    natural k 16s + i, so each lane dequantizes the code byte holding its
//    pair (k, k+1): prmt puts the byte and the byte shifted by a nibble side
//    by side, then LOP3 magic (128 + q), an exact subtract and one bf16 FMA
//    with the group's scale and offset, and one mma.m16n8k16 per group of 8
//    tokens uses that fragment.
//  * 2- and 8-bit codes (Optimum Quanto's int2 / int8 weights) use the same
//    unit with 4 KB / 16 KB of codes (one 64-byte-swizzled box / two
//    128-byte-swizzled boxes).  2 bits: each lane extracts the nibble holding
//    its pair and spreads its two codes into the two bf16 halves (one
//    multiply by 0x4001), then the LOP3 magic, subtract and FMA as above.
//    8 bits: a bf16 of 128 + q cannot hold q up to 255, so each code goes
//    through fp32 (prmt into 2^23 + q, exact subtract, FMA with s and o,
//    round to bf16): w' is then bf16(fp32(q s + o)), the dequantized weight
//    bit for bit.
//  * One token at 2 or 8 bits: seven of the MMA's eight token columns would
//    be zero, so they carry the unit's eight 32-k slices instead (as in the
//    4-bit one-token stream kernel): the ldmatrix row of column c points at
//    the token's X only while the MMA works on slice c, at a zero row
//    otherwise, and A is the raw code (128 + q at 2 bits, q at 8 bits, both
//    exact in bf16) with no per-weight subtract or FMA.  Each unit then adds
//    s (D - 128 xs) + o xs (8 bits: s D + o xs) per row and slice in fp32,
//    D the slice's MMA sum and xs the slice's sum of X.
//  * The (row group, k) units are cut into equal contiguous block ranges; a
//    row group split between blocks is finished by the block holding its
//    first unit: each of its warps adds the partial sums that warp w of every
//    later sharer left in its workspace slot (split_publish / split_collect,
//    w4_device.cuh), deterministic and without atomics.
#include "w4_device.cuh"
#include "w4_internal.h"

#include <algorithm>
#include <cuda.h>

namespace w4 {

constexpr int BT_WARPS = 4;       // 16-row tiles per unit, one per warp
constexpr int BT_THREADS = BT_WARPS * 32;
constexpr int BT_UK = 256;        // k per unit
constexpr int BT_ROWS = 16 * BT_WARPS;
constexpr uint64_t BT_WAIT_LIMIT_NS = 2000000000ull;
__device__ unsigned int g_batch_fault;

struct BatchArgs {
    const uint16_t* scales;  // the cp.async qparam route
    const uint16_t* offsets;
    uint16_t* Y;
    Epilogue ep;           // bias and output scale, applied before the rounding
    uint64_t* ws;            // split-tile slots, one per warp, zero between calls
    int M, N, K;
    int nkc;                 // units per row group = ceil(K / 256)
    long long units;         // row groups x nkc
    int ctas;                // blocks with work
};

// Shared-memory layout of one ring stage (every piece 1024-byte aligned for the swizzled boxes).
template <int G, int MT, int B, bool QT>
struct BatchLayout {
    static constexpr int MP = 8 * MT;                       // token rows staged (M padded)
    static constexpr int CROW = BT_UK * B / 8;              // bytes of one row of a unit's codes
    static constexpr int CODES = BT_ROWS * CROW;            // 64 rows x 256 k of codes
    static constexpr int XBOX = MP * 128;                   // one 64-k box of X
    static constexpr int XBYTES = 4 * XBOX;
    static constexpr int QROW = (BT_UK / G) * 2;            // bytes of one row of one qparam array (a unit's groups)
    // staged row pitch: by TMA a box of 8 groups (16 bytes) per row holding the unit's groups
    // (g = 64 / 128: also its neighbours'), by cp.async just the unit's groups
    static constexpr int SQROW = QT ? 16 : QROW;
    static constexpr int QBYTES = 2 * BT_ROWS * SQROW;      // scales, then offsets
    static constexpr int STAGE = (CODES + XBYTES + QBYTES + 1023) / 1024 * 1024;
    static constexpr int DEPTH = MT == 4 ? 2 : 3;
    static constexpr int SCRATCH = BT_WARPS * 16 * MP * 4;  // owners' own sums, per warp 16 x M fp32
    static constexpr int SMEM = DEPTH * STAGE + SCRATCH + 8 * DEPTH + 1024;  // + alignment slack
};

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t& r0, uint32_t& r1, uint32_t& r2, uint32_t& r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}
__device__ __forceinline__ void ldsm_x2(uint32_t addr, uint32_t& r0, uint32_t& r1) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x2.shared.b16 {%0,%1}, [%2];" : "=r"(r0), "=r"(r1) : "r"(addr));
}
__device__ __forceinline__ uint4 lds128_b(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds16_b(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ void cp_async_4b(uint32_t dst, const void* src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_arrive_noinc_b(uint32_t bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" :: "r"(bar) : "memory");
}
// The pair (k, k+1) held by byte `sel & 3` of a code word w, as a bf16 pair
// w' = bf16(q*s + o): prmt puts the byte (low nibble: k) and the same byte of
// w >> 4 (its high nibble: k+1) in the two 16-bit halves, LOP3 makes 128 + q,
// subtract 128 (exact), one FMA with (s, s) and (o, o).
__device__ __forceinline__ uint32_t nat_pair(uint32_t w, uint32_t sel, uint32_t s2, uint32_t o2, uint32_t cm,
                                             uint32_t cg) {
    uint32_t r;
    asm("{\n\t.reg .b32 t, u;\n\t"
        "shr.b32 u, %1, 4;\n\t"
        "prmt.b32 t, %1, u, %2;\n\t"
        "lop3.b32 t, t, %5, %6, 0xEA;\n\t"
        "sub.rn.bf16x2 t, t, %6;\n\t"
        "fma.rn.bf16x2 %0, t, %3, %4;\n\t}"
        : "=r"(r)
        : "r"(w), "r"(sel), "r"(s2), "r"(o2), "r"(cm), "r"(cg));
    return r;
}
__device__ __forceinline__ void mma_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 8-bit codes: bytes sel0 and sel0 + 1 of w (k, k+1) as a bf16 pair
// bf16(fp32(q*s + o)): prmt builds 2^23 + q, an exact subtract gives q, one
// fp32 FMA (q*s is exact), one rounding to bf16.
__device__ __forceinline__ uint32_t pair8(uint32_t w, uint32_t sel0, float s, float o, uint32_t mg) {
    uint32_t lo, hi, r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(w), "r"(mg), "r"(sel0));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(w), "r"(mg), "r"(sel0 + 1u));
    const float a = __fmaf_rn(__fsub_rn(__uint_as_float(lo), 8388608.0f), s, o);
    const float b = __fmaf_rn(__fsub_rn(__uint_as_float(hi), 8388608.0f), s, o);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}
// 2-bit codes: a lane's two pairs of one 16-code word as raw bf16 pairs, (128 + q_2t, 128 + q_2t+1) and
// (128 + q_8+2t, 128 + q_9+2t), t = sh / 4: one shift brings both nibbles down (bits 0-3 and 16-19), LOP3
// magic takes codes (2t, 8+2t) and, after a shift by 2, (2t+1, 9+2t), two PRMTs pair them in k order.
__device__ __forceinline__ void raw2x2(uint32_t w, uint32_t sh, uint32_t cg, uint32_t& lo, uint32_t& hi) {
    asm("{\n\t.reg .b32 t, p, q;\n\t"
        "shr.b32 t, %2, %3;\n\t"
        "lop3.b32 p, t, 0x00030003, %4, 0xEA;\n\t"
        "shr.b32 t, t, 2;\n\t"
        "lop3.b32 q, t, 0x00030003, %4, 0xEA;\n\t"
        "prmt.b32 %0, p, q, 0x5410;\n\t"
        "prmt.b32 %1, p, q, 0x7632;\n\t}"
        : "=r"(lo), "=r"(hi)
        : "r"(w), "r"(sh), "r"(cg));
}
// (128 + q) pair -> bf16 w' pair: exact subtract of 128, one bf16 FMA with (s, s) and (o, o)
__device__ __forceinline__ uint32_t deq_raw(uint32_t r, uint32_t s2, uint32_t o2, uint32_t cg) {
    uint32_t v;
    asm("{\n\t.reg .b32 t;\n\t"
        "sub.rn.bf16x2 t, %1, %4;\n\t"
        "fma.rn.bf16x2 %0, t, %2, %3;\n\t}"
        : "=r"(v)
        : "r"(r), "r"(s2), "r"(o2), "r"(cg));
    return v;
}
// 8-bit codes, one-token path: bytes sel0 and sel0 + 1 of w as the bf16 pair (q_k, q_k+1), exact.
__device__ __forceinline__ uint32_t raw8(uint32_t w, uint32_t sel0, uint32_t mg) {
    uint32_t lo, hi, r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(lo) : "r"(w), "r"(mg), "r"(sel0));
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(hi) : "r"(w), "r"(mg), "r"(sel0 + 1u));
    const float a = __fsub_rn(__uint_as_float(lo), 8388608.0f), b = __fsub_rn(__uint_as_float(hi), 8388608.0f);
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(b), "f"(a));
    return r;
}
__device__ __forceinline__ float bf16lo_b(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16hi_b(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }
__device__ __forceinline__ uint2 lds64_b(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t lds32_b(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}

// ONE: the one-token slice-sum path (M == 1, 2- and 8-bit codes).
template <int G, int MT, bool QT, int B, bool ONE>
__global__ void __launch_bounds__(BT_THREADS, MT == 1 ? 4 : 3)
batch_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_x,
             const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_o, const BatchArgs p) {
    static_assert(B == 2 || B == 4 || B == 8, "code width");
    static_assert(!ONE || (MT == 1 && B != 4), "the one-token path is for 2- and 8-bit codes");
    using L = BatchLayout<G, MT, B, QT>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    constexpr int PPR = L::QROW / 4;               // 4-byte qparam pieces per row and array
    constexpr int PIECES = 2 * BT_ROWS * PPR;      // per unit
    constexpr int PPT = (PIECES + BT_THREADS - 1) / BT_THREADS;
    constexpr int NE = 4 * MT;                     // split-slot words per lane (16 M / 32)

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tq = lane & 3;
    const int cta = blockIdx.x;

    griddep_launch_dependents();
    if (cta >= p.ctas) return;
    const long long u0 = p.units * cta / p.ctas;
    const long long u1 = p.units * (cta + 1) / p.ctas;
    if (u0 >= u1) return;
    const int nunits = (int)(u1 - u0);

    const uint32_t sbase = smem_u32(smem);
    float* scr = reinterpret_cast<float*>(smem + L::DEPTH * L::STAGE) + warp * 16 * L::MP;
    const uint32_t bars = smem_u32(smem + L::DEPTH * L::STAGE + L::SCRATCH);
    const int ng = p.K / G;

    if (threadIdx.x == 0) {  // arrivals per fill: thread 0's arrive (+ every thread's cp.async arrive)
        for (int d = 0; d < L::DEPTH; ++d) mbar_init(bars + 8 * d, QT ? 1 : 1 + BT_THREADS);
        mbar_fence_init();
    }
    __syncthreads();

    // this thread's qparam pieces (4 bytes each): fixed (array, row, piece) for every unit
    int prow[PPT], pcol[PPT];
    uint32_t pdst[PPT];
    const uint16_t* pbase[PPT];
#pragma unroll
    for (int q = 0; q < PPT; ++q) {
        const int i = threadIdx.x + BT_THREADS * q;
        const int arr = (i < PIECES) ? i / (PIECES / 2) : 0, rem = (i < PIECES) ? i % (PIECES / 2) : 0;
        prow[q] = rem / PPR;
        pcol[q] = 2 * (rem % PPR);
        pdst[q] = (uint32_t)(L::CODES + L::XBYTES + arr * BT_ROWS * L::SQROW + prow[q] * L::SQROW + 4 * (rem % PPR));
        pbase[q] = arr ? p.offsets : p.scales;
    }
    // codes and qparams of unit u into stage d (thread 0's TMA; every thread's cp.async when !QT)
    auto issue_w = [&](long long u, int d) {
        const int grp = (int)(u / p.nkc), kc = (int)(u - (long long)grp * p.nkc);
        const int row0 = grp * BT_ROWS, k = kc * BT_UK;
        const uint32_t st = sbase + d * L::STAGE, bar = bars + 8 * d;
        if (threadIdx.x == 0) {
            if (B == 8) {  // two boxes of 128 k
                tma_load_2d(st, &tm_w, bar, k, row0);
                tma_load_2d(st + L::CODES / 2, &tm_w, bar, k + 128, row0);
            } else {
                tma_load_2d(st, &tm_w, bar, k * B / 8, row0);
            }
            if (QT) {  // the 8-group box holding the unit's groups (its first group rounded down to 8)
                tma_load_2d(st + L::CODES + L::XBYTES, &tm_s, bar, (k / G) & ~7, row0);
                tma_load_2d(st + L::CODES + L::XBYTES + BT_ROWS * L::SQROW, &tm_o, bar, (k / G) & ~7, row0);
            }
        }
        if (!QT) {
            const bool edge = (row0 + BT_ROWS > p.N) || (k + BT_UK > p.K);
#pragma unroll
            for (int q = 0; q < PPT; ++q) {
                if (PIECES % BT_THREADS == 0 || (int)threadIdx.x + BT_THREADS * q < PIECES) {
                    int n = row0 + prow[q], j = k / G + pcol[q];
                    if (edge) {
                        n = min(n, p.N - 1);  // rows past N: any finite qparams (their codes are 0)
                        j = min(j, ng - 2);   // groups past K: likewise (X is 0 there)
                    }
                    cp_async_4b(st + pdst[q], pbase[q] + (int64_t)n * ng + j);
                }
            }
            cp_async_arrive_noinc_b(bar);
        }
    };
    // thread 0: the X slice of unit u into stage d (four 64-k boxes of the padded token rows)
    auto issue_x = [&](long long u, int d) {
        const int kc = (int)(u % p.nkc);
        const uint32_t st = sbase + d * L::STAGE + L::CODES, bar = bars + 8 * d;
#pragma unroll
        for (int b = 0; b < 4; ++b) tma_load_2d(st + b * L::XBOX, &tm_x, bar, kc * BT_UK + 64 * b, 0);
    };

    const int depth = nunits < L::DEPTH ? nunits : L::DEPTH;
    for (int d = 0; d < depth; ++d) {  // weights never depend on the previous kernel
        if (threadIdx.x == 0) mbar_expect_tx(bars + 8 * d, L::CODES + (QT ? L::QBYTES : 0));
        issue_w(u0 + d, d);
    }
    // activations may come from the previous kernel: wait for it, then their boxes (and the arrive)
    griddep_wait();
    if (threadIdx.x == 0)
        for (int d = 0; d < depth; ++d) {
            mbar_arrive_expect_tx(bars + 8 * d, L::XBYTES);
            issue_x(u0 + d, d);
        }

    uint32_t cm, cg;  // constants pinned in registers: nibble mask, bf16 128.0 pair (magic and bias)
    asm volatile("mov.b32 %0, %1;" : "=r"(cm) : "r"(0x000F000Fu));
    asm volatile("mov.b32 %0, %1;" : "=r"(cg) : "r"(0x43004300u));
    const uint32_t sel = (uint32_t)tq | ((uint32_t)(4 + tq) << 8);  // prmt: byte tq of w, byte tq of w >> 4
    const uint32_t sh2 = 4u * (uint32_t)tq;                          // 2 bits: nibble of the pair (2tq, 2tq+1)
    const uint32_t w8 = 4u * (uint32_t)(tq >> 1);                    // 8 bits: word of bytes 2tq, 2tq+1 in a chunk
    const uint32_t sel8 = 0x7540u | (2u * (uint32_t)(tq & 1));       // prmt: that byte, then 0x00, 0x00, 0x4B
    uint32_t mg;                                                     // 2^23 as fp32 bits
    asm volatile("mov.b32 %0, %1;" : "=r"(mg) : "r"(0x4B000000u));
    // ldmatrix row addresses of this lane: matrix i = lane / 8 (token group 2tp + i / 2, chunk c0 + i % 2),
    // row r = lane % 8 (token 8 (2tp + i / 2) + r); the 128-byte swizzle XORs the chunk with r
    const int lr = lane & 7, li = lane >> 3;
    const uint32_t xo0 = (uint32_t)(li & 1) << 4, xo1 = 128u + ((uint32_t)((li & 1) ^ 1) << 4);  // one-token path

    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    float ya = 0.f, yb = 0.f;  // one-token path: rows gid, gid + 8 over this lane's slices of the tile so far
    const long long g0 = u0 / p.nkc;
    int grp = (int)g0, kc = (int)(u0 - g0 * p.nkc), kc_first = kc;
    bool owner_split = false, ok = true;
    int d = 0;
    uint32_t phase = 0;
    long long next = u0 + depth;  // next unit to request

    for (int it = 0; it < nunits; ++it) {
        ok = mbar_wait_bounded(bars + 8 * d, phase, nullptr, &g_batch_fault, 1u, BT_WAIT_LIMIT_NS) && ok;
        const uint32_t st = sbase + d * L::STAGE;
        // code row gid of this warp's tile (8 bits: in the first of the two 128-k boxes)
        const uint32_t crow = st + (16 * warp + gid) * (uint32_t)(B == 8 ? 128 : L::CROW);
        // scales of row gid of this warp's tile, from the unit's first group (TMA box: byte 2 (first group % 8))
        const uint32_t qa = st + L::CODES + L::XBYTES + (16 * warp + gid) * L::SQROW +
                            (QT ? (uint32_t)(((kc * (BT_UK / G)) & 7) * 2) : 0u);
        const uint32_t xst = st + L::CODES;
        float dacc[4] = {0.f, 0.f, 0.f, 0.f};  // one-token path: D[row gid / gid+8][slice 2tq / 2tq+1]
        float xs0 = 0.f, xs1 = 0.f;            // one-token path: sums of X over slices 2tq, 2tq+1
        if constexpr (ONE) {  // lane l sums k 8l .. 8l+7 of the token (row 0 of the boxes: no swizzle shift)
            const uint4 xv = lds128_b(xst + (uint32_t)(lane >> 3) * L::XBOX + ((uint32_t)(lane & 7) << 4));
            float xsl = ((bf16lo_b(xv.x) + bf16hi_b(xv.x)) + (bf16lo_b(xv.y) + bf16hi_b(xv.y))) +
                        ((bf16lo_b(xv.z) + bf16hi_b(xv.z)) + (bf16lo_b(xv.w) + bf16hi_b(xv.w)));
            xsl += __shfl_xor_sync(0xffffffffu, xsl, 1);
            xsl += __shfl_xor_sync(0xffffffffu, xsl, 2);  // lanes 4c .. 4c+3: slice c
            xs0 = __shfl_sync(0xffffffffu, xsl, 8 * tq);
            xs1 = __shfl_sync(0xffffffffu, xsl, 8 * tq + 4);
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {  // 32 k of codes per row, two 16-k steps
            const uint32_t jq = (uint32_t)(((32 * q) / G) * 2);  // the piece's group, bytes into the row
            uint32_t sa2, oa2, sb2, ob2;  // (s,s), (o,o) bf16 pairs of rows gid and gid + 8 (2 and 4 bits)
            float saf, oaf, sbf, obf;     // the same as fp32 (8 bits)
            if constexpr (!ONE) {
                const uint32_t sa = lds16_b(qa + jq), oa = lds16_b(qa + BT_ROWS * L::SQROW + jq);
                const uint32_t sb = lds16_b(qa + 8 * L::SQROW + jq), ob = lds16_b(qa + 8 * L::SQROW + BT_ROWS * L::SQROW + jq);
                sa2 = __byte_perm(sa, 0, 0x1010), oa2 = __byte_perm(oa, 0, 0x1010);
                sb2 = __byte_perm(sb, 0, 0x1010), ob2 = __byte_perm(ob, 0, 0x1010);
                saf = __uint_as_float(sa << 16), oaf = __uint_as_float(oa << 16);
                sbf = __uint_as_float(sb << 16), obf = __uint_as_float(ob << 16);
            }
            uint32_t wa4[4], wb4[4];  // 4 bits: the row's 32 k as four words (8 k each)
            uint32_t wa2[2], wb2[2];  // 2 bits: two words (16 k each)
            if constexpr (B == 4) {
                const uint4 wa = lds128_b(crow + ((uint32_t)(q ^ gid) << 4));
                const uint4 wb = lds128_b(crow + 8 * 128 + ((uint32_t)(q ^ gid) << 4));
                wa4[0] = wa.x, wa4[1] = wa.y, wa4[2] = wa.z, wa4[3] = wa.w;
                wb4[0] = wb.x, wb4[1] = wb.y, wb4[2] = wb.z, wb4[3] = wb.w;
            } else if constexpr (B == 2) {  // 64-byte rows, 64-byte swizzle: chunk c at c ^ ((row >> 1) & 3)
                const uint32_t off = ((uint32_t)((q >> 1) ^ ((gid >> 1) & 3)) << 4) + 8u * (uint32_t)(q & 1);
                const uint2 wa = lds64_b(crow + off), wb = lds64_b(crow + 8 * L::CROW + off);
                wa2[0] = wa.x, wa2[1] = wa.y, wb2[0] = wb.x, wb2[1] = wb.y;
            }
#pragma unroll
            for (int s2 = 0; s2 < 2; ++s2) {  // 16-k step: chunks c0 = 4q + 2 s2 (k 0..7) and c0 + 1 (k 8..15)
                uint32_t a0, a1, a2, a3;
                if constexpr (ONE && B == 2) {  // raw 128 + q
                    raw2x2(wa2[s2], sh2, cg, a0, a2);
                    raw2x2(wb2[s2], sh2, cg, a1, a3);
                } else if constexpr (ONE) {  // raw q (8 bits)
                    const int c = 2 * (q & 3) + s2;
                    const uint32_t base = crow + (uint32_t)(q >> 2) * (L::CODES / 2) + ((uint32_t)(c ^ gid) << 4) + w8;
                    a0 = raw8(lds32_b(base), sel8, mg);
                    a1 = raw8(lds32_b(base + 8 * 128), sel8, mg);
                    a2 = raw8(lds32_b(base + 8), sel8, mg);
                    a3 = raw8(lds32_b(base + 8 * 128 + 8), sel8, mg);
                } else if constexpr (B == 4) {
                    a0 = nat_pair(wa4[2 * s2], sel, sa2, oa2, cm, cg);
                    a1 = nat_pair(wb4[2 * s2], sel, sb2, ob2, cm, cg);
                    a2 = nat_pair(wa4[2 * s2 + 1], sel, sa2, oa2, cm, cg);
                    a3 = nat_pair(wb4[2 * s2 + 1], sel, sb2, ob2, cm, cg);
                } else if constexpr (B == 2) {  // k 2tq, 2tq+1 at bits 4tq; k + 8 at bits 16 + 4tq
                    raw2x2(wa2[s2], sh2, cg, a0, a2);
                    raw2x2(wb2[s2], sh2, cg, a1, a3);
                    a0 = deq_raw(a0, sa2, oa2, cg);
                    a2 = deq_raw(a2, sa2, oa2, cg);
                    a1 = deq_raw(a1, sb2, ob2, cg);
                    a3 = deq_raw(a3, sb2, ob2, cg);
                } else {  // 128-byte rows in two boxes of 128 k, 128-byte swizzle: chunk c at c ^ (row & 7)
                    const int c = 2 * (q & 3) + s2;
                    const uint32_t base = crow + (uint32_t)(q >> 2) * (L::CODES / 2) + ((uint32_t)(c ^ gid) << 4) + w8;
                    const uint32_t xa = lds32_b(base), xa8 = lds32_b(base + 8);
                    const uint32_t xb = lds32_b(base + 8 * 128), xb8 = lds32_b(base + 8 * 128 + 8);
                    a0 = pair8(xa, sel8, saf, oaf, mg);
                    a1 = pair8(xb, sel8, sbf, obf, mg);
                    a2 = pair8(xa8, sel8, saf, oaf, mg);
                    a3 = pair8(xb8, sel8, sbf, obf, mg);
                }
                const int cg8 = 4 * q + 2 * s2 + (li & 1);  // this lane's ldmatrix chunk (8 k) in the unit
                const uint32_t xrow = xst + (uint32_t)(cg8 >> 3) * L::XBOX +
                                      ((uint32_t)((cg8 & 7) ^ lr) << 4) + (uint32_t)lr * 128;
                if constexpr (ONE) {  // column lr: the token's row 0 while on slice q = lr, zero row 1 otherwise
                    // chunk c0 + (li & 1) of row 0, or (c0 + (li & 1)) ^ 1 of row 1 (c0 = 4q + 2 s2 is even)
                    const int c0 = 4 * q + 2 * s2;
                    uint32_t b0, b1;
                    ldsm_x2(xst + (uint32_t)((c0 >> 3) * L::XBOX + ((c0 & 7) << 4)) + (lr == q ? xo0 : xo1), b0, b1);
                    mma_16816(dacc, a0, a1, a2, a3, b0, b1);
                } else if (MT == 1) {  // one token group: matrices 0, 1 (lanes 0-15 give the addresses)
                    uint32_t b0, b1;
                    ldsm_x2(xrow, b0, b1);
                    mma_16816(acc[0], a0, a1, a2, a3, b0, b1);
                } else {
#pragma unroll
                    for (int tp = 0; tp < MT / 2; ++tp) {
                        uint32_t b0a, b1a, b0b, b1b;  // token groups 2tp (chunks c0, c0+1) and 2tp + 1
                        ldsm_x4(xrow + (uint32_t)(16 * tp + 8 * (li >> 1)) * 128, b0a, b1a, b0b, b1b);
                        mma_16816(acc[2 * tp], a0, a1, a2, a3, b0a, b1a);
                        mma_16816(acc[2 * tp + 1], a0, a1, a2, a3, b0b, b1b);
                    }
                }
            }
        }
        if constexpr (ONE) {  // this unit's slices: scales and offsets applied in fp32 (before the refill)
            const uint32_t oq = (uint32_t)(BT_ROWS * L::SQROW);  // offsets after the scales
            float sA0, sA1, oA0, oA1, sB0, sB1, oB0, oB1;    // rows gid (A), gid + 8 (B); slices 2tq, 2tq + 1
            if constexpr (G == 32) {  // groups 2tq, 2tq + 1: adjacent in the row
                const uint32_t sa = lds32_b(qa + 4 * tq), oa = lds32_b(qa + oq + 4 * tq);
                const uint32_t sb = lds32_b(qa + 8 * L::SQROW + 4 * tq), ob = lds32_b(qa + 8 * L::SQROW + oq + 4 * tq);
                sA0 = bf16lo_b(sa), sA1 = bf16hi_b(sa), oA0 = bf16lo_b(oa), oA1 = bf16hi_b(oa);
                sB0 = bf16lo_b(sb), sB1 = bf16hi_b(sb), oB0 = bf16lo_b(ob), oB1 = bf16hi_b(ob);
            } else {  // both slices in group (64 tq) / G
                const uint32_t go = (uint32_t)(((64 * tq) / G) * 2);
                sA0 = sA1 = bf16lo_b(lds16_b(qa + go)), oA0 = oA1 = bf16lo_b(lds16_b(qa + oq + go));
                sB0 = sB1 = bf16lo_b(lds16_b(qa + 8 * L::SQROW + go));
                oB0 = oB1 = bf16lo_b(lds16_b(qa + 8 * L::SQROW + oq + go));
            }
            // 2 bits: D sums (128 + q) x, so D - 128 xs sums q x; 8 bits: D sums q x
            const float bias0 = B == 2 ? -128.f * xs0 : 0.f, bias1 = B == 2 ? -128.f * xs1 : 0.f;
            ya = fmaf(sA0, dacc[0] + bias0, ya);
            ya = fmaf(oA0, xs0, ya);
            ya = fmaf(sA1, dacc[1] + bias1, ya);
            ya = fmaf(oA1, xs1, ya);
            yb = fmaf(sB0, dacc[2] + bias0, yb);
            yb = fmaf(oB0, xs0, yb);
            yb = fmaf(sB1, dacc[3] + bias1, yb);
            yb = fmaf(oB1, xs1, yb);
        }
        __syncthreads();  // every warp is done with stage d
        if (next < u1) {  // refill it with the unit DEPTH ahead
            if (threadIdx.x == 0) {
                fence_proxy_async_smem();
                mbar_arrive_expect_tx(bars + 8 * d, L::CODES + L::XBYTES + (QT ? L::QBYTES : 0));
            }
            issue_w(next, d);
            if (threadIdx.x == 0) issue_x(next, d);
            ++next;
        }
        if (++d == L::DEPTH) {
            d = 0;
            phase ^= 1u;
        }

        // end of a row group or of the range: hand each tile's sums on
        if (it + 1 == nunits || kc == p.nkc - 1) {
            const int tile = grp * BT_WARPS + warp;
            const int nrows = min(16, p.N - tile * 16);
            if constexpr (ONE) {  // row sums over the four lanes of a row pair (slices 0..7) -> token 0's column
                ya += __shfl_xor_sync(0xffffffffu, ya, 1);
                ya += __shfl_xor_sync(0xffffffffu, ya, 2);
                yb += __shfl_xor_sync(0xffffffffu, yb, 1);
                yb += __shfl_xor_sync(0xffffffffu, yb, 2);
                acc[0][0] = ya;
                acc[0][2] = yb;
                acc[0][1] = acc[0][3] = 0.f;
                ya = yb = 0.f;
            }
            if (kc_first == 0 && kc == p.nkc - 1) {  // this block summed all of the group's k
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int m = 8 * t + 2 * tq + (i & 1), r = gid + (i & 2) * 4;
                        if (m < p.M && r < nrows)
                            p.Y[(int64_t)m * p.N + tile * 16 + r] =
                                (uint16_t)float_to_bf16_bits(epilogue_f32(p.ep, acc[t][i], m, (int64_t)tile * 16 + r));
                    }
            } else if (kc_first != 0) {  // a later share of the group (the first of this range): publish it
                split_publish<MT>(p.ws + ((size_t)cta * BT_WARPS + warp) * 16 * p.M, acc, p.M, nrows, gid, tq);
            } else {  // the group's owner: its range ends here (last iteration); finished after the loop
                owner_split = true;
                break;
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
            kc_first = 0;
        }
        if (++kc == p.nkc) {
            kc = 0;
            ++grp;
        }
    }
    if (owner_split) {  // add the later shares of the last group's tile of this warp, write Y
        const int tile = grp * BT_WARPS + warp;
        const int wl = split_warp_of((long long)grp * p.nkc + p.nkc - 1, p.units, p.ctas);
        ok = split_collect<MT, NE>(acc, scr, p.ws + (size_t)warp * 16 * p.M, (size_t)BT_WARPS * 16 * p.M, cta, wl,
                                   p.M, min(16, p.N - tile * 16), gid, tq, lane, p.Y + (int64_t)tile * 16, p.N,
                                   &g_batch_fault, 2u, BT_WAIT_LIMIT_NS, epilogue_at(p.ep, (int64_t)tile * 16)) &&
             ok;
    }
    if (!ok) {  // never leave with copies still landing in shared memory (the last DEPTH fills)
        for (int i = max(0, nunits - L::DEPTH); i < nunits; ++i)
            mbar_drain_bounded(bars + 8 * (i % L::DEPTH), (uint32_t)((i / L::DEPTH) & 1), BT_WAIT_LIMIT_NS);
    }
}

// ------------------------------------------------------------------ host side

template <int G, int MT, bool QT, int B, bool ONE = false>
static cudaError_t launch_batch_gm(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& ts,
                                   const CUtensorMap& to, BatchArgs a, size_t ws_bytes, cudaStream_t stream) {
    using L = BatchLayout<G, MT, B, QT>;
    auto kern = batch_kernel<G, MT, QT, B, ONE>;
    cudaError_t e = ensure_kernel_attrs(reinterpret_cast<const void*>(kern), L::SMEM, false);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    if ((e = resident_blocks(reinterpret_cast<const void*>(kern), BT_THREADS, L::SMEM, &sms, &per_sm)) != cudaSuccess)
        return e;
    // one wave, no more blocks than units, and a workspace slot (16 x M words) for every warp
    long long ctas = std::min<long long>((long long)sms * per_sm, a.units);
    ctas = std::min<long long>(ctas, (long long)(ws_bytes / ((size_t)BT_WARPS * 16 * 8 * a.M)));
    if (ctas < 1) return cudaErrorInvalidValue;
    a.ctas = (int)ctas;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(BT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = L::SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tw, tx, ts, to, a);
}

template <int G, bool QT, int B>
static cudaError_t launch_batch_g(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& ts,
                                  const CUtensorMap& to, BatchArgs a, size_t ws_bytes, cudaStream_t stream) {
    if constexpr (B != 4)
        if (a.M == 1) return launch_batch_gm<G, 1, QT, B, true>(tw, tx, ts, to, a, ws_bytes, stream);
    if (a.M <= 8) return launch_batch_gm<G, 1, QT, B>(tw, tx, ts, to, a, ws_bytes, stream);
    if (a.M <= 16) return launch_batch_gm<G, 2, QT, B>(tw, tx, ts, to, a, ws_bytes, stream);
    return launch_batch_gm<G, 4, QT, B>(tw, tx, ts, to, a, ws_bytes, stream);
}

template <int B>
static cudaError_t launch_batch_b(const CUtensorMap& tw, const CUtensorMap& tx, const CUtensorMap& ts,
                                  const CUtensorMap& to, BatchArgs a, size_t ws, bool qt, int g, cudaStream_t stream) {
    switch (g) {
        case 32:
            return qt ? launch_batch_g<32, true, B>(tw, tx, ts, to, a, ws, stream)
                      : launch_batch_g<32, false, B>(tw, tx, ts, to, a, ws, stream);
        case 64:
            return qt ? launch_batch_g<64, true, B>(tw, tx, ts, to, a, ws, stream)
                      : launch_batch_g<64, false, B>(tw, tx, ts, to, a, ws, stream);
        default:
            return qt ? launch_batch_g<128, true, B>(tw, tx, ts, to, a, ws, stream)
                      : launch_batch_g<128, false, B>(tw, tx, ts, to, a, ws, stream);
    }
}

cudaError_t launch_batch(const StreamPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                         const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, int bits, uint16_t* Y,
                         void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep) {
    const int64_t ng = K / g;
    // qparam rows whole 16-byte pieces: 8-group TMA boxes (K is then a multiple of 256); else cp.async
    const bool qt = ng % 8 == 0;
    const int mp = M <= 8 ? 8 : (M <= 16 ? 16 : 32);
    CUtensorMap tw, tx, ts, to;
    // codes: [N][K bits/8] bytes, box 64 rows x 128 bytes (2 bits: 64 bytes, 64-byte swizzle);
    // X: [M][K] bf16, box mp rows x 64 k (rows past M read 0)
    const uint64_t row_bytes = (uint64_t)(K * bits / 8);
    cudaError_t e = encode_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, row_bytes, (uint64_t)N, row_bytes,
                                         bits == 2 ? 64 : 128, BT_ROWS,
                                         bits == 2 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, detail);
    if (e == cudaSuccess)
        e = encode_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_UINT16, X, (uint64_t)K, (uint64_t)M, (uint64_t)K * 2,
                                 64, (uint32_t)mp, CU_TENSOR_MAP_SWIZZLE_128B, detail);
    if (e != cudaSuccess) return e;
    ts = tw;
    to = tw;
    if (qt) {
        e = encode_tensor_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, (uint64_t)ng, (uint64_t)N,
                                 (uint64_t)ng * 2, 8, BT_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e == cudaSuccess)
            e = encode_tensor_map_2d(&to, CU_TENSOR_MAP_DATA_TYPE_UINT16, offsets, (uint64_t)ng, (uint64_t)N,
                                     (uint64_t)ng * 2, 8, BT_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e != cudaSuccess) return e;
    }
    BatchArgs a;
    a.scales = scales;
    a.offsets = offsets;
    a.Y = Y;
    a.ep = ep;
    a.ws = static_cast<uint64_t*>(workspace);
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.nkc = plan.nkc;
    a.units = (N + BT_ROWS - 1) / BT_ROWS * (long long)plan.nkc;
    a.ctas = 0;
    const size_t ws = plan.ws_bytes;
    if (bits == 2) return launch_batch_b<2>(tw, tx, ts, to, a, ws, qt, g, stream);
    if (bits == 8) return launch_batch_b<8>(tw, tx, ts, to, a, ws, qt, g, stream);
    return launch_batch_b<4>(tw, tx, ts, to, a, ws, qt, g, stream);
}

cudaError_t read_and_clear_batch_fault(unsigned int* fault) {
    cudaError_t e = cudaMemcpyFromSymbol(fault, g_batch_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !*fault) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_batch_fault, &zero, sizeof(unsigned int));
}

}  // namespace w4
