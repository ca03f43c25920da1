// w4_decode.cu -- persistent stream-K bf16 x int4 linear for decode (M <= 32)
// on weights in the decode layout (include/w4.h, written by w4_repack).
//
// Y[m,n] = sum_k X[m,k] * w'[n,k], w' = bf16(q*s + o), fp32 accumulation
// (Optimum Quanto: bf16 x int4 matmul, result accumulated at higher precision,
// "Pitfalls when quantizing activations").
//
// The decode layout stores every 16-row x 256-k unit contiguously with each
// lane's fragments in lane order, so a unit is five fully coalesced 512-byte
// warp loads straight into registers: no shared memory at all, no copy
// engine, no barriers per unit.  The design otherwise follows the stream
// kernel on the canonical layout (w4_stream.cu):
//  * the (row tile, k) units are cut into equal contiguous ranges, one per
//    warp of a one-wave persistent grid;
//  * a warp holds two units' fragments in registers and refills a set with
//    the unit two ahead as soon as it has computed it; the first two units
//    are requested before the programmatic-dependent-launch wait;
//  * dequantization: LOP3 nibble pairs (128+q as bf16), an exact subtract of
//    128 and one bf16 FMA with (scale, offset), then mma.sync m16n8k16 with
//    the weights as A and the tokens as B, one MMA per group of 8 tokens on
//    the same dequantized fragment (M up to 32: four groups).  The
//    layout's nibble order makes every extracted pair two consecutive k, so
//    the B fragments are X's own 32-bit words, read straight from global
//    memory through L1 (X is tiny and shared by every warp of the SM);
//  * a tile split between warps is finished by its owner (the warp holding
//    its first unit) from the partial sums the other sharers leave in their
//    workspace slots (split_publish / split_collect in w4_device.cuh).
#include "w4_device.cuh"
#include "w4_internal.h"

#include <algorithm>

namespace w4 {

constexpr int DC_WARPS = 4;
constexpr int DC_THREADS = DC_WARPS * 32;
constexpr uint64_t DC_WAIT_LIMIT_NS = 2000000000ull;
__device__ unsigned int g_decode_fault;

struct DecodeArgs {
    const uint16_t* X;
    const uint8_t* packed;
    uint16_t* Y;
    uint64_t* ws;         // split-tile slots, one per warp (split_ws_bytes), zero between calls
    int M, N, K;
    int nkc;              // units per row tile = ceil(K / 256)
    long long units;      // row tiles x nkc
    int workers;          // warps of the grid with work
};

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
    uint4 r;
    asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}

// One MMA step from packed codes (see the stream kernel): nibble pairs of the
// code words of rows a and b -> four A-fragment registers -> mma.sync.
template <int SH>
__device__ __forceinline__ void dc_mma(float (&c)[4], uint32_t wa, uint32_t wb, uint32_t sa2, uint32_t oa2,
                                       uint32_t sb2, uint32_t ob2, uint32_t x0, uint32_t x1, uint32_t cm,
                                       uint32_t cg) {
    asm volatile(
        "{\n\t.reg .b32 a0, a1, b0, b1, t;\n\t"
        "shr.b32 t, %4, %14;\n\t"
        "lop3.b32 a0, t, %12, %13, 0xEA;\n\t"
        "shr.b32 t, %4, %15;\n\t"
        "lop3.b32 a1, t, %12, %13, 0xEA;\n\t"
        "shr.b32 t, %5, %14;\n\t"
        "lop3.b32 b0, t, %12, %13, 0xEA;\n\t"
        "shr.b32 t, %5, %15;\n\t"
        "lop3.b32 b1, t, %12, %13, 0xEA;\n\t"
        "sub.rn.bf16x2 a0, a0, %13;\n\t"
        "sub.rn.bf16x2 a1, a1, %13;\n\t"
        "sub.rn.bf16x2 b0, b0, %13;\n\t"
        "sub.rn.bf16x2 b1, b1, %13;\n\t"
        "fma.rn.bf16x2 a0, a0, %6, %7;\n\t"
        "fma.rn.bf16x2 a1, a1, %6, %7;\n\t"
        "fma.rn.bf16x2 b0, b0, %8, %9;\n\t"
        "fma.rn.bf16x2 b1, b1, %8, %9;\n\t"
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {a0,b0,a1,b1}, {%10,%11}, "
        "{%0,%1,%2,%3};\n\t}"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(wa), "r"(wb), "r"(sa2), "r"(oa2), "r"(sb2), "r"(ob2), "r"(x0), "r"(x1), "r"(cm), "r"(cg),
          "n"(SH), "n"(SH + 4));
}

// The four A-fragment registers of one MMA step (rows a, b; nibble pairs SH,
// SH+4 and SH+1, SH+5), dequantized once for every token group.
template <int SH>
__device__ __forceinline__ void dc_dequant(uint32_t wa, uint32_t wb, uint32_t sa2, uint32_t oa2, uint32_t sb2,
                                           uint32_t ob2, uint32_t cm, uint32_t cg, uint32_t (&A)[4]) {
    asm("{\n\t.reg .b32 t;\n\t"
        "shr.b32 t, %4, %12;\n\t"
        "lop3.b32 %0, t, %10, %11, 0xEA;\n\t"
        "shr.b32 t, %4, %13;\n\t"
        "lop3.b32 %2, t, %10, %11, 0xEA;\n\t"
        "shr.b32 t, %5, %12;\n\t"
        "lop3.b32 %1, t, %10, %11, 0xEA;\n\t"
        "shr.b32 t, %5, %13;\n\t"
        "lop3.b32 %3, t, %10, %11, 0xEA;\n\t"
        "sub.rn.bf16x2 %0, %0, %11;\n\t"
        "sub.rn.bf16x2 %1, %1, %11;\n\t"
        "sub.rn.bf16x2 %2, %2, %11;\n\t"
        "sub.rn.bf16x2 %3, %3, %11;\n\t"
        "fma.rn.bf16x2 %0, %0, %6, %7;\n\t"
        "fma.rn.bf16x2 %1, %1, %8, %9;\n\t"
        "fma.rn.bf16x2 %2, %2, %6, %7;\n\t"
        "fma.rn.bf16x2 %3, %3, %8, %9;\n\t}"
        : "=&r"(A[0]), "=&r"(A[1]), "=&r"(A[2]), "=&r"(A[3])
        : "r"(wa), "r"(wb), "r"(sa2), "r"(oa2), "r"(sb2), "r"(ob2), "r"(cm), "r"(cg), "n"(SH), "n"(SH + 4));
}
__device__ __forceinline__ void dc_mma_only(float (&c)[4], const uint32_t (&A)[4], uint32_t x0, uint32_t x1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(A[0]), "r"(A[1]), "r"(A[2]), "r"(A[3]), "r"(x0), "r"(x1));
}

// One unit's fragments of this lane: code words of rows a / b for the two
// 128-k halves, and the lane's eight qparams.
struct DcUnit {
    uint4 a0, b0, a1, b1, q;
};

// MT: groups of 8 tokens (M <= 8 MT).
// NE: slot words per lane of an owner's collect (16 M / 32): 1 for one token,
// 4 MT otherwise.
template <int G, int MT, int NE>
__global__ void __launch_bounds__(DC_THREADS, MT == 4 ? 4 : 5)
decode_kernel(const DecodeArgs p) {
    constexpr int SLOT16 = (2048 + 16 * 32 * 32 / G) / 16;  // 16-byte pieces per unit
    constexpr int QSH = (G == 32) ? 0 : (G == 64 ? 1 : 2);   // lanes sharing a qparam piece: 1 << QSH
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tq = lane & 3;
    const int worker = blockIdx.x * DC_WARPS + warp;
    __shared__ float scr[DC_WARPS][16 * 8 * MT];  // split-tile scratch of each warp (a tile's 16 x M sums)

    griddep_launch_dependents();
    if (worker >= p.workers) return;
    const long long u0 = p.units * worker / p.workers;
    const long long u1 = p.units * (worker + 1) / p.workers;
    const int nunits = (int)(u1 - u0);
    if (nunits <= 0) return;

    // the first two units' fragments: weights never depend on the previous kernel
    const uint4* wsrc = reinterpret_cast<const uint4*>(p.packed) + lane;
    const uint4* qsrc = reinterpret_cast<const uint4*>(p.packed) + 128 + (lane >> QSH);
    auto load = [&](long long u, DcUnit& f) {
        const int64_t o = u * SLOT16;
        f.a0 = ldg_stream_v4(wsrc + o);
        f.b0 = ldg_stream_v4(wsrc + o + 32);
        f.a1 = ldg_stream_v4(wsrc + o + 64);
        f.b1 = ldg_stream_v4(wsrc + o + 96);
        f.q = ldg_stream_v4(qsrc + o);
    };
    DcUnit fa, fb;
    load(u0, fa);
    if (nunits > 1) load(u0 + 1, fb);

    // activations may come from the previous kernel: wait for it
    griddep_wait();

    // B fragments straight from X (natural k order, L1-cached): lane (gid, tq)
    // needs token (8t + gid)'s 8-k chunks at 32 tq + 8 j of each 128-k half
    const uint16_t* xlane = p.X + (int64_t)gid * p.K + 32 * tq;

    uint32_t cm, cg;  // constants pinned in registers: nibble mask, bf16 128.0 pair (magic and bias)
    asm volatile("mov.b32 %0, %1;" : "=r"(cm) : "r"(0x000F000Fu));
    asm volatile("mov.b32 %0, %1;" : "=r"(cg) : "r"(0x43004300u));

    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    int tile = (int)(u0 / p.nkc), kc = (int)(u0 % p.nkc), kc_first = kc;
    bool owner_split = false;  // the range ends inside a tile whose first unit it holds

    auto compute = [&](const DcUnit& f, int it) {
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // two 128-k halves per unit
            const int kx = kc * 256 + 128 * h;  // first k of the half (its chunks lie inside K or wholly past it)
            const uint4 wa = h ? f.a1 : f.a0, wb = h ? f.b1 : f.b0;
            const uint32_t qwa = h ? f.q.z : f.q.x, qwb = h ? f.q.w : f.q.y;  // (scale | offset << 16)
            const uint32_t sa2 = __byte_perm(qwa, 0, 0x1010), oa2 = __byte_perm(qwa, 0, 0x3232);
            const uint32_t sb2 = __byte_perm(qwb, 0, 0x1010), ob2 = __byte_perm(qwb, 0, 0x3232);
            const uint32_t wa4[4] = {wa.x, wa.y, wa.z, wa.w};
            const uint32_t wb4[4] = {wb.x, wb.y, wb.z, wb.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                // nibbles (i, i+4) of a decode-layout word are the consecutive k (2i, 2i+1):
                // the B pairs are X's own 32-bit words
                const bool kin = kx + 32 * tq + 8 * j < p.K;
                uint4 xv[MT];
#pragma unroll
                for (int t = 0; t < MT; ++t)
                    xv[t] = (kin && 8 * t + gid < p.M) ? ldg_nc_v4(xlane + (int64_t)(8 * t) * p.K + kx + 8 * j)
                                                       : make_uint4(0u, 0u, 0u, 0u);
                if (MT == 1) {  // dequantization fused with the single MMA
                    dc_mma<0>(acc[0], wa4[j], wb4[j], sa2, oa2, sb2, ob2, xv[0].x, xv[0].y, cm, cg);
                    dc_mma<8>(acc[0], wa4[j], wb4[j], sa2, oa2, sb2, ob2, xv[0].z, xv[0].w, cm, cg);
                } else {
                    uint32_t A[4];
                    dc_dequant<0>(wa4[j], wb4[j], sa2, oa2, sb2, ob2, cm, cg, A);
#pragma unroll
                    for (int t = 0; t < MT; ++t) dc_mma_only(acc[t], A, xv[t].x, xv[t].y);
                    dc_dequant<8>(wa4[j], wb4[j], sa2, oa2, sb2, ob2, cm, cg, A);
#pragma unroll
                    for (int t = 0; t < MT; ++t) dc_mma_only(acc[t], A, xv[t].z, xv[t].w);
                }
            }
        }

        // end of a row tile or of the range: hand the tile's sums on
        if (it + 1 == nunits || kc == p.nkc - 1) {
            const int n_a = tile * 16 + gid, n_b = n_a + 8;
            // acc[t] = D[row n_a: tokens 8t + 2tq, +1 | row n_b: the same tokens]
            if (kc_first == 0 && kc == p.nkc - 1) {  // this warp summed all of the tile's k
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int m = 8 * t + 2 * tq + (i & 1), n = (i < 2) ? n_a : n_b;
                        if (m < p.M && n < p.N) p.Y[(int64_t)m * p.N + n] = (uint16_t)float_to_bf16_bits(acc[t][i]);
                    }
            } else if (kc_first != 0) {  // a later share of the tile (the first of this range): publish it
                split_publish<MT>(p.ws + (size_t)worker * 16 * p.M, acc, p.M, min(16, p.N - tile * 16), gid, tq);
            } else {  // the tile's owner: its range ends here (last unit); finished after the loop
                owner_split = true;
                return;
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
            kc_first = 0;
        }
        if (++kc == p.nkc) {
            kc = 0;
            ++tile;
        }
    };

    // two register sets: a set is refilled with the unit two ahead as soon as
    // it has been computed, so every unit's loads overlap the previous compute
    for (int it = 0; it < nunits; it += 2) {
        compute(fa, it);
        if (it + 2 < nunits) load(u0 + it + 2, fa);
        if (it + 1 >= nunits) break;
        compute(fb, it + 1);
        if (it + 3 < nunits) load(u0 + it + 3, fb);
    }
    if (owner_split) {  // add the later shares of the last tile (their warps publish without waiting), write Y
        const int wl = split_warp_of((long long)tile * p.nkc + p.nkc - 1, p.units, p.workers);
        split_collect<MT, NE>(acc, scr[warp], p.ws, (size_t)16 * p.M, worker, wl, p.M, min(16, p.N - tile * 16), gid,
                              tq, lane, p.Y + (int64_t)tile * 16, p.N, &g_decode_fault, 1u, DC_WAIT_LIMIT_NS);
    }
}

// ------------------------------------------------------------------ host side

bool plan_decode(int64_t M, int64_t N, int64_t K, int g, DecodePlan* plan) {
    if (M < 1 || M > DECODE_MAX_M) return false;
    const int64_t tiles = (N + 15) / 16;
    if (tiles > 0x3FFFFFFF) return false;
    plan->nkc = (int)((K + 255) / 256);
    plan->units = tiles * plan->nkc;
    plan->ws_bytes = split_ws_bytes(M, plan->units);
    (void)g;
    return true;
}

template <int G, int MT, int NE>
static cudaError_t launch_decode_gm(const DecodePlan& plan, DecodeArgs a, cudaStream_t stream) {
    auto kern = decode_kernel<G, MT, NE>;
    // one wave: as many resident warps as the SMs hold, but no more than there are units
    int sms = 0, per_sm = 0;
    cudaError_t e = resident_blocks(reinterpret_cast<const void*>(kern), DC_THREADS, 0, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const long long max_workers = std::min<long long>((long long)sms * per_sm * DC_WARPS, SPLIT_MAX_WORKERS);
    a.workers = (int)std::min<long long>(max_workers, plan.units);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((a.workers + DC_WARPS - 1) / DC_WARPS), 1, 1);
    cfg.blockDim = dim3(DC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int G>
static cudaError_t launch_decode_g(const DecodePlan& plan, DecodeArgs a, cudaStream_t stream) {
    if (a.M <= 1) return launch_decode_gm<G, 1, 1>(plan, a, stream);
    if (a.M <= 8) return launch_decode_gm<G, 1, 4>(plan, a, stream);
    if (a.M <= 16) return launch_decode_gm<G, 2, 8>(plan, a, stream);
    return launch_decode_gm<G, 4, 16>(plan, a, stream);
}

cudaError_t launch_decode(const DecodePlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* packed,
                          int64_t N, int g, uint16_t* Y, void* workspace, cudaStream_t stream) {
    DecodeArgs a;
    a.X = X;
    a.packed = packed;
    a.Y = Y;
    a.ws = static_cast<uint64_t*>(workspace);
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.nkc = plan.nkc;
    a.units = plan.units;
    a.workers = 0;
    switch (g) {
        case 32: return launch_decode_g<32>(plan, a, stream);
        case 64: return launch_decode_g<64>(plan, a, stream);
        default: return launch_decode_g<128>(plan, a, stream);
    }
}

cudaError_t read_and_clear_decode_fault(unsigned int* fault) {
    cudaError_t e = cudaMemcpyFromSymbol(fault, g_decode_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !*fault) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_decode_fault, &zero, sizeof(unsigned int));
}

}  // namespace w4
