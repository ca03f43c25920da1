// w4_stream.cu -- persistent stream-K bf16 x int4 linear for decode (M <= 4;
// 5 to 32 tokens go to the block-shared X kernel of w4_batch.cu).
//
// Y[m,n] = sum_k X[m,k] * w'[n,k], w' = bf16(q*s + o), fp32 accumulation
// (Optimum Quanto: bf16 x int4 matmul, result accumulated at higher precision,
// "Pitfalls when quantizing activations").  With one to eight tokens the
// packed codes are almost all of the traffic, and a launch is a few
// microseconds of HBM time, so the kernel is organised around keeping every
// SM streaming for the whole launch:
//
//  * Work unit = 16 weight rows x 256 k (2 KB of codes).  The units of the
//    problem, taken in (row tile, k) order, are cut into equal contiguous
//    ranges, one per warp of a one-wave persistent grid: every warp streams
//    the same number of bytes (within one unit), whatever N and K are.
//  * Each warp owns a ring of three unit slots.  Lane 0 fetches a unit's codes
//    with one 2-D TMA copy (16 rows x 128 bytes, 128-byte swizzle, zero fill
//    past N and K); the 32 lanes fetch its scales and offsets with 4-byte
//    cp.async; all complete on the slot's mbarrier.  The first three units are
//    requested before the programmatic-dependent-launch wait.
//  * X (only 256 k x M tokens per unit): loaded one unit ahead into
//    registers, permuted to the MMA k order and staged in the warp's shared
//    memory (tokens beyond M read a zero row).
//  * Dequantization and products as in the skinny kernel: LOP3 nibble pairs,
//    exact subtract + one bf16 FMA, mma.m16n8k16 with the weights as the A
//    operand and the tokens as B (swap AB).
//  * One token: the eight token columns of the MMA would hold seven zero
//    columns, so they hold the unit's eight 32-k slices instead.  Lane
//    (gid, tq) supplies X only where its column gid is the slice its codes
//    come from (gid = tq + 4h), zero elsewhere, so column c of D sums slice c
//    alone.  The A operand is the raw LOP3 value 128 + q (no subtract, no
//    scale, no offset): D[n][c] = sum (128 + q) x over the slice, and the
//    group's scale and offset are applied to those sums in fp32,
//    y += s (D - 128 xs) + o xs with xs the slice's sum of X.  That halves the
//    per-weight instructions, and the weights are never rounded to bf16.
//  * A warp that covers all of a row tile's k writes bf16 Y directly.  A tile
//    split between warps is finished by its owner, the warp holding its
//    first unit, from the partial sums the other sharers leave in their
//    workspace slots (flag and value in one 64-bit store, no atomics, no
//    fence; split_publish / split_collect in w4_device.cuh): one round trip
//    to L2 at the end of the owner's range instead of a chain of atomics,
//    and a fixed summation order.
#include "w4_device.cuh"
#include "w4_internal.h"
#include "w4_mma.cuh"

#include <algorithm>
#include <cuda.h>
#include <mutex>

namespace w4 {

constexpr int ST_WARPS = 4;
constexpr int ST_THREADS = ST_WARPS * 32;
constexpr int ST_UK = 256;                 // k per unit
constexpr int ST_DEPTH = 3;                // ring slots per warp (16-row units)
constexpr int ST_WSLOT = 16 * 128;         // codes of one unit: 16 rows x 128 bytes
constexpr int ST_XPITCH = ST_UK * 2 + 16;  // one staged token row of a unit (+16 bytes against bank conflicts)

struct StreamArgs {
    const uint16_t* X;
    const uint16_t* scales;
    const uint16_t* offsets;
    uint16_t* Y;
    Epilogue ep;           // bias and output scale, applied before the rounding
    uint64_t* ws;          // split-tile slots, one per warp (split_ws_bytes), zero between calls
    int M, N, K;
    int nkc;               // units per row tile = ceil(K / 256)
    long long units;       // row tiles x nkc
    int workers;           // warps of the grid with work
};

// per-warp shared memory after the code slots: qparam slots, X slots, zero row,
// split-tile scratch, barriers
__host__ __device__ inline int st_qslot_bytes(int g, int rt) { return 2 * 16 * rt * (ST_UK / g) * 2; }
// ring slots per warp: three 16-row units, or two 32-row units
__host__ __device__ inline int st_depth(int rt) { return rt == 1 ? ST_DEPTH : 2; }
// X slot (one unit x M token rows; a warp rewrites it only after its reads of the
// previous unit have returned); none beyond 8 tokens, which this kernel never
// runs.  The block's warps share one zero row after their areas.
__host__ __device__ inline int st_xslot_bytes(int M) { return M <= 8 ? M * ST_XPITCH : 0; }
__host__ __device__ inline int st_scratch_bytes(int M, int rt) { return 16 * rt * M * 4; }  // a tile's fp32 sums
__host__ __device__ inline int st_rest_bytes(int M, int g, int rt) {
    const int dp = st_depth(rt);
    const int b = dp * st_qslot_bytes(g, rt) + st_xslot_bytes(M) + st_scratch_bytes(M, rt) + 8 * dp;
    return (b + 127) & ~127;  // qparam slots are TMA destinations: 128-byte aligned
}
__host__ __device__ inline int st_smem_bytes(int M, int g, int rt) {
    return ST_WARPS * st_depth(rt) * ST_WSLOT * rt + ST_WARPS * st_rest_bytes(M, g, rt) + (M <= 8 ? ST_XPITCH : 0) +
           1024;  // zero row, alignment slack
}

__device__ unsigned int g_stream_fault;
constexpr uint64_t ST_WAIT_LIMIT_NS = 2000000000ull;

// 16 bytes of read-only data through L1 (the blocks of an SM that read the same lines share them)
__device__ __forceinline__ uint4 ldg_l1_v4(const void* ptr) {
    uint4 v;
    asm("ld.global.nc.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(ptr));
    return v;
}

// XM, what X holds: 0 bf16 activations; 1 int8 activation codes (p.X points at
// bytes), widened to bf16 when loaded, their scale applied by the epilogue
// (p.ep.yscale); 2 bf16 activations quantized here to int8 codes with the
// dynamic symmetric scale of w4_quantize_activation_i8 (one for the tensor, or
// one per token when p.ep.ys_stride is 1): each block finds the maximum
// magnitude of X first (after the dependency wait, with its weight copies in
// flight), then codes every X chunk as it loads it, exactly as the separate
// quantization would, and its epilogue applies the scale.
// The owner's part of a split tile on the one-token path, for all RT row tiles of the unit at once
// (a sharer's slot holds them one after another, 16 words each).  It is split_collect's
// owner collect with one token, but one batch of loads covers the same sharers' words of every
// row tile, so the owner pays one round trip to L2 per batch instead of one per row tile.  Lanes
// 0-15 take row lane of even sharers and lanes 16-31 the odd ones, 8 sharers each per batch.
// The sums are added in warp order (deterministic); each word is zeroed after use.  Returns false
// if a wait timed out.
template <int RT>
__device__ __forceinline__ bool collect_one_token(const float (&oacc)[RT][1][4], float* scr, uint64_t* ws, int worker,
                                                  int wl, const int (&nrows)[RT], int row_a, int tq, int lane,
                                                  uint16_t* Yt, unsigned int* fault_word, unsigned int code,
                                                  uint64_t limit_ns, const Epilogue ep_t) {
    constexpr int BC = 8;                   // sharers per half-warp and batch
    constexpr size_t STRIDE = (size_t)RT * 16;
    if (tq == 0) {  // token 0 of rows row_a, row_a + 8 of each row tile
#pragma unroll
        for (int rt = 0; rt < RT; ++rt) {
            scr[rt * 16 + row_a] = oacc[rt][0][0];
            scr[rt * 16 + row_a + 8] = oacc[rt][0][2];
        }
    }
    __syncwarp();
    const int sub = lane >> 4, e0 = lane & 15;
    bool ok = true;
    float sum[RT];
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) sum[rt] = sub == 0 ? scr[rt * 16 + e0] : 0.f;
    for (int c0 = worker + 1 + sub; c0 <= wl; c0 += 2 * BC) {
        uint64_t v[RT][BC];
#pragma unroll
        for (int rt = 0; rt < RT; ++rt)
#pragma unroll
            for (int j = 0; j < BC; ++j) {
                const int c = c0 + 2 * j;
                v[rt][j] = (c <= wl && e0 < nrows[rt]) ? ld_relaxed_u64(ws + (size_t)c * STRIDE + rt * 16 + e0)
                                                       : (1ull << 32);
            }
        uint64_t t0 = 0;
        for (;;) {  // re-poll together the words whose sharer has not published yet
            bool all = true;
#pragma unroll
            for (int rt = 0; rt < RT; ++rt)
#pragma unroll
                for (int j = 0; j < BC; ++j) all = all && (v[rt][j] >> 32) != 0u;
            if (all) break;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            if (now - t0 > limit_ns) {  // give up: count what is missing as zero
                atomicOr(fault_word, code);
                ok = false;
                break;
            }
#pragma unroll
            for (int rt = 0; rt < RT; ++rt)
#pragma unroll
                for (int j = 0; j < BC; ++j)
                    if ((v[rt][j] >> 32) == 0u)
                        v[rt][j] = ld_relaxed_u64(ws + (size_t)(c0 + 2 * j) * STRIDE + rt * 16 + e0);
        }
#pragma unroll
        for (int rt = 0; rt < RT; ++rt)
#pragma unroll
            for (int j = 0; j < BC; ++j) {
                const int c = c0 + 2 * j;
                if (c <= wl && e0 < nrows[rt]) {
                    sum[rt] += __uint_as_float((uint32_t)v[rt][j]);
                    st_relaxed_u64(ws + (size_t)c * STRIDE + rt * 16 + e0, 0ull);
                }
            }
    }
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) {
        sum[rt] += __shfl_xor_sync(0xffffffffu, sum[rt], 16);
        if (sub == 0 && e0 < nrows[rt])
            Yt[16 * rt + e0] = (uint16_t)float_to_bf16_bits(epilogue_f32(epilogue_at(ep_t, 16 * rt), sum[rt], 0, e0));
    }
    __syncwarp();
    return ok;
}

template <int G, int MX, bool QT, int RT, int XM>
__global__ void __launch_bounds__(ST_THREADS, RT == 2 ? 4 : 6)
stream_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
              const __grid_constant__ CUtensorMap tm_o, const StreamArgs p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    static_assert(RT == 1 || MX == 1, "two row tiles per unit only on the one-token path");
    static_assert(MX == 1 || MX == 2 || MX == 4, "one to four tokens");
    constexpr int ROWS = 16 * RT;                    // weight rows per unit
    constexpr int DEPTH = RT == 1 ? ST_DEPTH : 2;    // ring slots (st_depth)
    constexpr int WSLOT = ST_WSLOT * RT;             // codes of one unit
    constexpr int QSLOT = 2 * ROWS * (ST_UK / G) * 2;  // scales then offsets, ROWS rows x (256/G) groups each
    constexpr int QROW = (ST_UK / G) * 2;            // bytes of one row of one array
    constexpr int PPR = QROW / 4;                    // 4-byte pieces per row and array
    constexpr int PIECES = 2 * ROWS * PPR;           // 4-byte qparam pieces per unit
    constexpr int PPL = (PIECES + 31) / 32;          // pieces per lane

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tq = lane & 3;
    const int worker = blockIdx.x * ST_WARPS + warp;

    griddep_launch_dependents();
    const bool idle = worker >= p.workers;
    const long long u0 = idle ? 0 : p.units * worker / p.workers;
    const long long u1 = idle ? 0 : p.units * (worker + 1) / p.workers;
    // XM 2: the block's scale(s) of X, found by all of its warps (two block barriers)
    __shared__ uint32_t qx_red[ST_WARPS][MX];
    __shared__ float qx_scale[MX];
    auto find_scales = [&]() {
        uint32_t mx[MX];
#pragma unroll
        for (int m = 0; m < MX; ++m) {
            mx[m] = 0u;
            if (m < p.M)
                for (int c = threadIdx.x; c < p.K / 8; c += ST_THREADS)  // through L1: the SM's blocks share X
                    mx[m] = max(mx[m], act_mag_max8(ldg_l1_v4(p.X + (int64_t)m * p.K + 8 * c)));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mx[m] = max(mx[m], __shfl_xor_sync(0xffffffffu, mx[m], o));
            if (lane == 0) qx_red[warp][m] = mx[m];
        }
        __syncthreads();
        if (threadIdx.x == 0) {
            uint32_t all = 0u;  // one scale for the tensor: the maximum over its rows
            for (int m = 0; m < p.M; ++m)
                for (int w = 0; w < ST_WARPS; ++w) all = max(all, qx_red[w][m]);
            for (int m = 0; m < p.M; ++m) {
                uint32_t row = 0u;
                for (int w = 0; w < ST_WARPS; ++w) row = max(row, qx_red[w][m]);
                qx_scale[m] = act_scale_of(p.ep.ys_stride ? row : all);
            }
        }
        __syncthreads();
    };
    if (u0 >= u1) {
        if constexpr (XM == 2) {  // an idle warp still helps its block find the scales
            griddep_wait();
            find_scales();
        }
        return;
    }
    const int nunits = (int)(u1 - u0);
    Epilogue ep = p.ep;  // XM 2: the output scale is the block's own
    if constexpr (XM == 2) {
        ep.yscale = qx_scale;
        ep.ys_stride = p.ep.ys_stride ? 1 : 0;
    }

    const int rest = st_rest_bytes(p.M, G, RT);
    const uint32_t wslots = smem_u32(smem) + warp * (DEPTH * WSLOT);
    unsigned char* rbase = smem + ST_WARPS * DEPTH * WSLOT + warp * rest;
    const uint32_t qslots = smem_u32(rbase);
    constexpr int MT = 1;            // one group of 8 token columns
    constexpr bool DIAG = MX == 1;   // one token: slice sums in the MMA columns, scales in fp32
    unsigned char* xs = rbase + DEPTH * QSLOT;                          // X slot: M token rows
    unsigned char* zrow = smem + ST_WARPS * (DEPTH * WSLOT + rest);     // zeros for tokens >= M (shared)
    float* scr = reinterpret_cast<float*>(rbase + DEPTH * QSLOT + st_xslot_bytes(p.M));  // split-tile scratch
    const uint32_t bars = smem_u32(rbase + DEPTH * QSLOT + st_xslot_bytes(p.M) + st_scratch_bytes(p.M, RT));
    const int ng = p.K / G;

    if (lane == 0) {  // arrivals per fill: the TMA arrive (+ 32 cp.async arrivals when qparams go that way)
        for (int d = 0; d < DEPTH; ++d) mbar_init(bars + 8 * d, QT ? 1 : 33);
        mbar_fence_init();
    }
    // every warp writes the same zeros (no block barrier needed before its own reads)
    for (int c = lane; c < ST_XPITCH / 16; c += 32)
        *reinterpret_cast<uint4*>(zrow + 16 * c) = make_uint4(0u, 0u, 0u, 0u);
    __syncwarp();

    // this lane's qparam pieces: fixed (array, row, piece) for every unit
    int prow[PPL], pcol[PPL];  // row in the tile, first group of the piece
    uint32_t pdst[PPL];        // offset inside a qparam slot
    const uint16_t* pbase[PPL];
#pragma unroll
    for (int q = 0; q < PPL; ++q) {
        const int i = lane + 32 * q;
        const int arr = (i < PIECES) ? i / (PIECES / 2) : 0, rem = (i < PIECES) ? i % (PIECES / 2) : 0;
        prow[q] = rem / PPR;
        pcol[q] = 2 * (rem % PPR);
        pdst[q] = (uint32_t)(arr * ROWS * QROW + prow[q] * QROW + 4 * (rem % PPR));
        pbase[q] = arr ? p.offsets : p.scales;
    }

    // request the unit at (tile, kc) into ring slot d: codes by TMA, scales/offsets by 4-byte cp.async
    auto issue = [&](int tile, int kc, int d) {
        const int row0 = tile * ROWS, k = kc * ST_UK;
        const uint32_t bar = bars + 8 * d;
        if (QT) {  // qparams as two more TMA boxes of 16 rows x 8 groups (zero fill past N and K)
            if (lane == 0) {
                mbar_arrive_expect_tx(bar, WSLOT + QSLOT);
                tma_load_2d(wslots + d * WSLOT, &tm_w, bar, k / 2, row0);
                tma_load_2d(qslots + d * QSLOT, &tm_s, bar, k / G, row0);
                tma_load_2d(qslots + d * QSLOT + ROWS * QROW, &tm_o, bar, k / G, row0);
            }
            return;
        }
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, WSLOT);
            tma_load_2d(wslots + d * WSLOT, &tm_w, bar, k / 2, row0);
        }
        const bool edge = (row0 + ROWS > p.N) || (k + ST_UK > p.K);  // clamp into the tensor (finite fill values)
#pragma unroll
        for (int q = 0; q < PPL; ++q) {
            if (PIECES % 32 == 0 || lane + 32 * q < PIECES) {
                int n = row0 + prow[q], j = k / G + pcol[q];
                if (edge) {
                    n = min(n, p.N - 1);  // rows past N: any finite qparams (their codes are 0)
                    j = min(j, ng - 2);   // groups past K: likewise (X is 0 there)
                }
                cp_async_4(qslots + d * QSLOT + pdst[q], pbase[q] + (int64_t)n * ng + j);
            }
        }
        cp_async_arrive_noinc(bar);
    };

    // unit cursors, advanced without division
    const int tile0 = (int)(u0 / p.nkc), kc0 = (int)(u0 % p.nkc);
    int it_tile = tile0, it_kc = kc0;  // next unit to request
    auto advance = [&](int& tile, int& kc) {
        if (++kc == p.nkc) {
            kc = 0;
            ++tile;
        }
    };
    const int depth = nunits < DEPTH ? nunits : DEPTH;
    for (int d = 0; d < depth; ++d) {
        issue(it_tile, it_kc, d);
        advance(it_tile, it_kc);
    }

    // activations may come from the previous kernel: wait for it
    griddep_wait();
    float qs[MX];  // XM 2: the scale of each token's codes
#pragma unroll
    for (int m = 0; m < MX; ++m) qs[m] = 1.f;
    if constexpr (XM == 2) {
        find_scales();
#pragma unroll
        for (int m = 0; m < MX; ++m)
            if (m < p.M) qs[m] = qx_scale[m];
    }

    // X of a unit: lane c holds 8-k chunk c of every token (staged path)
    uint4 xr[MX];
    const uint16_t* xlane = p.X + 8 * lane;
    auto load_x = [&](int kc) {
        const int k = kc * ST_UK + 8 * lane;
#pragma unroll
        for (int m = 0; m < MX; ++m)
            if (m < p.M) {
                if constexpr (XM == 1)
                    xr[m] = (k < p.K) ? widen_i8x8(ldg_cg_v2(reinterpret_cast<const int8_t*>(p.X) + 8 * lane +
                                                             (int64_t)m * p.K + kc * ST_UK))
                                      : make_uint4(0u, 0u, 0u, 0u);
                else if constexpr (XM == 2)
                    xr[m] = (k < p.K) ? act_codes_bf16x8(ldg_cg_v4(xlane + (int64_t)m * p.K + kc * ST_UK), qs[m])
                                      : make_uint4(0u, 0u, 0u, 0u);
                else
                    xr[m] = (k < p.K) ? ldg_cg_v4(xlane + (int64_t)m * p.K + kc * ST_UK) : make_uint4(0u, 0u, 0u, 0u);
            }
    };
    const uint32_t xst = (uint32_t)(16 * st_x_slot(lane));
    auto store_x = [&](unsigned char* slot) {
#pragma unroll
        for (int m = 0; m < MX; ++m)
            if (m < p.M) {
                uint4 o;
                o.x = __byte_perm(xr[m].x, xr[m].z, 0x5410);  // (x0, x4)
                o.y = __byte_perm(xr[m].x, xr[m].z, 0x7632);  // (x1, x5)
                o.z = __byte_perm(xr[m].y, xr[m].w, 0x5410);  // (x2, x6)
                o.w = __byte_perm(xr[m].y, xr[m].w, 0x7632);  // (x3, x7)
                *reinterpret_cast<uint4*>(slot + m * ST_XPITCH + xst) = o;
            }
    };

    uint32_t cm, cg, c128;  // constants pinned in registers: nibble mask, bf16 128.0 pair (magic and bias)
    asm volatile("mov.b32 %0, %1;" : "=r"(cm) : "r"(0x000F000Fu));
    asm volatile("mov.b32 %0, %1;" : "=r"(cg) : "r"(0x43004300u));
    c128 = cg;

    const int pr = ((gid >> 1) | ((gid & 1) << 2));  // MMA row gid <- tile row pr (bank-conflict-free swizzled reads)
    const uint32_t cpos0 = ((uint32_t)tq ^ (uint32_t)pr) << 4, cpos1 = ((uint32_t)(4 + tq) ^ (uint32_t)pr) << 4;
    uint32_t boff[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) boff[j] = 16u * (uint32_t)((4 * tq + j) ^ ((tq >> 1) << 1));
    const uint32_t jq0 = (uint32_t)(((32 * tq) / G) * 2), jq1 = (uint32_t)(((128 + 32 * tq) / G) * 2);
    const uint32_t xrow_off = (uint32_t)(gid * ST_XPITCH);
    const uint32_t zaddr = smem_u32(zrow);

    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
    float ya[RT], yb[RT];      // one-token path: rows pr, pr + 8 (of each row tile) over this lane's slices
    float oacc[RT][1][4];      // one-token path: the owner's sums of its last tile, kept for after the loop
#pragma unroll
    for (int rt = 0; rt < RT; ++rt) ya[rt] = yb[rt] = 0.f;
    float xpart = 0.f;         // one-token path: sum of the lane's 8-k chunk of X
    int tile = tile0, kc = kc0, kc_first = kc0;  // unit being computed
    bool owner_split = false;                    // the range ends inside a tile whose first unit it holds
    int x_kc = kc0;                               // unit whose X sits in xr
    bool ok = true;
    int d = 0;
    uint32_t phase = 0;

    load_x(x_kc);
    for (int it = 0; it < nunits; ++it) {
        store_x(xs);
        if (DIAG) xpart = bf16x8_sum(xr[0]);
        if (it + 1 < nunits) {
            if (++x_kc == p.nkc) x_kc = 0;
            load_x(x_kc);
        }
        ok = mbar_wait_bounded(bars + 8 * d, phase, nullptr, &g_stream_fault, 1u, ST_WAIT_LIMIT_NS) && ok;
        __syncwarp();

        const uint32_t ws_a = wslots + d * WSLOT + pr * 128;   // row pr of the (first) row tile; row tile rt
        const uint32_t ws_b = ws_a + 8 * 128;                  // starts 16 rows (16 x 128 bytes) further
        const uint32_t qa = qslots + d * QSLOT + pr * QROW;  // scales of row pr; offsets ROWS rows further
        const uint32_t qb = qa + 8 * QROW;
        const uint32_t bbase = gid < p.M ? smem_u32(xs) + xrow_off : zaddr;
        float dacc[RT][4];  // one-token path: D[row][slice] of this unit, per row tile
#pragma unroll
        for (int h = 0; h < 2; ++h) {  // two 128-k steps per unit
            const uint32_t cpos = h ? cpos1 : cpos0;
            if constexpr (DIAG) {
                uint32_t wa4[RT][4], wb4[RT][4];
#pragma unroll
                for (int rt = 0; rt < RT; ++rt) {
                    const uint4 wa = lds128_st(ws_a + rt * 16 * 128 + cpos);
                    const uint4 wb = lds128_st(ws_b + rt * 16 * 128 + cpos);
                    wa4[rt][0] = wa.x, wa4[rt][1] = wa.y, wa4[rt][2] = wa.z, wa4[rt][3] = wa.w;
                    wb4[rt][0] = wb.x, wb4[rt][1] = wb.y, wb4[rt][2] = wb.z, wb4[rt][3] = wb.w;
                }
                // X only on the lane whose column is its own slice (gid = tq + 4h)
                const uint32_t bd = (gid == tq + 4 * h) ? smem_u32(xs) : zaddr;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    const uint4 xv = lds128_st(bd + 256u * h + boff[j]);
#pragma unroll
                    for (int rt = 0; rt < RT; ++rt) {  // one X fragment, every row tile of the unit
                        if (h == 0 && j == 0)
                            raw_mma<0, true>(dacc[rt], wa4[rt][j], wb4[rt][j], xv.x, xv.y, cm, cg);
                        else
                            raw_mma<0, false>(dacc[rt], wa4[rt][j], wb4[rt][j], xv.x, xv.y, cm, cg);
                        raw_mma<8, false>(dacc[rt], wa4[rt][j], wb4[rt][j], xv.z, xv.w, cm, cg);
                    }
                }
                continue;
            }
            const uint4 wa = lds128_st(ws_a + cpos);
            const uint4 wb = lds128_st(ws_b + cpos);
            const uint32_t wa4[4] = {wa.x, wa.y, wa.z, wa.w};
            const uint32_t wb4[4] = {wb.x, wb.y, wb.z, wb.w};
            const uint32_t jq = h ? jq1 : jq0;
            const uint32_t sa = lds_u16_st(qa + jq), oa = lds_u16_st(qa + ROWS * QROW + jq);
            const uint32_t sb = lds_u16_st(qb + jq), ob = lds_u16_st(qb + ROWS * QROW + jq);
            const uint32_t sa2 = __byte_perm(sa, 0, 0x1010), oa2 = __byte_perm(oa, 0, 0x1010);
            const uint32_t sb2 = __byte_perm(sb, 0, 0x1010), ob2 = __byte_perm(ob, 0, 0x1010);
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const uint4 xv = lds128_st(bbase + 256u * h + boff[j]);
                dq_mma<0>(acc[0], wa4[j], wb4[j], sa2, oa2, sb2, ob2, xv.x, xv.y, cm, cg, c128);
                dq_mma<8>(acc[0], wa4[j], wb4[j], sa2, oa2, sb2, ob2, xv.z, xv.w, cm, cg, c128);
            }
        }
        if constexpr (DIAG) {  // apply the groups' scales and offsets to the slice sums (before the slot refill)
            float xsl = xpart;
            xsl += __shfl_xor_sync(0xffffffffu, xsl, 1);
            xsl += __shfl_xor_sync(0xffffffffu, xsl, 2);  // lanes 4c .. 4c+3: sum of slice c
            const float xs0 = __shfl_sync(0xffffffffu, xsl, 8 * tq), xs1 = __shfl_sync(0xffffffffu, xsl, 8 * tq + 4);
#pragma unroll
            for (int rt = 0; rt < RT; ++rt) {
                // this lane's columns are slices 2tq and 2tq+1: D[pr][.] in dacc[rt][0..1], D[pr+8][.] in [2..3]
                const uint32_t qra = qa + rt * 16 * QROW, qrb = qb + rt * 16 * QROW;
                if constexpr (G == 32) {  // two groups, adjacent in the qparam rows
                    const uint32_t sA = lds_u32_st(qra + 4 * tq), oA = lds_u32_st(qra + ROWS * QROW + 4 * tq);
                    const uint32_t sB = lds_u32_st(qrb + 4 * tq), oB = lds_u32_st(qrb + ROWS * QROW + 4 * tq);
                    ya[rt] = fmaf(bf16_lo(sA), fmaf(-128.f, xs0, dacc[rt][0]), ya[rt]);
                    ya[rt] = fmaf(bf16_lo(oA), xs0, ya[rt]);
                    ya[rt] = fmaf(bf16_hi(sA), fmaf(-128.f, xs1, dacc[rt][1]), ya[rt]);
                    ya[rt] = fmaf(bf16_hi(oA), xs1, ya[rt]);
                    yb[rt] = fmaf(bf16_lo(sB), fmaf(-128.f, xs0, dacc[rt][2]), yb[rt]);
                    yb[rt] = fmaf(bf16_lo(oB), xs0, yb[rt]);
                    yb[rt] = fmaf(bf16_hi(sB), fmaf(-128.f, xs1, dacc[rt][3]), yb[rt]);
                    yb[rt] = fmaf(bf16_hi(oB), xs1, yb[rt]);
                } else {  // both slices in one group
                    const uint32_t go = (uint32_t)(((64 * tq) / G) * 2);
                    const float x01 = xs0 + xs1;
                    const float sa = bf16_lo(lds_u16_st(qra + go)), oa = bf16_lo(lds_u16_st(qra + ROWS * QROW + go));
                    const float sb = bf16_lo(lds_u16_st(qrb + go)), ob = bf16_lo(lds_u16_st(qrb + ROWS * QROW + go));
                    ya[rt] = fmaf(sa, fmaf(-128.f, x01, dacc[rt][0] + dacc[rt][1]), ya[rt]);
                    ya[rt] = fmaf(oa, x01, ya[rt]);
                    yb[rt] = fmaf(sb, fmaf(-128.f, x01, dacc[rt][2] + dacc[rt][3]), yb[rt]);
                    yb[rt] = fmaf(ob, x01, yb[rt]);
                }
            }
        }
        __syncwarp();
        if (it + DEPTH < nunits) {  // refill the slot (its reads are done: order them before the async writes)
            fence_proxy_async_smem();
            issue(it_tile, it_kc, d);
            advance(it_tile, it_kc);
        }
        if (++d == DEPTH) {
            d = 0;
            phase ^= 1u;
        }

        // end of a row tile or of the range: hand the tile's sums on
        if ((it + 1 == nunits || kc == p.nkc - 1) && DIAG) {
            // the row sums over the four lanes of a row pair (slices 0..7), per row tile
            float racc[RT][1][4];
#pragma unroll
            for (int rt = 0; rt < RT; ++rt) {
                ya[rt] += __shfl_xor_sync(0xffffffffu, ya[rt], 1);
                ya[rt] += __shfl_xor_sync(0xffffffffu, ya[rt], 2);
                yb[rt] += __shfl_xor_sync(0xffffffffu, yb[rt], 1);
                yb[rt] += __shfl_xor_sync(0xffffffffu, yb[rt], 2);
                racc[rt][0][0] = ya[rt];  // token 0 of rows pr, pr + 8 of row tile rt (the tq = 0 lanes write)
                racc[rt][0][2] = yb[rt];
                racc[rt][0][1] = racc[rt][0][3] = 0.f;
                ya[rt] = yb[rt] = 0.f;
            }
            if (kc_first == 0 && kc == p.nkc - 1) {  // this warp summed all of the tile's k
#pragma unroll
                for (int rt = 0; rt < RT; ++rt) {
                    const int n_a = tile * ROWS + 16 * rt + pr, n_b = n_a + 8;
                    if (tq == 0 && n_a < p.N)
                        p.Y[n_a] = (uint16_t)float_to_bf16_bits(epilogue_f32(ep, racc[rt][0][0], 0, n_a));
                    if (tq == 0 && n_b < p.N)
                        p.Y[n_b] = (uint16_t)float_to_bf16_bits(epilogue_f32(ep, racc[rt][0][2], 0, n_b));
                }
            } else if (kc_first != 0) {  // a later share of the tile (the first of this range): publish it
#pragma unroll
                for (int rt = 0; rt < RT; ++rt)
                    split_publish<1>(p.ws + ((size_t)worker * RT + rt) * 16, racc[rt], 1,
                                     min(16, p.N - (tile * ROWS + 16 * rt)), pr, tq);
            } else {  // the tile's owner: its range ends here (last iteration); finished after the loop
#pragma unroll
                for (int rt = 0; rt < RT; ++rt)
#pragma unroll
                    for (int i = 0; i < 4; ++i) oacc[rt][0][i] = racc[rt][0][i];
                owner_split = true;
                break;
            }
            kc_first = 0;
        } else if (it + 1 == nunits || kc == p.nkc - 1) {
            const int n_a = tile * 16 + pr, n_b = n_a + 8;
            // acc[t] = D[row n_a: tokens 8t + 2tq, +1 | row n_b: the same tokens]
            if (kc_first == 0 && kc == p.nkc - 1) {  // this warp summed all of the tile's k
#pragma unroll
                for (int t = 0; t < MT; ++t)
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int m = 8 * t + 2 * tq + (i & 1), n = (i < 2) ? n_a : n_b;
                        if (m < p.M && n < p.N)
                            p.Y[(int64_t)m * p.N + n] = (uint16_t)float_to_bf16_bits(epilogue_f32(ep, acc[t][i], m, n));
                    }
            } else if (kc_first != 0) {  // a later share of the tile (the first of this range): publish it
                split_publish<MT>(p.ws + (size_t)worker * 16 * p.M, acc, p.M, min(16, p.N - tile * 16), pr, tq);
            } else {  // the tile's owner: its range ends here (last iteration); finished after the loop
                owner_split = true;
                break;
            }
#pragma unroll
            for (int t = 0; t < MT; ++t) acc[t][0] = acc[t][1] = acc[t][2] = acc[t][3] = 0.f;
            kc_first = 0;
        }
        advance(tile, kc);
    }
    if (owner_split) {  // add the later shares of the last tile (their warps publish without waiting), write Y
        const int wl = split_warp_of((long long)tile * p.nkc + p.nkc - 1, p.units, p.workers);
        constexpr int NE = MX / 2 ? MX / 2 : 1;  // slot words per lane (16 M / 32)
        if constexpr (DIAG) {
            int nrows[RT];
#pragma unroll
            for (int rt = 0; rt < RT; ++rt) nrows[rt] = min(16, p.N - (tile * ROWS + 16 * rt));
            ok = collect_one_token<RT>(oacc, scr, p.ws, worker, wl, nrows, pr, tq, lane, p.Y + (int64_t)tile * ROWS,
                                       &g_stream_fault, 2u, ST_WAIT_LIMIT_NS, epilogue_at(ep, (int64_t)tile * ROWS)) &&
                 ok;
        } else {
            ok = split_collect<MT, NE>(acc, scr, p.ws, (size_t)16 * p.M, worker, wl, p.M, min(16, p.N - tile * 16), pr,
                                       tq, lane, p.Y + (int64_t)tile * 16, p.N, &g_stream_fault, 2u,
                                       ST_WAIT_LIMIT_NS, epilogue_at(ep, (int64_t)tile * 16)) &&
                 ok;
        }
    }
    if (!ok) {  // never leave with copies still landing in shared memory
        for (int it = max(0, nunits - DEPTH); it < nunits; ++it)
            mbar_drain_bounded(bars + 8 * (it % DEPTH), (uint32_t)((it / DEPTH) & 1), ST_WAIT_LIMIT_NS);
    }
}

// ------------------------------------------------------------------ host side

static_assert((size_t)SPLIT_MAX_WORKERS * 16 * STREAM_MAX_M * 8 <= I8_SCRATCH_OFFSET &&
                  (size_t)2 * SPLIT_MAX_WORKERS * 16 * 8 <= I8_SCRATCH_OFFSET,
              "the int8 linear's scratch must lie past every slot region");

bool plan_stream(int64_t M, int64_t N, int64_t K, int g, StreamPlan* plan) {
    if (M < 1 || M > STREAM_MAX_M) return false;
    const int64_t ng = K / g;
    if (ng % 2 != 0 || ng < 2) return false;  // 4-byte qparam pieces need an even group count
    const int64_t tiles = (N + 15) / 16;
    if (tiles > 0x3FFFFFFF) return false;
    plan->nkc = (int)((K + ST_UK - 1) / ST_UK);
    plan->units = tiles * plan->nkc;
    plan->tiles = tiles;
    plan->smem = (size_t)st_smem_bytes((int)M, g, 1);
    plan->ws_bytes = split_ws_bytes(M, plan->units);
    return true;
}

template <int G, int MX, bool QT, int RT, int XM>
static cudaError_t launch_stream_gm(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& to, StreamArgs a,
                                    cudaStream_t stream) {
    auto kern = stream_kernel<G, MX, QT, RT, XM>;
    const size_t smem = (size_t)st_smem_bytes(a.M, G, RT);
    cudaError_t e = ensure_kernel_attrs(reinterpret_cast<const void*>(kern), st_smem_bytes(MX, G, RT), false);
    if (e != cudaSuccess) return e;
    // one wave: as many resident warps as the SMs hold, but no more than there are units
    int sms = 0, per_sm = 0;
    if ((e = resident_blocks(reinterpret_cast<const void*>(kern), ST_THREADS, smem, &sms, &per_sm)) != cudaSuccess)
        return e;
    const long long max_workers = std::min<long long>((long long)sms * per_sm * ST_WARPS, SPLIT_MAX_WORKERS);
    a.workers = (int)std::min<long long>(max_workers, a.units);
    const int blocks = (a.workers + ST_WARPS - 1) / ST_WARPS;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(ST_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tw, ts, to, a);
}

template <int G, bool QT, int XM>
static cudaError_t launch_stream_g(const CUtensorMap& tw, const CUtensorMap& ts, const CUtensorMap& to, StreamArgs a,
                                   int rt, cudaStream_t stream) {
    if (rt == 2) return launch_stream_gm<G, 1, QT, 2, XM>(tw, ts, to, a, stream);
    if (a.M <= 1) return launch_stream_gm<G, 1, QT, 1, XM>(tw, ts, to, a, stream);
    if (a.M <= 2) return launch_stream_gm<G, 2, QT, 1, XM>(tw, ts, to, a, stream);
    return launch_stream_gm<G, 4, QT, 1, XM>(tw, ts, to, a, stream);
}

// One token takes 32-row units (two row tiles sharing the X staging, slice sums
// and ring work of a unit) when there are enough of them for at least half the
// resident warps, and the workspace holds two 16-row slots for each warp that
// runs.  Measured on the Llama-3-8B decode step: gate / up / down and q / o
// (4096 x 4096, 2048 units for about 2400 resident warps) are faster with them;
// k / v (512 units) are faster with 16-row units.
template <int G, bool QT>
static cudaError_t two_row_tiles(int64_t N, int nkc, size_t ws_bytes, bool* two) {
    auto kern = stream_kernel<G, 1, QT, 2, 0>;
    cudaError_t e = ensure_kernel_attrs(reinterpret_cast<const void*>(kern), st_smem_bytes(1, G, 2), false);
    int sms = 0, per_sm = 0;
    if (e == cudaSuccess)
        e = resident_blocks(reinterpret_cast<const void*>(kern), ST_THREADS, st_smem_bytes(1, G, 2), &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const long long max_workers = std::min<long long>((long long)sms * per_sm * ST_WARPS, SPLIT_MAX_WORKERS);
    const long long units = (N + 31) / 32 * (long long)nkc;
    *two = 2 * units >= max_workers && (size_t)std::min<long long>(max_workers, units) * 2 * 16 * 8 <= ws_bytes;
    return cudaSuccess;
}

template <int XM>
static cudaError_t launch_stream_t(const StreamPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                                   const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                                   void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep) {
    if (M > 4) {  // 5..32 tokens: the block-shared X kernel (w4_batch.cu), bf16 X only
        if (XM != 0) return cudaErrorInvalidValue;
        return launch_batch(plan, X, M, K, Wq, scales, offsets, N, g, 4, Y, workspace, stream, detail, ep);
    }
    const int64_t ng = K / g;
    const bool qt = (g == 32) && (ng % 8 == 0);  // qparam rows 16-byte aligned: 8-group TMA boxes
    cudaError_t e = cudaSuccess;
    bool two = false;
    if (M == 1) {
        e = g == 32 ? (qt ? two_row_tiles<32, true>(N, plan.nkc, plan.ws_bytes, &two)
                          : two_row_tiles<32, false>(N, plan.nkc, plan.ws_bytes, &two))
                    : g == 64 ? two_row_tiles<64, false>(N, plan.nkc, plan.ws_bytes, &two)
                              : two_row_tiles<128, false>(N, plan.nkc, plan.ws_bytes, &two);
        if (e != cudaSuccess) return e;
    }
    const int rt = two ? 2 : 1;
    // codes: [N][K/2] bytes, one box = 16 rt rows x 128 bytes (256 k), 128-byte swizzle
    CUtensorMap tw, ts, to;
    e = encode_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, (uint64_t)(K / 2), (uint64_t)N, (uint64_t)(K / 2),
                             128, 16 * rt, CU_TENSOR_MAP_SWIZZLE_128B, detail);
    if (e != cudaSuccess) return e;
    ts = tw;
    to = tw;
    if (qt) {
        e = encode_tensor_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, (uint64_t)ng, (uint64_t)N,
                                 (uint64_t)ng * 2, 8, 16 * rt, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e == cudaSuccess)
            e = encode_tensor_map_2d(&to, CU_TENSOR_MAP_DATA_TYPE_UINT16, offsets, (uint64_t)ng, (uint64_t)N,
                                     (uint64_t)ng * 2, 8, 16 * rt, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e != cudaSuccess) return e;
    }
    StreamArgs a;
    a.X = X;
    a.scales = scales;
    a.offsets = offsets;
    a.Y = Y;
    a.ep = ep;
    a.ws = static_cast<uint64_t*>(workspace);
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.nkc = plan.nkc;
    a.units = rt == 2 ? (N + 31) / 32 * (long long)plan.nkc : plan.units;
    a.workers = 0;
    switch (g) {
        case 32:
            return qt ? launch_stream_g<32, true, XM>(tw, ts, to, a, rt, stream)
                      : launch_stream_g<32, false, XM>(tw, ts, to, a, rt, stream);
        case 64: return launch_stream_g<64, false, XM>(tw, ts, to, a, rt, stream);
        default: return launch_stream_g<128, false, XM>(tw, ts, to, a, rt, stream);
    }
}

cudaError_t launch_stream(const StreamPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                          const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                          void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep) {
    return launch_stream_t<0>(plan, X, M, K, Wq, scales, offsets, N, g, Y, workspace, stream, detail, ep);
}

cudaError_t launch_stream_i8(const StreamPlan& plan, const int8_t* Xq, int64_t M, int64_t K, const uint8_t* Wq,
                             const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                             void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep) {
    return launch_stream_t<1>(plan, reinterpret_cast<const uint16_t*>(Xq), M, K, Wq, scales, offsets, N, g, Y,
                              workspace, stream, detail, ep);
}

cudaError_t launch_stream_qx(const StreamPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                             const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                             void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep) {
    return launch_stream_t<2>(plan, X, M, K, Wq, scales, offsets, N, g, Y, workspace, stream, detail, ep);
}


cudaError_t read_and_clear_stream_fault(unsigned int* fault) {
    cudaError_t e = cudaMemcpyFromSymbol(fault, g_stream_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !*fault) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_stream_fault, &zero, sizeof(unsigned int));
}

}  // namespace w4
