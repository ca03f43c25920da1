// w4_tcdec.cu -- bf16 x int4 linear for a batch of 5..32 tokens on the
// 5th-generation tensor cores (tcgen05) of sm_103a.
//
// Y[m,n] = sum_k X[m,k] * w'[n,k], w' = bf16(q*s + o), fp32 accumulation in
// tensor memory (Optimum Quanto: bf16 x int4 matmul with higher-precision
// accumulation, "Pitfalls when quantizing activations").  With up to 32
// tokens each weight feeds few products, so the work is the weights' bytes
// and their dequantization, not the multiplies.  The kernel keeps the prefill
// GEMM's division of labour, in which one thread issues every MMA and the
// weights go from registers straight into tensor memory, and gives it the
// decode kernels' partition of the work:
//   * A persistent grid, one block per SM, cuts the problem's units (128 weight
//     rows x 256 k) into equal contiguous ranges (stream-K).  A range is walked
//     in k order, tile after tile.
//   * warp 0    TMA producer: one ring stage per unit holds the code tile (128
//               rows x 128 bytes, 128-byte swizzle), four X sub-tiles (MT tokens x 64 k, 128-byte
//               swizzle, the UMMA B layout; rows past M read 0) and, when the
//               rows allow it, the scale / offset boxes of the unit's 8 groups.
//               The TMA unit's cost grows with the number of rows it fetches,
//               so whole 128-byte lines keep it off the critical path;
//     warp 1    tensor-memory owner and, on one lane, the UMMA issuer: per 64-k
//               sub-block 4 x tcgen05.mma (M=128 from tensor memory, N=MT,
//               K=16) into one fp32 accumulator of MT columns;
//     warps 2-9 dequantization: thread (row, 32-k half) of its tensor-memory
//               sub-partition turns 32 codes of a sub-block into 16 bf16 pairs
//               with LOP3 magic, one exact subtract and one bf16 FMA a pair,
//               and stores them with one tcgen05.st; at the end of each tile of
//               the range the same warps read the accumulator back
//               (tcgen05.ld) and finish it.
//   * A tile whose k the range covers whole is written to Y.  A tile split
//     between ranges is finished by the block holding its first unit (the
//     owner; the tile is the last of its range): every later block stores its
//     partial sums in its own workspace slot as 8-byte words {fp32 sum, flag}
//     (one naturally aligned store, so value and flag arrive together) and goes
//     on; the owner adds the slots in block order to its own sums, writes Y and
//     zeroes them.  No atomics; the order of the additions is fixed, so results
//     are deterministic on a given GPU.  All blocks of the grid are resident at
//     once (one per SM), so an owner never waits for a block that cannot run;
//     the wait is bounded anyway.
// Every wait is bounded in time; a block that gives up sets the device fault
// word, waits (bounded) for its own copies and MMAs, frees its tensor memory
// and exits.
#include "w4_device.cuh"
#include "w4_internal.h"
#include "w4_tc.cuh"

#include <algorithm>

namespace w4 {

constexpr int TD_BW = 128;        // weight rows per tile (UMMA M, tensor-memory lanes)
constexpr int TD_UK = 256;        // k per unit: one 128-byte line of codes per row
constexpr int TD_SK = 64;         // k per sub-block (one A stage, four UMMAs of K=16)
constexpr int TD_NSUB = TD_UK / TD_SK;
constexpr int TD_WSTAGES = 4;     // dequantized sub-blocks in tensor memory (the UMMA A operand)
constexpr int TD_DEQ_WARPS = 8;
constexpr int TD_THREADS = 64 + TD_DEQ_WARPS * 32;
constexpr int TD_TMEM_COLS = 256;
constexpr int TD_ACOL = 64;                 // first tensor-memory column of the A stages (D: columns 0 .. MT-1)
constexpr int TD_ASTAGE_COLS = TD_SK / 2;   // 64 bf16 of a row = 32 columns
constexpr int TD_P_BYTES = TD_BW * TD_UK / 2;  // 16 KB of codes per unit
constexpr int TD_QBOX_BYTES = TD_BW * 16;      // 2 KB: 8 bf16 per row
constexpr uint64_t TD_WAIT_LIMIT_NS = 2000000000ull;
constexpr uint64_t TD_DRAIN_LIMIT_NS = 1000000000ull;
static_assert(TD_ACOL + TD_WSTAGES * TD_ASTAGE_COLS <= TD_TMEM_COLS, "tensor-memory budget");

// One TMA stage per unit: the code tile (128 rows x 128 bytes, 128-byte swizzle),
// the X sub-tiles (four of MT tokens x 64 k, 128-byte swizzle, the UMMA B
// layout) and, when the rows allow it, the scale and offset boxes of the 8
// groups around the unit.  Every piece starts on a 1024-byte boundary.
template <int MT>
struct TdLayout {
    static constexpr int XSUB = MT * TD_SK * 2;  // 2 / 4 KB
    static constexpr int STAGE = TD_P_BYTES + TD_NSUB * XSUB + 2 * TD_QBOX_BYTES;
    static constexpr int TSTAGES = MT == 16 ? 6 : 5;
    static constexpr int NBAR = 2 * TSTAGES + 2 * TD_WSTAGES + 2;  // full / empty per stage and A stage; tile_done; drain
    static constexpr int OFF_BAR = TSTAGES * STAGE;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + alignment slack for the swizzle atoms
    static_assert(XSUB % 1024 == 0 && STAGE % 1024 == 0 && SMEM_BYTES <= 227 * 1024, "shared-memory layout");
};

struct TdArgs {
    const uint16_t* scales;
    const uint16_t* offsets;
    uint16_t* Y;
    Epilogue ep;
    uint64_t* ws;      // block c's slot: MT x 128 words at ws + c * MT * 128, zero between calls
    int M, N, K;
    int nkc;           // units per tile (ceil(K / 256))
    long long units;   // tiles x nkc
};

__device__ unsigned int g_tcdec_fault;

// tcgen05.mma kind::f16: D fp32, A and B bf16, both K-major, N = MT, M = 128.
template <int MT>
constexpr uint32_t td_idesc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(MT >> 3) << 17) | ((uint32_t)(TD_BW >> 4) << 24);
}

// unit cursor: tile and 256-k column of unit u, advanced without division
struct TdCursor {
    int tile, kc, nkc;
    __device__ void next() {
        if (++kc == nkc) {
            kc = 0;
            ++tile;
        }
    }
};

// first group of the 8-group qparam box that holds unit column kc (8-group aligned)
template <int G>
__device__ __forceinline__ int td_box_group(int kc) {
    return ((kc * TD_UK / G) / 8) * 8;
}

template <int G, bool QT, int MT>
__global__ void __launch_bounds__(TD_THREADS, 1)
tcdec_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_p,
             const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_o, const TdArgs p) {
    using L = TdLayout<MT>;
    constexpr int TS = L::TSTAGES;
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + L::OFF_BAR;
    auto stage_p = [&](int t) { return sbase + (uint32_t)(t * L::STAGE); };
    auto stage_x = [&](int t, int s) { return sbase + (uint32_t)(t * L::STAGE + TD_P_BYTES + s * L::XSUB); };
    auto stage_q = [&](int t) { return sbase + (uint32_t)(t * L::STAGE + TD_P_BYTES + TD_NSUB * L::XSUB); };
    auto full_tma = [&](int t) { return bar0 + 8u * t; };
    auto empty_tma = [&](int t) { return bar0 + 8u * (TS + t); };
    auto full_deq = [&](int w) { return bar0 + 8u * (2 * TS + w); };
    auto empty_w = [&](int w) { return bar0 + 8u * (2 * TS + TD_WSTAGES + w); };
    const uint32_t tile_done = bar0 + 8u * (2 * TS + 2 * TD_WSTAGES);
    const uint32_t drain = tile_done + 8u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int cta = blockIdx.x, nctas = gridDim.x;
    const long long u0 = p.units * cta / nctas, u1 = p.units * (cta + 1) / nctas;
    const int nunits = (int)(u1 - u0);  // >= 1: the host launches at most `units` blocks
    const TdCursor first = {(int)(u0 / p.nkc), (int)(u0 % p.nkc), p.nkc};
    // the next launch may start once every block of this one has (so all of this grid is resident)
    griddep_launch_dependents();

    if (threadIdx.x == 0) {
        for (int t = 0; t < TS; ++t) {
            mbar_init(full_tma(t), 1);
            mbar_init(empty_tma(t), 1);
        }
        for (int w = 0; w < TD_WSTAGES; ++w) {
            mbar_init(full_deq(w), TD_DEQ_WARPS * 32);
            mbar_init(empty_w(w), 1);
        }
        mbar_init(tile_done, 1);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TD_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    // X, Y and the workspace may belong to the kernel before this one
    griddep_wait();

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(&tm_p);
            if (QT) {
                tma_prefetch_desc(&tm_s);
                tma_prefetch_desc(&tm_o);
            }
            int issued = 0;
            TdCursor c = first;
            for (int i = 0; i < nunits; ++i, c.next()) {
                const int row0 = c.tile * TD_BW;
                const int t = i % TS;
                const uint32_t ph = (i / TS) & 1;
                if (!mbar_wait_bounded(empty_tma(t), ph ^ 1, abort_flag, &g_tcdec_fault, 1u, TD_WAIT_LIMIT_NS)) break;
                mbar_arrive_expect_tx(full_tma(t), TD_P_BYTES + TD_NSUB * L::XSUB + (QT ? 2 * TD_QBOX_BYTES : 0));
                tma_load_2d(stage_p(t), &tm_p, full_tma(t), c.kc * (TD_UK / 2), row0);
#pragma unroll
                for (int s = 0; s < TD_NSUB; ++s)
                    tma_load_2d(stage_x(t, s), &tm_x, full_tma(t), c.kc * TD_UK + s * TD_SK, 0);
                if (QT) {
                    const int gb = td_box_group<G>(c.kc);
                    tma_load_2d(stage_q(t), &tm_s, full_tma(t), gb, row0);
                    tma_load_2d(stage_q(t) + TD_QBOX_BYTES, &tm_o, full_tma(t), gb, row0);
                }
                ++issued;
            }
            // never leave the block with copies still landing in its shared memory
            for (int i = (issued > TS ? issued - TS : 0); i < issued; ++i)
                mbar_drain_bounded(full_tma(i % TS), (i / TS) & 1, TD_DRAIN_LIMIT_NS);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = td_idesc<MT>();
            int issued = 0;
            TdCursor c = first;
            bool ok = true;
            for (int i = 0; i < nunits && ok; ++i, c.next()) {
                const bool tile_first = i == 0 || c.kc == 0;
                const bool tile_last = i == nunits - 1 || c.kc == p.nkc - 1;
                const int t = i % TS;
                if (!mbar_wait_bounded(full_tma(t), (i / TS) & 1, abort_flag, &g_tcdec_fault, 2u, TD_WAIT_LIMIT_NS)) break;
                for (int s = 0; s < TD_NSUB; ++s) {
                    const int sb = i * TD_NSUB + s, w = sb % TD_WSTAGES;
                    if (!mbar_wait_bounded(full_deq(w), (sb / TD_WSTAGES) & 1, abort_flag, &g_tcdec_fault, 2u,
                                           TD_WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = sw128_kmajor_desc(stage_x(t, s));
                    const uint32_t a_tmem = tmem + (uint32_t)(TD_ACOL + w * TD_ASTAGE_COLS);
#pragma unroll
                    for (int kk = 0; kk < TD_SK / 16; ++kk)  // K=16 a step: 8 A columns, +32 bytes of B (+2 in the desc)
                        umma_bf16_tmem_a(tmem, a_tmem + 8u * kk, bdesc + 2u * kk, idesc,
                                         (tile_first && s == 0 && kk == 0) ? 0u : 1u);
                    umma_commit(empty_w(w));  // A stage consumed
                    ++issued;
                }
                if (!ok) break;
                umma_commit(empty_tma(t));  // codes, X and qparams of this unit consumed
                if (tile_last) umma_commit(tile_done);  // the tile's sums are complete when these MMAs are
            }
            // the MMAs must be finished before tensor memory is released
            if (issued > 0) {
                umma_commit(drain);
                mbar_drain_bounded(drain, 0, TD_DRAIN_LIMIT_NS);
            }
        }
    } else {
        // --------------------------------------------- dequantization and epilogue warps
        const int sp = warp & 3;         // tensor-memory sub-partition: lanes (weight rows) 32 sp .. 32 sp + 31
        const int hh = (warp - 2) >> 2;  // which 32-k half of each sub-block; which half of the tokens in the epilogue
        const int r = 32 * sp + lane;    // weight row within the tile
        const int ng = p.K / G;
        // scale and offset of this row for this thread's half of a sub-block, loaded four
        // sub-blocks ahead and kept raw until used (no-TMA variant); rows past N and groups
        // past K read as 0, so with the zero-filled codes those weights are exactly 0
        struct QRaw {
            uint32_t s, o;
        };
        TdCursor qc = first;
        int qs = 0, qi = 0;
        auto qload = [&]() {
            QRaw q = {0u, 0u};
            if (!QT && qi < nunits) {
                const int n = qc.tile * TD_BW + r, j = (qc.kc * TD_UK + qs * TD_SK + 32 * hh) / G;
                if (n < p.N && j < ng) {
                    q.s = ldg_nc_u16(p.scales + (int64_t)n * ng + j);
                    q.o = ldg_nc_u16(p.offsets + (int64_t)n * ng + j);
                }
            }
            if (++qs == TD_NSUB) {
                qs = 0;
                ++qi;
                qc.next();
            }
            return q;
        };
        QRaw q0 = qload(), q1 = qload(), q2 = qload(), q3 = qload();
        uint32_t cm, cg;  // LOP3 constants pinned in registers (0x4300 pairs are also the 128.0 bias)
        asm volatile("mov.b32 %0, %1;" : "=r"(cm) : "r"(0x000F000Fu));
        asm volatile("mov.b32 %0, %1;" : "=r"(cg) : "r"(0x43004300u));
        const uint32_t a_lane = tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)(TD_ACOL + 16 * hh);
        const uint32_t d_lane = tmem + ((uint32_t)(32 * sp) << 16);
        uint64_t* const my_slot = p.ws + (size_t)cta * MT * TD_BW;
        constexpr int MH = MT / 2;  // tokens of this thread in the epilogue: hh MH .. hh MH + MH - 1
        bool ok = true;
        int tiles_done = 0, tile_kc0 = first.kc;
        TdCursor c = first;
        for (int i = 0; i < nunits && ok; ++i, c.next()) {
            if (i > 0 && c.kc == 0) tile_kc0 = 0;
            const int t = i % TS;
            if (!mbar_wait_bounded(full_tma(t), (i / TS) & 1, abort_flag, &g_tcdec_fault, 4u, TD_WAIT_LIMIT_NS)) {
                ok = false;
                break;
            }
            uint4 sq = make_uint4(0u, 0u, 0u, 0u), oq = sq;  // TMA variant: this row's 8 groups
            if (QT) {
                sq = lds128(stage_q(t) + r * 16);
                oq = lds128(stage_q(t) + TD_QBOX_BYTES + r * 16);
            }
            const int gb = td_box_group<G>(c.kc);
            for (int s = 0; s < TD_NSUB; ++s) {
                const QRaw qr = q0;
                q0 = q1;
                q1 = q2;
                q2 = q3;
                q3 = qload();
                const int sb = i * TD_NSUB + s, w = sb % TD_WSTAGES;
                if (!mbar_wait_bounded(empty_w(w), ((sb / TD_WSTAGES) & 1) ^ 1, abort_flag, &g_tcdec_fault, 4u,
                                       TD_WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // the MMAs that read this A stage are complete
                uint32_t s2, o2;   // (s,s) and (o,o) bf16 pairs of this half's group
                if (QT) {
                    const int j = (c.kc * TD_UK + s * TD_SK + 32 * hh) / G - gb;  // group among the box's 8
                    const uint32_t sel = (j & 1) ? 0x3232u : 0x1010u;
                    s2 = __byte_perm(pick_word(sq, j >> 1), 0, sel);
                    o2 = __byte_perm(pick_word(oq, j >> 1), 0, sel);
                } else {
                    s2 = __byte_perm(qr.s, 0, 0x1010);
                    o2 = __byte_perm(qr.o, 0, 0x1010);
                }
                // 32 codes of this row: 16-byte chunk 2s + hh of its 128-byte line, 128-byte swizzle
                const uint32_t chunk = (uint32_t)((2 * s + hh) ^ (r & 7));
                const uint4 words = lds128(stage_p(t) + (uint32_t)(r * 128) + 16u * chunk);
                tmem_st_16cols(a_lane + (uint32_t)(w * TD_ASTAGE_COLS), dequant8(words.x, s2, o2, cm, cg),
                               dequant8(words.y, s2, o2, cm, cg), dequant8(words.z, s2, o2, cm, cg),
                               dequant8(words.w, s2, o2, cm, cg));
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(full_deq(w));
            }
            if (!ok) break;

            if (!(i == nunits - 1 || c.kc == p.nkc - 1)) continue;
            // ------------------------------------------------ end of a tile of the range
            if (!mbar_wait_bounded(tile_done, (uint32_t)(tiles_done & 1), abort_flag, &g_tcdec_fault, 8u,
                                   TD_WAIT_LIMIT_NS)) {
                ok = false;
                break;
            }
            ++tiles_done;
            tc_fence_after();
            uint32_t v[32];  // D[row r][token 0 .. 31] (tokens past MT: other columns, unused)
            tmem_ld_32cols(d_lane, v);
            tmem_ld_wait();
            tc_fence_before();  // the next tile's MMAs overwrite D only after these reads
            const int n = c.tile * TD_BW + r;
            const bool whole = tile_kc0 == 0 && c.kc == p.nkc - 1;
            if (tile_kc0 > 0) {  // a later share of the tile: publish it in this block's slot
#pragma unroll
                for (int e = 0; e < MH; ++e) {
                    const int m = hh * MH + e;
                    if (m < p.M) st_relaxed_u64(my_slot + (size_t)m * TD_BW + r, (1ull << 32) | (hh ? v[MH + e] : v[e]));
                }
                continue;
            }
            float y[MH];
#pragma unroll
            for (int e = 0; e < MH; ++e) y[e] = __uint_as_float(hh ? v[MH + e] : v[e]);  // register indices only
            if (!whole) {  // the owner: add the shares of the blocks after it, in block order
                const int wl = split_warp_of((long long)c.tile * p.nkc + p.nkc - 1, p.units, nctas);
                for (int sh = cta + 1; sh <= wl; ++sh) {
                    uint64_t* slot = p.ws + (size_t)sh * MT * TD_BW;
                    uint64_t wv[MH];
#pragma unroll
                    for (int e = 0; e < MH; ++e) {
                        const int m = hh * MH + e;
                        wv[e] = m < p.M ? ld_relaxed_u64(slot + (size_t)m * TD_BW + r) : (1ull << 32);
                    }
                    uint64_t t0 = 0;
                    for (;;) {  // re-poll together the words not published yet
                        bool all = true;
#pragma unroll
                        for (int e = 0; e < MH; ++e) all = all && (wv[e] >> 32) != 0u;
                        if (all) break;
                        const uint64_t now = globaltimer_ns();
                        if (t0 == 0) t0 = now;
                        if (now - t0 > TD_WAIT_LIMIT_NS || *abort_flag) {  // give up: count what is missing as zero
                            atomicOr(&g_tcdec_fault, 16u);
                            *abort_flag = 1;
                            ok = false;
                            break;
                        }
#pragma unroll
                        for (int e = 0; e < MH; ++e)
                            if ((wv[e] >> 32) == 0u) wv[e] = ld_relaxed_u64(slot + (size_t)(hh * MH + e) * TD_BW + r);
                    }
#pragma unroll
                    for (int e = 0; e < MH; ++e) {
                        const int m = hh * MH + e;
                        if (m < p.M) {
                            y[e] += (wv[e] >> 32) ? __uint_as_float((uint32_t)wv[e]) : 0.f;
                            st_relaxed_u64(slot + (size_t)m * TD_BW + r, 0ull);
                        }
                    }
                }
            }
            if (n < p.N) {
#pragma unroll
                for (int e = 0; e < MH; ++e) {
                    const int m = hh * MH + e;
                    if (m < p.M) p.Y[(int64_t)m * p.N + n] = (uint16_t)float_to_bf16_bits(epilogue_f32(p.ep, y[e], m, n));
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, TD_TMEM_COLS);
}

// ------------------------------------------------------------------ host side

bool plan_tcdec(int64_t M, int64_t N, int64_t K, int g, TcDecPlan* plan) {
    if (M < 1 || M > TCDEC_MAX_M || N < 1 || K < 1) return false;
    (void)g;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return false;
    plan->nkc = (int)((K + TD_UK - 1) / TD_UK);
    plan->units = (N + TD_BW - 1) / TD_BW * (long long)plan->nkc;
    plan->ctas = (int)std::min<long long>(sms, plan->units);
    plan->mt = M <= 16 ? 16 : 32;
    plan->ws_bytes = (size_t)plan->ctas * plan->mt * TD_BW * 8;
    return true;
}

template <int G, bool QT, int MT>
static cudaError_t launch_tcdec_g(const CUtensorMap& tx, const CUtensorMap& tp, const CUtensorMap& ts,
                                  const CUtensorMap& to, const TdArgs& a, int ctas, cudaStream_t stream) {
    auto kern = tcdec_kernel<G, QT, MT>;
    constexpr int SMEM = TdLayout<MT>::SMEM_BYTES;
    cudaError_t e = ensure_kernel_attrs(reinterpret_cast<const void*>(kern), SMEM, false);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)ctas, 1, 1);
    cfg.blockDim = dim3(TD_THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, tx, tp, ts, to, a);
}

template <int MT>
static cudaError_t launch_tcdec_m(const CUtensorMap& tx, const CUtensorMap& tp, const CUtensorMap& ts,
                                  const CUtensorMap& to, bool qt, int g, const TdArgs& a, int ctas,
                                  cudaStream_t stream) {
    switch (g) {
        case 32:
            return qt ? launch_tcdec_g<32, true, MT>(tx, tp, ts, to, a, ctas, stream)
                      : launch_tcdec_g<32, false, MT>(tx, tp, ts, to, a, ctas, stream);
        case 64:
            return qt ? launch_tcdec_g<64, true, MT>(tx, tp, ts, to, a, ctas, stream)
                      : launch_tcdec_g<64, false, MT>(tx, tp, ts, to, a, ctas, stream);
        default:
            return qt ? launch_tcdec_g<128, true, MT>(tx, tp, ts, to, a, ctas, stream)
                      : launch_tcdec_g<128, false, MT>(tx, tp, ts, to, a, ctas, stream);
    }
}

cudaError_t launch_tcdec(const TcDecPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                         const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                         void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep) {
    CUtensorMap tx, tp;
    // X: [M][K] bf16, box MT tokens x 64 k (128 bytes), 128-byte swizzle; token rows past M read 0
    cudaError_t e = encode_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)K, (uint64_t)M,
                                         (uint64_t)K * 2, TD_SK, (uint32_t)plan.mt, CU_TENSOR_MAP_SWIZZLE_128B,
                                         detail);
    if (e != cudaSuccess) return e;
    // codes: [N][K/2] bytes, box 128 rows x 128 bytes (256 k), 128-byte swizzle: one full line a row
    e = encode_tensor_map_2d(&tp, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, (uint64_t)(K / 2), (uint64_t)N,
                             (uint64_t)(K / 2), TD_UK / 2, TD_BW, CU_TENSOR_MAP_SWIZZLE_128B, detail);
    if (e != cudaSuccess) return e;
    const int64_t ng = K / g;
    const bool qt = ng % 8 == 0;  // qparam rows whole 16-byte pieces: 8-group boxes by TMA
    CUtensorMap ts = tp, to = tp;
    if (qt) {
        e = encode_tensor_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, (uint64_t)ng, (uint64_t)N,
                                 (uint64_t)ng * 2, 8, TD_BW, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e == cudaSuccess)
            e = encode_tensor_map_2d(&to, CU_TENSOR_MAP_DATA_TYPE_UINT16, offsets, (uint64_t)ng, (uint64_t)N,
                                     (uint64_t)ng * 2, 8, TD_BW, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e != cudaSuccess) return e;
    }
    TdArgs a;
    a.scales = scales;
    a.offsets = offsets;
    a.Y = Y;
    a.ep = ep;
    a.ws = static_cast<uint64_t*>(workspace);
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.nkc = plan.nkc;
    a.units = plan.units;
    return plan.mt == 16 ? launch_tcdec_m<16>(tx, tp, ts, to, qt, g, a, plan.ctas, stream)
                         : launch_tcdec_m<32>(tx, tp, ts, to, qt, g, a, plan.ctas, stream);
}

cudaError_t read_and_clear_tcdec_fault(unsigned int* fault) {
    cudaError_t e = cudaMemcpyFromSymbol(fault, g_tcdec_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !*fault) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_tcdec_fault, &zero, sizeof(unsigned int));
}

}  // namespace w4
