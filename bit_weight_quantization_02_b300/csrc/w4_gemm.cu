// w4_gemm.cu -- compute-bound bf16 x int4 linear for many tokens, on the
// 5th-generation tensor cores (tcgen05) of sm_103a.
//
// Y[m,n] = sum_k X[m,k] * w'[n,k], w' = bf16(q*s + o), fp32 accumulation in
// tensor memory (Optimum Quanto: bf16 x int4 matmul with higher-precision
// accumulation, "Pitfalls when quantizing activations").  With M in the
// thousands this is a dense contraction (2*M*N*K flops against ~0.6 bytes per
// weight), so the int4 codes are expanded to bf16 on chip and fed to UMMA.
//
// The weights are the MMA's A operand and live in tensor memory: the
// dequantization threads write w' straight from registers into TMEM
// (tcgen05.st), so the bf16 weight tile never passes through shared memory,
// and the tokens (X, through TMA) are the B operand in shared memory.  A tile
// is 128 weight rows x 256 tokens of Y^T (D in TMEM: lane = weight row,
// column = token), walked along K in 64-k steps; every dequantized weight
// feeds 256 tokens.  The grid is persistent: one block per SM takes tiles
// blockIdx.x, + gridDim.x, ..., and every ring below runs on across tiles.
//   warp 0      TMA producer: a 5-stage ring of the X tile (256 tokens x 64
//               k, 128-byte swizzle, the UMMA B layout) and the packed code
//               tile (128 rows x 32 bytes, 32-byte swizzle); every 8 groups,
//               when the rows allow it, a 2-deep ring of scale / offset boxes;
//   warp 1      TMEM owner (512 columns: D in 0..255, one 32-column A stage
//               per ring stage above) and, on one lane, the UMMA issuer: 4 x
//               tcgen05.mma (M=128 from TMEM, N=256, K=16) a step; one
//               tcgen05.commit a step frees the stage (the TMA buffers and the
//               A tile of the same index); it waits only for the A tile (the
//               dequantization threads waited for the TMA stage first), and
//               before a tile's first step for the epilogue to have read D;
//   warps 2..9  dequantization: thread (row, 32-k half) of its TMEM
//               sub-partition turns 32 codes into 16 bf16 pairs and stores
//               them with one tcgen05.st;
//   warps 10..17 epilogue, two per TMEM sub-partition (128 tokens each): D
//               -> scale / bias -> bf16 pairs in registers, then D goes back
//               to the issuer; the pairs go through a [token][row] slice of
//               128 tokens in shared memory to a TMA store (plain stores when
//               Y's rows are not 16-byte multiples), overlapping the next
//               tile's main loop.
// 2- and 8-bit codes (Optimum Quanto's int2 / int8 weights) run the same
// pipeline with a code tile of 128 rows x 16 / 64 bytes per k block (no
// swizzle / 64-byte swizzle).  2 bits: the pairs (q_i, q_i+8) of a 16-code
// word come out of LOP3 magic like the 4-bit nibble pairs, PRMTs restore k
// order.  8 bits: 128 + q does not fit a bf16, so each code goes through fp32
// (prmt into 2^23 + q, exact subtract, FMA with s and o) and the pairs are
// rounded to bf16 together: w' = bf16(fp32(q s + o)) exactly.
// Every mbarrier wait is bounded in time; a block that gives up sets the
// device fault word, waits (bounded) for its own copies and MMAs, frees its
// tensor memory and exits.
#include "w4_device.cuh"
#include "w4_internal.h"
#include "w4_tc.cuh"


namespace w4 {

constexpr int GM_BW = 128;  // weight rows per tile (UMMA M, TMEM lanes)
constexpr int GM_BT = 256;  // tokens per tile (UMMA N)
constexpr int GM_BK = 64;
constexpr int GM_STAGES = 5;   // TMA ring: X tile + packed code tile per k block; one TMEM A tile each
constexpr int GM_QSTAGES = 2;  // TMA ring of qparam boxes (8 groups x 128 rows of scales and offsets)
constexpr int GM_QPF = 4;      // k blocks of qparams prefetched by each thread (no-TMA variant)
constexpr int GM_DEQ_WARPS = 8;
constexpr int GM_EPI_WARPS = 8;
constexpr int GM_EPI_WARP0 = 2 + GM_DEQ_WARPS;  // first epilogue warp
constexpr int GM_THREADS = (GM_EPI_WARP0 + GM_EPI_WARPS) * 32;
constexpr int GM_EPI_BAR = 1;  // named barrier of the epilogue warps
constexpr int GM_TMEM_COLS = 512;
constexpr int GM_ACOL = GM_BT;             // first TMEM column of the A stages
constexpr int GM_ASTAGE_COLS = GM_BK / 2;  // 64 bf16 of a row = 32 columns
constexpr int GM_YT = GM_BT / 2;           // tokens of one staged Y slice (one epilogue warp's columns)

constexpr int GM_X_BYTES = GM_BT * GM_BK * 2;  // 32 KB
constexpr int GM_QBOX_BYTES = GM_BW * 16;      //  2 KB: 8 bf16 per row
constexpr int GM_Y_BYTES = GM_YT * GM_BW * 2;  // 32 KB: a bf16 [token][row] slice
// Shared-memory layout for B-bit codes.  Barriers: full_tma, empty_tma (which
// also frees the stage's A tile) and full_deq per stage; full_q, empty_q per
// qparam stage; tmem_full, tmem_empty, drain.
template <int B>
struct GmLayout {
    static constexpr int STAGES = B == 8 ? 4 : GM_STAGES;
    static constexpr int PROW = GM_BK * B / 8;                 // code bytes of one row per k block
    static constexpr int P_BYTES = GM_BW * PROW;               // 2 / 4 / 8 KB
    static constexpr int OFF_X = 0;
    static constexpr int OFF_P = OFF_X + STAGES * GM_X_BYTES;
    static constexpr int OFF_Q = OFF_P + STAGES * P_BYTES;     // per stage: scales box, offsets box
    static constexpr int OFF_Y = (OFF_Q + GM_QSTAGES * 2 * GM_QBOX_BYTES + 1023) / 1024 * 1024;
    static constexpr int NBAR = 3 * STAGES + 2 * GM_QSTAGES + 3;
    static constexpr int OFF_BAR = OFF_Y + GM_Y_BYTES;
    static constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
    static constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;    // + alignment slack for the swizzle atoms
    static_assert(SMEM_BYTES <= 227 * 1024, "shared memory budget");
    static_assert(GM_ACOL + STAGES * GM_ASTAGE_COLS <= GM_TMEM_COLS, "tensor memory budget");
    static_assert(STAGES * GM_X_BYTES >= 2 * GM_Y_BYTES, "an owner stages its whole Y tile in the X ring");
};

// A block's work list.  Tiles 0 .. dp_tiles-1 are computed whole, tile b, b + G, ... by block b
// of the G blocks.  With a workspace, the tiles after those (the last full round and the
// part-empty one) are cut by k blocks into G equal contiguous ranges, one per block, taken after
// its whole tiles (stream-K): at most 3 pieces, the end of a tile (the block shares it: it
// publishes its fp32 sums and a flag), whole tiles, and the start of a tile (it owns it: it adds
// the sums of the blocks after it that share it, in block order, and writes Y).
struct GmWork {
    int ntn;              // row tiles per token tile
    int ntiles;
    int dp_tiles;         // tiles computed whole (all of them without a split)
    long long sk_units;   // (ntiles - dp_tiles) * k blocks (0: no split)
    float* part;          // one slot of 128 x 256 fp32 sums per block
    unsigned int* flags;  // one word per block, zero between calls (an owner clears what it used)
};
struct GmItem {
    int tile, kb0, kb1;
};
constexpr size_t GM_PART_FLOATS = (size_t)GM_BW * GM_BT;  // 128 KB a slot

__device__ __forceinline__ long long gm_sk_start(const GmWork& wk, int b) {
    return wk.sk_units * b / (long long)gridDim.x;
}
// item k of this block's list (false past its end); the same list in every role
__device__ __forceinline__ bool gm_item(const GmWork& wk, int nkb, int k, GmItem* it) {
    const int G = gridDim.x, b = blockIdx.x;
    const int nwhole = wk.dp_tiles > b ? (wk.dp_tiles - 1 - b) / G + 1 : 0;
    if (k < nwhole) {
        *it = GmItem{b + G * k, 0, nkb};
        return true;
    }
    if (wk.sk_units == 0) return false;
    long long u = gm_sk_start(wk, b);
    const long long u1 = gm_sk_start(wk, b + 1);
    for (int p = k - nwhole; u < u1; --p) {  // the host keeps a range under two tiles: 3 pieces at most
        const int t = (int)(u / nkb), kb0 = (int)(u % nkb);
        const int kb1 = (int)(kb0 + (u1 - u) < nkb ? kb0 + (u1 - u) : nkb);
        if (p == 0) {
            *it = GmItem{wk.dp_tiles + t, kb0, kb1};
            return true;
        }
        u += kb1 - kb0;
    }
    return false;
}

constexpr uint64_t GM_WAIT_LIMIT_NS = 2000000000ull;   // 2 s per wait
constexpr uint64_t GM_DRAIN_LIMIT_NS = 1000000000ull;  // 1 s per drain wait

__device__ unsigned int g_gemm_fault;

// Tiled store of a shared-memory box to global memory (a bulk async group of
// this thread); elements outside the tensor are not written.  The start
// coordinates are never negative and x * element size is a multiple of 16.
__device__ __forceinline__ void tma_store_2d(const void* tmap, uint32_t src, int x, int y) {
    asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];"
                 :: "l"(tmap), "r"(src), "r"(x), "r"(y) : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// this thread's bulk stores have finished reading shared memory / are complete
__device__ __forceinline__ void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
// One test of an mbarrier phase that may suspend the thread until the phase
// completes or about `hint_ns` have passed (no polling while it sleeps).
__device__ __forceinline__ bool mbar_try_wait_sleep(uint32_t bar, uint32_t parity, uint32_t hint_ns) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity), "r"(hint_ns) : "memory");
    return ok != 0;
}
// 16 consecutive fp32 columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld_16cols(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
// mbar_wait_bounded with the thread suspended between tests (no spinning):
// woken when the phase completes, re-checks the abort flag and the time limit
// at least every ~20 us.
__device__ __forceinline__ bool gm_wait(uint32_t bar, uint32_t parity, volatile int* abort, unsigned int* fault_word,
                                        unsigned int code, uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (;;) {
        if (mbar_try_wait_sleep(bar, parity, 20000u)) return true;
        if (abort && *abort) return false;
        if (globaltimer_ns() - t0 > limit_ns) {
            if (abort) *abort = 1;
            atomicOr(fault_word, code);
            return false;
        }
    }
}
// Split-tile flags: published with a release store after the block's sums,
// read with acquire loads; the sums themselves are read at L2 (ld.global.cg).
__device__ __forceinline__ void st_release_gpu_u32(unsigned int* p, unsigned int v) {
    asm volatile("st.release.gpu.global.u32 [%0], %1;" :: "l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_gpu_u32(const unsigned int* p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}
__device__ __forceinline__ float ldcg_f32(const float* p) {
    float v;
    asm volatile("ld.global.cg.f32 %0, [%1];" : "=f"(v) : "l"(p) : "memory");
    return v;
}
// Wait until *flag != 0, bounded like every other wait: false after limit_ns or
// once another role has given up (*abort), raising *abort and the fault code.
__device__ __forceinline__ bool wait_flag_bounded(const unsigned int* flag, volatile int* abort, unsigned int* fault_word,
                                                  unsigned int code, uint64_t limit_ns) {
    if (ld_acquire_gpu_u32(flag) != 0u) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        __nanosleep(128);
        if (ld_acquire_gpu_u32(flag) != 0u) return true;
        if ((it & 15u) == 0u) {
            if (*abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                *abort = 1;
                atomicOr(fault_word, code);
                return false;
            }
        }
    }
}
// barrier `id` over `threads` threads of the block (a multiple of 32)
__device__ __forceinline__ void named_barrier(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// Instruction descriptor of tcgen05.mma kind::f16: D fp32 (bits 4-5 = 1),
// A and B bf16 (bits 7-9 = 1, 10-12 = 1), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t gm_idesc() {
    return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(GM_BT >> 3) << 17) | ((uint32_t)(GM_BW >> 4) << 24);
}

// Sixteen 2-bit codes of one word (k0..k15, k0 in the low bits) -> sixteen bf16
// w' = q*s + o in k order (two uint4): LOP3 on w >> 2i gives the pair
// (128 + q_i, 128 + q_i+8), exact subtract, one bf16 FMA, PRMTs restore k order.
__device__ __forceinline__ void dequant16_2b(uint32_t w, uint32_t s2, uint32_t o2, uint32_t cg, uint4& lo, uint4& hi) {
    uint32_t p[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        uint32_t t;
        asm("{\n\t.reg .b32 u;\n\t"
            "shr.b32 u, %1, %4;\n\t"
            "lop3.b32 u, u, 0x00030003, %2, 0xEA;\n\t"
            "sub.rn.bf16x2 u, u, %2;\n\t"
            "fma.rn.bf16x2 %0, u, %3, %5;\n\t}"
            : "=r"(t)
            : "r"(w), "r"(cg), "r"(s2), "r"(2 * i), "r"(o2));
        p[i] = t;
    }
    lo.x = __byte_perm(p[0], p[1], 0x5410), lo.y = __byte_perm(p[2], p[3], 0x5410);
    lo.z = __byte_perm(p[4], p[5], 0x5410), lo.w = __byte_perm(p[6], p[7], 0x5410);
    hi.x = __byte_perm(p[0], p[1], 0x7632), hi.y = __byte_perm(p[2], p[3], 0x7632);
    hi.z = __byte_perm(p[4], p[5], 0x7632), hi.w = __byte_perm(p[6], p[7], 0x7632);
}
// Four 8-bit codes of one word -> two bf16 pairs bf16(fp32(q*s + o)) in k order:
// prmt builds 2^23 + q, an exact subtract gives q, one fp32 FMA, one rounding.
__device__ __forceinline__ uint2 dequant4_8b(uint32_t w, float s, float o, uint32_t mg) {
    float f[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        uint32_t t;
        asm("prmt.b32 %0, %1, %2, %3;" : "=r"(t) : "r"(w), "r"(mg), "r"(0x7540 + i));
        f[i] = __fmaf_rn(__fsub_rn(__uint_as_float(t), 8388608.0f), s, o);
    }
    uint2 r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r.x) : "f"(f[1]), "f"(f[0]));
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r.y) : "f"(f[3]), "f"(f[2]));
    return r;
}
// QT: scales and offsets arrive by TMA (tm_s, tm_o); otherwise the
// dequantization threads load them from `scales` / `offsets`.  y_tma: Y is
// written by TMA stores (tm_y); otherwise by plain stores.
template <int G, bool QT, int B>
__global__ void __launch_bounds__(GM_THREADS, 1)
gemm_kernel(const __grid_constant__ CUtensorMap tm_x, const __grid_constant__ CUtensorMap tm_p,
            const __grid_constant__ CUtensorMap tm_s, const __grid_constant__ CUtensorMap tm_o,
            const __grid_constant__ CUtensorMap tm_y, const uint16_t* __restrict__ scales,
            const uint16_t* __restrict__ offsets, uint16_t* __restrict__ Y, const Epilogue ep, int M, int N, int K,
            const GmWork wk, int y_tma) {
    using LY = GmLayout<B>;
    constexpr int ST = LY::STAGES;
    constexpr int QSPAN = 8 * G / GM_BK;  // k blocks covered by one qparam box (8 groups)
    extern __shared__ unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t bar0 = sbase + LY::OFF_BAR;
    auto full_tma = [&](int t) { return bar0 + 8u * t; };
    auto empty_tma = [&](int t) { return bar0 + 8u * (ST + t); };
    auto full_deq = [&](int t) { return bar0 + 8u * (2 * ST + t); };
    auto full_q = [&](int q) { return bar0 + 8u * (3 * ST + q); };
    auto empty_q = [&](int q) { return bar0 + 8u * (3 * ST + GM_QSTAGES + q); };
    const uint32_t tmem_full = bar0 + 8u * (3 * ST + 2 * GM_QSTAGES);
    const uint32_t tmem_empty = tmem_full + 8u;
    const uint32_t drain = tmem_full + 16u;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + LY::OFF_MISC);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + LY::OFF_MISC + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nkb = (K + GM_BK - 1) / GM_BK;

    if (threadIdx.x == 0) {
        for (int t = 0; t < ST; ++t) {
            mbar_init(full_tma(t), 1);
            mbar_init(empty_tma(t), 1);
            mbar_init(full_deq(t), GM_DEQ_WARPS * 32);
        }
        for (int q = 0; q < GM_QSTAGES; ++q) {
            mbar_init(full_q(q), 1);
            mbar_init(empty_q(q), GM_DEQ_WARPS * 32);
        }
        mbar_init(tmem_full, 1);
        mbar_init(tmem_empty, GM_EPI_WARPS * 32);
        mbar_init(drain, 1);
        *abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), GM_TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;

    if (warp == 0) {
        // ---------------------------------------------------------------- TMA producer
        if (lane == 0) {
            tma_prefetch_desc(&tm_x);
            tma_prefetch_desc(&tm_p);
            if (QT) {
                tma_prefetch_desc(&tm_s);
                tma_prefetch_desc(&tm_o);
            }
            int issued = 0, q_issued = 0;  // k blocks and qparam boxes requested, over all tiles
            bool ok = true;
            GmItem it;
            for (int k = 0; ok && gm_item(wk, nkb, k, &it); ++k) {
                const int n0 = (it.tile % wk.ntn) * GM_BW, m0 = (it.tile / wk.ntn) * GM_BT;
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    if (QT && (kb % QSPAN == 0 || kb == it.kb0)) {  // scales and offsets of groups 8u .. 8u+7
                        const int q = q_issued % GM_QSTAGES;
                        if (!gm_wait(empty_q(q), ((q_issued / GM_QSTAGES) & 1) ^ 1, abort_flag,
                                               &g_gemm_fault, 1u, GM_WAIT_LIMIT_NS)) {
                            ok = false;
                            break;
                        }
                        mbar_arrive_expect_tx(full_q(q), 2 * GM_QBOX_BYTES);
                        const uint32_t qdst = sbase + LY::OFF_Q + q * 2 * GM_QBOX_BYTES;
                        tma_load_2d(qdst, &tm_s, full_q(q), 8 * (kb / QSPAN), n0);
                        tma_load_2d(qdst + GM_QBOX_BYTES, &tm_o, full_q(q), 8 * (kb / QSPAN), n0);
                        ++q_issued;
                    }
                    const int t = issued % ST;
                    if (!gm_wait(empty_tma(t), ((issued / ST) & 1) ^ 1, abort_flag, &g_gemm_fault, 1u,
                                           GM_WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_tma(t), GM_X_BYTES + LY::P_BYTES);
                    tma_load_2d(sbase + LY::OFF_X + t * GM_X_BYTES, &tm_x, full_tma(t), kb * GM_BK, m0);
                    tma_load_2d(sbase + LY::OFF_P + t * LY::P_BYTES, &tm_p, full_tma(t), kb * LY::PROW, n0);
                    ++issued;
                }
            }
            // never leave the block with copies still landing in its shared memory
            for (int g = (issued > ST ? issued - ST : 0); g < issued; ++g)
                mbar_drain_bounded(full_tma(g % ST), (g / ST) & 1, GM_DRAIN_LIMIT_NS);
            for (int u = (q_issued > GM_QSTAGES ? q_issued - GM_QSTAGES : 0); u < q_issued; ++u)
                mbar_drain_bounded(full_q(u % GM_QSTAGES), (u / GM_QSTAGES) & 1, GM_DRAIN_LIMIT_NS);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------------ UMMA issuer
        if (lane == 0) {
            constexpr uint32_t idesc = gm_idesc();
            int issued = 0, j = 0;
            bool ok = true;
            GmItem it;
            for (int k = 0; ok && gm_item(wk, nkb, k, &it); ++k, ++j) {
                // the epilogue has read the previous item's D out of tensor memory
                if (j > 0 && !gm_wait(tmem_empty, (j - 1) & 1, abort_flag, &g_gemm_fault, 2u,
                                                GM_WAIT_LIMIT_NS))
                    break;
                tc_fence_after();
                for (int kb = it.kb0; kb < it.kb1; ++kb) {
                    const int t = issued % ST;
                    // Only the A stage is waited for: every dequantization thread waited for this
                    // k block's TMA stage (X and codes) before its arrive, so full_deq orders the X
                    // tile too.  One wait less a step keeps the tensor pipe fed (each N=256 MMA
                    // takes ~128 cycles, and the issuing thread's gaps between steps leave it idle).
                    if (!gm_wait(full_deq(t), (issued / ST) & 1, abort_flag, &g_gemm_fault, 2u,
                                           GM_WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t bdesc = sw128_kmajor_desc(sbase + LY::OFF_X + t * GM_X_BYTES);
                    const uint32_t a_tmem = tmem + (uint32_t)(GM_ACOL + t * GM_ASTAGE_COLS);
#pragma unroll
                    for (int kk = 0; kk < GM_BK / 16; ++kk)  // K=16 a step: 8 A columns, +32 bytes of B (+2 in the desc)
                        umma_bf16_tmem_a(tmem, a_tmem + 8u * kk, bdesc + 2u * kk, idesc, (kb != it.kb0) | (kk != 0));
                    umma_commit(empty_tma(t));  // X, codes and the A tile of this k block consumed (one commit)
                    ++issued;
                }
                if (ok) umma_commit(tmem_full);  // D of this item is complete once its MMAs are
            }
            // the MMAs must be finished before tensor memory is released
            if (issued > 0) {
                umma_commit(drain);
                mbar_drain_bounded(drain, 0, GM_DRAIN_LIMIT_NS);
            }
        }
    } else if (warp < GM_EPI_WARP0) {
        // ------------------------------------------------------- dequantization warps
        const int sp = warp & 3;         // TMEM sub-partition: lanes (weight rows) 32 sp .. 32 sp + 31
        const int hh = (warp - 2) >> 2;  // which 32-k half of each k block
        const int r = 32 * sp + lane;    // weight row within the tile
        const int ng = K / G;
        uint32_t cm, cg, mg;  // LOP3 constants pinned in registers (0x4300 pairs are also the 128.0 bias); 2^23
        asm volatile("mov.b32 %0, %1;" : "=r"(cm) : "r"(0x000F000Fu));
        asm volatile("mov.b32 %0, %1;" : "=r"(cg) : "r"(0x43004300u));
        asm volatile("mov.b32 %0, %1;" : "=r"(mg) : "r"(0x4B000000u));
        // this thread's 32 codes of a k block in the code tile: 4 bits: 32-byte rows, 32-byte swizzle,
        // half hh of row r at 16 * (hh ^ bit 2 of r); 2 bits: 16-byte rows, half hh at 8 hh;
        // 8 bits: 64-byte rows, 64-byte swizzle, 16-byte chunks 2hh, 2hh+1 at 16 * (c ^ ((r >> 1) & 3))
        const uint32_t pcol = B == 4 ? (uint32_t)(r * 32 + 16 * (hh ^ ((r >> 2) & 1)))
                              : B == 2 ? (uint32_t)(r * 16 + 8 * hh)
                                       : (uint32_t)(r * 64 + 16 * ((2 * hh) ^ ((r >> 1) & 3)));
        const uint32_t pcol1 = (uint32_t)(r * 64 + 16 * ((2 * hh + 1) ^ ((r >> 1) & 3)));  // 8 bits: second chunk
        // this thread's 16 columns of an A stage, in its own TMEM lane
        const uint32_t a_lane = tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)(GM_ACOL + 16 * hh);
        uint4 sq = make_uint4(0u, 0u, 0u, 0u), oq = sq;  // TMA variant: this row's 8 groups
        int done = 0, q_done = 0;  // k blocks and qparam boxes consumed, over all tiles
        bool ok = true;
        GmItem it;
        for (int k = 0; ok && gm_item(wk, nkb, k, &it); ++k) {
            const int n = (it.tile % wk.ntn) * GM_BW + r;
            const bool nvalid = n < N;
            const int64_t qrow = (int64_t)(nvalid ? n : 0) * ng;
            // scale and offset of this row for this thread's half of a k block,
            // loaded GM_QPF blocks ahead and kept raw until used (no-TMA variant).
            // Groups past K read as 0: with the zero-filled codes those weights
            // are exactly 0.
            struct QRaw {
                uint32_t s, o;
            };
            auto qload = [&](int kb) {
                QRaw q = {0u, 0u};
                if (!QT && kb < nkb && nvalid) {
                    const int jg = (kb * GM_BK + 32 * hh) / G;
                    if (jg < ng) {
                        q.s = ldg_nc_u16(scales + qrow + jg);
                        q.o = ldg_nc_u16(offsets + qrow + jg);
                    }
                }
                return q;
            };
            QRaw q0 = qload(it.kb0), q1 = qload(it.kb0 + 1), q2 = qload(it.kb0 + 2), q3 = qload(it.kb0 + 3);
            for (int kb = it.kb0; kb < it.kb1; ++kb) {
                const QRaw qc = q0;
                q0 = q1;
                q1 = q2;
                q2 = q3;
                q3 = qload(kb + GM_QPF);
                if (QT && (kb % QSPAN == 0 || kb == it.kb0)) {
                    const int q = q_done % GM_QSTAGES;
                    if (!gm_wait(full_q(q), (q_done / GM_QSTAGES) & 1, abort_flag, &g_gemm_fault, 4u,
                                           GM_WAIT_LIMIT_NS)) {
                        ok = false;
                        break;
                    }
                    const uint32_t qsrc = sbase + LY::OFF_Q + q * 2 * GM_QBOX_BYTES + r * 16;
                    sq = lds128(qsrc);
                    oq = lds128(qsrc + GM_QBOX_BYTES);
                    mbar_arrive(empty_q(q));
                    ++q_done;
                }
                const int t = done % ST;
                const uint32_t pt = (done / ST) & 1;
                if (!gm_wait(full_tma(t), pt, abort_flag, &g_gemm_fault, 4u, GM_WAIT_LIMIT_NS) ||
                    !gm_wait(empty_tma(t), pt ^ 1, abort_flag, &g_gemm_fault, 4u, GM_WAIT_LIMIT_NS)) {
                    ok = false;
                    break;
                }
                tc_fence_after();  // the MMAs that read this A stage are complete
                const uint32_t ptile = sbase + LY::OFF_P + t * LY::P_BYTES;
                uint32_t s2, o2;  // (s,s) and (o,o) bf16 pairs of this half's group
                if (QT) {
                    const int jg = (kb % QSPAN) * GM_BK / G + (G == 32 ? hh : 0);  // group among the box's 8
                    const uint32_t sel = (jg & 1) ? 0x3232u : 0x1010u;
                    s2 = __byte_perm(pick_word(sq, jg >> 1), 0, sel);
                    o2 = __byte_perm(pick_word(oq, jg >> 1), 0, sel);
                } else {
                    s2 = __byte_perm(qc.s, 0, 0x1010);
                    o2 = __byte_perm(qc.o, 0, 0x1010);
                }
                // 32 weights of this row -> 16 columns (two bf16 of consecutive k each) of the A stage
                const uint32_t acol = a_lane + (uint32_t)(t * GM_ASTAGE_COLS);
                if constexpr (B == 4) {
                    const uint4 words = lds128(ptile + pcol);  // 32 codes of this half
                    tmem_st_16cols(acol, dequant8(words.x, s2, o2, cm, cg), dequant8(words.y, s2, o2, cm, cg),
                                   dequant8(words.z, s2, o2, cm, cg), dequant8(words.w, s2, o2, cm, cg));
                } else if constexpr (B == 2) {
                    const uint2 words = lds64(ptile + pcol);
                    uint4 c0, c1, c2, c3;
                    dequant16_2b(words.x, s2, o2, cg, c0, c1);
                    dequant16_2b(words.y, s2, o2, cg, c2, c3);
                    tmem_st_16cols(acol, c0, c1, c2, c3);
                } else {
                    const uint4 wa = lds128(ptile + pcol), wb = lds128(ptile + pcol1);
                    const float sf = __uint_as_float(s2 << 16), of = __uint_as_float(o2 << 16);
                    const uint2 d0 = dequant4_8b(wa.x, sf, of, mg), d1 = dequant4_8b(wa.y, sf, of, mg);
                    const uint2 d2 = dequant4_8b(wa.z, sf, of, mg), d3 = dequant4_8b(wa.w, sf, of, mg);
                    const uint2 d4 = dequant4_8b(wb.x, sf, of, mg), d5 = dequant4_8b(wb.y, sf, of, mg);
                    const uint2 d6 = dequant4_8b(wb.z, sf, of, mg), d7 = dequant4_8b(wb.w, sf, of, mg);
                    tmem_st_16cols(acol, make_uint4(d0.x, d0.y, d1.x, d1.y), make_uint4(d2.x, d2.y, d3.x, d3.y),
                                   make_uint4(d4.x, d4.y, d5.x, d5.y), make_uint4(d6.x, d6.y, d7.x, d7.y));
                }
                tmem_st_wait();
                tc_fence_before();
                mbar_arrive(full_deq(t));
                ++done;
            }
        }
    } else {
        // ----------------------------------------------------------------- epilogue warps
        // Warp e (0..7) takes the 32 rows of TMEM sub-partition warp & 3 and the 128 tokens
        // [128 half, 128 half + 128), half = e / 4.  It reads its part of D into registers as bf16
        // pairs of neighbouring tokens and hands D back; the two halves then go one after the
        // other through the [token][row] slice in shared memory to a TMA store.  A shared piece's
        // fp32 sums go to this block's workspace slot instead, [warp][16 tokens][token][lane].
        // Every epilogue warp passes the same named barriers per item, whatever happened to the
        // others (the item's kind is the same for all of them).
        const int e = warp - GM_EPI_WARP0;
        const int sp = warp & 3, half = e >> 2;
        const int row = 32 * sp + lane;
        unsigned char* ystage = smem + LY::OFF_Y;
        const bool storer = e == 0 && lane == 0;
        volatile int* tile_ok = reinterpret_cast<volatile int*>(smem + LY::OFF_MISC + 8);  // the waiter's verdict
        const int b = blockIdx.x;
        bool ok = true;
        int j = 0;
        GmItem it;
        for (int k = 0; gm_item(wk, nkb, k, &it); ++k, ++j) {
            const int n0 = (it.tile % wk.ntn) * GM_BW, m0 = (it.tile / wk.ntn) * GM_BT;
            const bool sharer = it.kb0 > 0;                    // its sums go to the owner
            const bool owner = it.kb0 == 0 && it.kb1 < nkb;   // adds the sums of the blocks after it
            int nsh = 0;
            if (owner) {
                const long long t_rel = it.tile - wk.dp_tiles;
                while (b + 1 + nsh < (int)gridDim.x && gm_sk_start(wk, b + 1 + nsh) / nkb == t_rel) ++nsh;
            }
            // one thread waits for the item's sums (suspended, not spinning) and, for an owner,
            // for its sharers' flags; the other epilogue threads are blocked on the named barrier
            if (storer) {
                bool got = ok && gm_wait(tmem_full, j & 1, abort_flag, &g_gemm_fault, 8u, GM_WAIT_LIMIT_NS);
                for (int sh = 0; got && sh < nsh; ++sh)
                    got = wait_flag_bounded(wk.flags + b + 1 + sh, abort_flag, &g_gemm_fault, 16u, GM_WAIT_LIMIT_NS);
                *tile_ok = got ? 1 : 0;
            }
            named_barrier(GM_EPI_BAR, GM_EPI_WARPS * 32);
            ok = *tile_ok != 0;
            if (sharer) {
                if (ok) {
                    tc_fence_after();
                    float* slot = wk.part + (size_t)b * GM_PART_FLOATS + (size_t)e * (GM_YT * 32) + lane;
#pragma unroll 1
                    for (int cc = 0; cc < 8; ++cc) {
                        uint32_t v[16];
                        tmem_ld_16cols(tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)(GM_YT * half + 16 * cc), v);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 16; ++i) slot[(cc * 16 + i) * 32] = __uint_as_float(v[i]);
                    }
                    tc_fence_before();
                    mbar_arrive(tmem_empty);  // the next item's MMAs may overwrite D
                }
                __threadfence();  // this thread's sums before the flag
                named_barrier(GM_EPI_BAR, GM_EPI_WARPS * 32);
                if (storer && ok && !*abort_flag) st_release_gpu_u32(wk.flags + b, 1u);
                continue;
            }
            if (owner) {
                // the block's last item (its range ends inside the tile), so the X ring is free: the
                // whole [token][row] tile is staged there, the sharers' sums added in block order
                // on the way (the first sharer's loads in flight during the TMEM read)
                unsigned char* ost = smem + LY::OFF_X;
                if (ok) {
                    tc_fence_after();
                    const float bl = n0 + row < N ? bias_f32(ep.bias, n0 + row) : 0.f;  // this lane's row
#pragma unroll 1
                    for (int cc = 0; cc < 8; ++cc) {
                        const int col = GM_YT * half + 16 * cc;  // first token (TMEM column) of the piece
                        const float fl = yscale_f32(ep, min(m0 + col + (lane & 15), M - 1));
                        uint32_t v[16];
#pragma unroll 1
                        for (int sh = 0; sh < nsh; ++sh) {
                            const float* src = wk.part + (size_t)(b + 1 + sh) * GM_PART_FLOATS +
                                               (size_t)e * (GM_YT * 32) + (size_t)(cc * 16) * 32 + lane;
                            float pv[16];
#pragma unroll
                            for (int i = 0; i < 16; ++i) pv[i] = ldcg_f32(src + i * 32);
                            if (sh == 0) {  // the first sharer's loads are in flight during the TMEM read
                                tmem_ld_16cols(tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)col, v);
                                tmem_ld_wait();
                            }
#pragma unroll
                            for (int i = 0; i < 16; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) + pv[i]);
                        }
                        unsigned char* dst = ost + col * (GM_BW * 2) + 2 * row;
#pragma unroll
                        for (int i = 0; i < 16; ++i)
                            *reinterpret_cast<uint16_t*>(dst + i * (GM_BW * 2)) = (uint16_t)float_to_bf16_bits(
                                fmaf(__uint_as_float(v[i]), __shfl_sync(0xffffffffu, fl, i), bl));
                    }
                    tc_fence_before();
                    mbar_arrive(tmem_empty);
                    if (storer)  // the consumed flags back to zero for the next call
                        for (int sh = 0; sh < nsh; ++sh) st_release_gpu_u32(wk.flags + b + 1 + sh, 0u);
                }
                if (y_tma) fence_proxy_async_smem();  // the tile's writes, seen by the TMA stores
                named_barrier(GM_EPI_BAR, GM_EPI_WARPS * 32);
                if (y_tma) {
                    if (storer && ok && !*abort_flag) {
                        tma_store_2d(&tm_y, smem_u32(ost), n0, m0);
                        tma_store_2d(&tm_y, smem_u32(ost) + GM_Y_BYTES, n0, m0 + GM_YT);
                        bulk_commit_group();
                    }
                } else if (ok) {
                    for (int x = threadIdx.x - GM_EPI_WARP0 * 32; x < GM_BT * GM_BW; x += GM_EPI_WARPS * 32) {
                        const int m = m0 + x / GM_BW, n = n0 + x % GM_BW;
                        if (m < M && n < N) Y[(int64_t)m * N + n] = *reinterpret_cast<const uint16_t*>(ost + 2 * x);
                    }
                }
                continue;
            }
            uint32_t pk[64];  // bf16 pairs (token 2i, token 2i + 1) of this lane's row
            if (ok) {
                tc_fence_after();
                const float bl = n0 + row < N ? bias_f32(ep.bias, n0 + row) : 0.f;  // this lane's row
#pragma unroll
                for (int cc = 0; cc < 8; ++cc) {
                    const int col = GM_YT * half + 16 * cc;  // first token (TMEM column) of the piece
                    uint32_t v[16];
                    tmem_ld_16cols(tmem + ((uint32_t)(32 * sp) << 16) + (uint32_t)col, v);
                    // the output scale of token col + (lane & 15) (lane i hands token i's to the warp)
                    const float fl = yscale_f32(ep, min(m0 + col + (lane & 15), M - 1));
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 8; ++i)
                        pk[8 * cc + i] =
                            (float_to_bf16_bits(fmaf(__uint_as_float(v[2 * i]), __shfl_sync(0xffffffffu, fl, 2 * i), bl))) |
                            (float_to_bf16_bits(
                                 fmaf(__uint_as_float(v[2 * i + 1]), __shfl_sync(0xffffffffu, fl, 2 * i + 1), bl))
                             << 16);
                }
                tc_fence_before();
                mbar_arrive(tmem_empty);  // the next item's MMAs may overwrite D
            }
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                if (storer && y_tma && (j > 0 || h > 0)) bulk_wait_read_all();  // the last slice has left
                named_barrier(GM_EPI_BAR, GM_EPI_WARPS * 32);
                if (ok && half == h) {  // stage[token t][row] for this warp's 128 tokens
#pragma unroll
                    for (int i = 0; i < 64; ++i) {
                        unsigned char* dst = ystage + (2 * i) * (GM_BW * 2) + 2 * row;
                        *reinterpret_cast<uint16_t*>(dst) = (uint16_t)(pk[i] & 0xFFFFu);
                        *reinterpret_cast<uint16_t*>(dst + GM_BW * 2) = (uint16_t)(pk[i] >> 16);
                    }
                }
                if (y_tma) fence_proxy_async_smem();  // the slice's writes, seen by the TMA store
                named_barrier(GM_EPI_BAR, GM_EPI_WARPS * 32);
                if (y_tma) {
                    if (storer && ok && !*abort_flag) {
                        tma_store_2d(&tm_y, smem_u32(ystage), n0, m0 + GM_YT * h);
                        bulk_commit_group();
                    }
                } else if (ok) {  // plain stores: consecutive rows of one token per warp, inside Y only
                    for (int x = threadIdx.x - GM_EPI_WARP0 * 32; x < GM_YT * GM_BW; x += GM_EPI_WARPS * 32) {
                        const int m = m0 + GM_YT * h + x / GM_BW, n = n0 + x % GM_BW;
                        if (m < M && n < N) Y[(int64_t)m * N + n] = *reinterpret_cast<const uint16_t*>(ystage + 2 * x);
                    }
                }
            }
        }
        if (storer && y_tma) bulk_wait_all();  // the last store is complete before the block exits
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) tmem_dealloc(tmem, GM_TMEM_COLS);
}

// ------------------------------------------------------------------ host side

// The stream-K tail for T tiles of nkb k blocks on `sms` SMs: the blocks, the whole tiles and
// the split units, or false when whole tiles are as good.  Split when the last round is
// part-empty and the estimate saves at least 3%.  The estimate counts k blocks of one block
// plus 40 for the split's fixed cost (measured: the sharers' partial tiles out and the owners'
// in, an extra tile boundary, the owners' waits; ~20 us at ~0.45 us a k block).  A split range
// stays under two tiles of k blocks (at most 3 pieces) and at least 8 k blocks.
static bool gemm_split_plan(int64_t T, int64_t nkb, int sms, int* blocks, int64_t* dp_tiles, int64_t* units) {
    if (sms < 2 || T < 1 || nkb < 8 || T % sms == 0) return false;
    const int64_t gw = std::min<int64_t>(T, sms);
    const double whole = (double)((T + gw - 1) / gw) * nkb;
    const int64_t rounds = T / sms;
    const int64_t dp = rounds >= 1 ? (rounds - 1) * sms : 0;  // whole tiles, the same count per block
    const int64_t u = (T - dp) * nkb;
    const int64_t g = std::min<int64_t>(sms, u / 8);
    if (g < 2 || (dp > 0 && g != sms)) return false;
    const int64_t span = (u + g - 1) / g;
    if (span > 2 * nkb - 1) return false;
    const double split = (double)(dp / g) * nkb + span + 40.0;
    if (split > 0.97 * whole) return false;
    *blocks = (int)g;
    *dp_tiles = dp;
    *units = u;
    return true;
}

cudaError_t gemm_split_bytes(int64_t M, int64_t N, int64_t K, size_t part_off, size_t* bytes) {
    *bytes = 0;
    int dev = 0, sms = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    int g = 0;
    int64_t dp = 0, u = 0;
    const int64_t T = ((N + GM_BW - 1) / GM_BW) * ((M + GM_BT - 1) / GM_BT);
    if (gemm_split_plan(T, (K + GM_BK - 1) / GM_BK, sms, &g, &dp, &u)) *bytes = part_off + g * GM_PART_FLOATS * 4;
    return cudaSuccess;
}

// one block per SM (persistent), no more blocks than tiles; the stream-K tail when the workspace
// holds its flags (from byte 0) and partial sums (from part_off)
template <int G, bool QT, int B>
static cudaError_t launch_gemm_g(const CUtensorMap& tx, const CUtensorMap& tp, const CUtensorMap& ts,
                                 const CUtensorMap& to, const CUtensorMap& ty, bool y_tma, const uint16_t* scales,
                                 const uint16_t* offsets, uint16_t* Y, const Epilogue& ep, int M, int N, int K,
                                 void* workspace, size_t workspace_bytes, size_t part_off, cudaStream_t stream) {
    auto kern = gemm_kernel<G, QT, B>;
    constexpr int SMEM = GmLayout<B>::SMEM_BYTES;
    cudaError_t e = ensure_kernel_attrs(reinterpret_cast<const void*>(kern), SMEM, false);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    if ((e = resident_blocks(reinterpret_cast<const void*>(kern), GM_THREADS, SMEM, &sms, &per_sm)) != cudaSuccess)
        return e;
    GmWork wk{};
    wk.ntn = (N + GM_BW - 1) / GM_BW;
    wk.ntiles = wk.ntn * ((M + GM_BT - 1) / GM_BT);
    wk.dp_tiles = wk.ntiles;
    int grid = std::max(1, std::min(wk.ntiles, sms * std::max(per_sm, 1)));
    int g = 0;
    int64_t dp = 0, u = 0;
    if (workspace != nullptr && per_sm == 1 && part_off % 16 == 0 &&
        gemm_split_plan(wk.ntiles, (K + GM_BK - 1) / GM_BK, sms, &g, &dp, &u) && (size_t)g * 4 <= part_off &&
        workspace_bytes >= part_off + (size_t)g * GM_PART_FLOATS * 4) {
        grid = g;
        wk.dp_tiles = (int)dp;
        wk.sk_units = u;
        wk.part = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + part_off);
        wk.flags = static_cast<unsigned int*>(workspace);
    }
    kern<<<grid, GM_THREADS, SMEM, stream>>>(tx, tp, ts, to, ty, scales, offsets, Y, ep, M, N, K, wk, y_tma ? 1 : 0);
    return cudaGetLastError();
}

template <int B>
static cudaError_t launch_gemm_b(const CUtensorMap& tx, const CUtensorMap& tp, const CUtensorMap& ts,
                                 const CUtensorMap& to, const CUtensorMap& ty, bool y_tma, bool qt,
                                 const uint16_t* scales, const uint16_t* offsets, uint16_t* Y, const Epilogue& ep,
                                 int m, int n, int k, int g, void* ws, size_t ws_bytes, size_t part_off,
                                 cudaStream_t stream) {
    switch (g) {
        case 32:
            return qt ? launch_gemm_g<32, true, B>(tx, tp, ts, to, ty, y_tma, scales, offsets, Y, ep, m, n, k, ws, ws_bytes, part_off, stream)
                      : launch_gemm_g<32, false, B>(tx, tp, ts, to, ty, y_tma, scales, offsets, Y, ep, m, n, k, ws, ws_bytes, part_off, stream);
        case 64:
            return qt ? launch_gemm_g<64, true, B>(tx, tp, ts, to, ty, y_tma, scales, offsets, Y, ep, m, n, k, ws, ws_bytes, part_off, stream)
                      : launch_gemm_g<64, false, B>(tx, tp, ts, to, ty, y_tma, scales, offsets, Y, ep, m, n, k, ws, ws_bytes, part_off, stream);
        default:
            return qt ? launch_gemm_g<128, true, B>(tx, tp, ts, to, ty, y_tma, scales, offsets, Y, ep, m, n, k, ws, ws_bytes, part_off, stream)
                      : launch_gemm_g<128, false, B>(tx, tp, ts, to, ty, y_tma, scales, offsets, Y, ep, m, n, k, ws, ws_bytes, part_off, stream);
    }
}

cudaError_t launch_gemm(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                        const uint16_t* offsets, int64_t N, int g, int bits, uint16_t* Y, cudaStream_t stream,
                        const char** detail, const Epilogue& ep, void* workspace, size_t workspace_bytes,
                        size_t part_off) {
    if ((N + GM_BW - 1) / GM_BW * ((M + GM_BT - 1) / GM_BT) > 0x7FFFFFFF) {
        *detail = "problem too large for the GEMM's tile count";
        return cudaErrorInvalidValue;
    }
    CUtensorMap tx, tp;
    // X: [M][K] bf16, box 256 tokens x 64 k (128 bytes), 128-byte swizzle (the UMMA B layout)
    cudaError_t e = encode_tensor_map_2d(&tx, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, X, (uint64_t)K, (uint64_t)M,
                                         (uint64_t)K * 2, GM_BK, GM_BT, CU_TENSOR_MAP_SWIZZLE_128B, detail);
    if (e != cudaSuccess) return e;
    // codes: [N][K bits/8] bytes, box 128 rows x (64 k of codes): 4 bits: 32 bytes, 32-byte swizzle
    // (the two 16-byte halves of rows 4..7 of every 8 trade places: conflict-free reads of one half
    // per thread); 2 bits: 16 bytes, no swizzle; 8 bits: 64 bytes, 64-byte swizzle
    const uint64_t row_bytes = (uint64_t)(K * bits / 8);
    e = encode_tensor_map_2d(&tp, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, row_bytes, (uint64_t)N, row_bytes,
                             (uint32_t)(GM_BK * bits / 8), GM_BW,
                             bits == 4   ? CU_TENSOR_MAP_SWIZZLE_32B
                             : bits == 2 ? CU_TENSOR_MAP_SWIZZLE_NONE
                                         : CU_TENSOR_MAP_SWIZZLE_64B,
                             detail);
    if (e != cudaSuccess) return e;
    // scales / offsets: [N][K/g] bf16, box 128 rows x 8 groups, when a row is
    // a whole number of 16-byte pieces (the tensor-map stride rule)
    const int64_t ng = K / g;
    const bool qt = ng % 8 == 0;
    CUtensorMap ts = tp, to = tp;
    if (qt) {
        e = encode_tensor_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, (uint64_t)ng, (uint64_t)N,
                                 (uint64_t)ng * 2, 8, GM_BW, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e == cudaSuccess)
            e = encode_tensor_map_2d(&to, CU_TENSOR_MAP_DATA_TYPE_UINT16, offsets, (uint64_t)ng, (uint64_t)N,
                                     (uint64_t)ng * 2, 8, GM_BW, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e != cudaSuccess) return e;
    }
    // Y: [M][N] bf16, box 128 rows x one 128-token slice, stored by TMA when the base and the row
    // pitch are 16-byte multiples (the tensor-map rules)
    const bool y_tma = (reinterpret_cast<uintptr_t>(Y) & 15u) == 0 && N % 8 == 0;
    CUtensorMap ty = tx;  // not read when !y_tma
    if (y_tma) {
        e = encode_tensor_map_2d(&ty, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, Y, (uint64_t)N, (uint64_t)M, (uint64_t)N * 2,
                                 GM_BW, GM_YT, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e != cudaSuccess) return e;
    }
    const int m = (int)M, n = (int)N, k = (int)K;
    if (bits == 2) return launch_gemm_b<2>(tx, tp, ts, to, ty, y_tma, qt, scales, offsets, Y, ep, m, n, k, g, workspace, workspace_bytes, part_off, stream);
    if (bits == 8) return launch_gemm_b<8>(tx, tp, ts, to, ty, y_tma, qt, scales, offsets, Y, ep, m, n, k, g, workspace, workspace_bytes, part_off, stream);
    return launch_gemm_b<4>(tx, tp, ts, to, ty, y_tma, qt, scales, offsets, Y, ep, m, n, k, g, workspace, workspace_bytes, part_off, stream);
}

cudaError_t read_and_clear_gemm_fault(unsigned int* fault) {
    cudaError_t e = cudaMemcpyFromSymbol(fault, g_gemm_fault, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (*fault) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_gemm_fault, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace w4
