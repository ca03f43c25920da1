// w4_device.cuh -- device-side helpers shared by the libw4 kernels:
// bf16 bit handling, cache-controlled loads, mbarrier waits with a time
// limit, TMA copies, tcgen05 (TMEM / UMMA) wrappers, programmatic dependent
// launch.  sm_103a only.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>

#include "w4_internal.h"  // Epilogue

namespace w4 {

// ---------------------------------------------------------------- bf16 bits
__device__ __forceinline__ float bf16_bits_to_float(uint32_t b) {
    return __uint_as_float(b << 16);
}
__device__ __forceinline__ uint32_t float_to_bf16_bits(float f) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(f));
}
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t*>(&v);
}

// ------------------------------------------------------------------- loads
// Streamed read-only data (weights): skip L1 allocation.
__device__ __forceinline__ uint4 ldg_stream_v4(const void* p) {
    uint4 r;
    asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
        : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
// Data another kernel may have just written (activations): cache in L2 only.
__device__ __forceinline__ uint4 ldg_cg_v4(const void* p) {
    uint4 r;
    asm volatile("ld.global.cg.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
    return r;
}
__device__ __forceinline__ uint2 ldg_cg_v2(const void* p) {
    uint2 r;
    asm volatile("ld.global.cg.v2.u32 {%0,%1}, [%2];" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}
// Eight int8 codes (bytes of v, lowest first) as eight bf16 values, exactly
// (|q| <= 128 has at most 8 significant bits), in the order of eight bf16 in memory.
__device__ __forceinline__ uint4 widen_i8x8(uint2 v) {
    uint32_t h[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q = (int)(int8_t)(((i < 4 ? v.x : v.y) >> (8 * (i & 3))) & 0xFFu);
        h[i] = __float_as_uint((float)q) >> 16;
    }
    return make_uint4(h[0] | (h[1] << 16), h[2] | (h[3] << 16), h[4] | (h[5] << 16), h[6] | (h[7] << 16));
}
// Dynamic int8 activation quantization (w4_act.cu, and the stream kernel's
// fused mode): the largest magnitude of eight bf16 values as magnitude bits
// (bits & 0x7FFF order like magnitudes for finite values), the scale
// s = max|x| / 127 (one IEEE division, at least 1e-6), and eight codes
// q = clamp(rne(x / s), -127, 127) (one IEEE division each).
__device__ __forceinline__ uint32_t act_mag_max8(uint4 v) {
    const uint32_t a = max(v.x & 0x7FFFu, (v.x >> 16) & 0x7FFFu), b = max(v.y & 0x7FFFu, (v.y >> 16) & 0x7FFFu);
    const uint32_t c = max(v.z & 0x7FFFu, (v.z >> 16) & 0x7FFFu), d = max(v.w & 0x7FFFu, (v.w >> 16) & 0x7FFFu);
    return max(max(a, b), max(c, d));
}
__device__ __forceinline__ float act_scale_of(uint32_t mag_bits) {
    const float s = __fdiv_rn(__uint_as_float(mag_bits << 16), 127.0f);
    return s < 1e-6f ? 1e-6f : s;
}
__device__ __forceinline__ int act_code(uint32_t h, float s) {
    const int q = __float2int_rn(__fdiv_rn(__uint_as_float(h << 16), s));
    return min(127, max(-127, q));
}
// eight bf16 values -> their eight codes as bf16 (exact), in the same order
__device__ __forceinline__ uint4 act_codes_bf16x8(uint4 v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t o[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo = __float_as_uint((float)act_code(w[i] & 0xFFFFu, s)) >> 16;
        const uint32_t hi = __float_as_uint((float)act_code(w[i] >> 16, s)) >> 16;
        o[i] = lo | (hi << 16);
    }
    return make_uint4(o[0], o[1], o[2], o[3]);
}
__device__ __forceinline__ uint32_t ldg_nc_u16(const uint16_t* p) {
    unsigned short v;
    asm("ld.global.nc.u16 %0, [%1];" : "=h"(v) : "l"(p));
    return v;
}
__device__ __forceinline__ uint32_t ldg_nc_u32(const void* p) {
    uint32_t v;
    asm("ld.global.nc.u32 %0, [%1];" : "=r"(v) : "l"(p));
    return v;
}

// The bias of output row n in fp32 (bf16 bits; no bias when b is null), added to
// the fp32 sum before the one rounding to bf16.
__device__ __forceinline__ float bias_f32(const uint16_t* b, int64_t n) {
    return b ? bf16_bits_to_float(ldg_nc_u16(b + n)) : 0.f;
}
// The output scale of token m (1 when there is none).  A plain load: the scale may
// come from the kernel before this one (read after the dependency wait).
__device__ __forceinline__ float yscale_f32(const Epilogue& ep, int m) {
    return ep.yscale ? ep.yscale[(int64_t)m * ep.ys_stride] : 1.f;
}
// The value rounded to bf16 for output (m, n): sum * yscale + bias in one fp32
// rounding (with neither, exactly the sum; with a bias only, sum + bias).
__device__ __forceinline__ float epilogue_f32(const Epilogue& ep, float sum, int m, int64_t n) {
    return fmaf(sum, yscale_f32(ep, m), bias_f32(ep.bias, n));
}
// The epilogue of a tile whose first output row is n0 (bias pointer moved to it).
__device__ __forceinline__ Epilogue epilogue_at(Epilogue ep, int64_t n0) {
    if (ep.bias) ep.bias += n0;
    return ep;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

// ------------------------------------------------- programmatic dependent launch
// Let the next kernel in the stream start launching (its blocks then run up to
// their own griddep_wait()).
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
// Wait until the previous kernel in the stream has completed and its memory
// is visible.  A no-op when the launch did not allow early start.
__device__ __forceinline__ void griddep_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" :: "r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" :: "r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" :: "r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ uint64_t globaltimer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

// Every wait on a barrier is bounded: after `limit_ns` of wall time (or as
// soon as another role of the block has given up, *abort != 0; `abort` may be
// null when no other role shares the wait) it returns false, having raised
// *abort and or-ed `code` into the device fault word.
__device__ __forceinline__ bool mbar_wait_bounded(uint32_t bar, uint32_t parity, volatile int* abort,
                                                  unsigned int* fault_word, unsigned int code,
                                                  uint64_t limit_ns) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 15u) == 0u) {
            if (abort && *abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                if (abort) *abort = 1;
                atomicOr(fault_word, code);
                return false;
            }
        }
    }
}
// Drain wait used on the way out: no abort check, only the time limit.
__device__ __forceinline__ bool mbar_drain_bounded(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
    const uint64_t t0 = globaltimer_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (globaltimer_ns() - t0 > limit_ns) return false;
    }
    return true;
}

// --------------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const void* tmap) {
    asm volatile("prefetch.tensormap [%0];" :: "l"(tmap) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4}], [%2];"
        :: "r"(dst), "l"(tmap), "r"(bar), "r"(x), "r"(y) : "memory");
}
// Plain (untiled) bulk copy global -> this block's shared memory, completing
// `bytes` on the mbarrier.  Both addresses 16-byte aligned, bytes % 16 == 0.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
    asm volatile("cp.async.bulk.shared::cta.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
                 :: "r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// Generic-proxy writes to shared memory become visible to the async proxy
// (tcgen05.mma operand reads) after this fence.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 :: "r"(dst_smem), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" :: "r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] . B[smem desc]^T, kind::f16 (bf16 inputs, fp32 accumulate).
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                          uint32_t accumulate) {
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "setp.ne.b32 p, %4, 0;\n\t"
                 "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
                 :: "r"(d_tmem), "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate) : "memory");
}
// Arrive on an mbarrier once all previously issued tcgen05.mma of this thread completed.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                 :: "r"(bar) : "memory");
}
// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld_32cols(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
        "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}

// ------------------------------------------------------- int4 -> bf16 pairs
// Nibbles i and i+4 of a 32-bit word of packed codes (bits 4i..4i+3 and
// 4i+16..4i+19 after the shift) become the bf16 pair (128 + q_i, 128 + q_{i+4}):
// 0x4300 is bf16 128.0, whose last mantissa bit weighs exactly 1.
__device__ __forceinline__ uint32_t nib_pair_biased(uint32_t w_shifted) {
    return (w_shifted & 0x000F000Fu) | 0x43004300u;  // one LOP3
}
// (128 + q) pair -> w' = bf16(q * s + o) pair: q = (128+q) - 128 is exact, then
// one fused multiply-add with a single rounding to bf16.
__device__ __forceinline__ uint32_t dequant_pair(uint32_t biased, uint32_t s2, uint32_t o2) {
    __nv_bfloat162 b = *reinterpret_cast<__nv_bfloat162*>(&biased);
    const __nv_bfloat162 c128 = __floats2bfloat162_rn(128.0f, 128.0f);
    __nv_bfloat162 q = __hsub2(b, c128);
    __nv_bfloat162 w = __hfma2(q, *reinterpret_cast<__nv_bfloat162*>(&s2), *reinterpret_cast<__nv_bfloat162*>(&o2));
    return *reinterpret_cast<uint32_t*>(&w);
}

// ------------------------------------------- split row tiles (stream-K decode)
// The decode kernels cut the (row tile, k) units into equal contiguous warp
// ranges, so several warps can share a row tile.  The tile's owner is the
// warp holding its first unit: the shared tile is the last of the owner's
// range and the first of every other sharer's.  A sharer leaves its partial
// sums in its own slot of the workspace (16 rows x M tokens of 8-byte words:
// the fp32 bits in the low half, 1 in the high half, one naturally aligned
// 64-bit store, so value and flag arrive together) and goes on without
// waiting.  The owner reads the slots of the warps after it (in one batch of
// loads; it waits only for a sharer that is still computing), adds them in
// warp order to its own sums (a fixed order: the result is deterministic),
// writes Y and stores zeros back, so the workspace is all zeros again after
// every call.  Liveness of the wait: a dependent grid starts only once every
// block of this grid has started, so no block an owner waits for can be kept
// off the GPU by work queued behind this grid; the wait is bounded anyway.
constexpr int SPLIT_MAX_WORKERS = 4096;

// workspace bytes: one 16-row slot per warp (at most SPLIT_MAX_WORKERS warps, no
// more than there are 16-row units), two per warp for one token (32-row units)
__host__ __device__ inline size_t split_ws_bytes(int64_t M, int64_t units) {
    const int64_t cap = M == 1 ? 2 * SPLIT_MAX_WORKERS : SPLIT_MAX_WORKERS;
    const int64_t w = units < cap ? units : cap;
    return (size_t)w * 16u * (size_t)M * 8u;
}
// the warp whose range [U w / W, U (w + 1) / W) holds unit u
__device__ __forceinline__ int split_warp_of(long long u, long long units, int workers) {
    return (int)(((u + 1) * workers - 1) / units);
}
__device__ __forceinline__ void st_relaxed_u64(uint64_t* p, uint64_t v) {
    asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" :: "l"(p), "l"(v) : "memory");
}
__device__ __forceinline__ uint64_t ld_relaxed_u64(const uint64_t* p) {
    uint64_t v;
    asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
    return v;
}
// A sharer's part: acc[t][i] holds rows row_a (i < 2) / row_a + 8 (i >= 2) of
// the tile for tokens 8t + 2tq + (i & 1) (the mma.m16n8k16 accumulator).
template <int MT>
__device__ __forceinline__ void split_publish(uint64_t* slot, const float (&acc)[MT][4], int M, int nrows, int row_a,
                                              int tq) {
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * t + 2 * tq + (i & 1), r = row_a + (i & 2) * 4;
            if (m < M && r < nrows) st_relaxed_u64(slot + m * 16 + r, (1ull << 32) | __float_as_uint(acc[t][i]));
        }
}

// The owner's part, after its own sums are in the warp's scratch (16 M floats
// of shared memory, element m * 16 + r): the slots of warps worker + 1 .. wl
// (warp c's words at ws + c * stride),
// then bf16 Y of the tile (Yt = first column of the tile, ldy = N; ep_t, the
// epilogue with its bias moved to the tile's first row, applied before the rounding).  The
// owner's shared tile is the last of its range, so the kernels call this after
// their main loop, when the loop's registers are free.  Each lane takes
// elements lane, lane + 32, ... (NE of them, at most NEMAX; with one token,
// lanes 16..31 take every other sharer instead) and loads 8 slot words per
// batch (NEMAX when that is larger), so a batch costs one round trip to L2.
// Returns false if a wait timed out.
template <int NEMAX>
__device__ __forceinline__ bool split_sum_shares(const float* scr, uint64_t* ws, size_t stride, int worker, int wl,
                                                 int M,
                                                 int nrows, int lane, uint16_t* Yt, int64_t ldy,
                                                 unsigned int* fault_word, unsigned int code, uint64_t limit_ns,
                                                 const Epilogue ep_t = Epilogue()) {
    constexpr int BC = NEMAX >= 8 ? 1 : 8 / NEMAX;  // sharers per batch (8 words per lane, 16 for NEMAX 16)
    bool ok = true;
    const int E = 16 * M;          // words per slot
    const bool halves = E == 16;   // one token: lanes 16..31 take every other sharer
    const int sub = halves ? lane >> 4 : 0, step = halves ? 2 : 1;
    const int e0 = halves ? (lane & 15) : lane;
    float sum[NEMAX];
#pragma unroll
    for (int i = 0; i < NEMAX; ++i) {
        const int e = e0 + 32 * i;
        sum[i] = (sub == 0 && e < E) ? scr[e] : 0.f;
    }
    for (int c0 = worker + 1 + sub; c0 <= wl; c0 += BC * step) {
        uint64_t v[NEMAX][BC];
#pragma unroll
        for (int i = 0; i < NEMAX; ++i)
#pragma unroll
            for (int j = 0; j < BC; ++j) {
                const int c = c0 + j * step, e = e0 + 32 * i;
                const bool use = c <= wl && e < E && (e & 15) < nrows;
                v[i][j] = use ? ld_relaxed_u64(ws + (size_t)c * stride + e) : (1ull << 32);
            }
        uint64_t t0 = 0;
        for (;;) {  // re-poll together the words whose sharer has not published yet
            bool all = true;
#pragma unroll
            for (int i = 0; i < NEMAX; ++i)
#pragma unroll
                for (int j = 0; j < BC; ++j) all = all && (v[i][j] >> 32) != 0u;
            if (all) break;
            const uint64_t now = globaltimer_ns();
            if (t0 == 0) t0 = now;
            if (now - t0 > limit_ns) {  // give up: count what is missing as zero
                atomicOr(fault_word, code);
                ok = false;
                break;
            }
#pragma unroll
            for (int i = 0; i < NEMAX; ++i)
#pragma unroll
                for (int j = 0; j < BC; ++j)
                    if ((v[i][j] >> 32) == 0u)
                        v[i][j] = ld_relaxed_u64(ws + (size_t)(c0 + j * step) * stride + e0 + 32 * i);
        }
#pragma unroll
        for (int i = 0; i < NEMAX; ++i)
#pragma unroll
            for (int j = 0; j < BC; ++j) {
                const int c = c0 + j * step, e = e0 + 32 * i;
                if (c <= wl && e < E && (e & 15) < nrows) {
                    sum[i] += __uint_as_float((uint32_t)v[i][j]);
                    st_relaxed_u64(ws + (size_t)c * stride + e, 0ull);
                }
            }
    }
    if (halves) sum[0] += __shfl_xor_sync(0xffffffffu, sum[0], 16);
#pragma unroll
    for (int i = 0; i < NEMAX; ++i) {
        const int e = e0 + 32 * i;
        if (sub == 0 && e < E && (e & 15) < nrows)
            Yt[(int64_t)(e >> 4) * ldy + (e & 15)] = (uint16_t)float_to_bf16_bits(epilogue_f32(ep_t, sum[i], e >> 4, e & 15));
    }
    return ok;
}
// The owner's part: its own sums into the scratch, then split_sum_shares
// (NEMAX: elements per lane for the largest M of the kernel, 16 M / 32, at least 1).
template <int MT, int NEMAX>
__device__ __forceinline__ bool split_collect(const float (&acc)[MT][4], float* scr, uint64_t* ws, size_t stride,
                                              int worker, int wl,
                                              int M, int nrows, int row_a, int tq, int lane, uint16_t* Yt,
                                              int64_t ldy, unsigned int* fault_word, unsigned int code,
                                              uint64_t limit_ns, const Epilogue ep_t = Epilogue()) {
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * t + 2 * tq + (i & 1), r = row_a + (i & 2) * 4;
            if (m < M) scr[m * 16 + r] = acc[t][i];
        }
    __syncwarp();
    const bool ok =
        split_sum_shares<NEMAX>(scr, ws, stride, worker, wl, M, nrows, lane, Yt, ldy, fault_word, code, limit_ns, ep_t);
    __syncwarp();
    return ok;
}

}  // namespace w4
