// w4_pair.cu -- bf16 x int4 linear for one token on pairs of SMs: no workspace.
//
// Y[n] = sum_k X[k] * w'[n,k], w' = q*s + o, fp32 accumulation (Optimum Quanto:
// bf16 x int4 matmul, accumulation at higher precision, "Pitfalls when
// quantizing activations").  This is w4_linear's one-token kernel when the
// caller passes no workspace: the partial sums of split rows meet in shared
// memory, never in global memory.  With one token the packed codes are nearly
// all of the bytes, so the kernel is built around the memory system:
//
//  * Thread-block clusters of two.  Cluster c owns the output rows of the
//    8-row blocks [rb[c], rb[c+1]) (the problem's 8-row blocks cut into equal
//    contiguous ranges on the host).  Block r (rank in the cluster) takes half
//    of K: the 512-k stages [0, ceil(S/2)) or [ceil(S/2), S).  Both blocks of a
//    pair stream the same number of bytes; the two partial sums of a row meet
//    in distributed shared memory (st.async, counted on the partner's mbarrier).
//  * One block per SM, under half of its registers and shared memory, so the
//    next launch's block is resident beside it and streams its first stages
//    (weights do not depend on this launch) before its programmatic-dependent-
//    launch wait returns.
//  * A cluster's rows are cut into groups of at most 64 rows (multiples of 8,
//    as equal as possible).  A producer warp streams stages of one group x 512 k
//    into a ring of four slots with three TMA copies a stage: the codes as one
//    box of a 3-D view [N][K/256][128 bytes] (h rows x two 128-byte chunks,
//    128-byte swizzle), then one box of scales and one of offsets.  Few, large
//    copies matter: the SM's TMA unit spends a fixed cost on every copy.
//  * X (the block's half of K) is staged once per block after the dependency
//    wait, permuted to the MMA fragment order, with the sum of every 32-k slice.
//  * Sixteen consumer warps take every stage: warp w computes rows 16 t .. +15
//    (t = (w / 4) % 4) over the 128-k quarter w % 4 of the stage.  It copies its
//    codes and qparams into registers, releases the slot, then runs eight
//    mma.m16n8k16 steps whose eight token columns carry 16-k halves of the
//    lane's 32-k slice (lane (gid, tq) supplies X only where its column is a
//    half of the slice its codes come from): A is the raw LOP3 value 128 + q, so
//    each column sums (128 + q) x over its half, and the group's scale and
//    offset are applied in fp32, y += s (D - 128 xs) + o xs, xs the slice's sum
//    of X.  No weight is rounded to bf16.
//  * Row partials are summed in a fixed order (a warp's stages in k order, then
//    the four quarters, then block 0's sum + block 1's sum), so results are
//    deterministic on a given GPU and do not depend on timing.
#include "w4_device.cuh"
#include "w4_internal.h"

#include <algorithm>
#include <cuda.h>

namespace w4 {

constexpr int PK_CW = 16;                       // consumer warps
constexpr int PK_THREADS = (PK_CW + 1) * 32;    // + the producer warp
constexpr int PK_ROWS = 64;                     // rows of a full stage
constexpr int PK_KS = 512;                      // k of a stage
constexpr int PK_DEPTH = 4;                     // ring slots (a power of two)
constexpr int PK_PASS = 256;                    // rows between two exchanges of partial sums
constexpr int PK_MAXK = 16384;                  // X of a block's half of K fits its shared memory
constexpr uint64_t PK_WAIT_LIMIT_NS = 2000000000ull;

// Tensor maps with box heights 8, 16, ..., 64 (index h / 8 - 1): the codes as a
// 3-D view [N][K / 256][128 bytes] (one box = h rows x two 128-byte chunks = 512 k),
// the scales and offsets as [N][K / g] with boxes of pk_qbox(g) groups.
struct PairMaps {
    CUtensorMap w[8], s[8], o[8];
};
constexpr int PK_MAX_CLUSTERS = 128;
struct PairArgs {
    const uint16_t* X;
    uint16_t* Y;
    const uint16_t* bias;  // [N] bf16 added before the rounding, or null
    int N, K;
    int nks;        // 512-k stages per row
    int nclusters;  // gridDim.x / 2
    int rb[PK_MAX_CLUSTERS + 1];  // cluster c owns the 8-row blocks [rb[c], rb[c + 1])
};

// groups of a stage's qparam box: 16 at g = 32 (512 k), 8 above (512 k at g = 64,
// 1024 k at g = 128); host and device
__host__ __device__ constexpr int pk_qbox(int g) { return g == 32 ? 16 : 8; }

// Shared-memory layout (byte offsets from a 1024-aligned base), the same on
// host and device.  A code slot is [row][two 128-byte chunks]; a qparam slot is
// the scales box then the offsets box, [row][pk_qbox(g) groups].
struct PairLayout {
    int qw, qslot, xunits;
    int codes, qp, x, xsum, zrow, part, recv, bars, total;
};
__host__ __device__ inline PairLayout pair_layout(int g, int nks) {
    PairLayout L;
    L.qw = 2 * pk_qbox(g);
    L.qslot = 2 * PK_ROWS * L.qw;
    L.xunits = 2 * ((nks + 1) / 2);          // 256-k units of X of the larger half
    L.codes = 0;                             // PK_DEPTH x (64 x 256) bytes, 1024-aligned
    L.qp = L.codes + PK_DEPTH * PK_ROWS * 256;
    L.x = L.qp + PK_DEPTH * L.qslot;
    L.xsum = L.x + L.xunits * 512;
    L.zrow = L.xsum + L.xunits * 8 * 4;
    L.part = L.zrow + 256;
    L.recv = L.part + 4 * PK_PASS * 4;       // part: [k quarter][pass row]
    L.bars = L.recv + 2 * PK_PASS * 4;
    L.total = L.bars + (2 * PK_DEPTH + 2) * 8;
    return L;
}

__device__ unsigned int g_pair_fault;

// ------------------------------------------------------------ cluster helpers
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_arrive_release() {
    asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory");
}
// the same, one thread at a time (threads of a warp may arrive at different points)
__device__ __forceinline__ void cluster_arrive_release_thread() {
    asm volatile("barrier.cluster.arrive.release;" ::: "memory");
}
__device__ __forceinline__ void cluster_wait_acquire() {
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// address of the same shared-memory location in block `rank` of the cluster
__device__ __forceinline__ uint32_t map_to_rank(uint32_t addr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
// 4 bytes into the partner's shared memory, counted on the partner's mbarrier (both cluster addresses)
__device__ __forceinline__ void st_async_remote_f32(uint32_t addr, float v, uint32_t remote_bar) {
    asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.f32 [%0], %1, [%2];"
                 :: "r"(addr), "f"(v), "r"(remote_bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait_cluster(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\t"
                 "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}
__device__ __forceinline__ void named_bar_sync(int id, int threads) {
    asm volatile("bar.sync %0, %1;" :: "r"(id), "r"(threads) : "memory");
}

// -------------------------------------------------------------- MMA helpers
__device__ __forceinline__ uint4 pk_lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}
// 16 bytes of shared memory where `pred`, zeros elsewhere (lanes that read nothing cost no bandwidth)
__device__ __forceinline__ uint4 pk_lds128_if(bool pred, uint32_t addr) {
    uint4 v = make_uint4(0u, 0u, 0u, 0u);
    asm volatile("{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
                 "@p ld.shared.v4.u32 {%0,%1,%2,%3}, [%5];\n\t}"
                 : "+r"(v.x), "+r"(v.y), "+r"(v.z), "+r"(v.w) : "r"((uint32_t)pred), "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t pk_lds32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ uint32_t pk_lds16(uint32_t addr) {
    unsigned short v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(addr));
    return v;
}
__device__ __forceinline__ float2 pk_lds64f(uint32_t addr) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0,%1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
    return v;
}
__device__ __forceinline__ float pk_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float pk_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

// One m16n8k16 step on raw codes: A = (128 + q) pairs straight from LOP3 of
// nibbles (SH, SH+4) and (SH+1, SH+5) of the code words of rows a and b, B = X
// or zero per lane.  ZC starts from a zero accumulator.
template <int SH, bool ZC>
__device__ __forceinline__ void pk_mma(float (&c)[4], uint32_t wa, uint32_t wb, uint32_t x0, uint32_t x1, uint32_t cm,
                                       uint32_t cg) {
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

// position of 8-k chunk c (0..31) of a 256-k unit in its staged X: a bank swizzle
__device__ __forceinline__ int pk_x_slot(int c) { return c ^ (((c >> 3) & 1) << 1); }

// Row groups of a cluster's range: ng = ceil(nb / 8) groups of whole 8-row
// blocks; group i holds blocks [nb * i / ng, nb * (i + 1) / ng) of the range.
struct PkGroups {
    int nb, ng;
    __device__ __forceinline__ int start(int i) const {
        return nb < 65536 ? 8 * (int)((unsigned)(nb * i) / (unsigned)ng) : 8 * (int)((long long)nb * i / ng);
    }
};
constexpr int PK_GPP = PK_PASS / PK_ROWS;  // row groups per pass (exchange)

// Walks a block's stages in order: row group gi (rows [gs, ge) of the cluster's range), k stage ks.
struct PkCursor {
    int gi, ks, gs, ge;
    __device__ __forceinline__ void init(const PkGroups& grp, int ks0) {
        gi = 0;
        ks = ks0;
        gs = grp.start(0);
        ge = grp.start(1);
    }
    __device__ __forceinline__ void next(const PkGroups& grp, int ks0, int ks1) {
        if (++ks == ks1) {
            ks = ks0;
            ++gi;
            gs = ge;
            ge = grp.start(gi + 1);
        }
    }
};
// first group of the qparam box that holds 512-k stage ks
template <int G>
__device__ __forceinline__ int pk_qbox_x(int ks) {
    return G == 32 ? 16 * ks : G == 64 ? 8 * ks : 8 * (ks >> 1);
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* tmap, uint32_t bar, int x, int y, int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%3, %4, %5}], [%2];"
        :: "r"(dst), "l"(tmap), "r"(bar), "r"(x), "r"(y), "r"(z) : "memory");
}

// rows [0, pk_split(h)) of an h-row group are finished by block 0, the rest by block 1
__device__ __forceinline__ int pk_split(int h) { return 8 * ((h / 8 + 1) / 2); }

// Sets the bytes this block receives in pass ps (4 per row of the pass it finishes, below N)
// on its exchange barrier: the one arrival of the pass's phase.
__device__ __forceinline__ void pk_expect_pass(uint32_t bar, const PkGroups& grp, int ps, int r0, int N,
                                               uint32_t rank) {
    int rows = 0;
    for (int gi = ps * PK_GPP; gi < min(grp.ng, (ps + 1) * PK_GPP); ++gi) {
        const int gs = grp.start(gi), h = grp.start(gi + 1) - gs;
        const int lo = rank == 0 ? 0 : pk_split(h), hi = rank == 0 ? pk_split(h) : h;
        rows += max(0, min(hi, N - r0 - gs) - lo);
    }
    mbar_arrive_expect_tx(bar, (uint32_t)(4 * rows));
}

// L2 prefetch of a tensor-map box (no shared memory, no completion)
__device__ __forceinline__ void tma_prefetch_l2(const void* tmap, int x, int y) {
    asm volatile("cp.async.bulk.prefetch.tensor.2d.L2.global.tile [%0, {%1, %2}];" :: "l"(tmap), "r"(x), "r"(y)
                 : "memory");
}

template <int G>
__global__ void __launch_bounds__(PK_THREADS, 2) pair_kernel(const __grid_constant__ PairMaps maps, const __grid_constant__ PairArgs p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-aligned base, kept as a shared-memory pointer (plain C++ accesses compile to shared loads/stores)
    unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const PairLayout L = pair_layout(G, p.nks);
    const uint32_t base = smem_u32(smem);
    const uint32_t full0 = base + L.bars, empty0 = full0 + 8 * PK_DEPTH, recv_bar = empty0 + 8 * PK_DEPTH;
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.bars + (2 * PK_DEPTH + 1) * 8);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const int cl = blockIdx.x >> 1;

    griddep_launch_dependents();

    // this cluster's rows, cut into row groups; this block's k stages
    const int rb0 = p.rb[cl];
    const int r0 = 8 * rb0;
    PkGroups grp;
    grp.nb = p.rb[cl + 1] - rb0;
    grp.ng = (grp.nb + PK_ROWS / 8 - 1) / (PK_ROWS / 8);
    const int half = (p.nks + 1) / 2;
    const int ks0 = rank ? half : 0, ks1 = rank ? p.nks : half;
    const int nk = ks1 - ks0;
    const int npass = (grp.ng + PK_GPP - 1) / PK_GPP;
    const int nstages = nk * grp.ng;  // stage s = row group s / nk, k stage ks0 + s % nk

    if (threadIdx.x == 0) {
        for (int d = 0; d < PK_DEPTH; ++d) {
            mbar_init(full0 + 8 * d, 1);
            mbar_init(empty0 + 8 * d, PK_CW);  // every consumer warp takes every stage
        }
        mbar_init(recv_bar, 1);  // one expect-tx arrival per pass; the partner's stores complete it
        *abort_flag = 0;
        mbar_fence_init();
        if (npass > 0) pk_expect_pass(recv_bar, grp, 0, r0, p.N, rank);
    }
    __syncthreads();

    if (warp == PK_CW) {
        // ------------------------------------------------------ producer
        // Every thread of both blocks arrives once on the cluster barrier, which the consumers
        // wait on before their first access to the partner's shared memory.  Lane 0 arrives once
        // its first stages are requested (the arrive orders memory, so it should not delay them).
        if (lane != 0) {
            cluster_arrive_release_thread();
            return;
        }
        PkCursor cur;  // the stage to load
        cur.init(grp, ks0);
        bool arrived = false;
        int s = 0;
        for (; s < nstages; ++s) {
            const int slot = s & (PK_DEPTH - 1);
            if (s == PK_DEPTH) {
                cluster_arrive_release_thread();
                arrived = true;
            }
            if (s >= PK_DEPTH &&
                !mbar_wait_bounded(empty0 + 8 * slot, (uint32_t)(((s / PK_DEPTH) - 1) & 1), abort_flag,
                                   &g_pair_fault, 1u, PK_WAIT_LIMIT_NS))
                break;
            const int h = cur.ge - cur.gs;  // rows of the boxes (rows past N are zero-filled)
            const int row0 = r0 + cur.gs, mi = h / 8 - 1;
            const uint32_t bar = full0 + 8 * slot;
            mbar_arrive_expect_tx(bar, (uint32_t)h * (PK_KS / 2 + 2 * L.qw));  // the three boxes below
            tma_load_3d(base + L.codes + slot * (PK_ROWS * 256), &maps.w[mi], bar, 0, 2 * cur.ks, row0);
            const uint32_t qdst = base + L.qp + slot * L.qslot;
            tma_load_2d(qdst, &maps.s[mi], bar, pk_qbox_x<G>(cur.ks), row0);
            tma_load_2d(qdst + PK_ROWS * L.qw, &maps.o[mi], bar, pk_qbox_x<G>(cur.ks), row0);
            cur.next(grp, ks0, ks1);
        }
        if (!arrived) cluster_arrive_release_thread();
        // leave no copy landing in shared memory after the block exits (the consumers have
        // waited for every stage unless a wait gave up)
        for (int t = max(0, s - PK_DEPTH); t < s; ++t)
            mbar_drain_bounded(full0 + 8 * (t % PK_DEPTH), (uint32_t)((t / PK_DEPTH) & 1), PK_WAIT_LIMIT_NS);
        return;
    }
    cluster_arrive_release();  // the partner may arrive on recv_bar once it has waited for this

    // ------------------------------------------------------------ consumers
    // Every consumer warp takes every stage: warp w computes rows 16 t .. 16 t + 15, t = (w / 4) % 4,
    // over the 128-k quarter q = w % 4 of the stage (256-k chunk q / 2, its half q % 2): one item
    // of eight m16n8k16 steps.  The four warps of a tile sit on the four schedulers of the SM, so a
    // short row group (one tile) still spreads over all of them.  A warp copies its codes and qparams into registers and releases the ring
    // slot before it computes, so the ring is refilled while the products run.
    const int ctid = threadIdx.x;              // 0 .. 511
    const int gid = lane >> 2, tq = lane & 3;
    const int t = (warp >> 2) & 3, q = warp & 3, b2 = q >> 1, hq = q & 1;

    // activations may come from the previous kernel: wait for it, then stage X
    griddep_wait();
    {
        const int k0 = ks0 * PK_KS, nu = 2 * nk;  // this block's 256-k units
        float* xsum = reinterpret_cast<float*>(smem + L.xsum);
        for (int c = ctid; c < nu * 32; c += PK_CW * 32) {  // 8-k chunk c: unit c / 32, chunk c % 32
            const int k = k0 + 8 * c;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (k < p.K) v = ldg_cg_v4(p.X + k);  // K % 32 == 0: a chunk is all in or all out
            float part = ((pk_lo(v.x) + pk_hi(v.x)) + (pk_lo(v.y) + pk_hi(v.y))) +
                         ((pk_lo(v.z) + pk_hi(v.z)) + (pk_lo(v.w) + pk_hi(v.w)));
            uint4 o;  // (x0, x4), (x1, x5), (x2, x6), (x3, x7): the nibble-pair order of the codes
            o.x = __byte_perm(v.x, v.z, 0x5410);
            o.y = __byte_perm(v.x, v.z, 0x7632);
            o.z = __byte_perm(v.y, v.w, 0x5410);
            o.w = __byte_perm(v.y, v.w, 0x7632);
            const int u = c >> 5, cc = c & 31;
            *reinterpret_cast<uint4*>(smem + L.x + u * 512 + 16 * pk_x_slot(cc)) = o;
            // slice sums: four consecutive chunks (lanes 4i .. 4i+3) make a 32-k slice
            part += __shfl_xor_sync(0xffffffffu, part, 1);
            part += __shfl_xor_sync(0xffffffffu, part, 2);
            if ((c & 3) == 0) xsum[c >> 2] = part;
        }
    }
    named_bar_sync(1, PK_CW * 32);

    uint32_t cm, cg;  // nibble mask and bf16 128.0 pair, pinned in registers
    asm volatile("mov.b32 %0, %1;" : "=r"(cm) : "r"(0x000F000Fu));
    asm volatile("mov.b32 %0, %1;" : "=r"(cg) : "r"(0x43004300u));
    // MMA row gid <- tile row pr.  A code slot line is (row, chunk) = 2 row + b2, swizzled by its
    // low three bits; the two rows a phase of eight lanes reads (gid 2i, 2i + 1) then differ in
    // bit 2 of that key, so their 16-byte reads never share a bank.
    const int pr = ((gid & 1) << 1) | ((gid >> 1) & 1) | (gid & 4);
    // X words j of the lane's slice (4 hq + tq of its 256-k chunk): the MMA's column 2 tq + (j >> 1)
    // is the 16-k half of slice tq that word j belongs to, so the lane supplies X for j < 2 when
    // gid == 2 tq, for j >= 2 when gid == 2 tq + 1
    const bool selA = gid == 2 * tq, selB = gid == 2 * tq + 1;
    uint32_t boff[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) boff[j] = 16u * (uint32_t)((4 * tq + j) ^ ((tq >> 1) << 1));
    // codes: 16-byte chunk 4 hq + tq of line (row, b2), rows 16 t + pr and + 8 (same swizzle key)
    const int lna = 2 * (16 * t + pr) + b2;
    const uint32_t coff = (uint32_t)(lna * 128) + (((uint32_t)(4 * hq + tq) ^ (uint32_t)(lna & 7)) << 4);
    const uint32_t rowa = (uint32_t)((16 * t + pr) * L.qw), rowb = rowa + 8u * (uint32_t)L.qw;  // qparam box rows
    const int kq = 256 * b2 + 128 * hq + 32 * tq;  // k of the lane's slice inside a stage
    const float* xsum = reinterpret_cast<const float*>(smem + L.xsum);
    float* part = reinterpret_cast<float*>(smem + L.part);
    float* recv = reinterpret_cast<float*>(smem + L.recv);
    const uint32_t partner = rank ^ 1u;
    bool ok = true;
    bool cluster_synced = false;
    int s = 0;

    for (int ps = 0; ps < npass; ++ps) {
        const int g0 = ps * PK_GPP, g1 = min(grp.ng, g0 + PK_GPP);
        for (int gi = g0; gi < g1; ++gi) {
            const int h = grp.start(gi + 1) - grp.start(gi);
            const bool active = 16 * t < h;
            float ya = 0.f, yb = 0.f;  // rows pr, pr + 8 of the warp's tile over its slices
            for (int ks = ks0; ks < ks1; ++ks, ++s) {
                const uint32_t slot = (uint32_t)(s & (PK_DEPTH - 1));
                if (ok)
                    ok = mbar_wait_bounded(full0 + 8 * slot, (uint32_t)((s / PK_DEPTH) & 1), abort_flag,
                                           &g_pair_fault, 2u, PK_WAIT_LIMIT_NS);
                uint4 wa = make_uint4(0u, 0u, 0u, 0u), wb = wa;
                float sA = 0.f, oA = 0.f, sB = 0.f, oB = 0.f;
                const bool work = ok && active;
                if (work) {
                    const uint32_t ra = base + L.codes + slot * (PK_ROWS * 256) + coff;
                    wa = pk_lds128(ra);
                    wb = pk_lds128(ra + 16 * 128);  // row + 8: 16 lines further, same swizzle key
                    const uint32_t qs = base + L.qp + slot * (uint32_t)L.qslot +
                                        (uint32_t)(2 * (kq / G + (G == 128 ? 4 * (ks & 1) : 0)));
                    const uint32_t qo = qs + PK_ROWS * L.qw;
                    sA = pk_lo(pk_lds16(qs + rowa));
                    oA = pk_lo(pk_lds16(qo + rowa));
                    sB = pk_lo(pk_lds16(qs + rowb));
                    oB = pk_lo(pk_lds16(qo + rowb));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(empty0 + 8 * slot);  // the item is in registers: refill the slot
                if (work) {
                    const int unit = 2 * (ks - ks0) + b2;
                    const uint32_t xu = base + L.x + (uint32_t)unit * 512u + 256u * (uint32_t)hq;
                    const uint4 x0 = pk_lds128_if(selA, xu + boff[0]), x1 = pk_lds128_if(selA, xu + boff[1]);
                    const uint4 x2 = pk_lds128_if(selB, xu + boff[2]), x3 = pk_lds128_if(selB, xu + boff[3]);
                    const float xs = xsum[unit * 8 + 4 * hq + tq];
                    float dE[4], dO[4];  // even columns (words 0, 1), odd columns (words 2, 3)
                    pk_mma<0, true>(dE, wa.x, wb.x, x0.x, x0.y, cm, cg);
                    pk_mma<0, true>(dO, wa.z, wb.z, x2.x, x2.y, cm, cg);
                    pk_mma<8, false>(dE, wa.x, wb.x, x0.z, x0.w, cm, cg);
                    pk_mma<8, false>(dO, wa.z, wb.z, x2.z, x2.w, cm, cg);
                    pk_mma<0, false>(dE, wa.y, wb.y, x1.x, x1.y, cm, cg);
                    pk_mma<0, false>(dO, wa.w, wb.w, x3.x, x3.y, cm, cg);
                    pk_mma<8, false>(dE, wa.y, wb.y, x1.z, x1.w, cm, cg);
                    pk_mma<8, false>(dO, wa.w, wb.w, x3.z, x3.w, cm, cg);
                    // columns 2tq (dE) and 2tq + 1 (dO): the two 16-k halves of the lane's slice
                    const float Da = dE[0] + dO[1], Db = dE[2] + dO[3];
                    ya = fmaf(sA, fmaf(-128.f, xs, Da), ya);
                    ya = fmaf(oA, xs, ya);
                    yb = fmaf(sB, fmaf(-128.f, xs, Db), yb);
                    yb = fmaf(oB, xs, yb);
                }
            }
            // the row group's sums of this warp's quarter: over the four lanes of a row pair
            ya += __shfl_xor_sync(0xffffffffu, ya, 1);
            ya += __shfl_xor_sync(0xffffffffu, ya, 2);
            yb += __shfl_xor_sync(0xffffffffu, yb, 1);
            yb += __shfl_xor_sync(0xffffffffu, yb, 2);
            if (tq == 0 && active) {
                const int gp = (gi - g0) * PK_ROWS + 16 * t + pr;
                part[q * PK_PASS + gp] = ya;
                part[q * PK_PASS + gp + 8] = yb;
            }
        }
        // ---- exchange: in each row group the first rows are finished by block 0, the rest by block 1.
        // A block pushes its sums of the partner's rows into the partner's shared memory with
        // st.async, each store counted on the partner's barrier, whose expected byte count the
        // partner set before it pushed anything of this pass (so no store of a later pass can
        // arrive before it).
        named_bar_sync(1, PK_CW * 32);
        if (!cluster_synced) {
            cluster_wait_acquire();  // the partner's barrier is initialised
            cluster_synced = true;
        }
        const int gi = g0 + ((ctid & (PK_PASS - 1)) >> 6), r = ctid & (PK_ROWS - 1);
        const int gs = gi < g1 ? grp.start(gi) : 0;
        const int h = gi < g1 ? grp.start(gi + 1) - gs : 0;
        const int row = r0 + gs + r;
        const int i = ctid & (PK_PASS - 1);
        const bool valid = ctid < PK_PASS && r < h && row < p.N;
        const bool mine = valid && ((r < pk_split(h)) == (rank == 0));
        float sv = 0.f;
        if (valid) sv = (part[i] + part[PK_PASS + i]) + (part[2 * PK_PASS + i] + part[3 * PK_PASS + i]);
        const uint32_t slotoff = (uint32_t)(((ps & 1) * PK_PASS + i) * 4);
        if (valid && !mine)
            st_async_remote_f32(map_to_rank(base + L.recv + slotoff, partner), sv, map_to_rank(recv_bar, partner));
        bool got = true;
        if (mine && !mbar_try_wait_cluster(recv_bar, (uint32_t)(ps & 1))) {
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_try_wait_cluster(recv_bar, (uint32_t)(ps & 1))) {
                if (globaltimer_ns() - t0 > PK_WAIT_LIMIT_NS) {
                    atomicOr(&g_pair_fault, 4u);
                    got = false;
                    break;
                }
            }
        }
        if (mine) {
            const float other = got ? recv[(ps & 1) * PK_PASS + i] : 0.f;
            const float y = rank == 0 ? sv + other : other + sv;  // block 0's sum first, on either block
            p.Y[row] = (uint16_t)float_to_bf16_bits(y + bias_f32(p.bias, row));
        }
        if (!got) *abort_flag = 1;
        named_bar_sync(1, PK_CW * 32);
        if (*abort_flag) ok = false;
        // the next pass's expected bytes, now that this pass's phase has completed
        if (ctid == 0 && ps + 1 < npass) pk_expect_pass(recv_bar, grp, ps + 1, r0, p.N, rank);
    }
    if (!cluster_synced) cluster_wait_acquire();
}

// ------------------------------------------------------------------ host side

// codes [N][K/2] bytes seen as [N][K/256][128]: a box of h rows x 2 chunks holds 512 k of h rows
static cudaError_t encode_codes_map_3d(CUtensorMap* map, const uint8_t* Wq, int64_t N, int64_t K, uint32_t h,
                                       const char** detail) {
    const uint64_t dims[3] = {128, (uint64_t)(K / 256), (uint64_t)N};
    const uint64_t strides[2] = {128, (uint64_t)(K / 2)};
    const uint32_t box[3] = {128, 2, h};
    return encode_tensor_map_3d(map, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B,
                                detail);
}

bool plan_pair(int64_t M, int64_t N, int64_t K, int g, PairPlan* plan) {
    if (M != 1 || N < 1 || K < 32) return false;
    if (K > PK_MAXK) return false;
    if ((K / g) % 8 != 0) return false;  // qparam rows whole 16-byte pieces (TMA row stride); K % 256 == 0
    const int nks = (int)((K + PK_KS - 1) / PK_KS);
    plan->nks = nks;
    plan->smem = (size_t)pair_layout(g, nks).total + 1024;
    return true;
}

template <int G>
static cudaError_t launch_pair_g(const PairMaps& maps, PairArgs a, size_t smem, cudaStream_t stream) {
    auto kern = pair_kernel<G>;
    cudaError_t e = ensure_kernel_attrs(reinterpret_cast<const void*>(kern),
                                        pair_layout(G, (PK_MAXK + PK_KS - 1) / PK_KS).total + 1024, false);
    if (e != cudaSuccess) return e;
    int sms = 0, per_sm = 0;
    if ((e = resident_blocks(reinterpret_cast<const void*>(kern), PK_THREADS, smem, &sms, &per_sm)) != cudaSuccess)
        return e;
    // one cluster per SM pair, but no more clusters than there are 8-row groups
    const int64_t n8 = (a.N + 7) / 8;
    a.nclusters = (int)std::max<int64_t>(1, std::min<int64_t>(std::min(sms / 2, PK_MAX_CLUSTERS), n8));
    for (int c = 0; c <= a.nclusters; ++c) a.rb[c] = (int)(n8 * c / a.nclusters);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)(2 * a.nclusters), 1, 1);
    cfg.blockDim = dim3(PK_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 2;
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kern, maps, a);
}

cudaError_t launch_pair(const PairPlan& plan, const uint16_t* X, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                        const uint16_t* offsets, int64_t N, int g, uint16_t* Y, cudaStream_t stream,
                        const char** detail, const uint16_t* bias) {
    PairMaps maps;
    const int64_t ng = K / g;
    cudaError_t e = cudaSuccess;
    const uint32_t qbox = (uint32_t)pk_qbox(g);  // groups of a stage's qparam box (as the device expects)
    for (int mi = 0; mi < 8 && e == cudaSuccess; ++mi) {
        const uint32_t h = (uint32_t)(8 * (mi + 1));
        // codes as [N][K/256][128 bytes]: boxes of h rows x 2 chunks (512 k), 128-byte swizzle, zero
        // fill past N and past the last chunk (K % 256 == 0, so every chunk is whole)
        e = encode_codes_map_3d(&maps.w[mi], Wq, N, K, h, detail);
        if (e == cudaSuccess)
            e = encode_tensor_map_2d(&maps.s[mi], CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, (uint64_t)ng, (uint64_t)N,
                                     (uint64_t)ng * 2, qbox, h, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e == cudaSuccess)
            e = encode_tensor_map_2d(&maps.o[mi], CU_TENSOR_MAP_DATA_TYPE_UINT16, offsets, (uint64_t)ng, (uint64_t)N,
                                     (uint64_t)ng * 2, qbox, h, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
    }
    if (e != cudaSuccess) return e;
    PairArgs a;
    a.X = X;
    a.Y = Y;
    a.bias = bias;
    a.N = (int)N;
    a.K = (int)K;
    a.nks = plan.nks;
    a.nclusters = 0;
    switch (g) {
        case 32: return launch_pair_g<32>(maps, a, plan.smem, stream);
        case 64: return launch_pair_g<64>(maps, a, plan.smem, stream);
        default: return launch_pair_g<128>(maps, a, plan.smem, stream);
    }
}

cudaError_t read_and_clear_pair_fault(unsigned int* fault) {
    cudaError_t e = cudaMemcpyFromSymbol(fault, g_pair_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !*fault) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_pair_fault, &zero, sizeof(unsigned int));
}

}  // namespace w4
