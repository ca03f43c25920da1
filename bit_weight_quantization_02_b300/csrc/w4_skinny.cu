// w4_skinny.cu -- memory-bound bf16 x int4 linear for few tokens (M <= 32).
//
// Y[m,n] = sum_k X[m,k] * w'[n,k], w' = bf16(q*s + o), fp32 accumulation
// (Optimum Quanto: bf16 x int4 matmul, result accumulated at higher precision,
// "Pitfalls when quantizing activations").  At M <= 32 the packed weights
// dominate the traffic (0.5 + 4/g bytes per weight against 2 bytes per token
// and k), so the kernel is built to stream them at HBM speed:
//
//  * Thread block = 4 warps = 64 output rows x one K slice.  A warp owns 16
//    rows; each lane streams 16 bytes (32 codes) of two rows per 128-k step
//    with 128-bit non-allocating loads, software-pipelined one step group ahead.
//  * In-register dequantization: one LOP3 turns a 32-bit word of codes into
//    the bf16 pairs (128+q_i, 128+q_{i+4}); an exact subtract and one bf16 FMA
//    give w' = bf16(q*s + o) with a single rounding.
//  * The products run on the tensor cores with warp-level mma.m16n8k16
//    (bf16 in, fp32 accumulate) with the weights as the 16-row A operand and
//    the tokens as the 8-column B operand ("swap AB"), so M = 1..32 costs one
//    to four MMAs per A fragment.  The k order inside each 8-k chunk is
//    permuted identically for A (nibble pairs) and B (staged activations), so
//    no register shuffles are needed.
//  * X of the slice is staged once per block in shared memory, permuted and
//    xor-swizzled so the B-fragment loads are bank-conflict free.
//  * Split K: grid.y slices of K write fp32 partial sums to the caller's
//    workspace; the last block to finish a row tile (atomic ticket, no waiting)
//    adds the slices in a fixed order and writes bf16 Y, then resets its
//    ticket to zero for the next call.
//  * Programmatic dependent launch: the block lets the next kernel start at
//    once, and issues its first weight loads before griddepcontrol.wait, so
//    consecutive linears overlap their weight streams.  X, Y and the
//    workspace are only touched after the wait.
#include "w4_device.cuh"
#include "w4_internal.h"

#include <algorithm>

namespace w4 {

constexpr int SK_WARPS = 4;
constexpr int SK_THREADS = SK_WARPS * 32;
constexpr int SK_KSTEP = 128;  // k per step: 4 lanes x 32 codes
constexpr int SK_UNROLL = 4;   // steps per pipelined load group

static_assert(SKINNY_ROWS == 16 * SK_WARPS, "row tile");

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// 16-byte slot of 8-k chunk c inside a token's staged row: chunks of lanes
// with tq in {2,3} (bit 3 of c) swap slots pairwise so that, together with
// the 16-byte row padding, each quarter-warp of B loads hits 8 distinct banks.
__device__ __forceinline__ int x_slot(int c) { return c ^ (((c >> 3) & 1) << 1); }

struct SkinnyArgs {
    const uint16_t* X;
    const uint8_t* Wq;
    const uint16_t* scales;
    const uint16_t* offsets;
    uint16_t* Y;
    float* ws_part;           // [splits][M][N] fp32 partial sums
    unsigned int* ws_ticket;  // [tiles] arrival counters, zero between calls
    int M, N, K, ks, splits;
};

template <int MT, int G>
__global__ void __launch_bounds__(SK_THREADS)
skinny_kernel(const SkinnyArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];
    __shared__ int s_last;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tq = lane & 3;
    const int tile = blockIdx.x, slice = blockIdx.y;
    const int k0 = slice * p.ks;
    const int klen = min(p.K, k0 + p.ks) - k0;  // multiple of 32
    const int nsteps = (klen + SK_KSTEP - 1) / SK_KSTEP;
    const int ngroups = (nsteps + SK_UNROLL - 1) / SK_UNROLL;
    const int pitch = p.ks * 2 + 16;  // bytes per staged token row
    const int qpitch = p.ks / G + 1;  // 32-bit qparam words per staged row (+1 pad)

    unsigned char* xs = smem;                                                // [M][pitch]
    uint32_t* qs = reinterpret_cast<uint32_t*>(smem + (size_t)p.M * pitch);  // [64][qpitch]

    griddep_launch_dependents();

    const int row0 = tile * SKINNY_ROWS;
    const int ra = row0 + warp * 16 + gid;
    const int rb = ra + 8;
    const bool va = ra < p.N, vb = rb < p.N;
    const int64_t rowbytes = p.K / 2;
    const uint8_t* wa = p.Wq + (int64_t)(va ? ra : 0) * rowbytes + k0 / 2;
    const uint8_t* wb = p.Wq + (int64_t)(vb ? rb : 0) * rowbytes + k0 / 2;

    // load group `grp` of SK_UNROLL steps: 16 bytes of rows a and b per step
    auto load_group = [&](int grp, uint4 (&A)[SK_UNROLL], uint4 (&B)[SK_UNROLL]) {
#pragma unroll
        for (int u = 0; u < SK_UNROLL; ++u) {
            const int kk = (grp * SK_UNROLL + u) * SK_KSTEP + 32 * tq;
            const bool in = kk < klen;
            A[u] = (in && va) ? ldg_stream_v4(wa + kk / 2) : make_uint4(0u, 0u, 0u, 0u);
            B[u] = (in && vb) ? ldg_stream_v4(wb + kk / 2) : make_uint4(0u, 0u, 0u, 0u);
        }
    };

    uint4 curA[SK_UNROLL], curB[SK_UNROLL];
    load_group(0, curA, curB);

    // qparams of the block's 64 rows for this slice -> smem as (s | o << 16)
    {
        const int ng = p.K / G;
        const int j0 = k0 / G;
        const int nq = klen / G > 0 ? (klen + G - 1) / G : 1;
        for (int i = threadIdx.x; i < SKINNY_ROWS * nq; i += SK_THREADS) {
            const int r = i / nq, j = i - r * nq;
            const int n = row0 + r;
            uint32_t v = 0;
            if (n < p.N && j0 + j < ng) {
                const int64_t idx = (int64_t)n * ng + j0 + j;
                v = ldg_nc_u16(p.scales + idx) | (ldg_nc_u16(p.offsets + idx) << 16);
            }
            qs[r * qpitch + j] = v;
        }
    }

    // activations may come from the previous kernel: wait for it
    griddep_wait();

    // stage X[:, k0:k0+klen], each 8-k chunk permuted to (x0,x4),(x1,x5),(x2,x6),(x3,x7)
    {
        const int nch = klen / 8;
        for (int i = threadIdx.x; i < p.M * nch; i += SK_THREADS) {
            const int m = i / nch, c = i - m * nch;
            const uint4 v = ldg_cg_v4(p.X + (int64_t)m * p.K + k0 + c * 8);
            uint4 o;
            o.x = __byte_perm(v.x, v.z, 0x5410);
            o.y = __byte_perm(v.x, v.z, 0x7632);
            o.z = __byte_perm(v.y, v.w, 0x5410);
            o.w = __byte_perm(v.y, v.w, 0x7632);
            *reinterpret_cast<uint4*>(xs + (size_t)m * pitch + 16 * x_slot(c)) = o;
        }
    }
    __syncthreads();

    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;

    const uint32_t* qa = qs + (warp * 16 + gid) * qpitch;
    const uint32_t* qb = qa + 8 * qpitch;

    for (int grp = 0; grp < ngroups; ++grp) {
        uint4 nxtA[SK_UNROLL], nxtB[SK_UNROLL];
        if (grp + 1 < ngroups) load_group(grp + 1, nxtA, nxtB);
#pragma unroll
        for (int u = 0; u < SK_UNROLL; ++u) {
            const int step = grp * SK_UNROLL + u;
            const int kk = step * SK_KSTEP + 32 * tq;  // this lane's 32 codes
            if (step < nsteps) {
                const bool in = kk < klen;
                const int jl = in ? kk / G : 0;
                const uint32_t qpa = qa[jl], qpb = qb[jl];
                const uint32_t sa2 = __byte_perm(qpa, 0, 0x1010), oa2 = __byte_perm(qpa, 0, 0x3232);
                const uint32_t sb2 = __byte_perm(qpb, 0, 0x1010), ob2 = __byte_perm(qpb, 0, 0x3232);
                const uint32_t wa4[4] = {curA[u].x, curA[u].y, curA[u].z, curA[u].w};
                const uint32_t wb4[4] = {curB[u].x, curB[u].y, curB[u].z, curB[u].w};
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    // A fragments: (n0,n4),(n1,n5),(n2,n6),(n3,n7) of rows a and b
                    const uint32_t a0 = dequant_pair(nib_pair_biased(wa4[j]), sa2, oa2);
                    const uint32_t a1 = dequant_pair(nib_pair_biased(wa4[j] >> 4), sa2, oa2);
                    const uint32_t a2 = dequant_pair(nib_pair_biased(wa4[j] >> 8), sa2, oa2);
                    const uint32_t a3 = dequant_pair(nib_pair_biased(wa4[j] >> 12), sa2, oa2);
                    const uint32_t b0 = dequant_pair(nib_pair_biased(wb4[j]), sb2, ob2);
                    const uint32_t b1 = dequant_pair(nib_pair_biased(wb4[j] >> 4), sb2, ob2);
                    const uint32_t b2 = dequant_pair(nib_pair_biased(wb4[j] >> 8), sb2, ob2);
                    const uint32_t b3 = dequant_pair(nib_pair_biased(wb4[j] >> 12), sb2, ob2);
                    const int c = step * (SK_KSTEP / 8) + 4 * tq + j;  // 8-k chunk within the slice
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const int m = 8 * t + gid;
                        uint4 xv = make_uint4(0u, 0u, 0u, 0u);
                        if (in && m < p.M)
                            xv = *reinterpret_cast<const uint4*>(xs + (size_t)m * pitch + 16 * x_slot(c));
                        mma_bf16_16816(acc[t], a0, b0, a1, b1, xv.x, xv.y);
                        mma_bf16_16816(acc[t], a2, b2, a3, b3, xv.z, xv.w);
                    }
                }
            }
        }
        if (grp + 1 < ngroups) {
#pragma unroll
            for (int u = 0; u < SK_UNROLL; ++u) {
                curA[u] = nxtA[u];
                curB[u] = nxtB[u];
            }
        }
    }

    // acc[t] = D[row gid, gid+8][token 8t + 2tq, +1]
    if (p.splits == 1) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
            const int m0 = 8 * t + 2 * tq;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = m0 + (i & 1);
                const int n = (i < 2) ? ra : rb;
                if (m < p.M && n < p.N)
                    p.Y[(int64_t)m * p.N + n] = (uint16_t)float_to_bf16_bits(acc[t][i]);
            }
        }
        return;
    }

#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int m0 = 8 * t + 2 * tq;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = m0 + (i & 1);
            const int n = (i < 2) ? ra : rb;
            if (m < p.M && n < p.N)
                __stcg(p.ws_part + ((int64_t)slice * p.M + m) * p.N + n, acc[t][i]);
        }
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) {
        const unsigned int prev = atomicAdd(p.ws_ticket + tile, 1u);
        s_last = (prev == (unsigned int)(p.splits - 1));
    }
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    const int rows = min(SKINNY_ROWS, p.N - row0);
    for (int i = threadIdx.x; i < p.M * SKINNY_ROWS; i += SK_THREADS) {
        const int m = i / SKINNY_ROWS, r = i - m * SKINNY_ROWS;
        if (r >= rows) continue;
        const int64_t n = row0 + r;
        float s = 0.0f;
        for (int sl = 0; sl < p.splits; ++sl) s += __ldcg(p.ws_part + ((int64_t)sl * p.M + m) * p.N + n);
        p.Y[(int64_t)m * p.N + n] = (uint16_t)float_to_bf16_bits(s);
    }
    if (threadIdx.x == 0) p.ws_ticket[tile] = 0u;
}

// ------------------------------------------------------------------ host side

static size_t skinny_smem_bytes(int M, int ks, int g) {
    return (size_t)M * (ks * 2 + 16) + (size_t)SKINNY_ROWS * (ks / g + 1) * 4;
}
// Workspace layout: a fixed region of SK_MAX_TICKETS arrival counters at the
// start (the same bytes for every problem, so a workspace shared by calls of
// different shapes keeps its counters at zero), then [splits][M][N] fp32
// partial sums.
static constexpr int SK_MAX_TICKETS = 16384;  // row tiles: N <= 1,048,576
static constexpr size_t SK_TICKET_BYTES = SK_MAX_TICKETS * 4;
static size_t skinny_ws_bytes(int M, int64_t N, int splits) {
    if (splits <= 1) return 0;
    return SK_TICKET_BYTES + (size_t)splits * M * N * 4;
}

static constexpr int SK_TARGET_BLOCKS = 148 * 8;  // 8 blocks per SM on a 148-SM B300
static constexpr size_t SK_SMEM_CAP = 64 * 1024;  // keeps >= 3 blocks per SM
// attribute limit: the cap, or the smallest slice (128 k) when even that exceeds it
static constexpr size_t SK_SMEM_LIMIT = 96 * 1024;

bool plan_skinny(int64_t M, int64_t N, int64_t K, int g, size_t ws_avail, SkinnyPlan* plan) {
    if (M < 1 || M > SKINNY_MAX_M) return false;
    const int tiles = (int)((N + SKINNY_ROWS - 1) / SKINNY_ROWS);
    const int kchunks = (int)((K + SK_KSTEP - 1) / SK_KSTEP);
    // largest slice whose activations fit the shared-memory cap
    int ks_cap = SK_KSTEP;
    while (ks_cap + SK_KSTEP <= kchunks * SK_KSTEP &&
           skinny_smem_bytes((int)M, ks_cap + SK_KSTEP, g) <= SK_SMEM_CAP)
        ks_cap += SK_KSTEP;
    int splits = std::max(1, std::min(kchunks, (SK_TARGET_BLOCKS + tiles - 1) / tiles));
    int ks = (int)(((K + splits - 1) / splits + SK_KSTEP - 1) / SK_KSTEP) * SK_KSTEP;
    ks = std::min(ks, ks_cap);
    splits = (int)((K + ks - 1) / ks);
    // shrink the split until the workspace holds it (larger slices, fewer blocks)
    if (tiles > SK_MAX_TICKETS) splits = 1;  // no split for more rows than the ticket region covers
    while (splits > 1 && skinny_ws_bytes((int)M, N, splits) > ws_avail) {
        if (ks + SK_KSTEP > ks_cap) return false;
        ks += SK_KSTEP;
        splits = (int)((K + ks - 1) / ks);
    }
    if (splits > 65535) return false;  // grid.y limit
    plan->tiles = tiles;
    plan->splits = splits;
    plan->ks = ks;
    plan->smem = skinny_smem_bytes((int)M, ks, g);
    plan->ws_bytes = skinny_ws_bytes((int)M, N, splits);
    return true;
}

template <int MT, int G>
static cudaError_t launch_one(const SkinnyPlan& plan, const SkinnyArgs& a, cudaStream_t stream) {
    auto kern = skinny_kernel<MT, G>;
    cudaError_t e = ensure_smem_limit(reinterpret_cast<const void*>(kern), (int)SK_SMEM_LIMIT);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.tiles, (unsigned)plan.splits, 1);
    cfg.blockDim = dim3(SK_THREADS, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, a);
}

template <int G>
static cudaError_t launch_g(const SkinnyPlan& plan, const SkinnyArgs& a, cudaStream_t stream) {
    switch ((a.M + 7) / 8) {
        case 1: return launch_one<1, G>(plan, a, stream);
        case 2: return launch_one<2, G>(plan, a, stream);
        case 3: return launch_one<3, G>(plan, a, stream);
        default: return launch_one<4, G>(plan, a, stream);
    }
}

cudaError_t launch_skinny(const SkinnyPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                          const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                          void* workspace, cudaStream_t stream) {
    SkinnyArgs a;
    a.X = X;
    a.Wq = Wq;
    a.scales = scales;
    a.offsets = offsets;
    a.Y = Y;
    a.ws_ticket = plan.splits > 1 ? static_cast<unsigned int*>(workspace) : nullptr;
    a.ws_part = plan.splits > 1 ? reinterpret_cast<float*>(static_cast<char*>(workspace) + SK_TICKET_BYTES) : nullptr;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.ks = plan.ks;
    a.splits = plan.splits;
    switch (g) {
        case 32: return launch_g<32>(plan, a, stream);
        case 64: return launch_g<64>(plan, a, stream);
        default: return launch_g<128>(plan, a, stream);
    }
}

}  // namespace w4
