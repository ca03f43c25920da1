// w4_skinny.cu -- memory-bound bf16 x int4 linear for few tokens (M <= 32).
//
// Y[m,n] = sum_k X[m,k] * w'[n,k], w' = bf16(q*s + o), fp32 accumulation
// (Optimum Quanto: bf16 x int4 matmul, result accumulated at higher precision,
// "Pitfalls when quantizing activations").  At M <= 32 the packed weights
// dominate the traffic (0.5 + 4/g bytes per weight against 2 bytes per token
// and k), so the kernel is built to stream them at HBM speed with as few
// instructions per weight as possible:
//
//  * Thread block = 4 warps = 64 output rows x one K slice.  A warp owns 16
//    rows; each lane streams 16 bytes (32 codes) of two rows per 128-k step
//    with 128-bit non-allocating loads, plus the two rows' scale and offset,
//    ping-ponging between two register buffers a few steps ahead.
//  * In-register dequantization: one LOP3 turns a 32-bit word of codes into
//    the bf16 pairs (128+q_i, 128+q_{i+4}); an exact subtract and one bf16 FMA
//    give w' = bf16(q*s + o) with a single rounding.
//  * The products run on the tensor cores with warp-level mma.m16n8k16
//    (bf16 in, fp32 accumulate) with the weights as the 16-row A operand and
//    the tokens as the 8-column B operand ("swap AB"), so M = 1..32 costs one
//    to four MMAs per A fragment.  The k order inside each 8-k chunk is
//    permuted identically for A (nibble pairs) and B (staged activations).
//  * X of the slice is staged in shared memory (in sub-chunks when it would
//    not fit), permuted and xor-swizzled so B-fragment loads are bank-conflict
//    free; tokens beyond M read a zero row, so the inner loop has no branches.
//  * Split K without global scratch: the S slices of a row tile form one
//    thread-block cluster; each block leaves its fp32 partial tile in its own
//    shared memory, and after a cluster barrier every block sums a share of
//    the outputs over the S ranks through distributed shared memory, in rank
//    order (deterministic), and writes bf16 Y.
//  * Programmatic dependent launch: the block lets the next kernel start at
//    once and issues its first weight loads before griddepcontrol.wait, so
//    consecutive linears overlap their weight streams.  X and Y are only
//    touched after the wait.
#include "w4_device.cuh"
#include "w4_internal.h"

#include <algorithm>
#include <cooperative_groups.h>

namespace cg = cooperative_groups;

namespace w4 {

constexpr int SK_WARPS = 4;
constexpr int SK_THREADS = SK_WARPS * 32;
constexpr int SK_KSTEP = 128;  // k per step: 4 lanes x 32 codes
constexpr int SK_U = 2;        // steps per register buffer

static_assert(SKINNY_ROWS == 16 * SK_WARPS, "row tile");

__device__ __forceinline__ void mma_bf16_16816(float (&c)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1) {
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// 16-byte slot of 8-k chunk c inside a token's staged row: the chunks of lanes
// with tq in {2,3} (bit 3 of c) swap slots pairwise so that, with the 16-byte
// row padding, each quarter-warp of B loads hits 8 distinct bank groups.
__device__ __forceinline__ int x_slot(int c) { return c ^ (((c >> 3) & 1) << 1); }

struct SkinnyArgs {
    const uint16_t* X;
    const uint8_t* Wq;
    const uint16_t* scales;
    const uint16_t* offsets;
    uint16_t* Y;
    int M, N, K;
    int ks;      // k per slice (multiple of SK_KSTEP * SK_U)
    int kc;      // k per staged X sub-chunk (multiple of SK_KSTEP * SK_U, divides ks)
    int splits;  // K slices = cluster size along grid.y
};

template <int U>
struct WBuf {
    uint4 a[U], b[U];       // 16 bytes of codes of rows a and b per step
    uint32_t qa[U], qb[U];  // (scale | offset << 16) of rows a and b per step
};

template <int MT, int G>
__global__ void __launch_bounds__(SK_THREADS)
skinny_kernel(const SkinnyArgs p) {
    extern __shared__ __align__(16) unsigned char smem[];

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tq = lane & 3;
    const int tile = blockIdx.x, slice = blockIdx.y;
    const int k0 = slice * p.ks;
    const int klen = min(p.K - k0, p.ks);  // multiple of 32
    const int nsteps = (klen + SK_KSTEP - 1) / SK_KSTEP;
    const int nbuf = (nsteps + SK_U - 1) / SK_U;  // register buffers to consume
    const int pitch = p.kc * 2 + 16;              // bytes per staged token row

    unsigned char* xs = smem;                              // [M][pitch]
    unsigned char* zrow = smem + (size_t)p.M * pitch;      // [pitch] zeros
    float* part = reinterpret_cast<float*>(zrow + pitch);  // [M][64]

    griddep_launch_dependents();

    const int row0 = tile * SKINNY_ROWS;
    const int ra = row0 + warp * 16 + gid;
    const int rb = ra + 8;
    const bool va = ra < p.N, vb = rb < p.N;
    const uint8_t* wa = p.Wq + (int64_t)(va ? ra : 0) * (p.K / 2) + k0 / 2;
    const uint8_t* wb = p.Wq + (int64_t)(vb ? rb : 0) * (p.K / 2) + k0 / 2;
    const int ng = p.K / G;
    const int64_t qoffa = (int64_t)(va ? ra : 0) * ng + k0 / G;
    const int64_t qoffb = (int64_t)(vb ? rb : 0) * ng + k0 / G;

    auto load = [&](int buf, WBuf<SK_U>& w) {
#pragma unroll
        for (int u = 0; u < SK_U; ++u) {
            const int kk = (buf * SK_U + u) * SK_KSTEP + 32 * tq;  // this lane's 32 codes, within the slice
            const bool in = kk < klen;
            const int j = kk / G;
            w.a[u] = (in && va) ? ldg_stream_v4(wa + kk / 2) : make_uint4(0u, 0u, 0u, 0u);
            w.b[u] = (in && vb) ? ldg_stream_v4(wb + kk / 2) : make_uint4(0u, 0u, 0u, 0u);
            w.qa[u] = (in && va) ? (ldg_nc_u16(p.scales + qoffa + j) | (ldg_nc_u16(p.offsets + qoffa + j) << 16)) : 0u;
            w.qb[u] = (in && vb) ? (ldg_nc_u16(p.scales + qoffb + j) | (ldg_nc_u16(p.offsets + qoffb + j) << 16)) : 0u;
        }
    };

    WBuf<SK_U> w0, w1;
    load(0, w0);

    // activations may come from the previous kernel: wait for it
    griddep_wait();

    // stage X[:, k0 + c0 : k0 + c0 + kc] into the token rows; zeros past the slice end
    const int kc_chunks = p.kc / 8;
    auto stage = [&](int c0) {  // c0 = first k of the sub-chunk, relative to k0
        const int valid = max(0, min(p.kc, klen - c0)) / 8;
        for (int m = 0; m < p.M; ++m) {
            const uint16_t* xrow = p.X + (int64_t)m * p.K + k0 + c0;
            unsigned char* srow = xs + (size_t)m * pitch;
            for (int c = threadIdx.x; c < kc_chunks; c += SK_THREADS) {
                uint4 o = make_uint4(0u, 0u, 0u, 0u);
                if (c < valid) {
                    const uint4 v = ldg_cg_v4(xrow + c * 8);
                    o.x = __byte_perm(v.x, v.z, 0x5410);  // (x0, x4)
                    o.y = __byte_perm(v.x, v.z, 0x7632);  // (x1, x5)
                    o.z = __byte_perm(v.y, v.w, 0x5410);  // (x2, x6)
                    o.w = __byte_perm(v.y, v.w, 0x7632);  // (x3, x7)
                }
                *reinterpret_cast<uint4*>(srow + 16 * x_slot(c)) = o;
            }
        }
    };
    for (int c = threadIdx.x; c < kc_chunks; c += SK_THREADS)
        *reinterpret_cast<uint4*>(zrow + 16 * c) = make_uint4(0u, 0u, 0u, 0u);
    stage(0);
    __syncthreads();

    // per-lane B addresses: token row (or the zero row) + swizzled chunk offsets
    uint32_t bbase[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int m = 8 * t + gid;
        bbase[t] = smem_u32(m < p.M ? xs + (size_t)m * pitch : zrow);
    }
    uint32_t boff[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) boff[j] = 16u * (uint32_t)((4 * tq + j) ^ ((tq >> 1) << 1));

    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;

    const int bufs_per_chunk = p.kc / (SK_KSTEP * SK_U);

    auto compute = [&](int buf, const WBuf<SK_U>& w) {
        if (buf > 0 && buf % bufs_per_chunk == 0) {  // next X sub-chunk (block-uniform)
            __syncthreads();
            stage((buf / bufs_per_chunk) * p.kc);
            __syncthreads();
        }
        const int sbase = (buf % bufs_per_chunk) * SK_U;  // first step of this buffer inside the sub-chunk
#pragma unroll
        for (int u = 0; u < SK_U; ++u) {
            if (buf * SK_U + u < nsteps) {
                const uint32_t sa2 = __byte_perm(w.qa[u], 0, 0x1010), oa2 = __byte_perm(w.qa[u], 0, 0x3232);
                const uint32_t sb2 = __byte_perm(w.qb[u], 0, 0x1010), ob2 = __byte_perm(w.qb[u], 0, 0x3232);
                const uint32_t wa4[4] = {w.a[u].x, w.a[u].y, w.a[u].z, w.a[u].w};
                const uint32_t wb4[4] = {w.b[u].x, w.b[u].y, w.b[u].z, w.b[u].w};
                const uint32_t soff = (uint32_t)(sbase + u) * 256u;  // 16 chunks of 16 bytes per step
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
#pragma unroll
                    for (int t = 0; t < MT; ++t) {
                        const uint4 xv = lds128(bbase[t] + soff + boff[j]);
                        mma_bf16_16816(acc[t], a0, b0, a1, b1, xv.x, xv.y);
                        mma_bf16_16816(acc[t], a2, b2, a3, b3, xv.z, xv.w);
                    }
                }
            }
        }
    };

    for (int buf = 0; buf < nbuf; buf += 2) {
        if (buf + 1 < nbuf) load(buf + 1, w1);
        compute(buf, w0);
        if (buf + 1 < nbuf) {
            if (buf + 2 < nbuf) load(buf + 2, w0);
            compute(buf + 1, w1);
        }
    }

    // acc[t][i] = D[row gid (i<2) or gid+8][token 8t + 2tq + (i&1)]
    if (p.splits == 1) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = 8 * t + 2 * tq + (i & 1);
                const int n = (i < 2) ? ra : rb;
                if (m < p.M && n < p.N) p.Y[(int64_t)m * p.N + n] = (uint16_t)float_to_bf16_bits(acc[t][i]);
            }
        }
        return;
    }

    // split K: partial tile -> own shared memory, then a share of the sum over the cluster
#pragma unroll
    for (int t = 0; t < MT; ++t) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int m = 8 * t + 2 * tq + (i & 1);
            const int r = warp * 16 + gid + ((i < 2) ? 0 : 8);
            if (m < p.M) part[m * SKINNY_ROWS + r] = acc[t][i];
        }
    }
    cg::cluster_group cluster = cg::this_cluster();
    cluster.sync();
    const int total = p.M * SKINNY_ROWS;
    const int share = (total + p.splits - 1) / p.splits;
    const int rank = (int)cluster.block_rank();
    const int lo = rank * share, hi = min(total, lo + share);
    for (int idx = lo + threadIdx.x; idx < hi; idx += SK_THREADS) {
        float s = 0.0f;
        for (int q = 0; q < p.splits; ++q) s += cluster.map_shared_rank(part, q)[idx];
        const int m = idx / SKINNY_ROWS, r = idx % SKINNY_ROWS;
        const int n = row0 + r;
        if (n < p.N) p.Y[(int64_t)m * p.N + n] = (uint16_t)float_to_bf16_bits(s);
    }
    cluster.sync();  // no block leaves while its partials may still be read
}

// ------------------------------------------------------------------ host side

static constexpr int SK_TARGET_BLOCKS = 148 * 6;  // about 6 resident blocks on each of 148 SMs
static constexpr int SK_MAX_SPLIT = 8;            // portable cluster size
static constexpr size_t SK_SMEM_CAP = 40 * 1024;  // keeps >= 5 blocks per SM; below the default 48 KB

static size_t skinny_smem_bytes(int M, int kc, int splits) {
    return (size_t)(M + 1) * (kc * 2 + 16) + (splits > 1 ? (size_t)M * SKINNY_ROWS * 4 : 0);
}

bool plan_skinny(int64_t M, int64_t N, int64_t K, int g, SkinnyPlan* plan) {
    (void)g;
    if (M < 1 || M > SKINNY_MAX_M) return false;
    const int64_t tiles = (N + SKINNY_ROWS - 1) / SKINNY_ROWS;
    if (tiles > 0x7FFFFFFF) return false;
    const int quantum = SK_KSTEP * SK_U;  // slices and sub-chunks are whole register buffers
    const int64_t kq = (K + quantum - 1) / quantum;
    int splits = (int)std::min<int64_t>(SK_MAX_SPLIT, std::max<int64_t>(1, (SK_TARGET_BLOCKS + tiles - 1) / tiles));
    splits = (int)std::min<int64_t>(splits, kq);
    const int64_t ks = (kq + splits - 1) / splits * quantum;
    splits = (int)((K + ks - 1) / ks);
    // largest sub-chunk (whole quanta, dividing ks) whose staged X fits the cap
    int64_t kc = ks;
    while (kc > quantum && skinny_smem_bytes((int)M, (int)kc, splits) > SK_SMEM_CAP) {
        int64_t q = kc / quantum - 1;
        while (q > 1 && (ks / quantum) % q != 0) --q;
        kc = q * quantum;
    }
    plan->tiles = (int)tiles;
    plan->splits = splits;
    plan->ks = (int)ks;
    plan->kc = (int)kc;
    plan->smem = skinny_smem_bytes((int)M, (int)kc, splits);
    return true;
}

template <int MT, int G>
static cudaError_t launch_one(const SkinnyPlan& plan, const SkinnyArgs& a, cudaStream_t stream) {
    auto kern = skinny_kernel<MT, G>;  // dynamic shared memory <= SK_SMEM_CAP, under the default 48 KB
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)plan.tiles, (unsigned)plan.splits, 1);
    cfg.blockDim = dim3(SK_THREADS, 1, 1);
    cfg.dynamicSmemBytes = plan.smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = (unsigned)plan.splits;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
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
                          cudaStream_t stream) {
    SkinnyArgs a;
    a.X = X;
    a.Wq = Wq;
    a.scales = scales;
    a.offsets = offsets;
    a.Y = Y;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.ks = plan.ks;
    a.kc = plan.kc;
    a.splits = plan.splits;
    switch (g) {
        case 32: return launch_g<32>(plan, a, stream);
        case 64: return launch_g<64>(plan, a, stream);
        default: return launch_g<128>(plan, a, stream);
    }
}

}  // namespace w4
