// w4_skinny.cu -- memory-bound bf16 x int4 linear for few tokens (M <= 32).
//
// Y[m,n] = sum_k X[m,k] * w'[n,k], w' = bf16(q*s + o), fp32 accumulation
// (Optimum Quanto: bf16 x int4 matmul, result accumulated at higher precision,
// "Pitfalls when quantizing activations").  At M <= 32 the packed weights
// dominate the traffic (0.5 + 4/g bytes per weight against 2 bytes per token
// and k), so the kernel is built to stream them at HBM speed with as few
// instructions per weight as possible:
//
//  * Thread block = 4 warps = 64 output rows x one K slice of up to 2048 k.
//    At block start one thread issues the whole slice as 2-D TMA copies of
//    64 rows x 256 k (128 bytes, 128-byte swizzle), one mbarrier per copy,
//    plus the slice's scales and offsets: everything is in flight before the
//    block even waits for the previous kernel, and compute on the first 256 k
//    starts as soon as it lands.  TMA zero-fills rows past N and k past K.
//    Warps read 16 bytes (32 codes) of two rows per 128-k step from shared
//    memory; the rows of an MMA tile are permuted so the swizzled reads of a
//    quarter-warp fall in distinct banks.
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
#include <cuda.h>

namespace cg = cooperative_groups;

namespace w4 {

constexpr int SK_WARPS = 4;
constexpr int SK_THREADS = SK_WARPS * 32;
constexpr int SK_KSTEP = 128;  // k per step: 4 lanes x 32 codes

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
    const uint16_t* scales;   // used by the plain-load qparam path only
    const uint16_t* offsets;
    uint16_t* Y;
    const uint16_t* bias;  // [N] bf16 added before the rounding, or null
    int M, N, K;
    int ks;      // k per slice (multiple of 256)
    int kc;      // k per staged X sub-chunk (multiple of 256, divides ks)
    int splits;  // K slices = cluster size along grid.y
    int qtma;    // 1: qparams arrive by TMA with the first chunk; 0: plain loads
};

constexpr int SK_CHUNK = 256;                    // k per TMA chunk: 64 rows x 128 bytes of codes
constexpr int SK_CHUNK_BYTES = SKINNY_ROWS * 128;
constexpr int SK_MAX_CHUNKS = 8;                 // slices up to 2048 k

// Byte offsets inside the dynamic shared memory of one block (host and device
// compute the same layout).  The code chunks come first, 1024-byte aligned
// for the 128-byte TMA swizzle.
struct SkLayout {
    int qpitch, xpitch;
    int off_s, off_o, off_x, off_z, off_part, off_bar, total;
};
__host__ __device__ inline SkLayout sk_layout(int M, int ks, int kc, int g, int splits) {
    SkLayout L;
    L.qpitch = 2 * (ks / g);  // bytes per row of staged scales (or offsets); TMA writes rows back to back
    L.xpitch = kc * 2 + 16;
    int off = (ks / SK_CHUNK) * SK_CHUNK_BYTES;
    L.off_s = off;  // TMA destinations: 128-byte aligned
    off += SKINNY_ROWS * L.qpitch;
    off = (off + 127) & ~127;
    L.off_o = off;
    off += SKINNY_ROWS * L.qpitch;
    off = (off + 127) & ~127;
    L.off_x = off;
    off += M * L.xpitch;
    L.off_z = off;
    off += L.xpitch;
    L.off_part = off;
    off += splits > 1 ? M * SKINNY_ROWS * 4 : 0;
    L.off_bar = off;
    off += 8 * SK_MAX_CHUNKS + 16;
    L.total = off;
    return L;
}

__device__ unsigned int g_skinny_fault;
constexpr uint64_t SK_WAIT_LIMIT_NS = 2000000000ull;

template <int MT, int G>
__global__ void __launch_bounds__(SK_THREADS)
skinny_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_s,
              const __grid_constant__ CUtensorMap tm_o, const SkinnyArgs p) {
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char* smem = reinterpret_cast<unsigned char*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const SkLayout L = sk_layout(p.M, p.ks, p.kc, G, p.splits);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gid = lane >> 2, tq = lane & 3;
    const int tile = blockIdx.x, slice = blockIdx.y;
    const int k0 = slice * p.ks;
    const int klen = min(p.K - k0, p.ks);  // multiple of 32
    const int nsteps = (klen + SK_KSTEP - 1) / SK_KSTEP;
    const int nchunks = (klen + SK_CHUNK - 1) / SK_CHUNK;
    const int row0 = tile * SKINNY_ROWS;
    const int nqs = klen / G;  // groups of this slice (>= 1)

    uint16_t* ssm = reinterpret_cast<uint16_t*>(smem + L.off_s);  // [64][ks/G] scales
    uint16_t* osm = reinterpret_cast<uint16_t*>(smem + L.off_o);  // [64][ks/G] offsets
    unsigned char* xs = smem + L.off_x;                            // [M][xpitch] staged X
    unsigned char* zrow = smem + L.off_z;                          // [xpitch] zeros
    float* part = reinterpret_cast<float*>(smem + L.off_part);     // [M][64] partial sums
    const uint32_t bar0 = smem_u32(smem + L.off_bar);               // one mbarrier per chunk
    volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L.off_bar + 8 * SK_MAX_CHUNKS);

    griddep_launch_dependents();

    // ---- every chunk of the slice in flight at once, before waiting on the previous kernel
    if (threadIdx.x == 0) {
        for (int c = 0; c < nchunks; ++c) mbar_init(bar0 + 8 * c, 1);
        *abort_flag = 0;
        mbar_fence_init();
        tma_prefetch_desc(&tm_w);
        const uint32_t qbytes = p.qtma ? (uint32_t)(2 * SKINNY_ROWS * L.qpitch) : 0u;
        for (int c = 0; c < nchunks; ++c) {
            const uint32_t bar = bar0 + 8 * c;
            mbar_arrive_expect_tx(bar, SK_CHUNK_BYTES + (c == 0 ? qbytes : 0u));
            tma_load_2d(smem_u32(smem) + c * SK_CHUNK_BYTES, &tm_w, bar, (k0 + c * SK_CHUNK) / 2, row0);
            if (c == 0 && p.qtma) {
                tma_load_2d(smem_u32(ssm), &tm_s, bar, k0 / G, row0);
                tma_load_2d(smem_u32(osm), &tm_o, bar, k0 / G, row0);
            }
        }
    }
    if (!p.qtma) {  // qparams by plain loads; zeros for rows past N and groups past the slice
        const int nrows = min(SKINNY_ROWS, p.N - row0);
        const int qcols = L.qpitch / 2;
        const int ng = p.K / G;
        for (int r = 0; r < SKINNY_ROWS; ++r)
            for (int j = threadIdx.x; j < qcols; j += SK_THREADS) {
                uint16_t sv = 0, ov = 0;
                if (r < nrows && j < nqs) {
                    const int64_t idx = (int64_t)(row0 + r) * ng + k0 / G + j;
                    sv = (uint16_t)ldg_nc_u16(p.scales + idx);
                    ov = (uint16_t)ldg_nc_u16(p.offsets + idx);
                }
                ssm[r * qcols + j] = sv;
                osm[r * qcols + j] = ov;
            }
    }

    // ---- activations may come from the previous kernel: wait for it, then stage X
    griddep_wait();
    const int kc_chunks = p.kc / 8;
    auto stage = [&](int c0) {  // X[:, k0 + c0 : k0 + c0 + kc], each 8-k chunk permuted; zeros past the slice
        const int valid = max(0, min(p.kc, klen - c0)) / 8;
        for (int m = 0; m < p.M; ++m) {
            const uint16_t* xrow = p.X + (int64_t)m * p.K + k0 + c0;
            unsigned char* srow = xs + (size_t)m * L.xpitch;
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

    uint32_t bbase[MT];
#pragma unroll
    for (int t = 0; t < MT; ++t) {
        const int m = 8 * t + gid;
        bbase[t] = smem_u32(m < p.M ? xs + (size_t)m * L.xpitch : zrow);
    }
    uint32_t boff[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) boff[j] = 16u * (uint32_t)((4 * tq + j) ^ ((tq >> 1) << 1));

    // A-row gid of the warp's MMA tile is weight row pi(gid) = {0,4,1,5,2,6,3,7}[gid] (+8 for gid+8):
    // the two rows a quarter-warp reads then differ in bit 2, which the 128-byte swizzle turns into
    // different bank halves.
    const int pr = ((gid >> 1) | ((gid & 1) << 2));
    const int ra = warp * 16 + pr;  // local rows ra and ra + 8
    const uint32_t wsm = smem_u32(smem);
    const uint32_t wa_row = wsm + ra * 128, wb_row = wa_row + 8 * 128;
    const uint32_t swz = (uint32_t)(ra & 7);  // rows ra and ra + 8 share it
    const int qcols = L.qpitch / 2;
    const uint16_t* sa_p = ssm + ra * qcols;
    const uint16_t* oa_p = osm + ra * qcols;
    const uint16_t* sb_p = sa_p + 8 * qcols;
    const uint16_t* ob_p = oa_p + 8 * qcols;

    float acc[MT][4];
#pragma unroll
    for (int t = 0; t < MT; ++t)
#pragma unroll
        for (int i = 0; i < 4; ++i) acc[t][i] = 0.0f;

    bool ok = true;
    const int steps_per_chunk = p.kc / SK_KSTEP;
    int sc = 0;       // step inside the staged X sub-chunk
    uint32_t xo = 0;  // its byte offset in a staged row
#pragma unroll 2
    for (int s = 0; s < nsteps; ++s) {
        if (sc == steps_per_chunk) {  // next X sub-chunk (block-uniform)
            __syncthreads();
            stage(s * SK_KSTEP);
            __syncthreads();
            sc = 0;
            xo = 0;
        }
        if ((s & 1) == 0)  // first step of a TMA chunk: wait for it (bounded)
            ok = mbar_wait_bounded(bar0 + 8 * (s >> 1), 0, abort_flag, &g_skinny_fault, 1u, SK_WAIT_LIMIT_NS) && ok;
        const uint32_t cbase = (uint32_t)(s >> 1) * SK_CHUNK_BYTES;
        const uint32_t cpos = (((uint32_t)(4 * (s & 1) + tq)) ^ swz) << 4;
        const uint4 wa = lds128(wa_row + cbase + cpos);
        const uint4 wb = lds128(wb_row + cbase + cpos);
        const int jg = (s * SK_KSTEP + 32 * tq) / G;
        const uint32_t sa2 = __byte_perm(sa_p[jg], 0, 0x1010), oa2 = __byte_perm(oa_p[jg], 0, 0x1010);
        const uint32_t sb2 = __byte_perm(sb_p[jg], 0, 0x1010), ob2 = __byte_perm(ob_p[jg], 0, 0x1010);
        const uint32_t wa4[4] = {wa.x, wa.y, wa.z, wa.w};
        const uint32_t wb4[4] = {wb.x, wb.y, wb.z, wb.w};
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
                const uint4 xv = lds128(bbase[t] + xo + boff[j]);
                mma_bf16_16816(acc[t], a0, b0, a1, b1, xv.x, xv.y);
                mma_bf16_16816(acc[t], a2, b2, a3, b3, xv.z, xv.w);
            }
        }
        ++sc;
        xo += 256u;  // 16 chunks of 16 bytes per step
    }

    // acc[t][i] = D[row ra (i<2) or ra+8][token 8t + 2tq + (i&1)]
    if (p.splits == 1) {
#pragma unroll
        for (int t = 0; t < MT; ++t) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = 8 * t + 2 * tq + (i & 1);
                const int n = row0 + ra + ((i < 2) ? 0 : 8);
                if (m < p.M && n < p.N)
                    p.Y[(int64_t)m * p.N + n] = (uint16_t)float_to_bf16_bits(acc[t][i] + bias_f32(p.bias, n));
            }
        }
    } else {
        // split K: partial tile -> own shared memory, then a share of the sum over the cluster
#pragma unroll
        for (int t = 0; t < MT; ++t) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const int m = 8 * t + 2 * tq + (i & 1);
                if (m < p.M) part[m * SKINNY_ROWS + ra + ((i < 2) ? 0 : 8)] = acc[t][i];
            }
        }
        cg::cluster_group cluster = cg::this_cluster();
        cluster.sync();
        const int total = p.M * SKINNY_ROWS;
        const int share = (total + p.splits - 1) / p.splits;
        const int rank = (int)cluster.block_rank();
        const int lo = rank * share, hi = min(total, lo + share);
        for (int idx = lo + threadIdx.x; idx < hi; idx += SK_THREADS) {
            float sum = 0.0f;
            for (int q = 0; q < p.splits; ++q) sum += cluster.map_shared_rank(part, q)[idx];
            const int m = idx / SKINNY_ROWS, r = idx % SKINNY_ROWS;
            const int n = row0 + r;
            if (n < p.N) p.Y[(int64_t)m * p.N + n] = (uint16_t)float_to_bf16_bits(sum + bias_f32(p.bias, n));
        }
        cluster.sync();  // no block leaves while its partials may still be read
    }
    if (!ok)  // never leave with copies still landing in shared memory
        for (int c = 0; c < nchunks; ++c) mbar_drain_bounded(bar0 + 8 * c, 0, SK_WAIT_LIMIT_NS);
}

// ------------------------------------------------------------------ host side

static constexpr int SK_TARGET_BLOCKS = 148 * 4;  // ~4-5 resident blocks (~45 KB of shared memory each) per SM
static constexpr int SK_MAX_SPLIT = 16;           // cluster size (above 8 needs the non-portable opt-in)
static constexpr int SK_MAX_KS = SK_CHUNK * SK_MAX_CHUNKS;
static constexpr int SK_XCAP = 16 * 1024;         // staged X budget
static constexpr int SK_SMEM_MAX = 200 * 1024;

bool plan_skinny(int64_t M, int64_t N, int64_t K, int g, SkinnyPlan* plan) {
    if (M < 1 || M > SKINNY_MAX_M) return false;
    const int64_t tiles = (N + SKINNY_ROWS - 1) / SKINNY_ROWS;
    if (tiles > 0x7FFFFFFF) return false;
    const int64_t kq = (K + SK_CHUNK - 1) / SK_CHUNK;
    int64_t splits = std::min<int64_t>(SK_MAX_SPLIT, std::max<int64_t>(1, (K + 1023) / 1024));
    // few row tiles: more, shorter slices (down to 512 k) so the launch fills the GPU
    while (splits < SK_MAX_SPLIT && tiles * splits < SK_TARGET_BLOCKS && (kq + splits) / (splits + 1) >= 2) ++splits;
    int64_t ks = (kq + splits - 1) / splits * SK_CHUNK;
    if (ks > SK_MAX_KS) return false;  // K too long for 16 slices: the tensor-core path takes it
    splits = (K + ks - 1) / ks;
    int64_t kc = ks;  // largest sub-chunk (whole 256-k units, dividing ks) whose staged X fits
    while (kc > SK_CHUNK && (M + 1) * (2 * kc + 16) > SK_XCAP) {
        int64_t q = kc / SK_CHUNK - 1;
        while (q > 1 && (ks / SK_CHUNK) % q != 0) --q;
        kc = q * SK_CHUNK;
    }
    const SkLayout L = sk_layout((int)M, (int)ks, (int)kc, g, (int)splits);
    if (L.total + 1024 > SK_SMEM_MAX) return false;
    const int64_t ng = K / g;
    plan->tiles = (int)tiles;
    plan->splits = (int)splits;
    plan->ks = (int)ks;
    plan->kc = (int)kc;
    plan->smem = (size_t)L.total + 1024;  // + slack to align the swizzled chunks to 1024 bytes
    // qparams by TMA: row pitch and every slice start 16-byte aligned
    plan->qtma = (ng % 8 == 0) && ((ks / g) % 8 == 0);
    return true;
}

template <int MT, int G>
static cudaError_t launch_one(const SkinnyPlan& plan, const CUtensorMap& tw, const CUtensorMap& ts,
                              const CUtensorMap& to, const SkinnyArgs& a, cudaStream_t stream) {
    auto kern = skinny_kernel<MT, G>;
    cudaError_t e = ensure_kernel_attrs(reinterpret_cast<const void*>(kern), SK_SMEM_MAX, true);
    if (e != cudaSuccess) return e;
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
    return cudaLaunchKernelEx(&cfg, kern, tw, ts, to, a);
}

template <int G>
static cudaError_t launch_g(const SkinnyPlan& plan, const CUtensorMap& tw, const CUtensorMap& ts,
                            const CUtensorMap& to, const SkinnyArgs& a, cudaStream_t stream) {
    switch ((a.M + 7) / 8) {
        case 1: return launch_one<1, G>(plan, tw, ts, to, a, stream);
        case 2: return launch_one<2, G>(plan, tw, ts, to, a, stream);
        case 3: return launch_one<3, G>(plan, tw, ts, to, a, stream);
        default: return launch_one<4, G>(plan, tw, ts, to, a, stream);
    }
}

cudaError_t launch_skinny(const SkinnyPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                          const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                          cudaStream_t stream, const char** detail, const uint16_t* bias) {
    // codes: [N][K/2] bytes, one box = 64 rows x 128 bytes (256 k), 128-byte swizzle
    CUtensorMap tw, ts, to;
    cudaError_t e = encode_tensor_map_2d(&tw, CU_TENSOR_MAP_DATA_TYPE_UINT8, Wq, (uint64_t)(K / 2), (uint64_t)N,
                                         (uint64_t)(K / 2), 128, SKINNY_ROWS, CU_TENSOR_MAP_SWIZZLE_128B, detail);
    if (e != cudaSuccess) return e;
    ts = tw;
    to = tw;  // placeholders when the qparams go by plain loads
    if (plan.qtma) {
        const uint64_t ng = (uint64_t)(K / g);
        e = encode_tensor_map_2d(&ts, CU_TENSOR_MAP_DATA_TYPE_UINT16, scales, ng, (uint64_t)N, ng * 2,
                                 (uint32_t)(plan.ks / g), SKINNY_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e == cudaSuccess)
            e = encode_tensor_map_2d(&to, CU_TENSOR_MAP_DATA_TYPE_UINT16, offsets, ng, (uint64_t)N, ng * 2,
                                     (uint32_t)(plan.ks / g), SKINNY_ROWS, CU_TENSOR_MAP_SWIZZLE_NONE, detail);
        if (e != cudaSuccess) return e;
    }
    SkinnyArgs a;
    a.X = X;
    a.scales = scales;
    a.offsets = offsets;
    a.Y = Y;
    a.bias = bias;
    a.M = (int)M;
    a.N = (int)N;
    a.K = (int)K;
    a.ks = plan.ks;
    a.kc = plan.kc;
    a.splits = plan.splits;
    a.qtma = plan.qtma ? 1 : 0;
    switch (g) {
        case 32: return launch_g<32>(plan, tw, ts, to, a, stream);
        case 64: return launch_g<64>(plan, tw, ts, to, a, stream);
        default: return launch_g<128>(plan, tw, ts, to, a, stream);
    }
}

cudaError_t read_and_clear_skinny_fault(unsigned int* fault) {
    cudaError_t e = cudaMemcpyFromSymbol(fault, g_skinny_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !*fault) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_skinny_fault, &zero, sizeof(unsigned int));
}

}  // namespace w4
