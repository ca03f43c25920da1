// w4_repack.cu -- canonical codes / scales / offsets -> the decode layout.
//
// The decode layout (byte-exact description in include/w4.h) stores each
// 16-row x 256-k unit of the weights contiguously, in the order the lanes of
// the stream-K decode kernel read it: four 512-byte blocks of code fragments
// (16 bytes per lane, the lane's row and 32-k slice), then the unit's scales
// and offsets, 16 bytes per lane group.  One unit is then five coalesced
// 512-byte warp loads instead of 16 separate 128-byte rows plus 16-byte qparam
// pieces.  The
// pages name such load-time rearrangements without defining one (torchao
// README "Quick start": tile_packed_to_4d; TorchAO 0.14.0 release notes:
// Int4PreshuffledTensor, Int4TilePackedTo4dTensor); this one is ours.
//
// The conversion is a pure gather: one thread writes one 16-byte piece of the
// output (a code fragment, its 32-bit words' nibbles reordered so that nibbles
// i and i + 4 hold two consecutive k; or eight qparams), zeros where the unit
// runs past N, K or the last group.
#include "w4_device.cuh"
#include "w4_internal.h"

namespace w4 {

constexpr int RP_THREADS = 256;

// Eight codes of one canonical word (nibble i = k0 + i) -> the decode layout's
// order k0, k0+2, k0+4, k0+6, k0+1, k0+3, k0+5, k0+7.
__device__ __forceinline__ uint32_t unzip_nibbles(uint32_t w) {
    uint32_t r = 0;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        r |= ((w >> (8 * i)) & 0xFu) << (4 * i);             // even k: low nibble of byte i
        r |= ((w >> (8 * i + 4)) & 0xFu) << (16 + 4 * i);    // odd k: high nibble of byte i
    }
    return r;
}

int64_t repacked_unit_bytes(int g) { return 2048 + 16 * 32 * 32 / g; }

int64_t repacked_bytes(int64_t N, int64_t K, int g) {
    const int64_t tiles = (N + 15) / 16, nkc = (K + 255) / 256;
    return tiles * nkc * repacked_unit_bytes(g);
}

template <int G>
__global__ void __launch_bounds__(RP_THREADS)
repack_kernel(const uint8_t* __restrict__ Wq, const uint16_t* __restrict__ scales,
              const uint16_t* __restrict__ offsets, int64_t N, int64_t K, uint8_t* __restrict__ packed,
              int64_t pieces) {
    constexpr int QPIECES = 1024 / G;          // 16-byte qparam pieces per unit
    constexpr int PIECES = 128 + QPIECES;      // 16-byte pieces per unit
    constexpr int LPP = G / 32;                // lanes sharing one qparam piece
    const int64_t nkc = (K + 255) / 256, ng = K / G, kb = K / 2;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < pieces;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t u = i / PIECES;
        const int piece = (int)(i - u * PIECES);
        const int64_t tile = u / nkc, kc = u - tile * nkc;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (piece < 128) {  // code fragment j of lane l
            const int j = piece >> 5, l = piece & 31;
            const int64_t row = tile * 16 + (l >> 2) + 8 * (j & 1);
            const int64_t k0 = kc * 256 + 128 * (j >> 1) + 32 * (l & 3);
            if (row < N && k0 < K) {
                v = *reinterpret_cast<const uint4*>(Wq + row * kb + k0 / 2);
                v = make_uint4(unzip_nibbles(v.x), unzip_nibbles(v.y), unzip_nibbles(v.z), unzip_nibbles(v.w));
            }
        } else {  // qparams of the lanes l0 .. l0 + LPP - 1
            const int l0 = (piece - 128) * LPP;
            const int64_t ra = tile * 16 + (l0 >> 2), rb = ra + 8;
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int64_t grp = (kc * 256 + 128 * h + 32 * (l0 & 3)) / G;
                const bool in_k = grp < ng;
                const uint32_t sa = (in_k && ra < N) ? scales[ra * ng + grp] : 0u;
                const uint32_t oa = (in_k && ra < N) ? offsets[ra * ng + grp] : 0u;
                const uint32_t sb = (in_k && rb < N) ? scales[rb * ng + grp] : 0u;
                const uint32_t ob = (in_k && rb < N) ? offsets[rb * ng + grp] : 0u;
                w[2 * h] = sa | (oa << 16);
                w[2 * h + 1] = sb | (ob << 16);
            }
            v = make_uint4(w[0], w[1], w[2], w[3]);
        }
        *reinterpret_cast<uint4*>(packed + i * 16) = v;
    }
}

cudaError_t launch_repack(const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N, int64_t K,
                          int g, uint8_t* packed, cudaStream_t stream) {
    const int64_t pieces = repacked_bytes(N, K, g) / 16;
    int sms = 0, dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    const int64_t want = (pieces + RP_THREADS - 1) / RP_THREADS;
    const unsigned blocks = (unsigned)(want < (int64_t)sms * 8 ? want : (int64_t)sms * 8);
    switch (g) {
        case 32: repack_kernel<32><<<blocks, RP_THREADS, 0, stream>>>(Wq, scales, offsets, N, K, packed, pieces); break;
        case 64: repack_kernel<64><<<blocks, RP_THREADS, 0, stream>>>(Wq, scales, offsets, N, K, packed, pieces); break;
        default: repack_kernel<128><<<blocks, RP_THREADS, 0, stream>>>(Wq, scales, offsets, N, K, packed, pieces); break;
    }
    return cudaGetLastError();
}

}  // namespace w4
