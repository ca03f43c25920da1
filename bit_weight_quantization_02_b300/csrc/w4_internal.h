// w4_internal.h -- host-side launchers shared between the libw4 translation
// units.  Arguments are already validated by w4_api.cu; launchers only pick a
// launch shape, enqueue on `stream` and return the launch error.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace w4 {

// What a linear kernel does to the fp32 sum of output (m, n) before its one
// rounding to bf16: y = sum * yscale[m * ys_stride] + bias[n].  A null yscale is
// the factor 1 and a null bias adds 0, so the default is the plain product.
// yscale is the activation scale of int8 activation codes (ys_stride 0: one
// for the tensor, 1: one per token); kernels read it after their dependency
// wait, so the kernel before them may write it.
struct Epilogue {
    const uint16_t* bias = nullptr;  // [N] bf16
    const float* yscale = nullptr;
    int ys_stride = 0;
};

// bits: code width, 2, 4 or 8
cudaError_t launch_quantize(const uint16_t* W, int64_t N, int64_t K, int g, int bits, uint8_t* Wq, uint16_t* scales,
                            uint16_t* offsets, cudaStream_t stream);
cudaError_t launch_dequantize(const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N,
                              int64_t K, int g, int bits, uint16_t* W_out, cudaStream_t stream);

// Skinny (M <= 32) decode kernel.
struct SkinnyPlan {
    int tiles;    // row tiles of SKINNY_ROWS rows (grid.x)
    int splits;   // K slices (grid.y), one thread-block cluster per row tile
    int ks;       // k per slice
    int kc;       // k per staged activation sub-chunk
    size_t smem;  // dynamic shared memory bytes
    bool qtma;    // qparam rows 16-byte aligned: copied by TMA with the codes
};
constexpr int SKINNY_ROWS = 64;
constexpr int SKINNY_MAX_M = 32;
bool plan_skinny(int64_t M, int64_t N, int64_t K, int g, SkinnyPlan* plan);
cudaError_t launch_skinny(const SkinnyPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                          const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                          cudaStream_t stream, const char** detail, const uint16_t* bias = nullptr);

// Persistent stream-K decode kernel (M <= 4; launch_stream hands 5 <= M <= 32
// to launch_batch with the same plan): needs a zero-initialized,
// self-cleaning workspace of split_ws_bytes(M, units) bytes (w4_device.cuh).
struct StreamPlan {
    int nkc;          // 256-k units per 16-row tile
    int64_t tiles;    // 16-row tiles
    int64_t units;    // tiles * nkc
    size_t smem;      // dynamic shared memory bytes per block
    size_t ws_bytes;  // workspace bytes
};
constexpr int STREAM_MAX_M = 32;
constexpr int DECODE_MAX_M = 32;  // decode-layout kernel
// Where the int8 linear puts its bf16 copy of the codes in a caller's
// workspace: past the largest slot region any linear keeps at zero (4096 warps
// x 16 rows x 32 tokens x 8 bytes), so calls of any shape can share one workspace.
constexpr size_t I8_SCRATCH_OFFSET = size_t(16) << 20;
bool plan_stream(int64_t M, int64_t N, int64_t K, int g, StreamPlan* plan);
// bias: [N] bf16 added in fp32 before the one rounding of Y, or null; ep: the same
// and an output scale (the stream, batch and GEMM launchers).
cudaError_t launch_stream(const StreamPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                          const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                          void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep = Epilogue());
// The same kernel on int8 activation codes (M <= 4; Xq [M][K] bytes), widened to
// bf16 as they are loaded; ep carries their scale.
cudaError_t launch_stream_i8(const StreamPlan& plan, const int8_t* Xq, int64_t M, int64_t K, const uint8_t* Wq,
                             const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                             void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep);
// The same kernel on bf16 X that it quantizes to int8 codes itself (M <= 4), with
// w4_quantize_activation_i8's scale (ep.ys_stride 1: one per token, else one for
// the tensor); ep.yscale is ignored (each block uses the scale it computes).
cudaError_t launch_stream_qx(const StreamPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                             const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                             void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep);
cudaError_t read_and_clear_stream_fault(unsigned int* fault);
// Batched decode (5 <= M <= 32): 64-row units, the block's X slice staged once
// by TMA; same plan and workspace as the stream kernel (launch_stream calls it).
cudaError_t launch_batch(const StreamPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                         const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, int bits, uint16_t* Y,
                         void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep = Epilogue());
cudaError_t read_and_clear_batch_fault(unsigned int* fault);

// Decode layout (see w4.h): bytes of one 16-row x 256-k unit, of the whole
// layout, and the repack launch.
int64_t repacked_unit_bytes(int g);
int64_t repacked_bytes(int64_t N, int64_t K, int g);
cudaError_t launch_repack(const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N, int64_t K,
                          int g, uint8_t* packed, cudaStream_t stream);

// Persistent stream-K decode kernel on the decode layout (M <= 32), same
// workspace as the stream kernel.
struct DecodePlan {
    int nkc;          // 256-k units per 16-row tile
    int64_t units;    // tiles * nkc
    size_t ws_bytes;  // workspace bytes
};
bool plan_decode(int64_t M, int64_t N, int64_t K, int g, DecodePlan* plan);
cudaError_t launch_decode(const DecodePlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* packed,
                          int64_t N, int g, uint16_t* Y, void* workspace, cudaStream_t stream);

// One-token decode on pairs of SMs (thread-block clusters of two), no
// workspace: M == 1, K <= 16384, K / g a multiple of 8.
struct PairPlan {
    int nks;      // 512-k stages per row
    size_t smem;  // dynamic shared memory bytes per block
};
bool plan_pair(int64_t M, int64_t N, int64_t K, int g, PairPlan* plan);
cudaError_t launch_pair(const PairPlan& plan, const uint16_t* X, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                        const uint16_t* offsets, int64_t N, int g, uint16_t* Y, cudaStream_t stream,
                        const char** detail, const uint16_t* bias = nullptr);
cudaError_t read_and_clear_pair_fault(unsigned int* fault);
cudaError_t read_and_clear_selftest_fault(unsigned int* fault);  // w4_selftest.cu

// int8 activations (w4_act.cu): dynamic symmetric quantization, per token
// (per_token) or per tensor, and the widening of codes to bf16 for the kernels
// that stage X by TMA.  `partials` holds ACT_MAX_PARTIALS 32-bit words, used
// per tensor when M > 1.
constexpr int ACT_MAX_PARTIALS = 1024;
cudaError_t launch_quantize_activation(const uint16_t* X, int64_t M, int64_t K, bool per_token, int8_t* Xq,
                                       float* x_scale, uint32_t* partials, cudaStream_t stream);
cudaError_t launch_widen_i8(const int8_t* Xq, int64_t n, uint16_t* Xb, cudaStream_t stream);

// SM count of the current device and resident blocks per SM for a kernel
// launch shape (cached per device, kernel and shared-memory size).
cudaError_t resident_blocks(const void* kernel, int threads, size_t smem, int* sms, int* per_sm);

// Batched decode on the tcgen05 tensor cores (1 <= M <= 32, 4-bit codes): a
// persistent grid of one block per SM over 128-row x 256-k units (stream-K),
// split tiles finished by their owner block from a zero-initialized,
// self-cleaning workspace of ws_bytes.
constexpr int TCDEC_MAX_M = 32;
struct TcDecPlan {
    int nkc;          // 256-k units per 128-row tile
    long long units;  // tiles * nkc
    int ctas;         // blocks (at most one per SM and per unit)
    int mt;           // token tile: 16 or 32
    size_t ws_bytes;  // workspace bytes
};
bool plan_tcdec(int64_t M, int64_t N, int64_t K, int g, TcDecPlan* plan);
cudaError_t launch_tcdec(const TcDecPlan& plan, const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                         const uint16_t* scales, const uint16_t* offsets, int64_t N, int g, uint16_t* Y,
                         void* workspace, cudaStream_t stream, const char** detail, const Epilogue& ep = Epilogue());
cudaError_t read_and_clear_tcdec_fault(unsigned int* fault);

// tcgen05 tensor-core GEMM (any M).  With a workspace that holds them, a
// part-empty last round of tiles is split by k blocks over the blocks
// (stream-K): flags from the workspace's start (zero between calls, under
// part_off bytes), fp32 partial tiles from byte part_off on (16-byte aligned).
cudaError_t launch_gemm(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                        const uint16_t* offsets, int64_t N, int g, int bits, uint16_t* Y, cudaStream_t stream,
                        const char** detail, const Epilogue& ep = Epilogue(), void* workspace = nullptr,
                        size_t workspace_bytes = 0, size_t part_off = 0);
// Workspace bytes a GEMM call with its partial tiles at part_off uses on the
// current device (0: it splits nothing).
cudaError_t gemm_split_bytes(int64_t M, int64_t N, int64_t K, size_t part_off, size_t* bytes);
// Read and clear the kernels' device fault words (bounded-wait timeouts); the
// caller has synchronized the stream.
cudaError_t read_and_clear_gemm_fault(unsigned int* fault);
cudaError_t read_and_clear_skinny_fault(unsigned int* fault);
cudaError_t read_and_clear_decode_fault(unsigned int* fault);

// Raises a kernel's dynamic shared-memory limit to `smem_bytes` (and allows
// cluster sizes above 8 if asked), once per device and kernel: later calls,
// e.g. during CUDA-graph capture, make no CUDA call.
cudaError_t ensure_kernel_attrs(const void* kernel, int smem_bytes, bool big_clusters);

// The same for a 3-D [outer][mid][inner] tensor: dims and box innermost first,
// strides of the two outer dimensions in bytes.
cudaError_t encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, const uint64_t dims[3],
                                 const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle,
                                 const char** detail);

// Sets the text w4_last_error_detail() returns on this host thread.
void set_error_detail(const char* msg);

// Encodes a 2-D tiled TMA descriptor for a row-major [outer][inner] tensor
// (driver entry point fetched once; a host-only call, fine during capture).
cudaError_t encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                                 uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                                 CUtensorMapSwizzle swizzle, const char** detail);

}  // namespace w4
