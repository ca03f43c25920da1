// w4_act.cu -- dynamic int8 quantization of activations, for the linear on
// int8 activation codes and int4 weights.
//
// torchao's Int8DynamicActivationInt4WeightConfig quantizes the activations to
// int8 at run time beside int4 group-wise weights (torchao README "Training /
// QAT", torchao guide); Optimum Quanto quantizes activations symmetrically,
// with one scale per tensor ("Design overview / Modules", "Pitfalls when
// quantizing activations"), and rounds half to even ("Design overview /
// Tensors").  Per tensor, or per row of X (token):
//   a = max |x|,   s = a / 127 (fp32 IEEE division, at least 1e-6),
//   q = clamp(rne(x / s), -127, 127) (fp32 IEEE division, round half to even).
// The largest magnitude codes to +-127 and zero to 0.  Every step is one IEEE
// fp32 operation and the maximum does not depend on the order of the scan, so
// codes and scales are exact: the same bits on any launch shape.
//
// A bf16's magnitude bits (bits & 0x7FFF) order like its magnitude (finite
// values), so the maximum runs on integers.
#include "w4_device.cuh"
#include "w4_internal.h"

#include <algorithm>

namespace w4 {

constexpr int ACT_THREADS = 256;

// the maximum over the block's ACT_THREADS threads (red: ACT_THREADS / 32 words)
__device__ __forceinline__ uint32_t block_max(uint32_t v, uint32_t* red) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) red[warp] = v;
    __syncthreads();
    if (warp == 0) {
        v = lane < ACT_THREADS / 32 ? red[lane] : 0u;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
        if (lane == 0) red[0] = v;
    }
    __syncthreads();
    return red[0];
}

// eight bf16 values -> eight int8 codes (the lowest k in the lowest byte)
__device__ __forceinline__ uint2 act_codes8(uint4 v, float s) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
    uint32_t out[2] = {0u, 0u};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const int q = act_code((w[i >> 1] >> (16 * (i & 1))) & 0xFFFFu, s);
        out[i >> 2] |= ((uint32_t)q & 0xFFu) << (8 * (i & 3));
    }
    return make_uint2(out[0], out[1]);
}

// one block per row of X: its maximum, its scale, its codes
__global__ void __launch_bounds__(ACT_THREADS) act_rows_kernel(const uint16_t* X, int K, int8_t* Xq, float* x_scale) {
    __shared__ uint32_t red[ACT_THREADS / 32];
    griddep_launch_dependents();  // the linear after this may start streaming its weights now
    griddep_wait();               // X may come from the kernel before this one
    const uint16_t* x = X + (int64_t)blockIdx.x * K;
    int8_t* q = Xq + (int64_t)blockIdx.x * K;
    const int nch = K / 8;
    uint32_t mx = 0u;
    for (int c = threadIdx.x; c < nch; c += ACT_THREADS) mx = max(mx, act_mag_max8(ldg_cg_v4(x + 8 * c)));
    const float s = act_scale_of(block_max(mx, red));
    for (int c = threadIdx.x; c < nch; c += ACT_THREADS)
        *reinterpret_cast<uint2*>(q + 8 * c) = act_codes8(ldg_cg_v4(x + 8 * c), s);
    if (threadIdx.x == 0) x_scale[blockIdx.x] = s;
}

// one scale for the whole tensor: each block's maximum (grid-stride over 8-value chunks) ...
__global__ void __launch_bounds__(ACT_THREADS) act_partial_max_kernel(const uint16_t* X, int64_t nch,
                                                                       uint32_t* partials) {
    __shared__ uint32_t red[ACT_THREADS / 32];
    griddep_launch_dependents();
    griddep_wait();
    uint32_t mx = 0u;
    for (int64_t c = (int64_t)blockIdx.x * ACT_THREADS + threadIdx.x; c < nch; c += (int64_t)gridDim.x * ACT_THREADS)
        mx = max(mx, act_mag_max8(ldg_cg_v4(X + 8 * c)));
    mx = block_max(mx, red);
    if (threadIdx.x == 0) partials[blockIdx.x] = mx;
}

// ... then every block takes the maximum of the partials and codes its chunks
__global__ void __launch_bounds__(ACT_THREADS) act_tensor_codes_kernel(const uint16_t* X, int64_t nch,
                                                                        const uint32_t* partials, int nparts,
                                                                        int8_t* Xq, float* x_scale) {
    __shared__ uint32_t red[ACT_THREADS / 32];
    griddep_launch_dependents();
    griddep_wait();
    uint32_t mx = 0u;
    for (int i = threadIdx.x; i < nparts; i += ACT_THREADS) mx = max(mx, partials[i]);
    const float s = act_scale_of(block_max(mx, red));
    for (int64_t c = (int64_t)blockIdx.x * ACT_THREADS + threadIdx.x; c < nch; c += (int64_t)gridDim.x * ACT_THREADS)
        *reinterpret_cast<uint2*>(Xq + 8 * c) = act_codes8(ldg_cg_v4(X + 8 * c), s);
    if (blockIdx.x == 0 && threadIdx.x == 0) x_scale[0] = s;
}

// int8 codes -> the same values in bf16 (exact), eight a thread per step
__global__ void __launch_bounds__(ACT_THREADS) widen_kernel(const int8_t* Xq, int64_t n8, uint16_t* Xb) {
    griddep_launch_dependents();
    griddep_wait();
    for (int64_t i = (int64_t)blockIdx.x * ACT_THREADS + threadIdx.x; i < n8; i += (int64_t)gridDim.x * ACT_THREADS)
        *reinterpret_cast<uint4*>(Xb + 8 * i) = widen_i8x8(*reinterpret_cast<const uint2*>(Xq + 8 * i));
}

// launch with programmatic dependent launch: the kernel waits for the one before it
// (griddepcontrol.wait) before reading its input, and lets the one after it start
template <typename... Args>
static cudaError_t launch_pdl(void (*kern)(Args...), int blocks, cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(ACT_THREADS, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, args...);
}

// blocks of a grid-stride launch: one wave, no more than the chunks need
static cudaError_t wave_blocks(const void* kern, int64_t nch, int cap, int* blocks) {
    int sms = 0, per_sm = 0;
    const cudaError_t e = resident_blocks(kern, ACT_THREADS, 0, &sms, &per_sm);
    if (e != cudaSuccess) return e;
    const int64_t need = (nch + ACT_THREADS - 1) / ACT_THREADS;
    *blocks = (int)std::max<int64_t>(1, std::min<int64_t>({need, (int64_t)sms * per_sm, (int64_t)cap}));
    return cudaSuccess;
}

cudaError_t launch_quantize_activation(const uint16_t* X, int64_t M, int64_t K, bool per_token, int8_t* Xq,
                                       float* x_scale, uint32_t* partials, cudaStream_t stream) {
    if (per_token || M == 1) {
        return launch_pdl(act_rows_kernel, (int)M, stream, X, (int)K, Xq, x_scale);
    }
    const int64_t nch = M * K / 8;
    int blocks = 0;
    cudaError_t e = wave_blocks(reinterpret_cast<const void*>(act_partial_max_kernel), nch, ACT_MAX_PARTIALS, &blocks);
    if (e != cudaSuccess) return e;
    if ((e = launch_pdl(act_partial_max_kernel, blocks, stream, X, nch, partials)) != cudaSuccess) return e;
    const int nparts = blocks;
    if ((e = wave_blocks(reinterpret_cast<const void*>(act_tensor_codes_kernel), nch, 1 << 30, &blocks)) != cudaSuccess)
        return e;
    return launch_pdl(act_tensor_codes_kernel, blocks, stream, X, nch, (const uint32_t*)partials, nparts, Xq, x_scale);
}

cudaError_t launch_widen_i8(const int8_t* Xq, int64_t n, uint16_t* Xb, cudaStream_t stream) {
    const int64_t n8 = n / 8;
    int blocks = 0;
    const cudaError_t e = wave_blocks(reinterpret_cast<const void*>(widen_kernel), n8, 1 << 30, &blocks);
    if (e != cudaSuccess) return e;
    return launch_pdl(widen_kernel, blocks, stream, Xq, n8, Xb);
}

}  // namespace w4
