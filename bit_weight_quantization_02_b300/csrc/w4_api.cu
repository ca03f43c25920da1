// w4_api.cu -- the C ABI of libw4 (include/w4.h): argument checks on the
// host, kernel choice, launch, error reporting.  No allocation, no
// synchronization (except w4_device_fault), no state kept between calls.
#include "w4.h"
#include "w4_internal.h"

#include <cstdarg>
#include <cstdio>
#include <cstring>

namespace {

thread_local char g_detail[256] = "";

w4_status fail(w4_status s, const char* fmt, ...) {
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_detail, sizeof g_detail, fmt, ap);
    va_end(ap);
    return s;
}

w4_status cuda_fail(cudaError_t e, const char* what) {
    return fail(W4_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Shape and group checks shared by every call.
w4_status check_shape(int64_t N, int64_t K, int g) {
    if (g != 32 && g != 64 && g != 128) return fail(W4_ERR_UNSUPPORTED, "group_size %d not in {32, 64, 128}", g);
    if (K <= 0) return fail(W4_ERR_INVALID_ARG, "K = %lld must be positive", (long long)K);
    if (N < 0) return fail(W4_ERR_INVALID_ARG, "N = %lld must not be negative", (long long)N);
    if (K % g != 0) return fail(W4_ERR_INVALID_ARG, "K = %lld is not a multiple of group_size %d", (long long)K, g);
    if (K > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL)
        return fail(W4_ERR_INVALID_ARG, "N and K must be below 2^31");
    if (N > 0 && K > (int64_t(1) << 62) / N) return fail(W4_ERR_INVALID_ARG, "N*K overflows");
    return W4_OK;
}

w4_status check_ptr(const void* p, const char* name) {
    if (p == nullptr) return fail(W4_ERR_INVALID_ARG, "%s is NULL", name);
    if (!aligned16(p)) return fail(W4_ERR_MISALIGNED, "%s is not 16-byte aligned", name);
    return W4_OK;
}

#define W4_TRY(expr)                     \
    do {                                 \
        w4_status _s = (expr);           \
        if (_s != W4_OK) return _s;      \
    } while (0)

}  // namespace

extern "C" {

w4_status w4_quantize(const uint16_t* W, int64_t N, int64_t K, int group_size, uint8_t* Wq, uint16_t* scales,
                      uint16_t* offsets, void* stream) {
    W4_TRY(check_shape(N, K, group_size));
    if (N == 0) return W4_OK;
    W4_TRY(check_ptr(W, "W"));
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    cudaError_t e = w4::launch_quantize(W, N, K, group_size, Wq, scales, offsets, (cudaStream_t)stream);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "quantize launch");
}

w4_status w4_dequantize(const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N, int64_t K,
                        int group_size, uint16_t* W_out, void* stream) {
    W4_TRY(check_shape(N, K, group_size));
    if (N == 0) return W4_OK;
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    W4_TRY(check_ptr(W_out, "W_out"));
    cudaError_t e = w4::launch_dequantize(Wq, scales, offsets, N, K, group_size, W_out, (cudaStream_t)stream);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "dequantize launch");
}

w4_status w4_linear_ex(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                       const uint16_t* offsets, int64_t N, int group_size, uint16_t* Y, w4_kernel kernel,
                       void* stream) {
    W4_TRY(check_shape(N, K, group_size));
    if (M < 0) return fail(W4_ERR_INVALID_ARG, "M = %lld must not be negative", (long long)M);
    if (M > 0x7FFFFFFFLL) return fail(W4_ERR_INVALID_ARG, "M must be below 2^31");
    if (kernel != W4_KERNEL_AUTO && kernel != W4_KERNEL_SKINNY && kernel != W4_KERNEL_GEMM)
        return fail(W4_ERR_INVALID_ARG, "unknown kernel choice %d", (int)kernel);
    if (kernel == W4_KERNEL_SKINNY && M > w4::SKINNY_MAX_M)
        return fail(W4_ERR_INVALID_ARG, "the skinny kernel takes M <= %d, got %lld", w4::SKINNY_MAX_M, (long long)M);
    if (M == 0 || N == 0) return W4_OK;
    W4_TRY(check_ptr(X, "X"));
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    W4_TRY(check_ptr(Y, "Y"));

    const bool use_skinny = (kernel == W4_KERNEL_SKINNY) || (kernel == W4_KERNEL_AUTO && M <= w4::SKINNY_MAX_M);
    cudaError_t e;
    if (use_skinny) {
        w4::SkinnyPlan plan;
        if (!w4::plan_skinny(M, N, K, group_size, &plan)) return fail(W4_ERR_INVALID_ARG, "no skinny launch plan");
        const char* detail = "";
        e = w4::launch_skinny(plan, X, M, K, Wq, scales, offsets, N, group_size, Y, (cudaStream_t)stream, &detail);
        if (e != cudaSuccess) return fail(W4_ERR_CUDA, "skinny linear: %s %s", cudaGetErrorString(e), detail);
        return W4_OK;
    }
    const char* detail = "";
    e = w4::launch_gemm(X, M, K, Wq, scales, offsets, N, group_size, Y, (cudaStream_t)stream, &detail);
    if (e != cudaSuccess) return fail(W4_ERR_CUDA, "tensor-core linear: %s %s", cudaGetErrorString(e), detail);
    return W4_OK;
}

w4_status w4_linear(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                    const uint16_t* offsets, int64_t N, int group_size, uint16_t* Y, void* stream) {
    return w4_linear_ex(X, M, K, Wq, scales, offsets, N, group_size, Y, W4_KERNEL_AUTO, stream);
}

size_t w4_packed_bytes(int64_t N, int64_t K) {
    if (N < 0 || K <= 0 || (K & 1) || (N > 0 && K > (int64_t(1) << 62) / N)) return 0;
    return (size_t)(N * (K / 2));
}

size_t w4_qparam_bytes(int64_t N, int64_t K, int group_size) {
    if (check_shape(N, K, group_size) != W4_OK) return 0;
    return (size_t)(N * (K / group_size) * 2);
}

w4_status w4_device_fault(void* stream) {
    cudaError_t e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "synchronizing the stream");
    unsigned int gemm = 0, skinny = 0;
    e = w4::read_and_clear_gemm_fault(&gemm);
    if (e == cudaSuccess) e = w4::read_and_clear_skinny_fault(&skinny);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device fault words");
    if (gemm || skinny)
        return fail(W4_ERR_TIMEOUT, "a block gave up a bounded wait (tensor-core linear 0x%x, skinny linear 0x%x)",
                    gemm, skinny);
    return W4_OK;
}

const char* w4_status_string(w4_status s) {
    switch (s) {
        case W4_OK: return "W4_OK";
        case W4_ERR_INVALID_ARG: return "W4_ERR_INVALID_ARG";
        case W4_ERR_UNSUPPORTED: return "W4_ERR_UNSUPPORTED";
        case W4_ERR_MISALIGNED: return "W4_ERR_MISALIGNED";
        case W4_ERR_CUDA: return "W4_ERR_CUDA";
        case W4_ERR_TIMEOUT: return "W4_ERR_TIMEOUT";
    }
    return "unknown w4_status";
}

const char* w4_last_error_detail(void) { return g_detail; }

int w4_format_version(void) { return W4_FORMAT_VERSION; }

}  // extern "C"

// ------------------------------------------------------------------ internal
#include <mutex>
#include <unordered_map>

#include <cuda.h>

namespace w4 {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

cudaError_t encode_tensor_map_2d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, uint64_t inner,
                                 uint64_t outer, uint64_t row_stride_bytes, uint32_t box_inner, uint32_t box_outer,
                                 CUtensorMapSwizzle swizzle, const char** detail) {
    EncodeTiledFn encode = encode_fn();
    if (!encode) {
        *detail = "cuTensorMapEncodeTiled is not available from the driver";
        return cudaErrorNotSupported;
    }
    const cuuint64_t dims[2] = {inner, outer};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_inner, box_outer};
    const cuuint32_t estr[2] = {1, 1};
    if (encode(map, dtype, 2, const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        *detail = "tensor map rejected by the driver";
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

cudaError_t ensure_kernel_attrs(const void* kernel, int smem_bytes, bool big_clusters) {
    static std::mutex mu;
    static std::unordered_map<const void*, uint64_t> done;  // kernel -> bitmask of devices already set
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
    std::lock_guard<std::mutex> lock(mu);
    if (bit && (done[kernel] & bit)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e == cudaSuccess && big_clusters) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess && bit) done[kernel] |= bit;
    return e;
}

}  // namespace w4
