// w4_api.cu -- the C ABI of libw4 (include/w4.h): argument checks on the
// host, kernel choice, launch, error reporting.  No allocation, no
// synchronization (except w4_device_fault), no state kept between calls.
#include "w4.h"
#include "w4_internal.h"

#include <algorithm>
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
    cudaError_t e = w4::launch_quantize(W, N, K, group_size, 4, Wq, scales, offsets, (cudaStream_t)stream);
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
    cudaError_t e = w4::launch_dequantize(Wq, scales, offsets, N, K, group_size, 4, W_out, (cudaStream_t)stream);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "dequantize launch");
}

size_t w4_linear_workspace_bytes(int64_t M, int64_t N, int64_t K, int group_size) {
    if (check_shape(N, K, group_size) != W4_OK || M < 1 || N == 0) return 0;
    w4::StreamPlan plan;
    w4::TcDecPlan tp;  // the tensor-core decode kernel's slots, when a device is there to size them
    const size_t tc = M <= w4::TCDEC_MAX_M && w4::plan_tcdec(M, N, K, group_size, &tp) ? tp.ws_bytes : 0;
    if (M <= w4::STREAM_MAX_M && w4::plan_stream(M, N, K, group_size, &plan)) return std::max(plan.ws_bytes, tc);
    if (tc) return tc;
    w4::DecodePlan dp;  // decode layout (w4_linear_repacked)
    if (w4::plan_decode(M, N, K, group_size, &dp)) return dp.ws_bytes;
    size_t gb = 0;  // the tensor-core GEMM's split tail (flags at 0, partial tiles past the slot region)
    if (w4::gemm_split_bytes(M, N, K, w4::I8_SCRATCH_OFFSET, &gb) != cudaSuccess) {
        cudaGetLastError();  // no device to size it for: the GEMM then splits nothing
        return 0;
    }
    return gb;
}

}  // extern "C"

namespace {

// The linear with an optional bias (null: none): argument checks, kernel choice, launch.
w4_status linear_impl(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                      const uint16_t* offsets, int64_t N, int group_size, const uint16_t* bias, uint16_t* Y,
                      void* workspace, size_t workspace_bytes, w4_kernel kernel, void* stream) {
    W4_TRY(check_shape(N, K, group_size));
    if (M < 0) return fail(W4_ERR_INVALID_ARG, "M = %lld must not be negative", (long long)M);
    if (M > 0x7FFFFFFFLL) return fail(W4_ERR_INVALID_ARG, "M must be below 2^31");
    if (kernel < W4_KERNEL_AUTO || kernel > W4_KERNEL_TC_DECODE)
        return fail(W4_ERR_INVALID_ARG, "unknown kernel choice %d", (int)kernel);
    if ((kernel == W4_KERNEL_SKINNY || kernel == W4_KERNEL_SKINNY_CLUSTER) && M > w4::SKINNY_MAX_M)
        return fail(W4_ERR_INVALID_ARG, "the skinny kernels take M <= %d, got %lld", w4::SKINNY_MAX_M, (long long)M);
    if (kernel == W4_KERNEL_STREAM && M > w4::STREAM_MAX_M)
        return fail(W4_ERR_INVALID_ARG, "the stream kernel takes M <= %d, got %lld", w4::STREAM_MAX_M, (long long)M);
    if (M == 0 || N == 0) return W4_OK;
    W4_TRY(check_ptr(X, "X"));
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    W4_TRY(check_ptr(Y, "Y"));
    if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1u))
        return fail(W4_ERR_MISALIGNED, "bias is not 2-byte aligned");
    if (workspace == nullptr) workspace_bytes = 0;
    if (workspace_bytes > 0 && !aligned16(workspace)) return fail(W4_ERR_MISALIGNED, "workspace is not 16-byte aligned");

    const char* detail = "";
    cudaError_t e;
    w4::Epilogue ep;
    ep.bias = bias;
    if (kernel == W4_KERNEL_TC_DECODE) {  // the tensor-core decode kernel, on request
        w4::TcDecPlan tp;
        if (!w4::plan_tcdec(M, N, K, group_size, &tp) || workspace_bytes < tp.ws_bytes)
            return fail(W4_ERR_INVALID_ARG, "the tensor-core decode kernel takes M <= %d and %zu workspace bytes",
                        w4::TCDEC_MAX_M, w4_linear_workspace_bytes(M, N, K, group_size));
        e = w4::launch_tcdec(tp, X, M, K, Wq, scales, offsets, N, group_size, Y, workspace, (cudaStream_t)stream,
                             &detail, ep);
        if (e != cudaSuccess) return fail(W4_ERR_CUDA, "tensor-core decode linear: %s %s", cudaGetErrorString(e), detail);
        return W4_OK;
    }
    // one token without a workspace (or when asked for): the SM-pair kernel, which needs none
    w4::StreamPlan sp0;
    const bool stream_ws = M <= w4::STREAM_MAX_M && w4::plan_stream(M, N, K, group_size, &sp0) &&
                           workspace_bytes >= sp0.ws_bytes;
    if (kernel == W4_KERNEL_PAIR || ((kernel == W4_KERNEL_AUTO || kernel == W4_KERNEL_SKINNY) && !stream_ws)) {
        w4::PairPlan pp;
        const bool can = w4::plan_pair(M, N, K, group_size, &pp);
        if (kernel == W4_KERNEL_PAIR && !can)
            return fail(W4_ERR_INVALID_ARG,
                        "the pair kernel takes M == 1, K <= 16384 and K / group_size a multiple of 8");
        if (can) {
            e = w4::launch_pair(pp, X, K, Wq, scales, offsets, N, group_size, Y, (cudaStream_t)stream, &detail, bias);
            if (e != cudaSuccess) return fail(W4_ERR_CUDA, "pair linear: %s %s", cudaGetErrorString(e), detail);
            return W4_OK;
        }
    }
    // stream kernel: M <= 32 with a large enough workspace
    if (kernel == W4_KERNEL_AUTO || kernel == W4_KERNEL_SKINNY || kernel == W4_KERNEL_STREAM) {
        w4::StreamPlan sp;
        const bool can = M <= w4::STREAM_MAX_M && w4::plan_stream(M, N, K, group_size, &sp) &&
                         workspace_bytes >= sp.ws_bytes;
        if (kernel == W4_KERNEL_STREAM && !can)
            return fail(W4_ERR_INVALID_ARG, "the stream kernel needs an even K/group_size and %zu workspace bytes",
                        w4_linear_workspace_bytes(M, N, K, group_size));
        if (can) {
            e = w4::launch_stream(sp, X, M, K, Wq, scales, offsets, N, group_size, Y, workspace, (cudaStream_t)stream,
                                  &detail, ep);
            if (e != cudaSuccess) return fail(W4_ERR_CUDA, "stream linear: %s %s", cudaGetErrorString(e), detail);
            return W4_OK;
        }
    }
    // cluster-split skinny kernel: M <= 32, no workspace
    if (kernel == W4_KERNEL_SKINNY_CLUSTER || ((kernel == W4_KERNEL_AUTO || kernel == W4_KERNEL_SKINNY) &&
                                               M <= w4::SKINNY_MAX_M)) {
        w4::SkinnyPlan plan;
        if (w4::plan_skinny(M, N, K, group_size, &plan)) {
            e = w4::launch_skinny(plan, X, M, K, Wq, scales, offsets, N, group_size, Y, (cudaStream_t)stream, &detail,
                                  bias);
            if (e != cudaSuccess) return fail(W4_ERR_CUDA, "skinny linear: %s %s", cudaGetErrorString(e), detail);
            return W4_OK;
        }
        if (kernel != W4_KERNEL_AUTO) return fail(W4_ERR_INVALID_ARG, "no skinny launch plan for this shape");
    }
    e = w4::launch_gemm(X, M, K, Wq, scales, offsets, N, group_size, 4, Y, (cudaStream_t)stream, &detail, ep, workspace,
                        workspace_bytes, w4::I8_SCRATCH_OFFSET);
    if (e != cudaSuccess) return fail(W4_ERR_CUDA, "tensor-core linear: %s %s", cudaGetErrorString(e), detail);
    return W4_OK;
}

}  // namespace

extern "C" {

w4_status w4_linear_ex(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                       const uint16_t* offsets, int64_t N, int group_size, uint16_t* Y, void* workspace,
                       size_t workspace_bytes, w4_kernel kernel, void* stream) {
    return linear_impl(X, M, K, Wq, scales, offsets, N, group_size, nullptr, Y, workspace, workspace_bytes, kernel,
                       stream);
}

w4_status w4_linear_bias_ex(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                            const uint16_t* offsets, int64_t N, int group_size, const uint16_t* bias, uint16_t* Y,
                            void* workspace, size_t workspace_bytes, w4_kernel kernel, void* stream) {
    return linear_impl(X, M, K, Wq, scales, offsets, N, group_size, bias, Y, workspace, workspace_bytes, kernel,
                       stream);
}

w4_status w4_linear_bias(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                         const uint16_t* offsets, int64_t N, int group_size, const uint16_t* bias, uint16_t* Y,
                         void* workspace, size_t workspace_bytes, void* stream) {
    return linear_impl(X, M, K, Wq, scales, offsets, N, group_size, bias, Y, workspace, workspace_bytes,
                       W4_KERNEL_AUTO, stream);
}

w4_status w4_linear(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                    const uint16_t* offsets, int64_t N, int group_size, uint16_t* Y, void* workspace,
                    size_t workspace_bytes, void* stream) {
    return w4_linear_ex(X, M, K, Wq, scales, offsets, N, group_size, Y, workspace, workspace_bytes, W4_KERNEL_AUTO,
                        stream);
}

// ---- int8 dynamic activations x int4 weights

size_t w4_quantize_activation_workspace_bytes(int64_t M, int64_t K, int per_token) {
    if (M <= 1 || K <= 0 || per_token) return 0;
    return (size_t)w4::ACT_MAX_PARTIALS * sizeof(uint32_t);
}

w4_status w4_quantize_activation_i8(const uint16_t* X, int64_t M, int64_t K, int per_token, int8_t* Xq,
                                    float* x_scale, void* workspace, size_t workspace_bytes, void* stream) {
    if (K <= 0 || K % 32 != 0) return fail(W4_ERR_INVALID_ARG, "K = %lld must be a positive multiple of 32", (long long)K);
    if (M < 0 || M > 0x7FFFFFFFLL || K > 0x7FFFFFFFLL) return fail(W4_ERR_INVALID_ARG, "M and K must lie in [0, 2^31)");
    if (M > 0 && K > (int64_t(1) << 62) / M) return fail(W4_ERR_INVALID_ARG, "M*K overflows");
    if (per_token != 0 && per_token != 1) return fail(W4_ERR_INVALID_ARG, "per_token must be 0 or 1");
    if (M == 0) return W4_OK;
    W4_TRY(check_ptr(X, "X"));
    W4_TRY(check_ptr(Xq, "Xq"));
    if (x_scale == nullptr) return fail(W4_ERR_INVALID_ARG, "x_scale is NULL");
    if (reinterpret_cast<uintptr_t>(x_scale) & 3u) return fail(W4_ERR_MISALIGNED, "x_scale is not 4-byte aligned");
    const size_t need = w4_quantize_activation_workspace_bytes(M, K, per_token);
    if (need > 0) {
        if (workspace == nullptr || workspace_bytes < need)
            return fail(W4_ERR_INVALID_ARG, "one scale for the tensor over %lld rows needs %zu workspace bytes",
                        (long long)M, need);
        if (!aligned16(workspace)) return fail(W4_ERR_MISALIGNED, "workspace is not 16-byte aligned");
    }
    const cudaError_t e = w4::launch_quantize_activation(X, M, K, per_token != 0, Xq, x_scale,
                                                         static_cast<uint32_t*>(workspace), (cudaStream_t)stream);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "activation quantize launch");
}

}  // extern "C"

namespace {

// How the int8 linear runs: codes read straight by the stream kernel (M <= 4), or
// widened to bf16 in the workspace first (then the batch or tensor-core kernel).
// The linear's own slots (zero between calls) start at 0; the bf16 copy of the
// codes (scratch) at I8_SCRATCH_OFFSET, past any call's slots.
struct I8Plan {
    bool direct;       // stream kernel on the int8 codes
    bool stream_ok;    // the stream / batch kernels take the shape (M <= 32, even K/g)
    w4::StreamPlan sp;
    size_t lin_bytes;  // the linear's own slots
    size_t wide_bytes; // the bf16 copy of the codes
    size_t part_off;   // the GEMM's partial tiles (past the bf16 codes)
    size_t total;      // workspace bytes the call needs
};

I8Plan plan_i8(int64_t M, int64_t N, int64_t K, int g) {
    I8Plan p{};
    p.stream_ok = M <= w4::STREAM_MAX_M && w4::plan_stream(M, N, K, g, &p.sp);
    p.direct = M <= 4 && p.stream_ok;
    p.lin_bytes = p.stream_ok ? p.sp.ws_bytes : 0;
    p.wide_bytes = p.direct ? 0 : (size_t)(M * K * 2);
    p.total = p.direct ? p.lin_bytes : w4::I8_SCRATCH_OFFSET + p.wide_bytes;
    p.part_off = (w4::I8_SCRATCH_OFFSET + p.wide_bytes + 255) / 256 * 256;
    size_t gb = 0;  // the tensor-core GEMM's split tail, when a device is there to size it
    if (!p.stream_ok && w4::gemm_split_bytes(M, N, K, p.part_off, &gb) != cudaSuccess) cudaGetLastError();
    p.total = std::max(p.total, gb);
    return p;
}

size_t round256(size_t b) { return (b + 255) / 256 * 256; }

// The int8 linear's launches, arguments already checked (the workspace holds p.total bytes).
w4_status linear_i8_run(const I8Plan& p, const int8_t* Xq, const float* x_scale, int per_token, int64_t M, int64_t K,
                        const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N, int group_size,
                        const uint16_t* bias, uint16_t* Y, void* workspace, void* stream) {
    w4::Epilogue ep;
    ep.bias = bias;
    ep.yscale = x_scale;
    ep.ys_stride = per_token ? 1 : 0;
    const char* detail = "";
    cudaError_t e;
    if (p.direct) {
        e = w4::launch_stream_i8(p.sp, Xq, M, K, Wq, scales, offsets, N, group_size, Y, workspace,
                                 (cudaStream_t)stream, &detail, ep);
        if (e != cudaSuccess) return fail(W4_ERR_CUDA, "int8 stream linear: %s %s", cudaGetErrorString(e), detail);
        return W4_OK;
    }
    uint16_t* Xb = reinterpret_cast<uint16_t*>(static_cast<unsigned char*>(workspace) + w4::I8_SCRATCH_OFFSET);
    e = w4::launch_widen_i8(Xq, M * K, Xb, (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "int8 widen launch");
    if (p.stream_ok)
        e = w4::launch_stream(p.sp, Xb, M, K, Wq, scales, offsets, N, group_size, Y, workspace, (cudaStream_t)stream,
                              &detail, ep);
    else
        e = w4::launch_gemm(Xb, M, K, Wq, scales, offsets, N, group_size, 4, Y, (cudaStream_t)stream, &detail, ep,
                            workspace, p.total, p.part_off);
    if (e != cudaSuccess) return fail(W4_ERR_CUDA, "int8 linear: %s %s", cudaGetErrorString(e), detail);
    return W4_OK;
}

// The dynamic int8 linear: up to 4 tokens one fused kernel (the stream kernel codes X
// itself); otherwise the activation quantization into the workspace (codes, scales and
// partial maxima after the int8 linear's own scratch), then the int8 linear.
struct DynI8Plan {
    bool fused;
    w4::StreamPlan sp;
    I8Plan lin;
    size_t xq_off, xs_off, part_off;  // composed path: offsets in the workspace
    size_t total;
};

DynI8Plan plan_dyn_i8(int64_t M, int64_t N, int64_t K, int g) {
    DynI8Plan d{};
    d.fused = M <= 4 && w4::plan_stream(M, N, K, g, &d.sp);
    if (d.fused) {
        d.total = d.sp.ws_bytes;
        return d;
    }
    d.lin = plan_i8(M, N, K, g);
    const size_t base = std::max(d.lin.total, (size_t)w4::I8_SCRATCH_OFFSET);
    d.xq_off = round256(base);
    d.xs_off = d.xq_off + round256((size_t)(M * K));
    d.part_off = d.xs_off + round256((size_t)M * 4);
    d.total = d.part_off + (size_t)w4::ACT_MAX_PARTIALS * 4;
    return d;
}

}  // namespace

extern "C" {

size_t w4_linear_i8_workspace_bytes(int64_t M, int64_t N, int64_t K, int group_size) {
    if (check_shape(N, K, group_size) != W4_OK || M < 1 || N == 0 || M > 0x7FFFFFFFLL) return 0;
    return plan_i8(M, N, K, group_size).total;
}

w4_status w4_linear_i8(const int8_t* Xq, const float* x_scale, int per_token, int64_t M, int64_t K,
                       const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N,
                       int group_size, const uint16_t* bias, uint16_t* Y, void* workspace, size_t workspace_bytes,
                       void* stream) {
    W4_TRY(check_shape(N, K, group_size));
    if (M < 0 || M > 0x7FFFFFFFLL) return fail(W4_ERR_INVALID_ARG, "M = %lld must lie in [0, 2^31)", (long long)M);
    if (per_token != 0 && per_token != 1) return fail(W4_ERR_INVALID_ARG, "per_token must be 0 or 1");
    if (M == 0 || N == 0) return W4_OK;
    W4_TRY(check_ptr(Xq, "Xq"));
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    W4_TRY(check_ptr(Y, "Y"));
    if (x_scale == nullptr) return fail(W4_ERR_INVALID_ARG, "x_scale is NULL");
    if (reinterpret_cast<uintptr_t>(x_scale) & 3u) return fail(W4_ERR_MISALIGNED, "x_scale is not 4-byte aligned");
    if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1u))
        return fail(W4_ERR_MISALIGNED, "bias is not 2-byte aligned");
    const I8Plan p = plan_i8(M, N, K, group_size);
    if (p.total > 0) {
        if (workspace == nullptr || workspace_bytes < p.total)
            return fail(W4_ERR_INVALID_ARG, "the int8 linear needs %zu workspace bytes (w4_linear_i8_workspace_bytes)",
                        p.total);
        if (!aligned16(workspace)) return fail(W4_ERR_MISALIGNED, "workspace is not 16-byte aligned");
    }
    return linear_i8_run(p, Xq, x_scale, per_token, M, K, Wq, scales, offsets, N, group_size, bias, Y, workspace,
                         stream);
}

size_t w4_linear_i8_dynamic_workspace_bytes(int64_t M, int64_t N, int64_t K, int group_size) {
    if (check_shape(N, K, group_size) != W4_OK || M < 1 || N == 0 || M > 0x7FFFFFFFLL) return 0;
    return plan_dyn_i8(M, N, K, group_size).total;
}

w4_status w4_linear_i8_dynamic(const uint16_t* X, int per_token, int64_t M, int64_t K, const uint8_t* Wq,
                               const uint16_t* scales, const uint16_t* offsets, int64_t N, int group_size,
                               const uint16_t* bias, uint16_t* Y, void* workspace, size_t workspace_bytes,
                               void* stream) {
    W4_TRY(check_shape(N, K, group_size));
    if (M < 0 || M > 0x7FFFFFFFLL) return fail(W4_ERR_INVALID_ARG, "M = %lld must lie in [0, 2^31)", (long long)M);
    if (M > 0 && K > (int64_t(1) << 62) / M) return fail(W4_ERR_INVALID_ARG, "M*K overflows");
    if (per_token != 0 && per_token != 1) return fail(W4_ERR_INVALID_ARG, "per_token must be 0 or 1");
    if (M == 0 || N == 0) return W4_OK;
    W4_TRY(check_ptr(X, "X"));
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    W4_TRY(check_ptr(Y, "Y"));
    if (bias != nullptr && (reinterpret_cast<uintptr_t>(bias) & 1u))
        return fail(W4_ERR_MISALIGNED, "bias is not 2-byte aligned");
    const DynI8Plan d = plan_dyn_i8(M, N, K, group_size);
    if (workspace == nullptr || workspace_bytes < d.total)
        return fail(W4_ERR_INVALID_ARG,
                    "the dynamic int8 linear needs %zu workspace bytes (w4_linear_i8_dynamic_workspace_bytes)",
                    d.total);
    if (!aligned16(workspace)) return fail(W4_ERR_MISALIGNED, "workspace is not 16-byte aligned");
    if (d.fused) {
        w4::Epilogue ep;
        ep.bias = bias;
        ep.ys_stride = per_token ? 1 : 0;
        const char* detail = "";
        const cudaError_t e = w4::launch_stream_qx(d.sp, X, M, K, Wq, scales, offsets, N, group_size, Y, workspace,
                                                   (cudaStream_t)stream, &detail, ep);
        if (e != cudaSuccess)
            return fail(W4_ERR_CUDA, "dynamic int8 stream linear: %s %s", cudaGetErrorString(e), detail);
        return W4_OK;
    }
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    int8_t* Xq = reinterpret_cast<int8_t*>(ws + d.xq_off);
    float* xs = reinterpret_cast<float*>(ws + d.xs_off);
    const cudaError_t e = w4::launch_quantize_activation(X, M, K, per_token != 0, Xq, xs,
                                                         reinterpret_cast<uint32_t*>(ws + d.part_off),
                                                         (cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "activation quantize launch");
    return linear_i8_run(d.lin, Xq, xs, per_token, M, K, Wq, scales, offsets, N, group_size, bias, Y, workspace,
                         stream);
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
    unsigned int gemm = 0, skinny = 0, strm = 0, dec = 0, bat = 0, pair = 0, self = 0, tcd = 0;
    e = w4::read_and_clear_gemm_fault(&gemm);
    if (e == cudaSuccess) e = w4::read_and_clear_skinny_fault(&skinny);
    if (e == cudaSuccess) e = w4::read_and_clear_stream_fault(&strm);
    if (e == cudaSuccess) e = w4::read_and_clear_decode_fault(&dec);
    if (e == cudaSuccess) e = w4::read_and_clear_batch_fault(&bat);
    if (e == cudaSuccess) e = w4::read_and_clear_pair_fault(&pair);
    if (e == cudaSuccess) e = w4::read_and_clear_selftest_fault(&self);
    if (e == cudaSuccess) e = w4::read_and_clear_tcdec_fault(&tcd);
    if (e != cudaSuccess) return cuda_fail(e, "reading the device fault words");
    if (gemm || skinny || strm || dec || bat || pair || self || tcd)
        return fail(W4_ERR_TIMEOUT,
                    "a block gave up a bounded wait (tensor-core 0x%x, skinny 0x%x, stream 0x%x, decode 0x%x, "
                    "batched 0x%x, pair 0x%x, self-test 0x%x, tensor-core decode 0x%x)",
                    gemm, skinny, strm, dec, bat, pair, self, tcd);
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

size_t w4_repacked_bytes(int64_t N, int64_t K, int group_size) {
    if (check_shape(N, K, group_size) != W4_OK) return 0;
    return (size_t)w4::repacked_bytes(N, K, group_size);
}

w4_status w4_repack(const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N, int64_t K,
                    int group_size, uint8_t* packed, void* stream) {
    W4_TRY(check_shape(N, K, group_size));
    if (N == 0) return W4_OK;
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    W4_TRY(check_ptr(packed, "packed"));
    cudaError_t e = w4::launch_repack(Wq, scales, offsets, N, K, group_size, packed, (cudaStream_t)stream);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "repack launch");
}

w4_status w4_linear_repacked(const uint16_t* X, int64_t M, int64_t K, const uint8_t* packed, int64_t N,
                             int group_size, uint16_t* Y, void* workspace, size_t workspace_bytes, void* stream) {
    W4_TRY(check_shape(N, K, group_size));
    if (M < 0) return fail(W4_ERR_INVALID_ARG, "M = %lld must not be negative", (long long)M);
    if (M > w4::DECODE_MAX_M)
        return fail(W4_ERR_INVALID_ARG, "the decode layout is read for M <= %d, got %lld", w4::DECODE_MAX_M,
                    (long long)M);
    if (M == 0 || N == 0) return W4_OK;
    W4_TRY(check_ptr(X, "X"));
    W4_TRY(check_ptr(packed, "packed"));
    W4_TRY(check_ptr(Y, "Y"));
    if (workspace == nullptr) workspace_bytes = 0;
    if (workspace_bytes > 0 && !aligned16(workspace)) return fail(W4_ERR_MISALIGNED, "workspace is not 16-byte aligned");
    w4::DecodePlan dp;
    if (!w4::plan_decode(M, N, K, group_size, &dp)) return fail(W4_ERR_INVALID_ARG, "no decode plan for this shape");
    if (workspace_bytes < dp.ws_bytes)
        return fail(W4_ERR_INVALID_ARG, "w4_linear_repacked needs %zu workspace bytes", dp.ws_bytes);
    cudaError_t e = w4::launch_decode(dp, X, M, K, packed, N, group_size, Y, workspace, (cudaStream_t)stream);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "repacked linear launch");
}

size_t w4_packed_bytes_bits(int64_t N, int64_t K, int bits) {
    if (bits != 2 && bits != 4 && bits != 8) return 0;
    if (N < 0 || K <= 0 || K % (8 / bits) != 0 || (N > 0 && K > (int64_t(1) << 62) / N)) return 0;
    return (size_t)(N * (K * bits / 8));
}

namespace {
w4_status check_bits(int bits) {
    if (bits != 2 && bits != 4 && bits != 8) return fail(W4_ERR_UNSUPPORTED, "bits %d not in {2, 4, 8}", bits);
    return W4_OK;
}
}  // namespace

w4_status w4_quantize_bits(const uint16_t* W, int64_t N, int64_t K, int group_size, int bits, uint8_t* Wq,
                           uint16_t* scales, uint16_t* offsets, void* stream) {
    W4_TRY(check_bits(bits));
    W4_TRY(check_shape(N, K, group_size));
    if (N == 0) return W4_OK;
    W4_TRY(check_ptr(W, "W"));
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    cudaError_t e = w4::launch_quantize(W, N, K, group_size, bits, Wq, scales, offsets, (cudaStream_t)stream);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "quantize launch");
}

w4_status w4_dequantize_bits(const uint8_t* Wq, const uint16_t* scales, const uint16_t* offsets, int64_t N, int64_t K,
                             int group_size, int bits, uint16_t* W_out, void* stream) {
    W4_TRY(check_bits(bits));
    W4_TRY(check_shape(N, K, group_size));
    if (N == 0) return W4_OK;
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    W4_TRY(check_ptr(W_out, "W_out"));
    cudaError_t e = w4::launch_dequantize(Wq, scales, offsets, N, K, group_size, bits, W_out, (cudaStream_t)stream);
    return e == cudaSuccess ? W4_OK : cuda_fail(e, "dequantize launch");
}

w4_status w4_linear_bits(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq, const uint16_t* scales,
                         const uint16_t* offsets, int64_t N, int group_size, int bits, uint16_t* Y, void* workspace,
                         size_t workspace_bytes, void* stream) {
    W4_TRY(check_bits(bits));
    if (bits == 4)
        return w4_linear(X, M, K, Wq, scales, offsets, N, group_size, Y, workspace, workspace_bytes, stream);
    W4_TRY(check_shape(N, K, group_size));
    if (M < 0) return fail(W4_ERR_INVALID_ARG, "M = %lld must not be negative", (long long)M);
    if (M > 0x7FFFFFFFLL) return fail(W4_ERR_INVALID_ARG, "M must be below 2^31");
    if (bits == 2 && K % 64 != 0)
        return fail(W4_ERR_UNSUPPORTED, "2-bit codes need K %% 64 == 0 (16-byte code rows), got K = %lld",
                    (long long)K);
    if (M == 0 || N == 0) return W4_OK;
    W4_TRY(check_ptr(X, "X"));
    W4_TRY(check_ptr(Wq, "Wq"));
    W4_TRY(check_ptr(scales, "scales"));
    W4_TRY(check_ptr(offsets, "offsets"));
    W4_TRY(check_ptr(Y, "Y"));
    if (workspace == nullptr) workspace_bytes = 0;
    if (workspace_bytes > 0 && !aligned16(workspace)) return fail(W4_ERR_MISALIGNED, "workspace is not 16-byte aligned");
    const char* detail = "";
    cudaError_t e;
    w4::StreamPlan sp;
    if (M <= w4::STREAM_MAX_M && w4::plan_stream(M, N, K, group_size, &sp) && workspace_bytes >= sp.ws_bytes) {
        e = w4::launch_batch(sp, X, M, K, Wq, scales, offsets, N, group_size, bits, Y, workspace, (cudaStream_t)stream,
                             &detail);
        if (e != cudaSuccess) return fail(W4_ERR_CUDA, "batched linear: %s %s", cudaGetErrorString(e), detail);
        return W4_OK;
    }
    e = w4::launch_gemm(X, M, K, Wq, scales, offsets, N, group_size, bits, Y, (cudaStream_t)stream, &detail,
                        w4::Epilogue(), workspace, workspace_bytes, w4::I8_SCRATCH_OFFSET);
    if (e != cudaSuccess) return fail(W4_ERR_CUDA, "tensor-core linear: %s %s", cudaGetErrorString(e), detail);
    return W4_OK;
}

int w4_format_version(void) { return W4_FORMAT_VERSION; }

}  // extern "C"

// ------------------------------------------------------------------ internal
#include <map>
#include <mutex>
#include <tuple>
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

cudaError_t encode_tensor_map_3d(CUtensorMap* map, CUtensorMapDataType dtype, const void* base, const uint64_t dims[3],
                                 const uint64_t strides_bytes[2], const uint32_t box[3], CUtensorMapSwizzle swizzle,
                                 const char** detail) {
    EncodeTiledFn encode = encode_fn();
    if (!encode) {
        *detail = "cuTensorMapEncodeTiled is not available from the driver";
        return cudaErrorNotSupported;
    }
    const cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
    const cuuint64_t st[2] = {strides_bytes[0], strides_bytes[1]};
    const cuuint32_t bx[3] = {box[0], box[1], box[2]};
    const cuuint32_t estr[3] = {1, 1, 1};
    if (encode(map, dtype, 3, const_cast<void*>(base), d, st, bx, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS) {
        *detail = "3-D tensor map rejected by the driver";
        return cudaErrorInvalidValue;
    }
    return cudaSuccess;
}

void set_error_detail(const char* msg) { snprintf(g_detail, sizeof g_detail, "%s", msg ? msg : ""); }

cudaError_t resident_blocks(const void* kernel, int threads, size_t smem, int* sms, int* per_sm) {
    static std::mutex mu;
    static std::map<std::tuple<int, const void*, int, size_t>, std::pair<int, int>> cache;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const auto key = std::make_tuple(dev, kernel, threads, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it == cache.end()) {
        int n = 0, b = 0;
        if ((e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&b, kernel, threads, smem)) != cudaSuccess) return e;
        it = cache.emplace(key, std::make_pair(n, b > 0 ? b : 1)).first;
    }
    *sms = it->second.first;
    *per_sm = it->second.second;
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
    // every kernel asks for the largest shared-memory carveout, so consecutive launches of
    // different shapes (different dynamic shared memory) never need the SM's L1 / shared split
    // changed between them, which would keep the next launch's blocks off an SM until it drains
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e == cudaSuccess && big_clusters) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess && bit) done[kernel] |= bit;
    return e;
}

}  // namespace w4
