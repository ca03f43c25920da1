// w4_noalloc.cu -- w4_linear_static: the stream-K decode linear with its
// workspace in a fixed device array owned by this library, for callers that
// cannot allocate device memory.
//
// Who needs it: code that must not call cudaMalloc (or any allocator) -- for
// example a plugin running inside another framework that owns every device
// allocation, or a service whose device memory is a fixed budget reserved up
// front.  w4_linear needs a caller-provided workspace; this entry point brings
// its own.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library's device code holds W4_STATIC_SCRATCH_BYTES of it until the process
// exits.  With lazy module loading (the CUDA default since 12.2) that code is
// loaded, and the array set aside, at its first use on a device -- here, the
// first call's cudaGetSymbolAddress -- so the first call on each device is where
// the array is allocated, and it can fail there when device memory is short;
// later calls allocate nothing.  Host code cannot use the array's name as a
// device address, so that first call (with the device current) asks the runtime
// for the address and caches it.
#include "w4.h"
#include "w4_internal.h"

#include <cstdio>
#include <mutex>

namespace {

static __device__ __align__(256) unsigned char g_w4_static_scratch[W4_STATIC_SCRATCH_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_mu;
void* g_scratch_ptr[kMaxDevices] = {};

w4_status static_fail(w4_status s, const char* msg) {
    w4::set_error_detail(msg);  // read back with w4_last_error_detail()
    return s;
}
w4_status static_cuda_fail(const char* what, cudaError_t e) {
    char msg[200];
    snprintf(msg, sizeof msg, "%s: %s", what, cudaGetErrorString(e));
    return static_fail(W4_ERR_CUDA, msg);
}

// Device address of the scratch array on the current device (looked up once per device).
cudaError_t scratch_address(void** ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_w4_static_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev] = p;
    }
    *ptr = g_scratch_ptr[dev];
    return cudaSuccess;
}

}  // namespace

extern "C" w4_status w4_linear_static(const uint16_t* X, int64_t M, int64_t K, const uint8_t* Wq,
                                      const uint16_t* scales, const uint16_t* offsets, int64_t N, int group_size,
                                      uint16_t* Y, void* stream) {
    if (group_size != 32 && group_size != 64 && group_size != 128)
        return static_fail(W4_ERR_UNSUPPORTED, "group_size not in {32, 64, 128}");
    if (K <= 0 || N < 0 || M < 0 || K % group_size != 0 || K > 0x7FFFFFFFLL || N > 0x7FFFFFFFLL)
        return static_fail(W4_ERR_INVALID_ARG, "bad shape (K > 0, N >= 0, M >= 0, K % group_size == 0)");
    if (M > 8) return static_fail(W4_ERR_INVALID_ARG, "w4_linear_static takes M <= 8");
    if (M == 0 || N == 0) return W4_OK;
    if (!X || !Wq || !scales || !offsets || !Y) return static_fail(W4_ERR_INVALID_ARG, "NULL pointer");
    if (((uintptr_t)X | (uintptr_t)Wq | (uintptr_t)scales | (uintptr_t)offsets | (uintptr_t)Y) & 15u)
        return static_fail(W4_ERR_MISALIGNED, "a pointer is not 16-byte aligned");
    w4::StreamPlan plan;
    if (!w4::plan_stream(M, N, K, group_size, &plan))
        return static_fail(W4_ERR_INVALID_ARG, "w4_linear_static needs an even K / group_size");
    if (plan.ws_bytes > (size_t)W4_STATIC_SCRATCH_BYTES)
        return static_fail(W4_ERR_INVALID_ARG,
                           "problem too large for the static scratch: needs w4_linear_workspace_bytes "
                           "<= W4_STATIC_SCRATCH_BYTES");
    void* scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess)
        return static_cuda_fail("looking up (and on a device's first call, loading) the static scratch array", e);
    // The kernel leaves what it used at zero, but a call that gave up mid-way
    // could not: clear the part this call uses first (an asynchronous memset,
    // no allocation).
    e = cudaMemsetAsync(scratch, 0, plan.ws_bytes, (cudaStream_t)stream);
    if (e != cudaSuccess) return static_cuda_fail("clearing the static scratch array", e);
    const char* detail = "";
    e = w4::launch_stream(plan, X, M, K, Wq, scales, offsets, N, group_size, Y, scratch, (cudaStream_t)stream,
                          &detail);
    if (e != cudaSuccess) return static_fail(W4_ERR_CUDA, detail && *detail ? detail : cudaGetErrorString(e));
    return W4_OK;
}
