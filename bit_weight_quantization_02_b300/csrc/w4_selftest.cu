// w4_selftest.cu -- a test hook that makes libw4's bounded waits run out on
// purpose, without faulting or hanging the GPU: one small block waits on an
// mbarrier that nothing completes and, as the owner of a split row tile, on a
// sharer slot that nobody publishes.  Both waits use the kernels' own helpers
// (mbar_wait_bounded, split_collect) with a short limit, give up, raise the
// fault word and return; the host then sees W4_ERR_TIMEOUT from
// w4_device_fault, exactly as after a timed-out linear.
#include "w4_selftest.h"
#include "w4_device.cuh"
#include "w4_internal.h"

#include <cstdio>

namespace w4 {

__device__ unsigned int g_selftest_fault;

// block of 64 threads: warp 0 waits on the mbarrier, warp 1 collects a split tile
__global__ void __launch_bounds__(64) selftest_kernel(uint64_t* ws, uint16_t* Y, uint64_t limit_ns) {
    __shared__ __align__(8) unsigned long long bar;
    __shared__ float scr[16];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t b = smem_u32(&bar);
    if (threadIdx.x == 0) {
        mbar_init(b, 1);  // one arrival that never comes
        mbar_fence_init();
    }
    __syncthreads();
    if (warp == 0) {
        mbar_wait_bounded(b, 0u, nullptr, &g_selftest_fault, 1u, limit_ns);
        return;
    }
    // warp 1: worker 0 owns a 16-row tile whose other share is worker 1's (slot 1 of the
    // workspace, never published).  Its own sums: row r (MMA layout) holds r + 0.5.
    const int gid = lane >> 2, tq = lane & 3;
    float acc[1][4];
    acc[0][0] = acc[0][1] = (float)gid + 0.5f;
    acc[0][2] = acc[0][3] = (float)(gid + 8) + 0.5f;
    split_collect<1, 1>(acc, scr, ws, (size_t)16, 0, 1, 1, 16, gid, tq, lane, Y, (int64_t)16, &g_selftest_fault, 2u,
                        limit_ns);
}

cudaError_t read_and_clear_selftest_fault(unsigned int* fault) {
    cudaError_t e = cudaMemcpyFromSymbol(fault, g_selftest_fault, sizeof(unsigned int));
    if (e != cudaSuccess || !*fault) return e;
    const unsigned int zero = 0;
    return cudaMemcpyToSymbol(g_selftest_fault, &zero, sizeof(unsigned int));
}

}  // namespace w4

extern "C" w4_status w4_selftest_bounded_waits(void* workspace, size_t workspace_bytes, uint16_t* Y,
                                               uint64_t limit_ns, void* stream) {
    if (workspace == nullptr || Y == nullptr) {
        w4::set_error_detail("workspace and Y must not be NULL");
        return W4_ERR_INVALID_ARG;
    }
    if (workspace_bytes < 2 * 16 * 8) {
        w4::set_error_detail("the self-test needs 256 workspace bytes (two 16-row slots)");
        return W4_ERR_INVALID_ARG;
    }
    if ((reinterpret_cast<uintptr_t>(workspace) | reinterpret_cast<uintptr_t>(Y)) & 15u) {
        w4::set_error_detail("workspace and Y must be 16-byte aligned");
        return W4_ERR_MISALIGNED;
    }
    if (limit_ns < 100000ull || limit_ns > 1000000000ull) {
        w4::set_error_detail("limit_ns must lie in [1e5, 1e9] (0.1 ms to 1 s)");
        return W4_ERR_INVALID_ARG;
    }
    w4::selftest_kernel<<<1, 64, 0, (cudaStream_t)stream>>>(static_cast<uint64_t*>(workspace), Y, limit_ns);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        char msg[160];
        snprintf(msg, sizeof msg, "self-test launch: %s", cudaGetErrorString(e));
        w4::set_error_detail(msg);
        return W4_ERR_CUDA;
    }
    return W4_OK;
}
