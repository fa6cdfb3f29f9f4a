// Failure-detection self-test: makes one of the library's bounded device
// waits run out on purpose, so that a test can check that the timeout is
// reported (through the caller's workspace status word, or om_device_status
// without a workspace) and that the context stays usable.
//
// The waits are the kernels' own: an mbarrier phase wait (the TMA / cp.async
// pipelines) and a flag acquire (the balanced schedule's k-block
// continuation). Here nothing ever arrives on the mbarrier and nothing ever
// sets the flag, and the limit is short, so the wait gives up, records the
// timeout bit and the kernel returns normally. No trap, no fault.

#include <cuda_runtime.h>

#include <cstdint>

#include "om_device.cuh"
#include "om_internal.h"

namespace om {

__device__ unsigned g_status_selftest;
__device__ unsigned g_flag_never_set;  // zero-initialised, never written

namespace {

__global__ void wait_timeout_kernel(int which, unsigned long long limit_ns, unsigned *status) {
    __shared__ uint64_t bar;
    if (threadIdx.x == 0) {
        mbar_init(&bar, 1);  // one arrival completes phase 0; none comes
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x != 0) return;
    const bool ok = which == 0 ? mbar_wait_limit(&bar, 0, limit_ns)
                               : acquire_flag(&g_flag_never_set, limit_ns);
    if (!ok) report_timeout(status, &g_status_selftest);
}

}  // namespace

cudaError_t launch_wait_timeout(int which, int limit_ms, unsigned *status, cudaStream_t s) {
    wait_timeout_kernel<<<1, 32, 0, s>>>(which, static_cast<unsigned long long>(limit_ms) * 1000000ull,
                                         status);
    return cudaGetLastError();
}

cudaError_t read_clear_status_selftest(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status_selftest, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*out) e = cudaMemcpyToSymbol(g_status_selftest, &zero, sizeof(unsigned));
    return e;
}

}  // namespace om
