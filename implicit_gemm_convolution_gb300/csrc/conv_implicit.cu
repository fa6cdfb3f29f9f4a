// conv_implicit.cu -- implicit-GEMM convolution (every call currently falls
// back to the direct kernel).
#include "om_device.cuh"
#include "om_internal.h"

namespace om {

__device__ unsigned g_status_conv;

cudaError_t launch_conv_implicit(const ConvProblem &, int, int, cudaStream_t) {
    return cudaErrorNotSupported;
}

cudaError_t read_clear_status_conv(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status_conv, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*out) e = cudaMemcpyToSymbol(g_status_conv, &zero, sizeof(unsigned));
    return e;
}

}  // namespace om
