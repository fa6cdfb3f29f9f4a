// simple_kernels.cu -- one-thread-per-output kernels (the plain configuration
// every tiled kernel is compared against for identical bits), and the weight
// packing kernel.
//
// The per-output loops are the OneModel "Exact mode" page's definitions
// (section "Matrix product" and section "Convolution"): accumulate from +0
// over k (taps in channel, kernel row, kernel column order), store NaN as
// 0x7FC00000.
#include "om_device.cuh"
#include "om_internal.h"

namespace om {

template <int MODE>
__global__ void gemm_naive_kernel(GemmProblem p) {
    const int64_t j = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
    if (j >= p.n) return;
    for (int64_t i = blockIdx.y; i < p.m; i += gridDim.y) {
        const float *a = p.A + i * p.lda;
        const float *b = p.B + j;
        float acc = 0.0f;
        for (int64_t q = 0; q < p.k; ++q) {
            acc = term<MODE>(acc, a[q], b[q * p.ldb]);
        }
        if (p.ep.bias || p.ep.res || p.ep.act)
            acc = epilogue_value(acc, p.ep.bias ? p.ep.bias + j : nullptr,
                                 p.ep.res ? p.ep.res + i * p.ep.ldr + j : nullptr, p.ep.act);
        p.C[i * p.ldc + j] = canonical_nan(acc);
    }
}

cudaError_t launch_gemm_naive(const GemmProblem &p, int mode, cudaStream_t s) {
    const int threads = 128;
    const int64_t gx = (p.n + threads - 1) / threads;
    if (gx > 0x7FFFFFFF) return cudaErrorInvalidValue;
    dim3 grid(static_cast<unsigned>(gx), static_cast<unsigned>(p.m < 65535 ? p.m : 65535));
    if (mode == kFast)
        gemm_naive_kernel<kFast><<<grid, threads, 0, s>>>(p);
    else
        gemm_naive_kernel<kExact><<<grid, threads, 0, s>>>(p);
    return cudaGetLastError();
}

template <int MODE>
__global__ void conv_naive_kernel(ConvProblem p) {
    const int64_t total = p.N * p.Cout * p.OH * p.OW;
    const int64_t cin_g = p.Cin / p.G, cout_g = p.Cout / p.G;
    for (int64_t o = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; o < total;
         o += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t ox = o % p.OW;
        const int64_t oy = (o / p.OW) % p.OH;
        const int64_t oc = (o / (p.OW * p.OH)) % p.Cout;
        const int64_t n = o / (p.OW * p.OH * p.Cout);
        const int64_t g = oc / cout_g;
        const float *wrow = p.w + oc * p.w_ld;
        float acc = 0.0f;
        int64_t t = 0;
        for (int64_t c = 0; c < cin_g; ++c) {
            const float *plane = p.x + ((n * p.Cin + g * cin_g + c) * p.H) * p.W;
            for (int64_t ky = 0; ky < p.KH; ++ky) {
                const int64_t iy = oy * p.sH - p.pT + ky * p.dH;
                for (int64_t kx = 0; kx < p.KW; ++kx, ++t) {
                    const int64_t ix = ox * p.sW - p.pL + kx * p.dW;
                    float v = 0.0f;
                    if (iy >= 0 && iy < p.H && ix >= 0 && ix < p.W) v = plane[iy * p.W + ix];
                    acc = term<MODE>(acc, wrow[t], v);
                }
            }
        }
        if (p.ep.bias || p.ep.res || p.ep.act)
            acc = epilogue_value(acc, p.ep.bias ? p.ep.bias + oc : nullptr,
                                 p.ep.res ? p.ep.res + o : nullptr, p.ep.act);
        p.y[o] = canonical_nan(acc);
    }
}

cudaError_t launch_conv_naive(const ConvProblem &p, int mode, cudaStream_t s) {
    const int64_t total = p.N * p.Cout * p.OH * p.OW;
    const int threads = 128;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 64;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    if (mode == kFast)
        conv_naive_kernel<kFast><<<static_cast<unsigned>(blocks), threads, 0, s>>>(p);
    else
        conv_naive_kernel<kExact><<<static_cast<unsigned>(blocks), threads, 0, s>>>(p);
    return cudaGetLastError();
}

// Packed layout: row oc of the weight matrix (K taps) at oc*Kp, columns
// K..Kp-1 set to +0. Rows of one group are consecutive and groups follow in
// order, so group g's block starts at g*(Cout/G)*Kp.
__global__ void pack_weights_kernel(int64_t Cout, int64_t K, int64_t Kp, const float *w,
                                    float *out) {
    const int64_t total = Cout * Kp;
    for (int64_t e = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; e < total;
         e += static_cast<int64_t>(gridDim.x) * blockDim.x) {
        const int64_t oc = e / Kp, q = e % Kp;
        out[e] = (q < K) ? w[oc * K + q] : 0.0f;
    }
}

cudaError_t launch_pack_conv_weights(int64_t Cout, int64_t K, int64_t Kp, const float *w,
                                     float *w_packed, cudaStream_t s) {
    const int64_t total = Cout * Kp;
    if (total == 0) return cudaSuccess;
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = static_cast<int64_t>(num_sms()) * 32;
    if (blocks > cap) blocks = cap;
    pack_weights_kernel<<<static_cast<unsigned>(blocks), threads, 0, s>>>(Cout, K, Kp, w, w_packed);
    return cudaGetLastError();
}

}  // namespace om
