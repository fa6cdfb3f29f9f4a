// om_internal.h -- host-side interface between the C ABI (om_api.cu) and the
// kernel translation units. Not installed; not part of the public ABI.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>

namespace om {

// Output epilogue, applied to each finished output before its NaN is made
// canonical: v = v + bias[channel]; v = v + residual; v = relu(v). Every
// pointer may be NULL (step skipped); act 0 = none, 1 = ReLU. For a product
// the bias is per column and the residual has row stride ldr; for a
// convolution the bias is per output channel and the residual has y's layout.
struct Epilogue {
    const float *bias;
    const float *res;
    int64_t ldr;
    int act;
};

// A validated row-major product problem (device pointers).
struct GemmProblem {
    int64_t m, n, k;
    const float *A;
    int64_t lda;
    const float *B;
    int64_t ldb;
    float *C;
    int64_t ldc;
    Epilogue ep;
    unsigned *status;  // the call's status word in a caller workspace, or NULL
};

// A validated convolution problem. Weights are read as the matrix
// w[oc][p] with row stride w_ld (K for the caller's layout, Kp for the
// packed layout), p = (c*KH + ky)*KW + kx.
struct ConvProblem {
    int64_t N, Cin, H, W, Cout, G, KH, KW;
    int64_t sH, sW, pT, pL, dH, dW;
    int64_t OH, OW;
    int64_t K;     // Cin/G*KH*KW
    int64_t w_ld;  // row stride of the weight matrix (>= K)
    const float *x;
    const float *w;
    float *y;
    Epilogue ep;
    unsigned *status;  // the call's status word in a caller workspace, or NULL
};

// Kernel configurations the dispatcher can choose. A test-only environment
// override (OM_FORCE_GEMM_CFG / OM_FORCE_CONV_CFG) forces one; every
// configuration gives identical bits.
enum GemmCfg : int {
    kCfgAuto = -1,
    kCfgNaive = 0,             // one thread per output
    kCfgTma128x256 = 1,        // TMA-fed SIMT tiles, 128x256, paired-lane fp32
    kCfgTma128x128 = 2,        // TMA-fed SIMT tiles, 128x128, paired-lane fp32
    kCfgAsync128x128 = 3,      // 4-byte cp.async-fed SIMT tiles (any alignment)
    kCfgTmaScalar128x256 = 4,  // as 1 with one-lane fp32 instructions
    kCfgGemv = 5,              // matrix-vector kernel (at most 8 rows or 8 columns)
    kCfgMixed128x256 = 6,      // A by TMA, B by 4-byte cp.async (B rows not 16-byte aligned)
    kCfgMixed128x128 = 7,      // as 6 with 128x128 tiles
};

// The matrix-vector kernels take products with at most kGemvMaxSmall rows
// or columns (and 1x1 convolutions over 1x1 inputs of at most that many
// images).
constexpr int kGemvMaxSmall = 8;

enum ConvCfg : int {
    kConvAuto = -1,
    kConvNaive = 0,     // one thread per output, direct loops
    kConvImplicit = 1,  // implicit GEMM with gathered patches, 64 x 256 tiles
    kConvDirect = 2,    // one thread per output pixel and group, all of its channels
    kConvGemv = 3,      // 1x1 over a 1x1 input: matrix-vector kernel
    kConvSkinny = 4,    // few output pixels: one pixel per thread, channels streamed in chunks
    kConvColumns = 5,   // blocks of 32 channels x 8 pixels, weights by TMA, patches gathered
    kConvRows = 6,      // stride 1: warps own output-row segments of 64 channels, windows by TMA
    kConvGroup = 7,     // up to 16 channels per group, KS x KS taps: a band's window by one TMA copy
};

// The direct kernel serves groups of up to kConvDirectMaxM output channels
// whose weights, tap table and an input window of at least one output row
// fit in its shared memory; the dispatcher takes it by itself up to
// kConvDirectAutoM channels per group.
constexpr int kConvDirectMaxM = 32;
constexpr int kConvDirectAutoM = 16;
// Channels the direct kernel computes per thread for M channels per group
// (M rounded up to a power of two), or 0 above kConvDirectMaxM.
int conv_direct_channels(int64_t M);
cudaError_t launch_conv_direct(const ConvProblem &p, int mode, cudaStream_t s);
// Groups of at most 16 output channels with 1x1, 3x3 or 5x5 taps (any
// stride, dilation and padding) whose input rows are 16-byte aligned: one
// block per band of output rows of one group and image, its input window
// copied by one TMA load with zero fill; cudaErrorNotSupported otherwise.
cudaError_t launch_conv_group(const ConvProblem &p, int mode, cudaStream_t s);
cudaError_t read_clear_status_dw(unsigned *out, cudaStream_t s);
// Few output pixels (output rows of at most 128 pixels), many output channels.
cudaError_t launch_conv_skinny(const ConvProblem &p, int mode, cudaStream_t s);

// Matrix-vector kernels; cudaErrorNotSupported when the shape is not theirs.
cudaError_t launch_gemm_gemv(const GemmProblem &p, int mode, cudaStream_t s);
cudaError_t launch_conv_gemv(const ConvProblem &p, int mode, cudaStream_t s);
// A convolution as per-image, per-group products in blocks of 32 output
// channels by 8 output pixels (the few-columns matrix-vector kernel): 1x1
// unpadded kernels read the input directly, others of up to 64 taps gather
// their patches during the copy.
// choose: decline gathered layers with a short k loop or too few blocks.
cudaError_t launch_conv_columns(const ConvProblem &p, int mode, bool choose, cudaStream_t s);
cudaError_t read_clear_status_gemv(unsigned *out, cudaStream_t s);

// Stride-1 convolutions (3x3 with padding 1 or 1x1 unpadded, any kernel
// height up to 7) whose output rows split into 14-pixel segments and whose
// groups have a multiple of 64 output channels: each warp owns four row
// segments of 64 channels, input windows by 4-D TMA with zero fill, the
// weight block resident in shared memory. choose: decline when the warp
// tasks would fill less than 80 % of the last round.
cudaError_t launch_conv_rows(const ConvProblem &p, int mode, bool choose, cudaStream_t s);
cudaError_t read_clear_status_rows(unsigned *out, cudaStream_t s);

// Failure-detection self-test (selftest.cu): a one-block kernel whose
// bounded wait (0: mbarrier phase, 1: global flag) runs out after limit_ms.
cudaError_t launch_wait_timeout(int which, int limit_ms, unsigned *status, cudaStream_t s);
cudaError_t read_clear_status_selftest(unsigned *out, cudaStream_t s);

cudaError_t launch_gemm_naive(const GemmProblem &p, int mode, cudaStream_t s);
cudaError_t launch_conv_naive(const ConvProblem &p, int mode, cudaStream_t s);
cudaError_t launch_pack_conv_weights(int64_t Cout, int64_t K, int64_t Kp, const float *w,
                                     float *w_packed, cudaStream_t s);

// Tiled kernels. Return cudaErrorNotSupported when the configuration cannot
// run this problem (the dispatcher then picks another one).
// flags: NULL for whole tiles only, or kMaxScheduleCtas words of caller
// scratch for the balanced schedule with k-block continuation.
cudaError_t launch_gemm_tiled(const GemmProblem &p, int mode, int cfg, unsigned *flags,
                              cudaStream_t s);
cudaError_t launch_conv_implicit(const ConvProblem &p, int mode, int cfg, unsigned *flags,
                                 cudaStream_t s);

// OM_MODE_TF32X3 on the tensor cores (needs 16-byte aligned A, B and lda,
// ldb multiples of 4; cudaErrorNotSupported otherwise).
cudaError_t launch_gemm_tf32x3(const GemmProblem &p, cudaStream_t s);
cudaError_t read_clear_status_tc(unsigned *out, cudaStream_t s);

// The checks and dispatch of om_gemm_f32_ws with scratch supplied by the
// library itself (see om_gemm_f32_no_alloc).
int gemm_with_scratch(int64_t m, int64_t n, int64_t k, const float *A, int64_t lda,
                      const float *B, int64_t ldb, float *C, int64_t ldc, int mode,
                      void *scratch, size_t scratch_bytes, void *stream);

// Read and clear the device status word of the tiled translation units
// (synchronises s).
cudaError_t read_clear_status_gemm(unsigned *out, cudaStream_t s);
cudaError_t read_clear_status_conv(unsigned *out, cudaStream_t s);

// Largest dynamic shared memory a block may opt in to on the current device.
int max_smem_optin();
int num_sms();

// Caller workspace of the *_ws / *_ex entry points: kWorkspaceWords 32-bit
// words; words [0, kMaxScheduleCtas) are the balanced schedule's flags (one
// per CTA), word kWsStatusWord the status word of the calls that use the
// workspace.
constexpr int kWorkspaceWords = 1024;
constexpr int kMaxScheduleCtas = 1023;
constexpr int kWsStatusWord = 1023;

// Bit of the device status words set by a bounded wait that ran out.
constexpr unsigned kDevErrTimeoutHost = 1u;

}  // namespace om
