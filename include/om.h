/*
 * om.h -- C ABI of the GB300 (sm_103a) fp32 matrix product and NCHW 2-D
 * convolution library (libom_gpu.so).
 *
 * What is computed (OneModel documentation):
 *   - "Exact mode", section "Matrix product (C = A * B, row-major, A is m x k,
 *     B is k x n)": for every output, acc = +0; for p = 0 .. k-1 in increasing
 *     order, acc = round(acc + round(A[i][p] * B[p][j])); a NaN result is
 *     stored as the bits 0x7FC00000; k = 0 gives +0.
 *   - "Matrix product and convolution kernels", section "Fast mode": the same
 *     order (one accumulator, increasing k, from +0) with one fused
 *     multiply-add per term.
 *   - "Exact mode", section "Convolution (2-D, NCHW, weights [Cout, Cin/G,
 *     KH, KW])": output (n, oc, y, x) of group g = oc / (Cout/G) sums over
 *     c, then ky, then kx of weight[oc][c][ky][kx] * v, where
 *     v = input[n][g*Cin/G + c][y*stride - pad + ky*dil][x*stride - pad + kx*dil]
 *     inside the plane and +0 outside (padding taps are real products);
 *     output size floor((size + 2*pad - dil*(K-1) - 1) / stride) + 1.
 *   - "Exact mode", rules 1-5: binary32 round-to-nearest-even, no fused
 *     multiply-add in exact mode, subnormals kept (no flush-to-zero), start
 *     from +0, canonical NaN, results independent of blocking and threads.
 *
 * Both OM_MODE_EXACT and OM_MODE_FAST produce exactly one bit pattern per
 * output, whatever kernel configuration, grid or stream runs the call. Fast
 * mode also stores NaN as 0x7FC00000 (the documentation lets fast mode keep
 * the hardware payload; this library canonicalises in both modes).
 * OM_MODE_TF32X3 is a separate tolerance mode on the tensor cores (see
 * om_gemm_f32); it is never bit-exact.
 *
 * Conventions for every entry point:
 *   - Pointers named A, B, C, x, w, w_packed, y, workspace are DEVICE
 *     pointers to memory owned by the caller. The library allocates no device
 *     memory and keeps no per-call state; it only caches device properties.
 *   - stream is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream). Calls are asynchronous on that stream and never synchronise;
 *     a kernel fault surfaces on the stream as CUDA reports it.
 *   - Sizes are int64_t; every size and stride is validated on the host
 *     before anything is launched. A call that fails validation launches
 *     nothing and leaves every output untouched.
 *   - Output ranges must not overlap input ranges (OM_ERR_ALIAS).
 *   - The return value is an om_status; om_status_string() names it.
 */
#ifndef OM_H
#define OM_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define OM_API __attribute__((visibility("default")))
#else
#define OM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

#define OM_VERSION 10000 /* 1.0.0 */

typedef enum om_status {
    OM_OK = 0,
    OM_ERR_INVALID_ARG = 1, /* negative size, short leading dimension, stride/dil < 1, pad < 0, bad groups */
    OM_ERR_NULL_PTR = 2,    /* NULL pointer for a non-empty operand */
    OM_ERR_ALIAS = 3,       /* the output range overlaps an input range */
    OM_ERR_UNSUPPORTED = 4, /* unknown mode, or a mode with no kernel for this call (reported, never approximated) */
    OM_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
    OM_ERR_TIMEOUT = 6,     /* a bounded device-side wait gave up (om_device_status, om_workspace_status) */
    OM_ERR_ALIGNMENT = 7,   /* a pointer is not 4-byte aligned, or packed weights not 16-byte aligned */
    OM_ERR_TOO_LARGE = 8    /* a size exceeds what the kernels index (see each entry point) */
} om_status;

typedef enum om_mode {
    OM_MODE_EXACT = 0,  /* round(acc + round(a*b)), no fused multiply-add */
    OM_MODE_FAST = 1,   /* acc = fma(a, b, acc), same order */
    OM_MODE_TF32X3 = 2  /* tensor-core 3xTF32 split; tolerance, not bit-exact */
} om_mode;

typedef enum om_activation {
    OM_ACT_NONE = 0,
    OM_ACT_RELU = 1  /* max(v, +0); NaN stays NaN, -0 becomes +0 */
} om_activation;

/* Library version, OM_VERSION of the build. */
OM_API int om_version(void);

/* Static name of a status code ("OM_OK", ...); "OM_UNKNOWN" for other values. */
OM_API const char *om_status_string(int status);

/*
 * Output size of one convolution axis:
 *   floor((size + 2*pad - dil*(ksize-1) - 1) / stride) + 1, or 0 when the
 * numerator is negative ("Exact mode", section "Convolution", output size).
 * Returns -1 for invalid arguments (size < 0, ksize < 1, stride < 1, pad < 0,
 * dil < 1) or sizes beyond 2^40.
 */
OM_API int64_t om_conv_out_dim(int64_t size, int64_t ksize, int64_t stride, int64_t pad, int64_t dil);

/*
 * C = A * B ("Exact mode", section "Matrix product"; "Fast mode").
 *   A: m x k row-major, row stride lda >= k (elements).
 *   B: k x n row-major, row stride ldb >= n.
 *   C: m x n row-major, row stride ldc >= n. Only C[i][j] with i < m and
 *      j < n is written; columns n .. ldc-1 are never touched.
 *   mode: OM_MODE_EXACT, OM_MODE_FAST or OM_MODE_TF32X3.
 * m == 0 or n == 0: OM_OK, nothing launched. k == 0: C[:m, :n] = +0.
 * Leading dimensions are checked only where the dimension is used (lda when
 * k > 0, ldb when k > 0, ldc always for a non-empty C).
 * Any 4-byte alignment of A, B, C and any lda, ldb, ldc is accepted; 16-byte
 * aligned operands with lda, ldb multiples of 4 take the TMA-fed kernel,
 * others a kernel fed by TMA for A and 4-byte copies for B, or by 4-byte
 * copies for both; products with at most 8 rows or 8 columns run as
 * matrix-vector products. Every path gives identical bits.
 * OM_MODE_TF32X3: each operand is split into a TF32 high part (truncated)
 * and a low part (the remainder, of which the tensor cores read the TF32
 * part); C accumulates hi*hi + hi*lo + lo*hi in fp32 on the tensor cores.
 * Bound, for outputs whose exact-mode result is finite:
 *   |C - C_exact| <= 1e-5 * sqrt(k) * sum_p |A[i][p]| * |B[p][j]|.
 * Non-finite inputs give non-finite outputs where the exact result is
 * non-finite (the class, NaN or infinity, may differ). The tensor-core
 * kernel fetches A and B with TMA, which needs them 16-byte aligned with lda
 * and ldb multiples of 4; other operands are computed by the fast-mode
 * CUDA-core kernel, whose result lies inside the same bound.
 */
OM_API int om_gemm_f32(int64_t m, int64_t n, int64_t k,
                       const float *A, int64_t lda,
                       const float *B, int64_t ldb,
                       float *C, int64_t ldc,
                       int mode, void *stream);

/*
 * Bytes of device scratch the *_ws and *_ex entry points take (a constant,
 * 4096): 1024 32-bit words; words 0..1022 hold one flag per CTA of the
 * balanced schedule (grids of up to 1023 CTAs), word 1023 is the status word
 * of the calls that use the workspace. A bounded device wait that runs out in
 * such a call records OM_ERR_TIMEOUT in that word -- not in the device-wide
 * words of om_device_status -- so every caller with its own workspace sees
 * only its own calls' timeouts (om_workspace_status). Zero a new workspace
 * once before its first use; afterwards the library keeps the flags and
 * om_workspace_status clears the status word.
 */
OM_API size_t om_workspace_bytes(void);

/*
 * Synchronises stream, then reads and clears the status word of workspace
 * (the word every *_ws / *_ex call given this workspace, and
 * om_selftest_wait_timeout_ws, reports a timed-out device wait in). Returns
 * OM_OK, OM_ERR_TIMEOUT if one of those calls' kernels gave up a bounded
 * wait (its outputs are then incomplete), OM_ERR_NULL_PTR / OM_ERR_INVALID_ARG
 * / OM_ERR_ALIGNMENT for a missing, short or misaligned workspace, or
 * OM_ERR_CUDA if the copy or the synchronisation failed. The pages have no
 * counterpart: this is the library's per-call failure report.
 */
OM_API int om_workspace_status(void *workspace, size_t workspace_bytes, void *stream);

/*
 * om_gemm_f32 with caller scratch for a balanced schedule. Output tiles are
 * handed out whole for all but the last one or two rounds of the SMs; the
 * k-loops of the remaining tiles are cut into equal contiguous ranges, one
 * per SM. A range that ends inside a tile computes that tile's first
 * k-stages and stores the raw accumulators to C; the next range finishes the
 * tile from those stored accumulators ("Matrix product and convolution
 * kernels" page, item 3 "Microkernel": a later k-block starts from the C
 * values the earlier blocks stored). Every output is still one sequential
 * loop over k from +0, so the bits are identical to om_gemm_f32; only the
 * load balance across SMs changes (no idle SMs in a last, partial round).
 *   workspace: device memory, 16-byte aligned, at least om_workspace_bytes(),
 *   not overlapping A, B or C. The call clears what it uses on stream before
 *   the kernel runs. Calls that may run at the same time on the GPU need
 *   distinct workspaces.
 * Problems whose tiles fill whole rounds of the SMs, or that have fewer tiles
 * than SMs, run the plain schedule. Errors as om_gemm_f32, plus
 * OM_ERR_NULL_PTR for a NULL workspace, OM_ERR_INVALID_ARG for a short one
 * and OM_ERR_ALIGNMENT for a misaligned one. OM_MODE_TF32X3 ignores the
 * workspace.
 */
OM_API int om_gemm_f32_ws(int64_t m, int64_t n, int64_t k,
                          const float *A, int64_t lda,
                          const float *B, int64_t ldb,
                          float *C, int64_t ldc,
                          int mode, void *workspace, size_t workspace_bytes, void *stream);

/*
 * om_gemm_f32_ws for callers that cannot allocate device memory. The paper has
 * no counterpart: it describes CPU kernels, with no device memory to manage.
 * Some callers of a GPU library may not call cudaMalloc at all: plugins and
 * kernels run by a host framework that hands out only buffers it planned
 * itself, or latency-critical paths where an allocation (and the
 * synchronisation it can bring) is not allowed. They pass only A, B and C.
 * Same arguments, results (bit for bit) and errors as om_gemm_f32 /
 * om_gemm_f32_ws.
 * Scratch: the balanced schedule's flags live in a 4 KiB static device array
 * (1024 words, one per SM used) that every GPU loading the library holds
 * until the process exits. OM_ERR_TOO_LARGE if the device has more than 1024
 * SMs.
 * The first call on a device (and the first call after the device's
 * context changed, e.g. after cudaDeviceReset) looks up that array's device
 * address with the device current (cudaGetSymbolAddress); make that first
 * call before any stream capture. No call allocates or frees device memory.
 * All calls share the one array and it keeps the previous call's contents;
 * each call clears the words it needs on its stream before its kernel runs.
 * Calls that may overlap on the GPU (other streams, other threads) race on
 * the array: run them on one stream, or use om_gemm_f32_ws with a workspace
 * per stream.
 */
OM_API int om_gemm_f32_no_alloc(int64_t m, int64_t n, int64_t k,
                                const float *A, int64_t lda,
                                const float *B, int64_t ldb,
                                float *C, int64_t ldc,
                                int mode, void *stream);

/*
 * 2-D convolution, NCHW ("Exact mode", section "Convolution"; "Convolution
 * (fast mode)", section "What each output is"), computed as an implicit
 * matrix product: per image and group, A = the group's weights
 * (Cout/G x Cin/G*KH*KW), B = the input patches gathered straight into
 * on-chip memory with the zero border written during the gather, C = the
 * group's output planes. Padding is never materialised. Shapes the
 * implicit product would run poorly go to other kernels with the same
 * per-output loop and the same bits: groups of at most 16 output channels
 * (depthwise included), stride-1 3x3 layers whose output-row segments fill
 * the GPU, and layers with few output pixels run from input windows staged
 * in on-chip memory (zero border written at copy time; by TMA with its
 * out-of-range fill where input rows are 16-byte aligned), and a 1x1 kernel
 * over a 1x1 input of at most 8 images runs as a matrix-vector product.
 *   x: [N][Cin][H][W] contiguous.
 *   w: [Cout][Cin/G][KH][KW] contiguous.
 *   y: [N][Cout][OutH][OutW] contiguous, OutH/OutW from om_conv_out_dim.
 *   Symmetric padding pad, one stride and one dilation for both axes.
 *   G >= 1 must divide Cin and Cout (depthwise, G == Cin, included).
 *   mode: OM_MODE_EXACT or OM_MODE_FAST (OM_MODE_TF32X3 -> OM_ERR_UNSUPPORTED).
 * An empty output (N, Cout, OutH or OutW zero) returns OM_OK with nothing
 * launched. Cin == 0 (an empty sum) writes +0 everywhere. No bias is added.
 * Element counts of x, w and y must each stay below 2^62; a per-image plane
 * block (Cin*H*W or Cout*OutH*OutW) and K = Cin/G*KH*KW must stay below
 * 2^31 (OM_ERR_TOO_LARGE otherwise).
 */
OM_API int om_conv2d_f32(int64_t N, int64_t Cin, int64_t H, int64_t W,
                         int64_t Cout, int64_t G, int64_t KH, int64_t KW,
                         int64_t stride, int64_t pad, int64_t dil,
                         const float *x, const float *w, float *y,
                         int mode, void *stream);

/*
 * om_conv2d_f32 with caller scratch for the balanced schedule (as
 * om_gemm_f32_ws: the taps of the last output tiles are split evenly over the
 * SMs with k-block continuation through y). Bit-identical to om_conv2d_f32.
 * Workspace rules and extra errors as om_gemm_f32_ws.
 */
OM_API int om_conv2d_f32_ws(int64_t N, int64_t Cin, int64_t H, int64_t W,
                            int64_t Cout, int64_t G, int64_t KH, int64_t KW,
                            int64_t stride, int64_t pad, int64_t dil,
                            const float *x, const float *w, float *y,
                            int mode, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Re-lays out convolution weights once for om_conv2d_f32_packed
 * ("Convolution (fast mode)", section "Layout of the work": weights packed
 * once, when the model is loaded).
 * Layout written: for each group g, a (Cout/G) x Kp row-major block with
 * Kp = K rounded up to a multiple of 4 (K = Cin/G*KH*KW), columns K..Kp-1
 * set to +0; groups follow one another. Every row then starts on a 16-byte
 * boundary, which lets the convolution fetch weights with TMA.
 * Two-call convention: with w_packed == NULL, only *packed_bytes is set
 * (the size the caller must allocate) and nothing is launched. Otherwise
 * *packed_bytes (if packed_bytes != NULL) is set again, and the packing
 * kernel is launched on stream. w_packed must be 16-byte aligned.
 */
OM_API int om_pack_conv_weights(int64_t Cout, int64_t Cin, int64_t G, int64_t KH, int64_t KW,
                                const float *w, float *w_packed, size_t *packed_bytes,
                                void *stream);

/*
 * om_conv2d_f32 with weights already packed by om_pack_conv_weights (same
 * Cout, Cin, G, KH, KW). The result is bit-identical to om_conv2d_f32 on the
 * unpacked weights. w_packed must be 16-byte aligned (OM_ERR_ALIGNMENT).
 */
OM_API int om_conv2d_f32_packed(int64_t N, int64_t Cin, int64_t H, int64_t W,
                                int64_t Cout, int64_t G, int64_t KH, int64_t KW,
                                int64_t stride, int64_t pad, int64_t dil,
                                const float *x, const float *w_packed, float *y,
                                int mode, void *stream);

/* om_conv2d_f32_packed with caller scratch for the balanced schedule. */
OM_API int om_conv2d_f32_packed_ws(int64_t N, int64_t Cin, int64_t H, int64_t W,
                                   int64_t Cout, int64_t G, int64_t KH, int64_t KW,
                                   int64_t stride, int64_t pad, int64_t dil,
                                   const float *x, const float *w_packed, float *y,
                                   int mode, void *workspace, size_t workspace_bytes,
                                   void *stream);

/*
 * Product with a fused output epilogue ("Convolution (fast mode)", sections
 * "Tiles and chunks" -- bias, then activation, on each finished tile -- and
 * "Single-column products" -- the bias, activation and residual epilogue).
 * Each output v of the product is finished as
 *   v = v + bias[j];  v = v + residual[i*ldr + j];  v = relu(v)
 * one binary32 round-to-nearest operation per step (bias and residual are
 * skipped when NULL; the pages do not fix the place of the residual, this
 * library adds it before the activation, as a residual block needs), then a
 * NaN is stored as 0x7FC00000. bias has n entries (one per column); residual
 * is m x n with row stride ldr >= n and must not overlap C.
 * activation: OM_ACT_NONE or OM_ACT_RELU. workspace may be NULL (the plain
 * schedule) or a workspace as for om_gemm_f32_ws. Modes and errors as
 * om_gemm_f32 / om_gemm_f32_ws; OM_ERR_INVALID_ARG for an unknown activation
 * or a short ldr, OM_ERR_ALIAS for a residual or bias overlapping C.
 */
OM_API int om_gemm_f32_ex(int64_t m, int64_t n, int64_t k,
                          const float *A, int64_t lda,
                          const float *B, int64_t ldb,
                          float *C, int64_t ldc,
                          const float *bias, const float *residual, int64_t ldr, int activation,
                          int mode, void *workspace, size_t workspace_bytes, void *stream);

/*
 * Convolution with a fused output epilogue: output (n, oc, oy, ox) is
 * finished as v + bias[oc], then + residual[n][oc][oy][ox], then the
 * activation, as om_gemm_f32_ex. bias has Cout entries; residual has y's
 * shape and must not overlap y. weights_packed != 0 takes w as laid out by
 * om_pack_conv_weights. workspace may be NULL or a workspace as for
 * om_conv2d_f32_ws. Errors as om_conv2d_f32 / om_conv2d_f32_ws, plus
 * OM_ERR_INVALID_ARG for an unknown activation and OM_ERR_ALIAS for a
 * residual or bias overlapping y.
 */
OM_API int om_conv2d_f32_ex(int64_t N, int64_t Cin, int64_t H, int64_t W,
                            int64_t Cout, int64_t G, int64_t KH, int64_t KW,
                            int64_t stride, int64_t pad, int64_t dil,
                            const float *x, const float *w, int weights_packed,
                            const float *bias, const float *residual, int activation,
                            float *y, int mode, void *workspace, size_t workspace_bytes,
                            void *stream);

/*
 * Synchronises stream, then reads and clears the library's device-wide status
 * words for the current device. Every device-side wait in the library's
 * kernels (mbarrier waits of the TMA and tensor-core pipelines) is bounded;
 * a wait that runs out records OM_ERR_TIMEOUT and the kernel returns early
 * instead of hanging. Calls given a workspace record it in the workspace's
 * status word (om_workspace_status); calls without one (om_gemm_f32,
 * om_conv2d_f32, om_conv2d_f32_packed, om_gemm_f32_no_alloc, the *_ex entry
 * points with a NULL workspace) record it in these device-wide words, which
 * every such call on the device shares: whichever caller reads them first
 * sees (and clears) any such timeout. Returns OM_OK, OM_ERR_TIMEOUT, or
 * OM_ERR_CUDA if the synchronisation itself failed.
 */
OM_API int om_device_status(void *stream);

/*
 * Failure-detection self-test (the pages have no counterpart: it exists so
 * that the timeout path of the kernels' bounded waits can be tested without
 * a GPU fault). Launches one block on `stream` whose wait runs out after
 * limit_ms milliseconds (1..1000): which = 0 waits on an mbarrier phase that
 * nothing completes (the kernels' pipeline wait), which = 1 acquires a
 * device flag that nothing sets (the balanced schedule's continuation
 * wait). The block then records the timeout and returns; a following
 * om_device_status(stream) reports OM_ERR_TIMEOUT (and clears it), and the
 * context stays usable. Returns OM_OK once launched, OM_ERR_INVALID_ARG for
 * other arguments, OM_ERR_CUDA on a launch error.
 */
OM_API int om_selftest_wait_timeout(int which, int limit_ms, void *stream);

/*
 * om_selftest_wait_timeout reporting into a caller workspace: the timeout is
 * recorded in the workspace's status word (om_workspace_status) and leaves
 * the device-wide words untouched. Errors as om_selftest_wait_timeout, plus
 * those of the workspace checks of om_gemm_f32_ws.
 */
OM_API int om_selftest_wait_timeout_ws(int which, int limit_ms, void *workspace,
                                       size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* OM_H */
