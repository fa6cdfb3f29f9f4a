// om_api.cu -- the C ABI declared in include/om.h: argument validation, shape
// derivation, kernel selection and launch on the caller's stream.
//
// The library allocates no device memory and keeps no state between calls
// besides a per-device cache of the SM count.
#include <cstdint>
#include <cstdlib>

#include "om.h"
#include "om_internal.h"

namespace om {

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 1;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int v = 1;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v < 1) v = 1;
    if (dev < 64) cached[dev] = v;
    return v;
}

int max_smem_optin() {
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) return 0;
    if (dev < 64 && cached[dev] > 0) return cached[dev];
    int v = 0;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) v = 0;
    if (dev < 64 && v > 0) cached[dev] = v;
    return v;
}

}  // namespace om

namespace {

using om::ConvProblem;
using om::GemmProblem;

// A test-only override of the kernel configuration; every configuration
// computes the same bits.
int forced(const char *name) {
    const char *v = std::getenv(name);
    if (!v || !*v) return -1;
    return std::atoi(v);
}

bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

// Byte range [lo, hi) touched by a row-major rows x cols block with row stride ld.
struct Range {
    uintptr_t lo, hi;
};

bool block_range(const void *base, int64_t rows, int64_t cols, int64_t ld, Range *r) {
    r->lo = r->hi = reinterpret_cast<uintptr_t>(base);
    if (rows <= 0 || cols <= 0) return true;
    const __int128 elems = static_cast<__int128>(rows - 1) * ld + cols;
    if (elems >= (static_cast<__int128>(1) << 60)) return false;
    r->hi = r->lo + static_cast<uintptr_t>(elems) * 4;
    return r->hi > r->lo;
}

Range span(const void *base, __int128 elems) {
    Range r;
    r.lo = reinterpret_cast<uintptr_t>(base);
    r.hi = r.lo + static_cast<uintptr_t>(elems) * 4;
    return r;
}

bool overlaps(const Range &a, const Range &b) {
    if (a.lo == a.hi || b.lo == b.hi) return false;
    return a.lo < b.hi && b.lo < a.hi;
}

int from_cuda(cudaError_t e) { return e == cudaSuccess ? OM_OK : OM_ERR_CUDA; }

int64_t out_dim(int64_t size, int64_t k, int64_t stride, int64_t pad, int64_t dil) {
    const int64_t num = size + 2 * pad - dil * (k - 1) - 1;
    if (num < 0) return 0;
    return num / stride + 1;
}

struct ConvArgs {
    int64_t N, Cin, H, W, Cout, G, KH, KW, stride, pad, dil;
};

// Validates a convolution call and fills the problem; returns an om_status.
int validate_conv(const ConvArgs &a, const float *x, const float *w, bool packed, float *y,
                  int mode, ConvProblem *p, bool *empty) {
    *empty = false;
    if (a.N < 0 || a.Cin < 0 || a.H < 0 || a.W < 0 || a.Cout < 0) return OM_ERR_INVALID_ARG;
    if (a.G < 1 || a.KH < 1 || a.KW < 1 || a.stride < 1 || a.dil < 1 || a.pad < 0)
        return OM_ERR_INVALID_ARG;
    if (a.Cin % a.G != 0 || a.Cout % a.G != 0) return OM_ERR_INVALID_ARG;
    if (mode != OM_MODE_EXACT && mode != OM_MODE_FAST) return OM_ERR_UNSUPPORTED;
    // Size bounds keep every derived quantity inside int64 and the kernels'
    // 32-bit per-image indices from overflowing.
    const int64_t lim31 = (int64_t(1) << 31) - 1;
    if (a.H > lim31 || a.W > lim31 || a.KH > 65535 || a.KW > 65535 || a.stride > 65535 ||
        a.dil > 65535 || a.pad > 65535)
        return OM_ERR_TOO_LARGE;
    // input coordinates oy*s - pad + ky*d stay inside 32-bit integers
    if (a.H + 2 * a.pad >= lim31 || a.W + 2 * a.pad >= lim31 ||
        (a.KH - 1) * a.dil >= lim31 - a.H || (a.KW - 1) * a.dil >= lim31 - a.W)
        return OM_ERR_TOO_LARGE;
    const int64_t OH = out_dim(a.H, a.KH, a.stride, a.pad, a.dil);
    const int64_t OW = out_dim(a.W, a.KW, a.stride, a.pad, a.dil);
    const int64_t cin_g = a.Cin / a.G;
    const __int128 K = static_cast<__int128>(cin_g) * a.KH * a.KW;
    const __int128 Kp = (K + 3) / 4 * 4;
    const __int128 w_ld = packed ? Kp : K;
    const __int128 xe = static_cast<__int128>(a.N) * a.Cin * a.H * a.W;
    const __int128 ye = static_cast<__int128>(a.N) * a.Cout * OH * OW;
    const __int128 we = static_cast<__int128>(a.Cout) * w_ld;
    const __int128 lim62 = static_cast<__int128>(1) << 62;
    if (K > lim31 || xe >= lim62 || ye >= lim62 || we >= lim62) return OM_ERR_TOO_LARGE;
    if (static_cast<__int128>(a.Cin) * a.H * a.W > lim31 ||
        static_cast<__int128>(a.Cout) * OH * OW > lim31)
        return OM_ERR_TOO_LARGE;
    if (ye == 0) {
        *empty = true;
        return OM_OK;
    }
    if (!y) return OM_ERR_NULL_PTR;
    if (xe > 0 && !x) return OM_ERR_NULL_PTR;
    if (K > 0 && !w) return OM_ERR_NULL_PTR;
    if (!aligned4(x) || !aligned4(w) || !aligned4(y)) return OM_ERR_ALIGNMENT;
    if (packed && (reinterpret_cast<uintptr_t>(w) & 15) != 0) return OM_ERR_ALIGNMENT;
    const Range ry = span(y, ye), rx = span(x, xe), rw = span(w, we);
    if ((xe > 0 && overlaps(ry, rx)) || (K > 0 && overlaps(ry, rw))) return OM_ERR_ALIAS;
    p->N = a.N; p->Cin = a.Cin; p->H = a.H; p->W = a.W; p->Cout = a.Cout; p->G = a.G;
    p->KH = a.KH; p->KW = a.KW;
    p->sH = p->sW = a.stride;
    p->pT = p->pL = a.pad;
    p->dH = p->dW = a.dil;
    p->OH = OH; p->OW = OW;
    p->K = static_cast<int64_t>(K);
    p->w_ld = static_cast<int64_t>(w_ld);
    p->x = x; p->w = w; p->y = y;
    return OM_OK;
}

// Output tiles are handed to a persistent grid of one CTA per SM. Without a
// workspace a launch costs whole rounds of tiles, so pick the tile shape with
// the fewer rounds times tile size (ties go to the larger tile, which reuses
// each operand load over more outputs). With a workspace the last rounds are
// balanced across the SMs and the larger tile is always taken.
int pick_gemm_cfg(const GemmProblem &p, bool balanced) {
    if (balanced) return om::kCfgTma128x256;
    const int64_t sms = om::num_sms();
    const int64_t tm = (p.m + 127) / 128;
    const int64_t t256 = tm * ((p.n + 255) / 256), t128 = tm * ((p.n + 127) / 128);
    const int64_t c256 = (t256 + sms - 1) / sms * 2;  // in units of a 128 x 128 tile
    const int64_t c128 = (t128 + sms - 1) / sms;
    return c128 < c256 ? om::kCfgTma128x128 : om::kCfgTma128x256;
}

// The implicit GEMM's 64 x 256 tiles would not give every SM a tile, and the
// k loop is long: the few-pixel kernel keeps one output pixel per thread.
bool few_pixels(const ConvProblem &p) {
    const int64_t M = p.Cout / p.G;
    const int64_t tiles = p.G * ((M + 63) / 64) * ((p.N * p.OH * p.OW + 255) / 256);
    return tiles < om::num_sms() && p.K >= 64 && p.OW <= 128;
}

int run_conv(const ConvProblem &p, int mode, unsigned *flags, cudaStream_t s) {
    const int cfg = forced("OM_FORCE_CONV_CFG");
    if (cfg == om::kConvNaive || p.K == 0) return from_cuda(om::launch_conv_naive(p, mode, s));
    cudaError_t e = cudaErrorNotSupported;
    if (cfg == om::kConvGemv || cfg < 0) e = om::launch_conv_gemv(p, mode, s);
    if (e == cudaErrorNotSupported &&
        (cfg == om::kConvGroup || (cfg < 0 && p.Cout / p.G <= om::kConvDirectAutoM)))
        e = om::launch_conv_group(p, mode, s);
    if (e == cudaErrorNotSupported &&
        (cfg == om::kConvDirect || (cfg < 0 && p.Cout / p.G <= om::kConvDirectAutoM)))
        e = om::launch_conv_direct(p, mode, s);
    if (e == cudaErrorNotSupported && (cfg == om::kConvRows || cfg < 0))
        e = om::launch_conv_rows(p, mode, cfg < 0, s);
    if (e == cudaErrorNotSupported && (cfg == om::kConvColumns || (cfg < 0 && few_pixels(p))))
        e = om::launch_conv_columns(p, mode, cfg < 0, s);
    if (e == cudaErrorNotSupported && (cfg == om::kConvSkinny || (cfg < 0 && few_pixels(p))))
        e = om::launch_conv_skinny(p, mode, s);
    if (e == cudaErrorNotSupported && cfg != om::kConvDirect && cfg != om::kConvGemv &&
        cfg != om::kConvSkinny && cfg != om::kConvColumns && cfg != om::kConvRows &&
        cfg != om::kConvGroup)
        e = om::launch_conv_implicit(p, mode, cfg < 0 ? om::kConvAuto : cfg, flags, s);
    if (e == cudaErrorNotSupported) e = om::launch_conv_naive(p, mode, s);
    return from_cuda(e);
}

// Validates a caller workspace; *flags stays NULL when none was given.
int check_workspace(void *ws, size_t bytes, unsigned **flags) {
    *flags = nullptr;
    if (!ws) return OM_OK;
    if ((reinterpret_cast<uintptr_t>(ws) & 15) != 0) return OM_ERR_ALIGNMENT;
    if (bytes < static_cast<size_t>(om::kWorkspaceWords) * sizeof(unsigned)) return OM_ERR_INVALID_ARG;
    *flags = static_cast<unsigned *>(ws);
    return OM_OK;
}

Range ws_range(const unsigned *flags) { return span(flags, flags ? om::kWorkspaceWords : 0); }

// The status word of the calls that use a workspace, or NULL without one
// (kernels then report into their translation unit's device-wide word).
unsigned *ws_status(unsigned *flags) { return flags ? flags + om::kWsStatusWord : nullptr; }

int gemm_impl(int64_t m, int64_t n, int64_t k, const float *A, int64_t lda, const float *B,
              int64_t ldb, float *C, int64_t ldc, int mode, void *workspace, size_t ws_bytes,
              void *stream, const om::Epilogue &ep = om::Epilogue{}, bool status_in_ws = true) {
    if (m < 0 || n < 0 || k < 0) return OM_ERR_INVALID_ARG;
    if (mode != OM_MODE_EXACT && mode != OM_MODE_FAST && mode != OM_MODE_TF32X3)
        return OM_ERR_UNSUPPORTED;
    unsigned *flags = nullptr;
    const int wst = check_workspace(workspace, ws_bytes, &flags);
    if (wst != OM_OK) return wst;
    if (m == 0 || n == 0) return OM_OK;
    const bool used = k > 0;
    if (used && (lda < k || ldb < n)) return OM_ERR_INVALID_ARG;
    if (ldc < n) return OM_ERR_INVALID_ARG;
    if (!C || (used && (!A || !B))) return OM_ERR_NULL_PTR;
    if (!aligned4(C) || (used && (!aligned4(A) || !aligned4(B)))) return OM_ERR_ALIGNMENT;
    Range rc, ra, rb;
    if (!block_range(C, m, n, ldc, &rc)) return OM_ERR_TOO_LARGE;
    if (used && !block_range(A, m, k, lda, &ra)) return OM_ERR_TOO_LARGE;
    if (used && !block_range(B, k, n, ldb, &rb)) return OM_ERR_TOO_LARGE;
    if (used && (overlaps(rc, ra) || overlaps(rc, rb))) return OM_ERR_ALIAS;
    const Range rw = ws_range(flags);
    if (flags && (overlaps(rw, rc) || (used && (overlaps(rw, ra) || overlaps(rw, rb)))))
        return OM_ERR_ALIAS;
    // Epilogue operands: read only, never overlapping C or the workspace.
    if (ep.act != 0 && ep.act != 1) return OM_ERR_INVALID_ARG;
    if (ep.bias) {
        if (!aligned4(ep.bias)) return OM_ERR_ALIGNMENT;
        const Range rbias = span(ep.bias, n);
        if (overlaps(rbias, rc) || (flags && overlaps(rbias, rw))) return OM_ERR_ALIAS;
    }
    if (ep.res) {
        if (!aligned4(ep.res)) return OM_ERR_ALIGNMENT;
        if (ep.ldr < n) return OM_ERR_INVALID_ARG;
        Range rres;
        if (!block_range(ep.res, m, n, ep.ldr, &rres)) return OM_ERR_TOO_LARGE;
        if (overlaps(rres, rc) || (flags && overlaps(rres, rw))) return OM_ERR_ALIAS;
    }
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    GemmProblem p{m, n, k, A, lda, B, ldb, C, ldc, ep, status_in_ws ? ws_status(flags) : nullptr};
    if (mode == OM_MODE_TF32X3) {
        if (k == 0) return from_cuda(om::launch_gemm_naive(p, OM_MODE_EXACT, s));  // +0
        cudaError_t e = om::launch_gemm_tf32x3(p, s);
        // Operands TMA cannot fetch take the fast-mode CUDA-core kernel: one
        // correctly rounded fused multiply-add per term is well inside the
        // tolerance mode's bound.
        if (e == cudaErrorNotSupported) e = om::launch_gemm_tiled(p, OM_MODE_FAST, om::kCfgAsync128x128, flags, s);
        if (e == cudaErrorNotSupported) e = om::launch_gemm_naive(p, OM_MODE_FAST, s);
        return from_cuda(e);
    }
    int cfg = forced("OM_FORCE_GEMM_CFG");
    if (k == 0 || cfg == om::kCfgNaive) return from_cuda(om::launch_gemm_naive(p, mode, s));
    if (cfg == om::kCfgGemv || (cfg < 0 && (m <= om::kGemvMaxSmall || n <= om::kGemvMaxSmall))) {
        const cudaError_t eg = om::launch_gemm_gemv(p, mode, s);
        if (eg != cudaErrorNotSupported) return from_cuda(eg);
        cfg = -1;
    }
    if (cfg < 0) cfg = pick_gemm_cfg(p, flags != nullptr);
    cudaError_t e = om::launch_gemm_tiled(p, mode, cfg, flags, s);
    // B rows not 16-byte aligned: A alone by TMA, same tile shape; then both
    // operands by 4-byte copies
    if (e == cudaErrorNotSupported)
        e = om::launch_gemm_tiled(p, mode, cfg == om::kCfgTma128x128 ? om::kCfgMixed128x128 : om::kCfgMixed128x256,
                                  flags, s);
    if (e == cudaErrorNotSupported) e = om::launch_gemm_tiled(p, mode, om::kCfgAsync128x128, flags, s);
    if (e == cudaErrorNotSupported) e = om::launch_gemm_naive(p, mode, s);
    return from_cuda(e);
}

int conv_impl(const ConvArgs &a, const float *x, const float *w, bool packed, float *y, int mode,
              void *workspace, size_t ws_bytes, void *stream,
              const om::Epilogue &ep = om::Epilogue{}) {
    unsigned *flags = nullptr;
    const int wst = check_workspace(workspace, ws_bytes, &flags);
    if (wst != OM_OK) return wst;
    if (ep.act != 0 && ep.act != 1) return OM_ERR_INVALID_ARG;
    ConvProblem p;
    bool empty = false;
    const int st = validate_conv(a, x, w, packed, y, mode, &p, &empty);
    if (st != OM_OK || empty) return st;
    const Range rw = ws_range(flags);
    const Range ry = span(y, static_cast<__int128>(p.N) * p.Cout * p.OH * p.OW);
    if (flags) {
        const Range rx = span(x, static_cast<__int128>(p.N) * p.Cin * p.H * p.W);
        const Range rwt = span(w, static_cast<__int128>(p.Cout) * p.w_ld);
        if (overlaps(rw, ry) || overlaps(rw, rx) || overlaps(rw, rwt)) return OM_ERR_ALIAS;
    }
    // Epilogue operands: read only, never overlapping y or the workspace.
    if (ep.bias) {
        if (!aligned4(ep.bias)) return OM_ERR_ALIGNMENT;
        const Range rb = span(ep.bias, p.Cout);
        if (overlaps(rb, ry) || (flags && overlaps(rb, rw))) return OM_ERR_ALIAS;
    }
    if (ep.res) {
        if (!aligned4(ep.res)) return OM_ERR_ALIGNMENT;
        const Range rr = span(ep.res, static_cast<__int128>(p.N) * p.Cout * p.OH * p.OW);
        if (overlaps(rr, ry) || (flags && overlaps(rr, rw))) return OM_ERR_ALIAS;
    }
    p.ep = ep;
    p.status = ws_status(flags);
    return run_conv(p, mode, flags, static_cast<cudaStream_t>(stream));
}

}  // namespace

namespace om {

// The argument checks and dispatch of om_gemm_f32_ws, for other entry points
// of the library that supply the scratch themselves.
int gemm_with_scratch(int64_t m, int64_t n, int64_t k, const float *A, int64_t lda,
                      const float *B, int64_t ldb, float *C, int64_t ldc, int mode,
                      void *scratch, size_t scratch_bytes, void *stream) {
    // the library's own scratch has no reader for a status word: timeouts go
    // to the device-wide words that om_device_status reads
    return gemm_impl(m, n, k, A, lda, B, ldb, C, ldc, mode, scratch, scratch_bytes, stream,
                     om::Epilogue{}, false);
}

}  // namespace om

extern "C" {

int om_version(void) { return OM_VERSION; }

const char *om_status_string(int status) {
    switch (status) {
        case OM_OK: return "OM_OK";
        case OM_ERR_INVALID_ARG: return "OM_ERR_INVALID_ARG";
        case OM_ERR_NULL_PTR: return "OM_ERR_NULL_PTR";
        case OM_ERR_ALIAS: return "OM_ERR_ALIAS";
        case OM_ERR_UNSUPPORTED: return "OM_ERR_UNSUPPORTED";
        case OM_ERR_CUDA: return "OM_ERR_CUDA";
        case OM_ERR_TIMEOUT: return "OM_ERR_TIMEOUT";
        case OM_ERR_ALIGNMENT: return "OM_ERR_ALIGNMENT";
        case OM_ERR_TOO_LARGE: return "OM_ERR_TOO_LARGE";
        default: return "OM_UNKNOWN";
    }
}

int64_t om_conv_out_dim(int64_t size, int64_t ksize, int64_t stride, int64_t pad, int64_t dil) {
    if (size < 0 || ksize < 1 || stride < 1 || pad < 0 || dil < 1) return -1;
    if (size > (int64_t(1) << 40) || ksize > (int64_t(1) << 20) || pad > (int64_t(1) << 40) ||
        dil > (int64_t(1) << 20) || stride > (int64_t(1) << 40))
        return -1;
    return out_dim(size, ksize, stride, pad, dil);
}

size_t om_workspace_bytes(void) {
    return static_cast<size_t>(om::kWorkspaceWords) * sizeof(unsigned);
}

int om_gemm_f32(int64_t m, int64_t n, int64_t k, const float *A, int64_t lda, const float *B,
                int64_t ldb, float *C, int64_t ldc, int mode, void *stream) {
    return gemm_impl(m, n, k, A, lda, B, ldb, C, ldc, mode, nullptr, 0, stream);
}

int om_gemm_f32_ws(int64_t m, int64_t n, int64_t k, const float *A, int64_t lda, const float *B,
                   int64_t ldb, float *C, int64_t ldc, int mode, void *workspace,
                   size_t workspace_bytes, void *stream) {
    if (!workspace) return OM_ERR_NULL_PTR;
    return gemm_impl(m, n, k, A, lda, B, ldb, C, ldc, mode, workspace, workspace_bytes, stream);
}

int om_conv2d_f32(int64_t N, int64_t Cin, int64_t H, int64_t W, int64_t Cout, int64_t G,
                  int64_t KH, int64_t KW, int64_t stride, int64_t pad, int64_t dil,
                  const float *x, const float *w, float *y, int mode, void *stream) {
    const ConvArgs a{N, Cin, H, W, Cout, G, KH, KW, stride, pad, dil};
    return conv_impl(a, x, w, false, y, mode, nullptr, 0, stream);
}

int om_conv2d_f32_ws(int64_t N, int64_t Cin, int64_t H, int64_t W, int64_t Cout, int64_t G,
                     int64_t KH, int64_t KW, int64_t stride, int64_t pad, int64_t dil,
                     const float *x, const float *w, float *y, int mode, void *workspace,
                     size_t workspace_bytes, void *stream) {
    if (!workspace) return OM_ERR_NULL_PTR;
    const ConvArgs a{N, Cin, H, W, Cout, G, KH, KW, stride, pad, dil};
    return conv_impl(a, x, w, false, y, mode, workspace, workspace_bytes, stream);
}

int om_pack_conv_weights(int64_t Cout, int64_t Cin, int64_t G, int64_t KH, int64_t KW,
                         const float *w, float *w_packed, size_t *packed_bytes, void *stream) {
    if (Cout < 0 || Cin < 0 || G < 1 || KH < 1 || KW < 1) return OM_ERR_INVALID_ARG;
    if (Cin % G != 0 || Cout % G != 0) return OM_ERR_INVALID_ARG;
    if (KH > 65535 || KW > 65535) return OM_ERR_TOO_LARGE;
    const __int128 K = static_cast<__int128>(Cin / G) * KH * KW;
    if (K > (int64_t(1) << 31) - 1) return OM_ERR_TOO_LARGE;
    const int64_t Kp = (static_cast<int64_t>(K) + 3) / 4 * 4;
    const __int128 bytes = static_cast<__int128>(Cout) * Kp * 4;
    if (bytes >= (static_cast<__int128>(1) << 62)) return OM_ERR_TOO_LARGE;
    if (!w_packed) {
        if (!packed_bytes) return OM_ERR_NULL_PTR;
        *packed_bytes = static_cast<size_t>(bytes);
        return OM_OK;
    }
    if (packed_bytes) *packed_bytes = static_cast<size_t>(bytes);
    if (bytes == 0) return OM_OK;
    if (K > 0 && !w) return OM_ERR_NULL_PTR;
    if ((reinterpret_cast<uintptr_t>(w_packed) & 15) != 0 || !aligned4(w)) return OM_ERR_ALIGNMENT;
    const Range rp = span(w_packed, bytes / 4), rw = span(w, static_cast<__int128>(Cout) * K);
    if (K > 0 && overlaps(rp, rw)) return OM_ERR_ALIAS;
    return from_cuda(om::launch_pack_conv_weights(Cout, static_cast<int64_t>(K), Kp, w, w_packed,
                                                  static_cast<cudaStream_t>(stream)));
}

int om_conv2d_f32_packed(int64_t N, int64_t Cin, int64_t H, int64_t W, int64_t Cout, int64_t G,
                         int64_t KH, int64_t KW, int64_t stride, int64_t pad, int64_t dil,
                         const float *x, const float *w_packed, float *y, int mode,
                         void *stream) {
    const ConvArgs a{N, Cin, H, W, Cout, G, KH, KW, stride, pad, dil};
    return conv_impl(a, x, w_packed, true, y, mode, nullptr, 0, stream);
}

int om_conv2d_f32_packed_ws(int64_t N, int64_t Cin, int64_t H, int64_t W, int64_t Cout, int64_t G,
                            int64_t KH, int64_t KW, int64_t stride, int64_t pad, int64_t dil,
                            const float *x, const float *w_packed, float *y, int mode,
                            void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace) return OM_ERR_NULL_PTR;
    const ConvArgs a{N, Cin, H, W, Cout, G, KH, KW, stride, pad, dil};
    return conv_impl(a, x, w_packed, true, y, mode, workspace, workspace_bytes, stream);
}

int om_gemm_f32_ex(int64_t m, int64_t n, int64_t k, const float *A, int64_t lda,
                   const float *B, int64_t ldb, float *C, int64_t ldc, const float *bias,
                   const float *residual, int64_t ldr, int activation, int mode, void *workspace,
                   size_t workspace_bytes, void *stream) {
    const om::Epilogue ep{bias, residual, ldr, activation};
    return gemm_impl(m, n, k, A, lda, B, ldb, C, ldc, mode, workspace, workspace_bytes, stream, ep);
}

int om_conv2d_f32_ex(int64_t N, int64_t Cin, int64_t H, int64_t W, int64_t Cout, int64_t G,
                     int64_t KH, int64_t KW, int64_t stride, int64_t pad, int64_t dil,
                     const float *x, const float *w, int weights_packed, const float *bias,
                     const float *residual, int activation, float *y, int mode, void *workspace,
                     size_t workspace_bytes, void *stream) {
    const ConvArgs a{N, Cin, H, W, Cout, G, KH, KW, stride, pad, dil};
    const om::Epilogue ep{bias, residual, 0, activation};
    return conv_impl(a, x, w, weights_packed != 0, y, mode, workspace, workspace_bytes, stream, ep);
}

int om_device_status(void *stream) {
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned a = 0, b = 0, c = 0, d = 0, e = 0, f = 0, h = 0;
    if (om::read_clear_status_gemm(&a, s) != cudaSuccess) return OM_ERR_CUDA;
    if (om::read_clear_status_dw(&h, s) != cudaSuccess) return OM_ERR_CUDA;
    if (om::read_clear_status_rows(&f, s) != cudaSuccess) return OM_ERR_CUDA;
    if (om::read_clear_status_conv(&b, s) != cudaSuccess) return OM_ERR_CUDA;
    if (om::read_clear_status_tc(&c, s) != cudaSuccess) return OM_ERR_CUDA;
    if (om::read_clear_status_gemv(&d, s) != cudaSuccess) return OM_ERR_CUDA;
    if (om::read_clear_status_selftest(&e, s) != cudaSuccess) return OM_ERR_CUDA;
    return ((a | b | c | d | e | f | h) & om::kDevErrTimeoutHost) ? OM_ERR_TIMEOUT : OM_OK;
}

int om_selftest_wait_timeout(int which, int limit_ms, void *stream) {
    if ((which != 0 && which != 1) || limit_ms < 1 || limit_ms > 1000) return OM_ERR_INVALID_ARG;
    return from_cuda(om::launch_wait_timeout(which, limit_ms, nullptr, static_cast<cudaStream_t>(stream)));
}

int om_selftest_wait_timeout_ws(int which, int limit_ms, void *workspace, size_t workspace_bytes,
                                void *stream) {
    if ((which != 0 && which != 1) || limit_ms < 1 || limit_ms > 1000) return OM_ERR_INVALID_ARG;
    if (!workspace) return OM_ERR_NULL_PTR;
    unsigned *flags = nullptr;
    const int wst = check_workspace(workspace, workspace_bytes, &flags);
    if (wst != OM_OK) return wst;
    return from_cuda(om::launch_wait_timeout(which, limit_ms, ws_status(flags), static_cast<cudaStream_t>(stream)));
}

int om_workspace_status(void *workspace, size_t workspace_bytes, void *stream) {
    if (!workspace) return OM_ERR_NULL_PTR;
    unsigned *flags = nullptr;
    const int wst = check_workspace(workspace, workspace_bytes, &flags);
    if (wst != OM_OK) return wst;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    unsigned word = 0;
    if (cudaMemcpyAsync(&word, ws_status(flags), sizeof(unsigned), cudaMemcpyDeviceToHost, s) != cudaSuccess)
        return OM_ERR_CUDA;
    if (cudaStreamSynchronize(s) != cudaSuccess) return OM_ERR_CUDA;
    if (word != 0) {
        if (cudaMemsetAsync(ws_status(flags), 0, sizeof(unsigned), s) != cudaSuccess) return OM_ERR_CUDA;
        if (cudaStreamSynchronize(s) != cudaSuccess) return OM_ERR_CUDA;
    }
    return (word & om::kDevErrTimeoutHost) ? OM_ERR_TIMEOUT : OM_OK;
}

}  // extern "C"
