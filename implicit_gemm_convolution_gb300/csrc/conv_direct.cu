// Direct convolution for groups with few output channels: depthwise
// (Cin/G = 1) and grouped convolutions with at most 32 output channels per
// group.
//
// The implicit-GEMM kernel tiles 64 output channels; a group with M = Cout/G
// of 8 would leave seven eighths of every tile idle, and a depthwise layer
// (K = KH*KW) has too little reuse to feed it. Here a block owns one group of
// one image and a band of output rows. It copies the input rows the band
// reads, for the group's channels, into shared memory with the zero border
// written at copy time (the pages' padding at gather time), then each thread
// computes all M output channels of a few pixels of the band from there,
// with the group's weights broadcast from shared memory.
//
// Each output is still the pages' per-output loop: one accumulator from +0,
// taps in (channel, kernel row, kernel column) order, the product formed at
// every tap (an input position outside the plane contributes w * (+0)),
// exact mode rounding the product and the sum separately, fast mode one
// fused multiply-add (OneModel operators page, "Convolution"; the depthwise
// workload of the convolution page).

#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "om_device.cuh"
#include "om_internal.h"

namespace om {
namespace {

constexpr int kDirectThreads = 128;
// Shared memory of one block: weights, tap table and input window.
constexpr int64_t kDirectWindowBytes = 64 * 1024;

struct DirectGeom {
    const float *x;
    const float *w;
    float *y;
    int H, W, HW, OH, OW, P;
    int Cin, Cout, cin_g, M, K, w_ld;
    int KH, KW, sH, sW, pT, pL, dH, dW;
    int R;       // output rows per band
    int WR, Wp;  // window rows (for R output rows) and columns
    int wfloats, tints;  // weight floats and table ints, each a multiple of 4
    int wshift;          // depthwise window: column j holds input column j - wshift
    int R_chunk;         // few-pixel kernel: input channels per chunk
    int ch_win, ch_w;    // few-pixel kernel: window and weight floats of one chunk buffer
    uint32_t plane_magic;  // few-pixel kernel: floor(2^32 / (WR*Wp)) + 1
    Epilogue ep;
};

// Adds one tap's products w[oc] * v for the MB output channels of a pixel.
template <int MODE, int MB>
__device__ __forceinline__ void direct_tap(float2 (&acc)[(MB + 1) / 2], float &acc1,
                                           const float *wt, float v) {
    if constexpr (MB == 1) {
        acc1 = term<MODE>(acc1, wt[0], v);
    } else if constexpr (MB == 2) {
        const float2 w2 = *reinterpret_cast<const float2 *>(wt);
        acc[0] = term2<MODE>(acc[0], w2, make_float2(v, v));
    } else {
        const float2 v2 = make_float2(v, v);
#pragma unroll
        for (int q = 0; q < MB / 4; ++q) {
            const float4 w4 = reinterpret_cast<const float4 *>(wt)[q];
            acc[2 * q] = term2<MODE>(acc[2 * q], make_float2(w4.x, w4.y), v2);
            acc[2 * q + 1] = term2<MODE>(acc[2 * q + 1], make_float2(w4.z, w4.w), v2);
        }
    }
}

// Grid: x over bands of R output rows, y over groups, z over images.
// Shared memory: the group's weights tap-major (MB per tap, +0 for channels
// past M); per tap its window offset c*WR*Wp + ky*dH*Wp + kx*dW; the window,
// channel-major, WR rows of Wp columns, column j holding input column
// j - pL (+0 outside the plane); then PX*sW floats of slack that only lanes
// past the last output column read.
// Thread pixels: unit (row r, q) covers columns q, q + QX, ... (QX =
// ceil(OW/PX)), so neighbouring lanes read neighbouring window columns.
template <int MODE, int MB, int PX>
__global__ void __launch_bounds__(kDirectThreads) conv_direct_kernel(const DirectGeom g) {
    extern __shared__ float4 smem4[];
    float *wsm = reinterpret_cast<float *>(smem4);
    int *tab = reinterpret_cast<int *>(wsm + g.wfloats);
    float *win = reinterpret_cast<float *>(tab + g.tints);
    const int grp = blockIdx.y;
    const int64_t img = blockIdx.z;
    const int oy0 = blockIdx.x * g.R;
    const int rows = min(g.R, g.OH - oy0);
    const int wr = (rows - 1) * g.sH + (g.KH - 1) * g.dH + 1;  // window rows this band reads
    const int iy_base = oy0 * g.sH - g.pT;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    // input window, zero border written here
    const float *xg = g.x + (img * g.Cin + static_cast<int64_t>(grp) * g.cin_g) * g.HW;
    const uint32_t win32 = smem_u32(win);
    for (int c = 0; c < g.cin_g; ++c) {
        const float *xc = xg + static_cast<int64_t>(c) * g.HW - g.pL;
        for (int r = warp; r < wr; r += kDirectThreads / 32) {
            const int iy = iy_base + r;
            const bool row_ok = static_cast<unsigned>(iy) < static_cast<unsigned>(g.H);
            const float *xrow = xc + static_cast<int64_t>(iy) * g.W;
            const uint32_t drow = win32 + static_cast<uint32_t>((c * g.WR + r) * g.Wp) * 4u;
            for (int j = lane; j < g.Wp; j += 32) {
                const int ix = j - g.pL;
                const bool ok = row_ok && static_cast<unsigned>(ix) < static_cast<unsigned>(g.W);
                cp_async_4_if(drow + j * 4u, ok ? xrow + j : g.x, ok);
            }
        }
    }
    for (int i = tid; i < g.K * MB; i += kDirectThreads) {
        const int t = i / MB, oc = i - (i / MB) * MB;
        wsm[i] = oc < g.M ? g.w[static_cast<int64_t>(grp * g.M + oc) * g.w_ld + t] : 0.0f;
    }
    const int taps = g.KH * g.KW;
    for (int t = tid; t < g.K; t += kDirectThreads) {
        const int c = t / taps, rr = t - (t / taps) * taps;
        const int ky = rr / g.KW, kx = rr - (rr / g.KW) * g.KW;
        tab[t] = (c * g.WR + ky * g.dH) * g.Wp + kx * g.dW;
    }
    cp_async_wait_all();
    __syncthreads();

    const int qx = (g.OW + PX - 1) / PX;
    for (int u = tid; u < rows * qx; u += kDirectThreads) {
        const int ry = u / qx, q = u - (u / qx) * qx;
        const float *wb = win + ry * g.sH * g.Wp + q * g.sW;
        float2 acc[PX][(MB + 1) / 2];
        float acc1[PX];
#pragma unroll
        for (int j = 0; j < PX; ++j) {
            acc1[j] = 0.0f;
#pragma unroll
            for (int h = 0; h < (MB + 1) / 2; ++h) acc[j][h] = make_float2(0.0f, 0.0f);
        }
        const int step = qx * g.sW;  // window columns between the thread's pixels
#pragma unroll 2
        for (int t = 0; t < g.K; ++t) {
            const float *src = wb + tab[t];
            const float *wt = wsm + t * MB;
#pragma unroll
            for (int j = 0; j < PX; ++j) direct_tap<MODE, MB>(acc[j], acc1[j], wt, src[j * step]);
        }
        const int oy = oy0 + ry;
        float *yp = g.y + (img * g.Cout + static_cast<int64_t>(grp) * g.M) * g.P +
                    static_cast<int64_t>(oy) * g.OW + q;
        const bool ep = g.ep.bias || g.ep.res || g.ep.act;
#pragma unroll
        for (int j = 0; j < PX; ++j) {
            if (q + j * qx >= g.OW) break;
#pragma unroll
            for (int oc = 0; oc < MB; ++oc) {
                if (oc < g.M) {
                    float v = MB == 1 ? acc1[j] : ((oc & 1) ? acc[j][oc / 2].y : acc[j][oc / 2].x);
                    float *o = yp + static_cast<int64_t>(oc) * g.P + j * qx;
                    if (ep)
                        v = epilogue_value(v, g.ep.bias ? g.ep.bias + grp * g.M + oc : nullptr,
                                           g.ep.res ? g.ep.res + (o - g.y) : nullptr, g.ep.act);
                    *o = canonical_nan(v);
                }
            }
        }
    }
}

// ------------------------------------------------------- few output pixels
// Convolutions with many output channels and few output pixels (a late
// layer at a small batch: 512 channels of 7 x 7 outputs), where the
// implicit-GEMM tiles would leave most SMs idle and k cannot be split. A
// block owns MB output channels of one group, one image and a band of output
// rows with at most kSkinnyThreads pixels; each thread owns one pixel and
// its MB outputs for the whole k loop. The group's input channels stream
// through shared memory in chunks of CC channels (window rows with the zero
// border written at copy time, the chunk's weights), double-buffered with
// cp.async groups so the next chunk's copy overlaps this chunk's taps. Taps
// run chunk by chunk, in (c, ky, kx) order within a chunk: the pages' one
// sequential loop per output.
constexpr int kSkinnyThreads = 128;

template <int MODE, int MB>
__global__ void __launch_bounds__(kSkinnyThreads) conv_skinny_kernel(const DirectGeom g) {
    extern __shared__ float4 smem4[];
    float *base = reinterpret_cast<float *>(smem4);
    const int buf_floats = g.ch_win + g.ch_w;  // window + weights of one buffer (multiples of 4)
    int *tab = reinterpret_cast<int *>(base + 2 * buf_floats);
    int *ftab = tab + g.R_chunk * g.KH * g.KW;  // per window element of a channel: input offset or -1
    const int mblocks = (g.M + MB - 1) / MB;
    const int grp = blockIdx.y / mblocks;
    const int oc0 = (blockIdx.y - grp * mblocks) * MB;
    const int64_t img = blockIdx.z;
    const int oy0 = blockIdx.x * g.R;
    const int rows = min(g.R, g.OH - oy0);
    const int wr = (rows - 1) * g.sH + (g.KH - 1) * g.dH + 1;
    const int iy_base = oy0 * g.sH - g.pT;
    const int tid = threadIdx.x;
    const int taps = g.KH * g.KW;
    const int cc_max = g.R_chunk;  // channels per chunk
    const int nchunks = (g.cin_g + cc_max - 1) / cc_max;

    // tap table of a chunk: offset of (c, ky, kx) in the chunk's window
    for (int t = tid; t < cc_max * taps; t += kSkinnyThreads) {
        const int c = t / taps, rr = t - (t / taps) * taps;
        const int ky = rr / g.KW, kx = rr - (rr / g.KW) * g.KW;
        tab[t] = (c * g.WR + ky * g.dH) * g.Wp + kx * g.dW;
    }
    // window element (r, j) of a channel: input offset iy*W + ix of the
    // band's plane position, or -1 outside the plane (and past this band's rows)
    const int plane = g.WR * g.Wp;
    for (int e = tid; e < plane; e += kSkinnyThreads) {
        const int r = e / g.Wp, j = e - (e / g.Wp) * g.Wp;
        const int iy = iy_base + r, ix = j - g.pL;
        const bool ok = r < wr && static_cast<unsigned>(iy) < static_cast<unsigned>(g.H) &&
                        static_cast<unsigned>(ix) < static_cast<unsigned>(g.W);
        ftab[e] = ok ? iy * g.W + ix : -1;
    }
    __syncthreads();
    const float *xg = g.x + (img * g.Cin + static_cast<int64_t>(grp) * g.cin_g) * g.HW;
    const float *wg = g.w + static_cast<int64_t>(grp * g.M + oc0) * g.w_ld;
    const uint32_t magic = g.plane_magic;  // e / plane == umulhi(e, magic) for e, plane < 2^16
    auto load_chunk = [&](int ch, int b) {
        float *win = base + b * buf_floats;
        float *wsm = win + g.ch_win;
        const uint32_t win32 = smem_u32(win), w32 = smem_u32(wsm);
        const int c0 = ch * cc_max, cc = min(cc_max, g.cin_g - c0);
        const float *xc0 = xg + static_cast<int64_t>(c0) * g.HW;
        for (int e = tid; e < cc * plane; e += kSkinnyThreads) {
            const int c = static_cast<int>(__umulhi(static_cast<uint32_t>(e), magic));
            const int off = ftab[e - c * plane];
            const bool ok = off >= 0;
            cp_async_4_if(win32 + e * 4u, ok ? xc0 + (static_cast<int64_t>(c) * g.HW + off) : g.x, ok);
        }
        // weights: tap t of the chunk for channel oc at wsm[t*MB + oc], +0 past M
        const int ntap = cc * taps;
        for (int i = tid; i < ntap * MB; i += kSkinnyThreads) {
            const int t = i / MB, oc = i - (i / MB) * MB;
            const bool ok = oc0 + oc < g.M;
            cp_async_4_if(w32 + i * 4u, ok ? wg + static_cast<int64_t>(oc) * g.w_ld + c0 * taps + t : g.w, ok);
        }
        asm volatile("cp.async.commit_group;" ::: "memory");
    };

    const int ry = tid / g.OW, ox = tid - (tid / g.OW) * g.OW;
    const bool active = tid < rows * g.OW;
    const int woff = (ry * g.sH) * g.Wp + ox * g.sW;
    float2 acc[(MB + 1) / 2];
    float acc1 = 0.0f;
#pragma unroll
    for (int h = 0; h < (MB + 1) / 2; ++h) acc[h] = make_float2(0.0f, 0.0f);

    load_chunk(0, 0);
    for (int ch = 0; ch < nchunks; ++ch) {
        const int b = ch & 1;
        if (ch + 1 < nchunks) {
            load_chunk(ch + 1, b ^ 1);
            asm volatile("cp.async.wait_group 1;" ::: "memory");
        } else {
            asm volatile("cp.async.wait_group 0;" ::: "memory");
        }
        __syncthreads();
        if (active) {
            const float *win = base + b * buf_floats;
            const float *wsm = win + g.ch_win;
            const int ntap = min(cc_max, g.cin_g - ch * cc_max) * taps;
            const float *src = win + woff;
#pragma unroll 4
            for (int t = 0; t < ntap; ++t) direct_tap<MODE, MB>(acc, acc1, wsm + t * MB, src[tab[t]]);
        }
        __syncthreads();  // the buffer is refilled two chunks on
    }
    if (!active) return;
    const int oy = oy0 + ry;
    float *yp = g.y + (img * g.Cout + static_cast<int64_t>(grp) * g.M + oc0) * g.P +
                static_cast<int64_t>(oy) * g.OW + ox;
    const bool ep = g.ep.bias || g.ep.res || g.ep.act;
#pragma unroll
    for (int oc = 0; oc < MB; ++oc) {
        if (oc0 + oc < g.M) {
            float v = MB == 1 ? acc1 : ((oc & 1) ? acc[oc / 2].y : acc[oc / 2].x);
            float *o = yp + static_cast<int64_t>(oc) * g.P;
            if (ep)
                v = epilogue_value(v, g.ep.bias ? g.ep.bias + grp * g.M + oc0 + oc : nullptr,
                                   g.ep.res ? g.ep.res + (o - g.y) : nullptr, g.ep.act);
            *o = canonical_nan(v);
        }
    }
}

// ------------------------------------------------------- depthwise KSxKS
// One input channel and one output channel per group (a depthwise layer
// with multiplier 1), a KS x KS kernel, stride SW on both axes, dilation 1.
// A block owns one channel of one image and a band of R output rows; its
// window holds the input rows the band reads, with the zero border, in rows
// of Wp floats (a multiple of 4, so 16-byte loads stay aligned). Each thread
// computes 8 consecutive outputs of one row: per kernel row it loads the
// 8*SW + KS - 1 window values those outputs read (as 16-byte loads) and the
// kernel row's weights come from registers, so each output's taps run in
// (ky, kx) order from +0 with one multiply-add (or multiply, add) apiece.
// The outputs are staged in shared memory and stored in one coalesced pass
// (a band's rows are contiguous in y), with the epilogue applied there.
constexpr int kDwRun = 8;  // outputs per thread
// Shared memory per depthwise block: about 12 blocks per SM, whose overlap
// hides the window copy's latency (measured: 18 KB bands beat 12, 28 and
// 64 KB ones on a 56 x 56 layer).
constexpr int64_t kDwBlockBytes = 18 * 1024;

template <int MODE, int KS, int SW, bool VEC, int C0>
__global__ void __launch_bounds__(kDirectThreads) conv_dw_kernel(const DirectGeom g) {
    constexpr int NV = kDwRun * SW + KS - 1;  // window values per kernel row and run
    constexpr int NL = (C0 + NV + 3) / 4;     // 16-byte loads covering them
    extern __shared__ float4 smem4[];
    float *win = reinterpret_cast<float *>(smem4);
    const int ch = blockIdx.y;
    const int64_t img = blockIdx.z;
    const int oy0 = blockIdx.x * g.R;
    const int rows = min(g.R, g.OH - oy0);
    const int wr = (rows - 1) * SW + KS;
    const int iy_base = oy0 * SW - g.pT;
    const int tid = threadIdx.x, warp = tid / 32, lane = tid % 32;

    // window: column j holds input column j - shift (shift = pL, or pL
    // rounded up to 4 so that 16-byte copies stay aligned); +0 outside
    const int shift = g.wshift;
    const float *xc = g.x + (img * g.Cin + ch) * static_cast<int64_t>(g.HW) - shift;
    const uint32_t win32 = smem_u32(win);
    constexpr int kStep = VEC ? 4 : 1;
    for (int r = warp; r < wr; r += kDirectThreads / 32) {
        const int iy = iy_base + r;
        const bool row_ok = static_cast<unsigned>(iy) < static_cast<unsigned>(g.H);
        const float *xrow = xc + static_cast<int64_t>(iy) * g.W;
        const uint32_t drow = win32 + static_cast<uint32_t>(r * g.Wp) * 4u;
        for (int j = lane * kStep; j < g.Wp; j += 32 * kStep) {
            const int ix = j - shift;
            const bool ok = row_ok && static_cast<unsigned>(ix) < static_cast<unsigned>(g.W);
            if constexpr (VEC)
                cp_async_16(drow + j * 4u, ok ? xrow + j : g.x, ok ? 16u : 0u);
            else
                cp_async_4_if(drow + j * 4u, ok ? xrow + j : g.x, ok);
        }
    }
    float wk[KS * KS];
#pragma unroll
    for (int t = 0; t < KS * KS; ++t) wk[t] = __ldg(g.w + static_cast<int64_t>(ch) * g.w_ld + t);
    cp_async_wait_all();
    __syncthreads();

    // outputs of the band are staged in shared memory (row pitch OW when
    // VEC, else OW rounded up to 8) and leave in one coalesced pass
    const int qx = (g.OW + kDwRun - 1) / kDwRun;
    const int pitch = VEC ? g.OW : qx * kDwRun;
    // window column of output 0's tap kx = 0 is C0 = shift - pL
    float *stage = win + g.WR * g.Wp;
    for (int u = tid; u < rows * qx; u += kDirectThreads) {
        const int ry = u / qx, ox0 = (u - (u / qx) * qx) * kDwRun;
        float acc[kDwRun];
#pragma unroll
        for (int j = 0; j < kDwRun; ++j) acc[j] = 0.0f;
#pragma unroll
        for (int ky = 0; ky < KS; ++ky) {
            const float4 *src = reinterpret_cast<const float4 *>(win + (ry * SW + ky) * g.Wp + ox0 * SW);
            float v[4 * NL];
#pragma unroll
            for (int q = 0; q < NL; ++q) {
                const float4 f = src[q];
                v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
            }
#pragma unroll
            for (int kx = 0; kx < KS; ++kx)
#pragma unroll
                for (int j = 0; j < kDwRun; ++j)
                    acc[j] = term<MODE>(acc[j], wk[ky * KS + kx], v[C0 + j * SW + kx]);
        }
        float4 *dst = reinterpret_cast<float4 *>(stage + ry * pitch + ox0);
        dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
        if (!VEC || ox0 + 4 < g.OW) dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
    }
    __syncthreads();
    // the band's outputs are rows oy0 .. oy0 + rows - 1 of the channel plane:
    // one contiguous run of rows * OW floats in y
    const int64_t ybase = (img * g.Cout + ch) * static_cast<int64_t>(g.P) + static_cast<int64_t>(oy0) * g.OW;
    const bool ep = g.ep.bias || g.ep.res || g.ep.act;
    const float *bias = g.ep.bias ? g.ep.bias + ch : nullptr;
    if constexpr (VEC) {
        const float4 *st4 = reinterpret_cast<const float4 *>(stage);
        float4 *y4 = reinterpret_cast<float4 *>(g.y + ybase);
        for (int i = tid; i < rows * g.OW / 4; i += kDirectThreads) {
            float4 v = st4[i];
            if (ep) {
                const float *res = g.ep.res ? g.ep.res + ybase + 4 * i : nullptr;
                v.x = epilogue_value(v.x, bias, res, g.ep.act);
                v.y = epilogue_value(v.y, bias, res ? res + 1 : nullptr, g.ep.act);
                v.z = epilogue_value(v.z, bias, res ? res + 2 : nullptr, g.ep.act);
                v.w = epilogue_value(v.w, bias, res ? res + 3 : nullptr, g.ep.act);
            }
            y4[i] = make_float4(canonical_nan(v.x), canonical_nan(v.y), canonical_nan(v.z), canonical_nan(v.w));
        }
    } else {
        for (int i = tid; i < rows * g.OW; i += kDirectThreads) {
            const int ry = i / g.OW, ox = i - (i / g.OW) * g.OW;
            float v = stage[ry * pitch + ox];
            if (ep) v = epilogue_value(v, bias, g.ep.res ? g.ep.res + ybase + i : nullptr, g.ep.act);
            g.y[ybase + i] = canonical_nan(v);
        }
    }
}

template <int MODE, int KS, int SW, bool VEC, int C0>
cudaError_t launch_dw(const DirectGeom &g, int64_t channels, int64_t images, size_t smem, cudaStream_t s) {
    auto kernel = conv_dw_kernel<MODE, KS, SW, VEC, C0>;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>((g.OH + g.R - 1) / g.R), static_cast<unsigned>(channels),
                    static_cast<unsigned>(images));
    kernel<<<grid, kDirectThreads, smem, s>>>(g);
    return cudaGetLastError();
}

// Instantiated: 4-byte window copies with the window starting at the left
// padding (C0 = 0), and 16-byte copies with the usual "same" paddings, 1 for
// 3 x 3 (C0 = 3) and 2 for 5 x 5 (C0 = 2), or none (C0 = 0).
template <int MODE>
cudaError_t launch_dw_mode(const DirectGeom &g, int ks, int sw, bool vec, int c0, int64_t channels,
                           int64_t images, size_t smem, cudaStream_t s) {
#define OM_DW(K, S, V, C)                                   \
    if (ks == K && sw == S && vec == V && c0 == C)          \
        return launch_dw<MODE, K, S, V, C>(g, channels, images, smem, s);
    OM_DW(3, 1, false, 0) OM_DW(3, 2, false, 0) OM_DW(5, 1, false, 0) OM_DW(5, 2, false, 0)
    OM_DW(3, 1, true, 0) OM_DW(3, 2, true, 0) OM_DW(5, 1, true, 0) OM_DW(5, 2, true, 0)
    OM_DW(3, 1, true, 3) OM_DW(3, 2, true, 3) OM_DW(5, 1, true, 2) OM_DW(5, 2, true, 2)
#undef OM_DW
    return cudaErrorNotSupported;
}

template <int MODE, int MB, int PX>
cudaError_t launch_direct(const DirectGeom &g, int64_t groups, int64_t images, size_t smem,
                          cudaStream_t s) {
    auto kernel = conv_direct_kernel<MODE, MB, PX>;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    const dim3 grid(static_cast<unsigned>((g.OH + g.R - 1) / g.R), static_cast<unsigned>(groups),
                    static_cast<unsigned>(images));
    kernel<<<grid, kDirectThreads, smem, s>>>(g);
    return cudaGetLastError();
}

// Pixels per thread PX (1, 2, 4 or 8): up to 32 accumulators (PX * MB) per thread.
template <int MODE, int MB>
cudaError_t launch_direct_px(const DirectGeom &g, int64_t groups, int64_t images, int px,
                             size_t smem, cudaStream_t s) {
    if constexpr (MB <= 4) {
        if (px == 8) return launch_direct<MODE, MB, 8>(g, groups, images, smem, s);
    }
    if constexpr (MB <= 8) {
        if (px == 4) return launch_direct<MODE, MB, 4>(g, groups, images, smem, s);
    }
    if constexpr (MB <= 16) {
        if (px == 2) return launch_direct<MODE, MB, 2>(g, groups, images, smem, s);
    }
    return launch_direct<MODE, MB, 1>(g, groups, images, smem, s);
}

template <int MODE>
cudaError_t launch_direct_mode(const DirectGeom &g, int64_t groups, int64_t images, int mb, int px,
                               size_t smem, cudaStream_t s) {
    switch (mb) {
        case 1: return launch_direct_px<MODE, 1>(g, groups, images, px, smem, s);
        case 2: return launch_direct_px<MODE, 2>(g, groups, images, px, smem, s);
        case 4: return launch_direct_px<MODE, 4>(g, groups, images, px, smem, s);
        case 8: return launch_direct_px<MODE, 8>(g, groups, images, px, smem, s);
        case 16: return launch_direct_px<MODE, 16>(g, groups, images, px, smem, s);
        case 32: return launch_direct_px<MODE, 32>(g, groups, images, px, smem, s);
        default: return cudaErrorNotSupported;
    }
}

template <int MODE, int MB>
cudaError_t launch_skinny(const DirectGeom &g, int64_t bands, int64_t gy, int64_t images, size_t smem,
                          cudaStream_t s) {
    auto kernel = conv_skinny_kernel<MODE, MB>;
    const cudaError_t e =
        cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    kernel<<<dim3(static_cast<unsigned>(bands), static_cast<unsigned>(gy), static_cast<unsigned>(images)),
             kSkinnyThreads, smem, s>>>(g);
    return cudaGetLastError();
}

template <int MODE>
cudaError_t launch_skinny_mb(const DirectGeom &g, int mb, int64_t bands, int64_t gy, int64_t images,
                             size_t smem, cudaStream_t s) {
    switch (mb) {
        case 1: return launch_skinny<MODE, 1>(g, bands, gy, images, smem, s);
        case 2: return launch_skinny<MODE, 2>(g, bands, gy, images, smem, s);
        case 4: return launch_skinny<MODE, 4>(g, bands, gy, images, smem, s);
        case 8: return launch_skinny<MODE, 8>(g, bands, gy, images, smem, s);
        case 16: return launch_skinny<MODE, 16>(g, bands, gy, images, smem, s);
        default: return cudaErrorNotSupported;
    }
}

// ---- depthwise KS x KS, "same" padding, stride 1 or 2, from a TMA window.
// A block owns a band of RB output rows of one channel of one image. One
// 4-D TMA copy (columns, rows, one channel, one image) brings the band's
// input window into shared memory (rows 4 (mod 32) floats wide); the box
// starts left of and above the plane as the padding needs and TMA writes +0
// for every element outside it
// (the zero border at copy time). Blocks are persistent: each walks its
// (image, channel, band) items with kDwTmaStages window copies in flight, so
// the copies of the next bands overlap this band's work. Thread s computes
// the 8 consecutive
// outputs of one strip of the band (row s % rows, columns 8 * (s / rows) ..): per
// kernel row, 16-byte window loads and KS * 8 multiply-adds in (ky, kx)
// order from +0, the weights in registers; the band's outputs are staged in
// shared memory and leave in one coalesced pass with the epilogue.
__device__ unsigned g_status_dw;

struct DwTmaGeom {
    float *y;
    const float *w;
    int OH, OW, Cout, w_ld;
    int RB;    // output rows per band
    int SPR;   // strips of 8 outputs per output row
    int x0;    // first window column (a multiple of 4)
    int BW, BH;
    int N, bands;
    int step_b, step_c, step_i;  // the grid size in (band, channel, image) digits
    Epilogue ep;
    unsigned *status;  // the call's status word in a caller workspace, or NULL
};

constexpr int kDwTmaMaxThreads = 512;
constexpr int kDwTmaStages = 3;  // window copies in flight per block

template <int MODE, int KS, int SW, int PAD>
__global__ void __launch_bounds__(kDwTmaMaxThreads) conv_dw_tma_kernel(const __grid_constant__ CUtensorMap map,
                                                                       const DwTmaGeom g) {
    // window column of output column 0, kernel column 0: -PAD - x0; its
    // offset in the 16-byte chunk every strip starts at
    constexpr int kX0 = -4 * ((PAD + 3) / 4);
    constexpr int C0 = -PAD - kX0;
    constexpr int NV = 7 * SW + KS;             // window values of a strip's row
    constexpr int NL = (C0 + NV + 3) / 4;       // 16-byte loads covering them
    extern __shared__ uint8_t dw_raw[];
    __shared__ uint64_t full[kDwTmaStages];
    __shared__ int stop_sh;  // a window copy never landed: every thread leaves
    uint8_t *ring = dw_raw + ((128u - (smem_u32(dw_raw) & 127u)) & 127u);
    const uint32_t box_bytes = static_cast<uint32_t>(g.BW * g.BH) * 4u;
    const uint32_t stage_bytes = (box_bytes + 127u) / 128u * 128u;
    float *outs = reinterpret_cast<float *>(ring + kDwTmaStages * stage_bytes);  // RB x (OW + 4)
    // items (image, channel, band), band fastest; this block takes
    // blockIdx.x, blockIdx.x + gridDim.x, ... Item numbers advance by the
    // grid size in mixed radix (band, channel, image), so no division is
    // needed per item.
    const int items = g.N * g.Cout * g.bands;
    const int mine = static_cast<int>(blockIdx.x) < items
                         ? (items - 1 - static_cast<int>(blockIdx.x)) / static_cast<int>(gridDim.x) + 1
                         : 0;
    const int b0 = static_cast<int>(blockIdx.x) % g.bands;
    const int c0 = (static_cast<int>(blockIdx.x) / g.bands) % g.Cout;
    const int i0 = static_cast<int>(blockIdx.x) / (g.bands * g.Cout);
    // the copy cursor (thread 0) runs kDwTmaStages items ahead of the compute cursor
    int qb = b0, qc = c0, qi = i0;
    auto advance = [&](int &b, int &c, int &i) {
        b += g.step_b;
        int carry = b >= g.bands;
        b -= carry ? g.bands : 0;
        c += g.step_c + carry;
        carry = c >= g.Cout;
        c -= carry ? g.Cout : 0;
        i += g.step_i + carry;
    };
    auto issue = [&](int j) {
        const int st = j % kDwTmaStages;
        mbar_arrive_expect_tx(&full[st], box_bytes);
        tma_load_4d(ring + st * stage_bytes, &map, &full[st], kX0, qb * g.RB * SW - PAD, qc, qi);
        advance(qb, qc, qi);
    };
    if (threadIdx.x == 0) {
        for (int st = 0; st < kDwTmaStages; ++st) mbar_init(&full[st], 1);
        stop_sh = 0;
        fence_mbar_init();
        for (int j = 0; j < kDwTmaStages && j < mine; ++j) issue(j);
    }
    __syncthreads();
    const int s = threadIdx.x;
    // this thread's strip in a full band and in the last band (which may be
    // shorter): lanes take consecutive rows of one strip column, so window
    // rows 4 (mod 32) floats apart put a quarter-warp's 16-byte loads on
    // distinct banks
    const int rows_last = g.OH - (g.bands - 1) * g.RB;
    const int seg_f = s / g.RB, ry_f = s - seg_f * g.RB;
    const int seg_l = s / rows_last, ry_l = s - seg_l * rows_last;
    int cb = b0, cc = c0, ci = i0;
    for (int j = 0; j < mine; ++j) {
        const bool last_band = cb == g.bands - 1;
        const int rows = last_band ? rows_last : g.RB;
        const int oy0 = cb * g.RB;
        const int st = j % kDwTmaStages;
        const bool landed = mbar_wait(&full[st], static_cast<uint32_t>((j / kDwTmaStages) & 1));
        if (!landed) atomicOr(&stop_sh, 1);
        if (landed && s < rows * g.SPR) {
            float wk[KS * KS];
#pragma unroll
            for (int t = 0; t < KS * KS; ++t) wk[t] = __ldg(g.w + static_cast<int64_t>(cc) * g.w_ld + t);
            const float *win = reinterpret_cast<const float *>(ring + st * stage_bytes);
            const int ry = last_band ? ry_l : ry_f;
            const int ox0 = (last_band ? seg_l : seg_f) * 8;
            float acc[8];
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
#pragma unroll
            for (int ky = 0; ky < KS; ++ky) {
                const float4 *src = reinterpret_cast<const float4 *>(win + (ry * SW + ky) * g.BW + ox0 * SW);
                float v[4 * NL];
#pragma unroll
                for (int q = 0; q < NL; ++q) {
                    const float4 f = src[q];
                    v[4 * q] = f.x; v[4 * q + 1] = f.y; v[4 * q + 2] = f.z; v[4 * q + 3] = f.w;
                }
#pragma unroll
                for (int kx = 0; kx < KS; ++kx)
#pragma unroll
                    for (int q = 0; q < 8; ++q) acc[q] = term<MODE>(acc[q], wk[ky * KS + kx], v[C0 + q * SW + kx]);
            }
            // staged by output row (pitch OW + 4 floats: a quarter-warp's
            // rows on distinct banks); the band leaves in one coalesced pass
            float4 *stg = reinterpret_cast<float4 *>(outs + ry * (g.OW + 4) + ox0);
            stg[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            stg[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
        }
        __syncthreads();
        if (landed) {
            // the band's output rows oy0 .. oy0 + rows - 1 are one contiguous
            // run of rows * OW floats in y
            const int64_t ybase = ((static_cast<int64_t>(ci) * g.Cout + cc) * g.OH + oy0) * g.OW;
            const int q4 = g.OW / 4;
            const float *bias = g.ep.bias ? g.ep.bias + cc : nullptr;
            const bool ep = g.ep.bias || g.ep.res || g.ep.act;
            for (int e = s; e < rows * q4; e += blockDim.x) {
                const int r = e / q4, c4 = e - r * q4;
                float4 v = *reinterpret_cast<const float4 *>(outs + r * (g.OW + 4) + 4 * c4);
                const int64_t o = ybase + static_cast<int64_t>(e) * 4;
                if (ep) {
                    const float *res = g.ep.res ? g.ep.res + o : nullptr;
                    v.x = epilogue_value(v.x, bias, res, g.ep.act);
                    v.y = epilogue_value(v.y, bias, res ? res + 1 : nullptr, g.ep.act);
                    v.z = epilogue_value(v.z, bias, res ? res + 2 : nullptr, g.ep.act);
                    v.w = epilogue_value(v.w, bias, res ? res + 3 : nullptr, g.ep.act);
                }
                *reinterpret_cast<float4 *>(g.y + o) =
                    make_float4(canonical_nan(v.x), canonical_nan(v.y), canonical_nan(v.z), canonical_nan(v.w));
            }
        }
        advance(cb, cc, ci);
        // every thread's reads of this stage and of the staged outputs are
        // done: hand the stage to the copy engine for the item kDwTmaStages
        // ahead
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(&stop_sh)) {
            // copies still in flight land (or give up) before the block leaves
            if (threadIdx.x == 0) {
                report_timeout(g.status, &g_status_dw);
                for (int jj = j; jj < mine && jj < j + kDwTmaStages; ++jj)
                    (void)mbar_wait_limit(&full[jj % kDwTmaStages],
                                          static_cast<uint32_t>((jj / kDwTmaStages) & 1), 1000000ull);
            }
            return;
        }
        if (threadIdx.x == 0 && j + kDwTmaStages < mine) {
            fence_proxy_async_smem();
            issue(j + kDwTmaStages);
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 dw_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

template <int MODE, int KS, int SW, int PAD>
cudaError_t launch_dw_tma(const CUtensorMap &map, const DwTmaGeom &g, int threads, int smem, cudaStream_t s) {
    auto kernel = conv_dw_tma_kernel<MODE, KS, SW, PAD>;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    int per_sm = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, threads, smem);
    if (e != cudaSuccess) return e;
    if (per_sm < 1) return cudaErrorNotSupported;
    const int64_t items = static_cast<int64_t>(g.N) * g.Cout * g.bands;
    int64_t grid = static_cast<int64_t>(num_sms()) * per_sm;
    if (grid > items) grid = items;
    DwTmaGeom gg = g;
    gg.step_b = static_cast<int>(grid % g.bands);
    gg.step_c = static_cast<int>((grid / g.bands) % g.Cout);
    gg.step_i = static_cast<int>(grid / (static_cast<int64_t>(g.bands) * g.Cout));
    kernel<<<static_cast<unsigned>(grid), threads, smem, s>>>(map, gg);
    return cudaGetLastError();
}

// The TMA-window depthwise path; cudaErrorNotSupported when the shape is
// not its own (then the 4-byte / 16-byte copy kernel below runs).
cudaError_t launch_conv_depthwise_tma(const ConvProblem &p, int mode, cudaStream_t s) {
    const int64_t ks = p.KH, sw = p.sH;
    auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    if (p.pL != ks / 2 || p.pT != ks / 2) return cudaErrorNotSupported;
    if (p.W % 4 != 0 || p.OW % 8 != 0 || !al16(p.x) || !al16(p.y) || (p.ep.res && !al16(p.ep.res)))
        return cudaErrorNotSupported;
    const int pad = static_cast<int>(p.pL);
    const int x0 = -4 * ((pad + 3) / 4);
    const int c0 = -pad - x0;
    const int nl = (c0 + 7 * static_cast<int>(sw) + static_cast<int>(ks) + 3) / 4;
    const int64_t spr = p.OW / 8;
    // the last strip's loads reach window column 8 * (spr - 1) * sw + 4 * nl - 1;
    // the box (and so the row pitch) is widened to 4 (mod 32) floats
    int64_t bw = (8 * (spr - 1) * sw + 4 * nl + 3) / 4 * 4;
    bw += ((4 - bw % 32) + 32) % 32;
    if (bw > 256) return cudaErrorNotSupported;
    // bands of at most 256 strips, as even as the rows allow
    const int64_t rb_max = std::max<int64_t>(1, 256 / spr);
    const int64_t nb = (p.OH + rb_max - 1) / rb_max;
    const int64_t rb = (p.OH + nb - 1) / nb;
    const int64_t bh = (rb - 1) * sw + ks;
    if (bh > 256 || rb * spr > kDwTmaMaxThreads) return cudaErrorNotSupported;
    auto fn = dw_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(p.W), static_cast<cuuint64_t>(p.H),
                          static_cast<cuuint64_t>(p.Cin), static_cast<cuuint64_t>(p.N)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.W) * 4, static_cast<cuuint64_t>(p.H * p.W) * 4,
                             static_cast<cuuint64_t>(p.Cin * p.H * p.W) * 4};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(bw), static_cast<cuuint32_t>(bh), 1, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(p.x), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    DwTmaGeom g{};
    g.y = p.y;
    g.w = p.w;
    g.OH = static_cast<int>(p.OH);
    g.OW = static_cast<int>(p.OW);
    g.Cout = static_cast<int>(p.Cout);
    g.w_ld = static_cast<int>(p.w_ld);
    g.RB = static_cast<int>(rb);
    g.SPR = static_cast<int>(spr);
    g.x0 = x0;
    g.BW = static_cast<int>(bw);
    g.BH = static_cast<int>(bh);
    g.N = static_cast<int>(p.N);
    g.bands = static_cast<int>(nb);
    g.ep = p.ep;
    g.status = p.status;
    const int threads = static_cast<int>((rb * spr + 31) / 32 * 32);
    const int smem = static_cast<int>(kDwTmaStages * ((bw * bh * 4 + 127) / 128 * 128) + rb * (p.OW + 4) * 4 + 128);
#define OM_DWT(K, S, P)                                                                               \
    if (ks == K && sw == S && pad == P)                                                               \
        return mode == kFast ? launch_dw_tma<kFast, K, S, P>(map, g, threads, smem, s) \
                             : launch_dw_tma<kExact, K, S, P>(map, g, threads, smem, s);
    OM_DWT(3, 1, 1) OM_DWT(3, 2, 1) OM_DWT(5, 1, 2) OM_DWT(5, 2, 2)
#undef OM_DWT
    return cudaErrorNotSupported;
}

// ---- groups of a few output channels (M <= 16) with KS x KS taps from a
// TMA window. A block owns a band of R output rows of one group of one
// image. One 4-D TMA copy (columns, rows, the group's input channels, one
// image) lands the band's input window in shared memory, rows BW floats
// wide, the box starting left of and above the plane as the padding needs,
// TMA writing +0 for every element outside the plane (the zero border at
// copy time); the group's weights arrive meanwhile by plain loads, stored
// tap-major (MT = OB * MB per tap, +0 past M). Thread u computes one output
// pixel of the band for one block of MB of the group's channels (OB blocks;
// a warp's threads share the block, so the weights of a tap are one
// broadcast read): per input channel and tap, in (c, ky, kx) order, the MB
// products of the window value and the tap's weights, so each output is one
// accumulator from +0 over (c, ky, kx) in the pages' order.
constexpr int kGrpMaxThreads = 256;

struct GrpGeom {
    float *y;
    const float *w;
    int OH, OW, P, Cout, M, K, w_ld, cin_g;
    int R;               // output rows per band
    int OB, MT;          // channel blocks of MB per pixel; channel slots OB * MB
    int BW, BH;          // window row pitch (= box width) and rows per channel
    int sH, sW, dH, dW;
    int pT, x0, c0;      // box origin column x0 (a multiple of 4); window column of input column -pL
    Epilogue ep;
    unsigned *status;
};

template <int MODE, int MB, int KS>
__global__ void __launch_bounds__(kGrpMaxThreads) conv_group_kernel(const __grid_constant__ CUtensorMap map,
                                                                    const GrpGeom g) {
    static_assert(MB % 4 == 0, "weights per tap are read 16 bytes at a time");
    extern __shared__ uint8_t gw_raw[];
    __shared__ uint64_t full;
    float *win = reinterpret_cast<float *>(gw_raw + ((128u - (smem_u32(gw_raw) & 127u)) & 127u));
    const int plane = g.BH * g.BW;
    const uint32_t win_bytes = static_cast<uint32_t>(g.cin_g * plane) * 4u;
    float *wsm = win + (g.cin_g * plane + 3) / 4 * 4;
    const int grp = blockIdx.y, img = blockIdx.z;
    const int oy0 = blockIdx.x * g.R;
    if (threadIdx.x == 0) {
        mbar_init(&full, 1);
        fence_mbar_init();
        mbar_arrive_expect_tx(&full, win_bytes);
        tma_load_4d(win, &map, &full, g.x0, oy0 * g.sH - g.pT, grp * g.cin_g, img);
    }
    // the group's weight rows, read along the taps (coalesced) while the
    // window is in flight, stored tap-major (+0 past M)
    {
        const float *wg = g.w + static_cast<int64_t>(grp) * g.M * g.w_ld;
        for (int i = threadIdx.x; i < g.MT * g.K; i += blockDim.x) {
            const int oc = i / g.K, t = i - oc * g.K;
            wsm[t * g.MT + oc] = oc < g.M ? __ldg(wg + static_cast<int64_t>(oc) * g.w_ld + t) : 0.0f;
        }
    }
    __syncthreads();
    const bool landed = mbar_wait(&full, 0);
    if (!landed) {
        if (threadIdx.x == 0) {
            report_timeout(g.status, &g_status_dw);
            // the copy, if it is still in flight, lands (or gives up) before the block leaves
            (void)mbar_wait_limit(&full, 0, 1000000ull);
        }
        return;
    }
    const int rows = min(g.R, g.OH - oy0);
    // thread u: channel block u / (R * OW), pixel u % (R * OW)
    const int ob = threadIdx.x / (g.R * g.OW);
    const int u = threadIdx.x - ob * (g.R * g.OW);
    if (ob >= g.OB || u >= rows * g.OW) return;
    const int ry = u / g.OW, ox = u - ry * g.OW;
    const float *src = win + ry * g.sH * g.BW + ox * g.sW + g.c0;
    int off[KS * KS];
#pragma unroll
    for (int ky = 0; ky < KS; ++ky)
#pragma unroll
        for (int kx = 0; kx < KS; ++kx) off[ky * KS + kx] = ky * g.dH * g.BW + kx * g.dW;
    float2 acc[MB / 2];
#pragma unroll
    for (int h = 0; h < MB / 2; ++h) acc[h] = make_float2(0.0f, 0.0f);
    const float *wblk = wsm + ob * MB;
#pragma unroll 1
    for (int c = 0; c < g.cin_g; ++c) {
        const float *sc = src + c * plane;
        const float4 *wt = reinterpret_cast<const float4 *>(wblk + c * (KS * KS * g.MT));
        float v[KS * KS];
#pragma unroll
        for (int t = 0; t < KS * KS; ++t) v[t] = sc[off[t]];
#pragma unroll
        for (int t = 0; t < KS * KS; ++t) {
            const float2 vv = make_float2(v[t], v[t]);
#pragma unroll
            for (int q = 0; q < MB / 4; ++q) {
                const float4 w4 = wt[t * (g.MT / 4) + q];
                acc[2 * q] = term2<MODE>(acc[2 * q], make_float2(w4.x, w4.y), vv);
                acc[2 * q + 1] = term2<MODE>(acc[2 * q + 1], make_float2(w4.z, w4.w), vv);
            }
        }
    }
    const int oc0 = ob * MB;
    const int64_t o0 = (static_cast<int64_t>(img) * g.Cout + static_cast<int64_t>(grp) * g.M + oc0) * g.P +
                       static_cast<int64_t>(oy0 + ry) * g.OW + ox;
    const bool ep = g.ep.bias || g.ep.res || g.ep.act;
#pragma unroll
    for (int oc = 0; oc < MB; ++oc) {
        if (oc0 + oc < g.M) {
            float v = (oc & 1) ? acc[oc / 2].y : acc[oc / 2].x;
            const int64_t o = o0 + static_cast<int64_t>(oc) * g.P;
            if (ep)
                v = epilogue_value(v, g.ep.bias ? g.ep.bias + grp * g.M + oc0 + oc : nullptr,
                                   g.ep.res ? g.ep.res + o : nullptr, g.ep.act);
            g.y[o] = canonical_nan(v);
        }
    }
}

template <int MODE, int MB, int KS>
cudaError_t launch_group(const CUtensorMap &map, const GrpGeom &g, int bands, int groups, int images, int threads,
                         int smem, cudaStream_t s) {
    auto kernel = conv_group_kernel<MODE, MB, KS>;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kernel<<<dim3(static_cast<unsigned>(bands), static_cast<unsigned>(groups), static_cast<unsigned>(images)),
             threads, smem, s>>>(map, g);
    return cudaGetLastError();
}

}  // namespace

int conv_direct_channels(int64_t M) {
    for (int mb = 1; mb <= kConvDirectMaxM; mb *= 2)
        if (M <= mb) return mb;
    return 0;
}

namespace {

// The depthwise KS x KS path: bands of R output rows whose window (rows of
// Wp floats) fits in the block's shared memory.
cudaError_t launch_conv_depthwise(const ConvProblem &p, int mode, cudaStream_t s) {
    {
        const cudaError_t e = launch_conv_depthwise_tma(p, mode, s);
        if (e != cudaErrorNotSupported) return e;
    }
    const int64_t ks = p.KH, sw = p.sH;
    // 16-byte window copies and output stores: input and output rows
    // 16-byte aligned (and the residual, when there is one)
    auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    const int64_t c0v = (p.pL + 3) / 4 * 4 - p.pL;
    const bool vec = p.W % 4 == 0 && p.OW % 4 == 0 && al16(p.x) && al16(p.y) &&
                     (!p.ep.res || al16(p.ep.res)) && (c0v == 0 || c0v == (ks == 3 ? 3 : 2));
    const int64_t shift = vec ? p.pL + c0v : p.pL;
    const int c0 = static_cast<int>(shift - p.pL);
    const int64_t qx = (p.OW + kDwRun - 1) / kDwRun;
    // the last run's 16-byte loads cover columns up to this one
    const int64_t last_col = kDwRun * (qx - 1) * sw + ((c0 + kDwRun * sw + ks - 1 + 3) / 4) * 4 - 1;
    // row pitch = 4 (mod 32) floats, so that the runs of neighbouring window
    // rows start in different shared-memory banks
    int64_t wp = (last_col + 1 + 3) / 4 * 4;
    wp += ((4 - wp % 32) + 32) % 32;
    const int64_t pitch = vec ? p.OW : qx * kDwRun;
    // window rows of the band plus its staged outputs
    auto window_bytes = [&](int64_t R) { return ((R - 1) * sw + ks) * wp * 4 + R * pitch * 4; };
    if (window_bytes(1) > kDirectWindowBytes) return cudaErrorNotSupported;
    // bands of at most kDwBlockBytes, at least one output row
    const int64_t budget = kDwBlockBytes;
    int64_t R = p.OH;
    while (R > 1 && window_bytes(R) > budget) R = (R + 1) / 2;
    while (R < p.OH && window_bytes(R + 1) <= budget) ++R;
    const int64_t want = 2 * static_cast<int64_t>(num_sms());
    const int64_t planes = p.N * p.Cout;
    if (planes * ((p.OH + R - 1) / R) < want) {
        const int64_t bands = std::min<int64_t>(p.OH, (want + planes - 1) / planes);
        R = std::max<int64_t>(1, (p.OH + bands - 1) / bands);
    }
    DirectGeom g{};
    g.x = p.x; g.w = p.w; g.y = p.y;
    g.H = static_cast<int>(p.H); g.W = static_cast<int>(p.W); g.HW = static_cast<int>(p.H * p.W);
    g.OH = static_cast<int>(p.OH); g.OW = static_cast<int>(p.OW); g.P = static_cast<int>(p.OH * p.OW);
    g.Cin = static_cast<int>(p.Cin); g.Cout = static_cast<int>(p.Cout);
    g.cin_g = 1; g.M = 1; g.K = static_cast<int>(p.K); g.w_ld = static_cast<int>(p.w_ld);
    g.KH = static_cast<int>(p.KH); g.KW = static_cast<int>(p.KW);
    g.sH = static_cast<int>(p.sH); g.sW = static_cast<int>(p.sW);
    g.pT = static_cast<int>(p.pT); g.pL = static_cast<int>(p.pL);
    g.dH = 1; g.dW = 1;
    g.R = static_cast<int>(R);
    g.WR = static_cast<int>((R - 1) * sw + ks);
    g.Wp = static_cast<int>(wp);
    g.wshift = static_cast<int>(shift);
    g.ep = p.ep;
    const size_t smem = static_cast<size_t>(window_bytes(R));
    const int k = static_cast<int>(ks), st = static_cast<int>(sw);
    return mode == kFast ? launch_dw_mode<kFast>(g, k, st, vec, c0, p.Cout, p.N, smem, s)
                         : launch_dw_mode<kExact>(g, k, st, vec, c0, p.Cout, p.N, smem, s);
}

}  // namespace

cudaError_t launch_conv_group(const ConvProblem &p, int mode, cudaStream_t s) {
    const int64_t M = p.Cout / p.G, cin_g = p.Cin / p.G;
    const int64_t ks = p.KH;
    auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    if (M < 1 || M > 16 || (M == 1 && cin_g == 1) || p.KW != ks || (ks != 1 && ks != 3 && ks != 5))
        return cudaErrorNotSupported;
    if (p.N == 0 || p.OH * p.OW == 0) return cudaSuccess;
    // one TMA box per band: rows 16-byte aligned, every box dimension <= 256
    constexpr int64_t kCoordMax = int64_t{1} << 24;
    if (p.W % 4 != 0 || !al16(p.x) || cin_g > 256 || p.H > kCoordMax || p.W > kCoordMax || p.pT > 1024 ||
        p.pL > 1024 || p.sH * p.dH > kCoordMax || p.sW * p.dW > kCoordMax || p.N > 65535 || p.G > 65535 ||
        p.w_ld > 0x7FFFFFFF || p.Cout * p.OH * p.OW > 0x7FFFFFFF)
        return cudaErrorNotSupported;
    const int64_t mb = M <= 4 ? 4 : 8, ob = (M + mb - 1) / mb;
    if (ob * p.OW > kGrpMaxThreads) return cudaErrorNotSupported;
    const int64_t x0 = -4 * ((p.pL + 3) / 4);
    const int64_t c0 = -p.pL - x0;
    // the last pixel's last tap reads window column c0 + (OW-1)*sW + (KW-1)*dW
    const int64_t bw = (c0 + (p.OW - 1) * p.sW + (ks - 1) * p.dW + 1 + 3) / 4 * 4;
    if (bw > 256) return cudaErrorNotSupported;
    const int64_t wfloats = p.K * ob * mb;
    auto bh_of = [&](int64_t R) { return (R - 1) * p.sH + (ks - 1) * p.dH + 1; };
    auto smem_for = [&](int64_t R) { return 128 + ((cin_g * bh_of(R) * bw + 3) / 4 * 4 + wfloats) * 4; };
    auto rows_ok = [&](int64_t R) {
        return ob * R * p.OW <= kGrpMaxThreads && bh_of(R) <= 256 && smem_for(R) <= 100 * 1024;
    };
    if (!rows_ok(1)) return cudaErrorNotSupported;
    // the most output rows per band that fit, evened out over the bands; then
    // more, shorter bands while the grid has fewer than two blocks per SM
    int64_t R = std::min<int64_t>(p.OH, kGrpMaxThreads / (ob * p.OW));
    while (R > 1 && !rows_ok(R)) --R;
    int64_t bands = (p.OH + R - 1) / R;
    R = (p.OH + bands - 1) / bands;
    const int64_t planes = p.N * p.G;
    const int64_t want = 2 * static_cast<int64_t>(num_sms());
    if (planes * bands < want) {
        bands = std::min<int64_t>(p.OH, (want + planes - 1) / planes);
        R = (p.OH + bands - 1) / bands;
        bands = (p.OH + R - 1) / R;
    }
    const int64_t bh = bh_of(R);
    auto fn = dw_encode_fn();
    if (!fn) return cudaErrorNotSupported;
    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(p.W), static_cast<cuuint64_t>(p.H),
                          static_cast<cuuint64_t>(p.Cin), static_cast<cuuint64_t>(p.N)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.W) * 4, static_cast<cuuint64_t>(p.H * p.W) * 4,
                             static_cast<cuuint64_t>(p.Cin * p.H * p.W) * 4};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(bw), static_cast<cuuint32_t>(bh),
                         static_cast<cuuint32_t>(cin_g), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    if (fn(&map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(p.x), dims, strides, box, estr,
           CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
           CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
        return cudaErrorNotSupported;
    GrpGeom g{};
    g.y = p.y;
    g.w = p.w;
    g.OH = static_cast<int>(p.OH);
    g.OW = static_cast<int>(p.OW);
    g.P = static_cast<int>(p.OH * p.OW);
    g.Cout = static_cast<int>(p.Cout);
    g.M = static_cast<int>(M);
    g.K = static_cast<int>(p.K);
    g.w_ld = static_cast<int>(p.w_ld);
    g.cin_g = static_cast<int>(cin_g);
    g.R = static_cast<int>(R);
    g.OB = static_cast<int>(ob);
    g.MT = static_cast<int>(ob * mb);
    g.BW = static_cast<int>(bw);
    g.BH = static_cast<int>(bh);
    g.sH = static_cast<int>(p.sH);
    g.sW = static_cast<int>(p.sW);
    g.dH = static_cast<int>(p.dH);
    g.dW = static_cast<int>(p.dW);
    g.pT = static_cast<int>(p.pT);
    g.x0 = static_cast<int>(x0);
    g.c0 = static_cast<int>(c0);
    g.ep = p.ep;
    g.status = p.status;
    const int threads = static_cast<int>(std::max<int64_t>(32, (ob * R * p.OW + 31) / 32 * 32));
    const int smem = static_cast<int>(smem_for(R));
    const int nb = static_cast<int>(bands), ng = static_cast<int>(p.G), ni = static_cast<int>(p.N);
#define OM_GR(MB_, KS_)                                                                          \
    if (mb == MB_ && ks == KS_)                                                                  \
        return mode == kFast ? launch_group<kFast, MB_, KS_>(map, g, nb, ng, ni, threads, smem, s) \
                             : launch_group<kExact, MB_, KS_>(map, g, nb, ng, ni, threads, smem, s);
    OM_GR(4, 1) OM_GR(4, 3) OM_GR(4, 5) OM_GR(8, 1) OM_GR(8, 3) OM_GR(8, 5)
#undef OM_GR
    return cudaErrorNotSupported;
}

cudaError_t launch_conv_direct(const ConvProblem &p, int mode, cudaStream_t s) {
    const int64_t M = p.Cout / p.G;
    const int mb = conv_direct_channels(M);
    if (mb == 0) return cudaErrorNotSupported;
    if (p.N == 0 || p.OH * p.OW == 0) return cudaSuccess;
    // all shared-memory offsets and per-image offsets in 32 bits
    constexpr int64_t kCoordMax = int64_t{1} << 24;
    if (p.H > kCoordMax || p.W > kCoordMax || p.pT > kCoordMax || p.pL > kCoordMax ||
        p.sH > kCoordMax || p.sW > kCoordMax || p.dH * p.KH > kCoordMax ||
        p.dW * p.KW > kCoordMax || p.G > 65535 || p.N > 65535 || p.w_ld > 0x7FFFFFFF ||
        p.Cin * p.H * p.W > 0x7FFFFFFF || p.Cout * p.OH * p.OW > 0x7FFFFFFF)
        return cudaErrorNotSupported;
    // Pixels per thread: the most (up to 32 accumulators) that still leave
    // about half of the GPU's thread slots busy.
    const int64_t pixels = p.N * p.G * p.OH;
    const int64_t busy = static_cast<int64_t>(num_sms()) * 1024;
    int64_t px = 1;
    for (int64_t c = 2; c <= 8 && c * mb <= 32; c *= 2)
        if (pixels * ((p.OW + c - 1) / c) >= busy) px = c;
    const int64_t cin_g = p.Cin / p.G;
    if (M == 1 && cin_g == 1 && p.KH == p.KW && (p.KH == 3 || p.KH == 5) && p.sH == p.sW &&
        (p.sH == 1 || p.sH == 2) && p.dH == 1 && p.dW == 1) {
        const cudaError_t e = launch_conv_depthwise(p, mode, s);
        if (e != cudaErrorNotSupported) return e;
    }
    const int64_t wp = (p.OW - 1) * p.sW + (p.KW - 1) * p.dW + 1;
    const int64_t wfloats = (p.K * mb + 3) / 4 * 4, tints = (p.K + 3) / 4 * 4;
    const int64_t fixed = (wfloats + tints + px * p.sW) * 4;
    auto window_bytes = [&](int64_t R) {
        return cin_g * ((R - 1) * p.sH + (p.KH - 1) * p.dH + 1) * wp * 4;
    };
    if (fixed + window_bytes(1) > kDirectWindowBytes) return cudaErrorNotSupported;
    // the most output rows whose window fits, then fewer if that leaves
    // fewer than two blocks per SM
    int64_t R = p.OH;
    while (R > 1 && fixed + window_bytes(R) > kDirectWindowBytes) R = (R + 1) / 2;
    while (fixed + window_bytes(R + 1) <= kDirectWindowBytes && R < p.OH) ++R;
    const int64_t want = 2 * static_cast<int64_t>(num_sms());
    const int64_t planes = p.N * p.G;
    if (planes * ((p.OH + R - 1) / R) < want) {
        const int64_t bands = std::min<int64_t>(p.OH, (want + planes - 1) / planes);
        R = std::max<int64_t>(1, (p.OH + bands - 1) / bands);
    }
    DirectGeom g;
    g.x = p.x; g.w = p.w; g.y = p.y;
    g.H = static_cast<int>(p.H); g.W = static_cast<int>(p.W); g.HW = static_cast<int>(p.H * p.W);
    g.OH = static_cast<int>(p.OH); g.OW = static_cast<int>(p.OW); g.P = static_cast<int>(p.OH * p.OW);
    g.Cin = static_cast<int>(p.Cin); g.Cout = static_cast<int>(p.Cout);
    g.cin_g = static_cast<int>(cin_g); g.M = static_cast<int>(M);
    g.K = static_cast<int>(p.K); g.w_ld = static_cast<int>(p.w_ld);
    g.KH = static_cast<int>(p.KH); g.KW = static_cast<int>(p.KW);
    g.sH = static_cast<int>(p.sH); g.sW = static_cast<int>(p.sW);
    g.pT = static_cast<int>(p.pT); g.pL = static_cast<int>(p.pL);
    g.dH = static_cast<int>(p.dH); g.dW = static_cast<int>(p.dW);
    g.R = static_cast<int>(R);
    g.WR = static_cast<int>((R - 1) * p.sH + (p.KH - 1) * p.dH + 1);
    g.Wp = static_cast<int>(wp);
    g.wfloats = static_cast<int>(wfloats); g.tints = static_cast<int>(tints);
    g.ep = p.ep;
    const size_t smem = static_cast<size_t>(fixed + window_bytes(R));
    const int pxi = static_cast<int>(px);
    return mode == kFast ? launch_direct_mode<kFast>(g, p.G, p.N, mb, pxi, smem, s)
                         : launch_direct_mode<kExact>(g, p.G, p.N, mb, pxi, smem, s);
}

}  // namespace om

namespace om {

cudaError_t launch_conv_skinny(const ConvProblem &p, int mode, cudaStream_t s) {
    if (p.N == 0 || p.OH * p.OW == 0) return cudaSuccess;
    const int64_t M = p.Cout / p.G, cin_g = p.Cin / p.G, taps = p.KH * p.KW;
    // one output pixel per thread: bands of whole output rows, at most
    // kSkinnyThreads pixels each; 32-bit offsets with room to spare
    constexpr int64_t kCoordMax = int64_t{1} << 24;
    if (p.OW > kSkinnyThreads || p.H > kCoordMax || p.W > kCoordMax || p.pT > kCoordMax ||
        p.pL > kCoordMax || p.sH > kCoordMax || p.sW > kCoordMax || p.dH * p.KH > kCoordMax ||
        p.dW * p.KW > kCoordMax || p.N > 65535 || p.w_ld > 0x7FFFFFFF ||
        p.Cin * p.H * p.W > 0x7FFFFFFF || p.Cout * p.OH * p.OW > 0x7FFFFFFF || p.K > 0x7FFFFFFF)
        return cudaErrorNotSupported;
    const int64_t R = std::min<int64_t>(p.OH, kSkinnyThreads / p.OW);
    const int64_t bands = (p.OH + R - 1) / R;
    const int64_t WR = (R - 1) * p.sH + (p.KH - 1) * p.dH + 1;
    const int64_t Wp = (p.OW - 1) * p.sW + (p.KW - 1) * p.dW + 1;
    // output channels per thread (up to 16): the most that still give every
    // SM a block. Each block streams the whole input window, so fewer blocks
    // with more channels each read less from L2 (measured on ResNet-50's
    // late layers: one block per SM beat two, and 16 channels beat 8).
    const int64_t want = static_cast<int64_t>(num_sms());
    int mb = 1;
    for (int c = 2; c <= 16; c *= 2)
        if (bands * p.G * ((M + c - 1) / c) * p.N >= want) mb = c;
    const int64_t gy = p.G * ((M + mb - 1) / mb);
    if (gy > 65535) return cudaErrorNotSupported;
    // channels per chunk: two buffers of (window + weights) and one tap table
    // in 48 KB; window and weights each rounded up to 4 floats, so that the
    // weights' 8- and 16-byte loads stay aligned in both buffers
    auto round4 = [](int64_t v) { return (v + 3) / 4 * 4; };
    const int64_t plane = WR * Wp;
    if (plane >= (1 << 15)) return cudaErrorNotSupported;
    const int64_t per_channel = 2 * (plane + taps * mb) + taps;
    int64_t cc = std::min<int64_t>(cin_g, (48 * 1024 / 4 - 32 - plane) / per_channel);
    if (cc < 1) return cudaErrorNotSupported;
    auto floats = [&](int64_t c) { return 2 * (round4(c * plane) + round4(c * taps * mb)) + c * taps + plane; };
    while (cc > 1 && floats(cc) > 48 * 1024 / 4) --cc;
    if (floats(cc) > 48 * 1024 / 4 || cc * plane >= (1 << 16)) return cudaErrorNotSupported;
    DirectGeom g{};
    g.x = p.x; g.w = p.w; g.y = p.y;
    g.H = static_cast<int>(p.H); g.W = static_cast<int>(p.W); g.HW = static_cast<int>(p.H * p.W);
    g.OH = static_cast<int>(p.OH); g.OW = static_cast<int>(p.OW); g.P = static_cast<int>(p.OH * p.OW);
    g.Cin = static_cast<int>(p.Cin); g.Cout = static_cast<int>(p.Cout);
    g.cin_g = static_cast<int>(cin_g); g.M = static_cast<int>(M);
    g.K = static_cast<int>(p.K); g.w_ld = static_cast<int>(p.w_ld);
    g.KH = static_cast<int>(p.KH); g.KW = static_cast<int>(p.KW);
    g.sH = static_cast<int>(p.sH); g.sW = static_cast<int>(p.sW);
    g.pT = static_cast<int>(p.pT); g.pL = static_cast<int>(p.pL);
    g.dH = static_cast<int>(p.dH); g.dW = static_cast<int>(p.dW);
    g.R = static_cast<int>(R);
    g.WR = static_cast<int>(WR);
    g.Wp = static_cast<int>(Wp);
    g.R_chunk = static_cast<int>(cc);
    g.ch_win = static_cast<int>(round4(cc * WR * Wp));
    g.ch_w = static_cast<int>(round4(cc * taps * mb));
    g.ep = p.ep;
    g.plane_magic = static_cast<uint32_t>((uint64_t{1} << 32) / static_cast<uint64_t>(plane) + 1);
    const size_t smem = static_cast<size_t>(floats(cc)) * 4;
    return mode == kFast ? launch_skinny_mb<kFast>(g, mb, bands, gy, p.N, smem, s)
                         : launch_skinny_mb<kExact>(g, mb, bands, gy, p.N, smem, s);
}

cudaError_t read_clear_status_dw(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status_dw, sizeof(unsigned), 0, cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*out) e = cudaMemcpyToSymbol(g_status_dw, &zero, sizeof(unsigned));
    return e;
}

}  // namespace om
