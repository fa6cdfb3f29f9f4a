// Matrix-vector products: a product with at most 8 rows (C = a . B, the
// decode-shaped GEMM) or at most 8 columns (C = A . b, which is also a 1x1
// convolution over a 1x1 input: a fully connected layer over a few images).
//
// Both are bound by streaming the large operand from HBM once. The tiled
// kernels would leave most of a 128-row (or 256-column) tile idle, so here a
// block owns a strip of 32 output columns (or rows): one producer warp
// streams the large operand's strip through a ring of shared-memory stages
// with TMA (cp.async when its rows are not 16-byte aligned) behind mbarrier
// full/empty pairs, and each of 32 consumer threads keeps all the few outputs
// of its own column (or row) in registers. Every output is still one
// sequential loop over k from +0, exact mode rounding product and sum
// separately, fast mode one fused multiply-add per term; rows past k are
// zero-filled on both operands, which adds +0 * +0 = +0 to an accumulator
// that is never -0 (OneModel operators page, "Matrix product"; the
// matrix-vector product page).

#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdint>
#include <cstring>

#include "om_device.cuh"
#include "om_internal.h"

namespace om {

__device__ unsigned g_status_gemv;

namespace {

constexpr int kGemvOut = 32;      // outputs (columns or rows) per block, one per consumer thread
// k per stage (tuning knob, a multiple of 32): a stage's fixed costs --
// barrier waits and arrivals, copy issue -- are paid once per this many
// terms on both the producer and the consumer side.
#ifndef OM_GEMV_STAGE_K
#define OM_GEMV_STAGE_K 64
#endif
constexpr int kGemvRS = OM_GEMV_STAGE_K;
constexpr int kGemvBox = 32;                    // k per 128-byte-swizzled box of A
constexpr int kGemvStages = 12 * 32 / kGemvRS;  // ring depth: 384 k in flight
static_assert(kGemvRS % kGemvBox == 0 && kGemvRS <= 256, "whole boxes per stage");
constexpr int kGemvThreads = kGemvOut + 32;  // consumers, then one producer warp
constexpr int kGemvConsumerWarps = kGemvOut / 32;
constexpr uint32_t kBigBytes = kGemvOut * kGemvRS * 4;  // large-operand tile of a stage

// Few columns: float index of A element (row r, k kk) in a stage's A tile --
// boxes of 32 k side by side, each [32 rows][32 k] with the 128-byte
// swizzle (16-byte chunk c of row r at chunk c ^ (r % 8)).
__host__ __device__ constexpr int gemv_a_index(int r, int kk) {
    return (kk / kGemvBox) * kGemvOut * kGemvBox + r * kGemvBox +
           ((((kk % kGemvBox) >> 2) ^ (r & 7)) << 2) + (kk & 3);
}

// Shared memory: the large operand's stages (1 KB aligned, as the 128-byte
// swizzle wants), the small operand's stages, then the full and empty
// barriers of the ring.
template <int R>
struct GemvSmem {
    static constexpr uint32_t kSmallBytes = kGemvRS * R * 4;
    static constexpr uint32_t kSmallOff = kGemvStages * kBigBytes;
    static constexpr uint32_t kBarOff = kSmallOff + kGemvStages * kSmallBytes;
    static constexpr uint32_t kBytes = 1024 + kBarOff + 2 * kGemvStages * 8;
};

// Strided operands: X(r, c) = X[r * sr + c * sc].
struct GemvProblem {
    int64_t m, n, k;
    const float *A;  // A(i, p)
    int64_t a_si, a_sp;
    const float *B;  // B(p, j) = B[p * b_sp + (j / b_jw) * b_sjy + (j % b_jw) * b_sj]
    int64_t b_sp, b_sj;
    int64_t b_jw, b_sjy;  // columns per row of B's column index (b_jw >= n: one row)
    float *C;  // C(i, j)
    int64_t c_si, c_sj;
    const float *bias;  // bias(i, j) = bias[i * bias_si + j * bias_sj]
    int64_t bias_si, bias_sj;
    const float *res;  // res(i, j) = res[i * res_si + j * res_sj]
    int64_t res_si, res_sj;
    int act;
    // per group offsets of A rows, B rows, C rows, bias and res, and the row
    // of the group's first A row in A's tensor map
    int64_t grp_a, grp_b, grp_c, grp_bias, grp_res;
    int64_t grp_map_rows;
    // few columns: blockIdx.y = group * col_groups + column group (columns
    // [R * cg, R * cg + R) of n); blockIdx.z = image, with these offsets of
    // B, C and res per image
    int col_groups, images;
    int col_width;  // columns per column group (a power of two up to 8)
    int64_t img_b, img_c, img_res;
    // few columns, im2col: B(p, j) is tap p = (c, ky, kx) of output pixel
    // j = (oy, ox) of a convolution: x[c][oy*sH - pT + ky*dH][ox*sW - pL + kx*dW],
    // +0 outside the plane (the zero border written during the copy)
    int im2col;
    int H, W, OW, KW, taps, sH, sW, pT, pL, dH, dW;
    int64_t HW;
    uint32_t magic_kw;  // t / KW = umulhi(t, magic_kw) for t < taps
    unsigned *status;   // the call's status word in a caller workspace, or NULL
};

struct GemvBlock {
    int grp, cg;
    int64_t img;
};

__device__ __forceinline__ GemvBlock gemv_block(const GemvProblem &g) {
    const int cg = blockIdx.y % g.col_groups;
    return GemvBlock{static_cast<int>(blockIdx.y / g.col_groups), cg, static_cast<int64_t>(blockIdx.z)};
}

__device__ __forceinline__ float gemv_epilogue(const GemvProblem &g, float v, int64_t i, int64_t j,
                                               const GemvBlock &bl) {
    if (g.bias || g.res || g.act)
        v = epilogue_value(v, g.bias ? g.bias + bl.grp * g.grp_bias + i * g.bias_si + j * g.bias_sj : nullptr,
                           g.res ? g.res + bl.grp * g.grp_res + bl.img * g.img_res + i * g.res_si + j * g.res_sj
                                 : nullptr,
                           g.act);
    return canonical_nan(v);
}

__device__ __forceinline__ uint8_t *gemv_smem_base(uint8_t *raw) {
    const uint32_t b = smem_u32(raw);
    return raw + ((1024u - (b & 1023u)) & 1023u);
}

__device__ __forceinline__ void gemv_record_timeout(unsigned *status) { report_timeout(status, &g_status_gemv); }

// Producer warp of both kernels. Stage kt: the large operand's tile by TMA
// (lane 0, when TMA) or by 4-byte copies of every lane, and the small
// operand's tile by 4-byte copies; each lane's copies arrive on the stage's
// full barrier as they land.
template <int R, bool ROWS, bool TMA>
__device__ __forceinline__ void gemv_produce(const GemvProblem &g, const CUtensorMap *map,
                                             uint8_t *base, uint64_t *full, uint64_t *empty,
                                             int nk, int lane) {
    using Sm = GemvSmem<R>;
    const GemvBlock bl = gemv_block(g);
    const int grp = bl.grp;
    const int64_t o0 = static_cast<int64_t>(blockIdx.x) * kGemvOut;  // first output column / row
    const float *A = g.A + grp * g.grp_a;
    const float *B = g.B + grp * g.grp_b;
    const float *Bg = B + bl.img * g.img_b;  // this block's image
    const int64_t n_here = ROWS ? g.n : min(static_cast<int64_t>(R), g.n - static_cast<int64_t>(bl.cg) * R);
    // im2col: lane r copies rows r + 32h of every stage (taps
    // p = kt * kGemvRS + r + 32h) for all R columns. Per column, the input
    // coordinates of its tap (0, 0); per lane, its next tap's channel c and
    // position t = ky * KW + kx in the kernel, advanced by 32 taps a row.
    int col_iy0[R], col_ix0[R];
    int tap_c = 0, tap_t = 0, step_c = 0, step_t = 0;
    if (!ROWS && g.im2col) {
#pragma unroll
        for (int q = 0; q < R; ++q) {
            const int j = bl.cg * R + q;
            const int jy = j / g.OW, jx = j - (j / g.OW) * g.OW;
            col_iy0[q] = jy * g.sH - g.pT;
            col_ix0[q] = jx * g.sW - g.pL;
        }
        tap_c = lane / g.taps;
        tap_t = lane - tap_c * g.taps;
        step_c = 32 / g.taps;
        step_t = 32 - step_c * g.taps;
    }
    // few columns, B read in place: the offset of this lane's column
    // j = cg * R + lane % R, split into (row, column) of its index
    int64_t col_off = 0;
    if (!ROWS && !g.im2col) {
        const int64_t j = static_cast<int64_t>(bl.cg) * R + lane % R;
        const int64_t jy = j / g.b_jw, jx = j - jy * g.b_jw;
        col_off = jy * g.b_sjy + jx * g.b_sj;
    }
    const uint32_t base32 = smem_u32(base);
    for (int kt = 0; kt < nk; ++kt) {
        const int s = kt % kGemvStages;
        if (!mbar_wait(&empty[s], ((kt / kGemvStages) & 1) ^ 1)) {
            gemv_record_timeout(g.status);
            cp_async_wait_all();
            if (TMA && lane == 0) {
                // let the tiles already requested land before leaving
                for (int s2 = 0; s2 < kGemvStages && s2 < kt; ++s2) {
                    const int last = s2 + ((kt - 1 - s2) / kGemvStages) * kGemvStages;
                    (void)mbar_wait(&full[s2], static_cast<uint32_t>((last / kGemvStages) & 1));
                }
            }
            return;
        }
        const int64_t p0 = static_cast<int64_t>(kt) * kGemvRS;
        uint8_t *big = base + s * kBigBytes;
        const uint32_t big32 = base32 + s * kBigBytes;
        const uint32_t small32 = base32 + Sm::kSmallOff + s * Sm::kSmallBytes;
        if constexpr (TMA) {
            if (lane == 0) {
                mbar_arrive_expect_tx(&full[s], kBigBytes);
                if constexpr (ROWS)
                    tma_load_2d(big, map, &full[s], static_cast<int>(o0), static_cast<int>(p0));
                else
                    for (int b = 0; b < kGemvRS / kGemvBox; ++b)
                        tma_load_2d(big + b * kGemvOut * kGemvBox * 4, map, &full[s],
                                    static_cast<int>(p0) + b * kGemvBox,
                                    static_cast<int>(grp * g.grp_map_rows + o0));
            }
        } else if constexpr (ROWS) {
            // B rows of the stage, [kGemvRS][32]
            for (int e = lane; e < kGemvRS * kGemvOut; e += 32) {
                const int r = e / kGemvOut, c = e % kGemvOut;
                const int64_t p = p0 + r, j = o0 + c;
                const bool ok = p < g.k && j < g.n;
                cp_async_4_if(big32 + e * 4, ok ? B + p * g.b_sp + j * g.b_sj : B, ok);
            }
        } else {
            // A rows of the block, laid out as the TMA boxes would be
            for (int e = lane; e < kGemvOut * kGemvRS; e += 32) {
                const int r = e / kGemvRS, kk = e % kGemvRS;
                const int64_t i = o0 + r, p = p0 + kk;
                const bool ok = i < g.m && p < g.k;
                const uint32_t off = static_cast<uint32_t>(gemv_a_index(r, kk)) * 4;
                cp_async_4_if(big32 + off, ok ? A + i * g.a_si + p * g.a_sp : A, ok);
            }
        }
        // the small operand: A columns [32][R] (few rows) or B rows [32][R] (few columns)
        if (!ROWS && g.im2col) {
#pragma unroll
            for (int h = 0; h < kGemvRS / 32; ++h) {
                const int r = lane + 32 * h;
                const bool p_ok = p0 + r < g.k;
                const int ky = g.KW == 1 ? tap_t
                                         : static_cast<int>(__umulhi(static_cast<uint32_t>(tap_t), g.magic_kw));
                const int dy = ky * g.dH, dx = (tap_t - ky * g.KW) * g.dW;
                const float *plane = Bg + (p_ok ? static_cast<int64_t>(tap_c) * g.HW : 0);
#pragma unroll
                for (int q = 0; q < R; ++q) {
                    const int iy = col_iy0[q] + dy, ix = col_ix0[q] + dx;
                    const bool ok = p_ok && q < n_here && static_cast<unsigned>(iy) < static_cast<unsigned>(g.H) &&
                                    static_cast<unsigned>(ix) < static_cast<unsigned>(g.W);
                    const float *src = ok ? plane + (static_cast<int64_t>(iy) * g.W + ix) : Bg;
                    cp_async_4_if(small32 + (r * R + q) * 4, src, ok);
                }
                tap_c += step_c;
                tap_t += step_t;
                if (tap_t >= g.taps) {
                    tap_t -= g.taps;
                    ++tap_c;
                }
            }
        } else {
            // lane copies column q = lane % R of rows lane / R + (32 / R) i
            const int q = lane % R;
#pragma unroll
            for (int i = 0; i < R * kGemvRS / 32; ++i) {
                const int r = lane / R + (32 / R) * i;
                const int64_t p = p0 + r;
                bool ok;
                const float *src;
                if constexpr (ROWS) {
                    ok = p < g.k && q < g.m;
                    src = ok ? A + q * g.a_si + p * g.a_sp : A;
                } else {
                    ok = p < g.k && q < n_here;
                    src = ok ? Bg + p * g.b_sp + col_off : Bg;
                }
                cp_async_4_if(small32 + (r * R + q) * 4, src, ok);
            }
        }
        cp_async_arrive_noinc(&full[s]);
    }
    cp_async_wait_all();
}

// Few columns: four k of a consumer thread's A row (from the stage's
// swizzled A tile) and the stage's four B rows of R columns.
template <int R>
struct GemvChunk {
    float4 a;
    float b[4][R];
};

template <int R>
__device__ __forceinline__ void gemv_load_chunk(GemvChunk<R> &ch, const float *big, const float *small,
                                                int c, int t) {
    ch.a = *reinterpret_cast<const float4 *>(big + gemv_a_index(t, 4 * c));
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float *brow = small + (4 * c + q) * R;
        if constexpr (R >= 4) {
#pragma unroll
            for (int u = 0; u < R / 4; ++u) {
                const float4 v = reinterpret_cast<const float4 *>(brow)[u];
                ch.b[q][4 * u] = v.x;
                ch.b[q][4 * u + 1] = v.y;
                ch.b[q][4 * u + 2] = v.z;
                ch.b[q][4 * u + 3] = v.w;
            }
        } else if constexpr (R == 2) {
            const float2 v = reinterpret_cast<const float2 *>(brow)[0];
            ch.b[q][0] = v.x;
            ch.b[q][1] = v.y;
        } else {
            ch.b[q][0] = brow[0];
        }
    }
}

// The chunk's four terms, in increasing k, for each of the R outputs.
template <int MODE, int R>
__device__ __forceinline__ void gemv_run_chunk(const GemvChunk<R> &ch, float2 (&acc)[(R + 1) / 2],
                                               float &acc1) {
#pragma unroll
    for (int q = 0; q < 4; ++q) {
        const float a = q == 0 ? ch.a.x : q == 1 ? ch.a.y : q == 2 ? ch.a.z : ch.a.w;
        if constexpr (R == 1) {
            acc1 = term<MODE>(acc1, a, ch.b[q][0]);
        } else {
            const float2 a2 = make_float2(a, a);
#pragma unroll
            for (int h = 0; h < R / 2; ++h)
                acc[h] = term2<MODE>(acc[h], a2, make_float2(ch.b[q][2 * h], ch.b[q][2 * h + 1]));
        }
    }
}

// C (m x n) = A (m x k) . B (k x n) with m <= R (ROWS: a block owns 32
// columns) or n <= R (!ROWS: a block owns 32 rows of group blockIdx.y).
// TMA: the large operand comes by a 2-D tensor map (ROWS: B, box 32 columns
// x kGemvRS rows; !ROWS: A, boxes of 32 k x 32 rows with the 128-byte
// swizzle, kGemvRS / 32 of them a stage).
template <int MODE, int R, bool ROWS, bool TMA>
__global__ void __launch_bounds__(kGemvThreads, 1)
    gemv_kernel(const __grid_constant__ CUtensorMap map, const GemvProblem g) {
    using Sm = GemvSmem<R>;
    extern __shared__ uint8_t gemv_raw[];
    uint8_t *base = gemv_smem_base(gemv_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(base + Sm::kBarOff);
    uint64_t *empty = full + kGemvStages;
    const int nk = static_cast<int>((g.k + kGemvRS - 1) / kGemvRS);
    const int t = threadIdx.x, warp = t / 32, lane = t % 32;
    if (t == 0) {
        for (int s = 0; s < kGemvStages; ++s) {
            mbar_init(&full[s], 32 + (TMA ? 1 : 0));
            mbar_init(&empty[s], kGemvConsumerWarps);
        }
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();
    if (warp == kGemvConsumerWarps) {
        if (TMA && lane == 0) prefetch_tensormap(&map);
        gemv_produce<R, ROWS, TMA>(g, &map, base, full, empty, nk, lane);
        return;
    }

    float2 acc[(R + 1) / 2];
    float acc1 = 0.0f;
#pragma unroll
    for (int h = 0; h < (R + 1) / 2; ++h) acc[h] = make_float2(0.0f, 0.0f);
    if constexpr (ROWS) {
#pragma unroll 1
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % kGemvStages;
            if (!mbar_wait(&full[s], (kt / kGemvStages) & 1)) {
                gemv_record_timeout(g.status);
                return;
            }
            const float *bcol = reinterpret_cast<const float *>(base + s * kBigBytes) + t;
            const float *small = reinterpret_cast<const float *>(base + Sm::kSmallOff + s * Sm::kSmallBytes);
#pragma unroll
            for (int r = 0; r < kGemvRS; ++r) {
                const float b = bcol[r * kGemvOut];
                if constexpr (R == 1) {
                    acc1 = term<MODE>(acc1, small[r], b);
                } else {
                    const float2 b2 = make_float2(b, b);
#pragma unroll
                    for (int h = 0; h < R / 2; ++h)
                        acc[h] = term2<MODE>(acc[h], reinterpret_cast<const float2 *>(small + r * R)[h], b2);
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    } else {
        // The thread's row runs in chunks of four k. Each chunk's operands are
        // loaded while the previous chunk computes, and the next stage's first
        // chunk while this stage's last one does, so shared-memory latency
        // stays off the accumulators' dependency chain.
        constexpr int kChunks = kGemvRS / 4;
        auto big_of = [&](int s) { return reinterpret_cast<const float *>(base + s * kBigBytes); };
        auto small_of = [&](int s) {
            return reinterpret_cast<const float *>(base + Sm::kSmallOff + s * Sm::kSmallBytes);
        };
        if (!mbar_wait(&full[0], 0)) {
            gemv_record_timeout(g.status);
            return;
        }
        GemvChunk<R> cur, nxt;
        gemv_load_chunk<R>(cur, big_of(0), small_of(0), 0, t);
#pragma unroll 1
        for (int kt = 0; kt < nk; ++kt) {
            const int s = kt % kGemvStages;
            const float *big = big_of(s), *small = small_of(s);
#pragma unroll
            for (int c = 0; c < kChunks - 1; ++c) {
                gemv_load_chunk<R>(nxt, big, small, c + 1, t);
                gemv_run_chunk<MODE, R>(cur, acc, acc1);
                cur = nxt;
            }
            if (kt + 1 < nk) {
                const int s1 = (kt + 1) % kGemvStages;
                if (!mbar_wait(&full[s1], ((kt + 1) / kGemvStages) & 1)) {
                    gemv_record_timeout(g.status);
                    return;
                }
                gemv_load_chunk<R>(nxt, big_of(s1), small_of(s1), 0, t);
            }
            gemv_run_chunk<MODE, R>(cur, acc, acc1);
            cur = nxt;
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[s]);
        }
    }

    const GemvBlock bl = gemv_block(g);
    const int64_t o = static_cast<int64_t>(blockIdx.x) * kGemvOut + t;
    if (o >= (ROWS ? g.n : g.m)) return;
    float *C = g.C + bl.grp * g.grp_c + bl.img * g.img_c;
    const int64_t j0 = ROWS ? 0 : static_cast<int64_t>(bl.cg) * R;  // first column of the block
#pragma unroll
    for (int q = 0; q < R; ++q) {
        if ((ROWS ? q : j0 + q) < (ROWS ? g.m : g.n)) {
            const float v = R == 1 ? acc1 : ((q & 1) ? acc[q / 2].y : acc[q / 2].x);
            const int64_t i = ROWS ? q : o, j = ROWS ? o : j0 + q;
            C[i * g.c_si + j * g.c_sj] = gemv_epilogue(g, v, i, j, bl);
        }
    }
}

PFN_cuTensorMapEncodeTiled_v12000 gemv_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    return fn;
}

// Row-major matrix (rows x cols, row stride ld floats) with box
// box_cols x box_rows; +0 outside. False when TMA cannot describe it.
bool gemv_map(CUtensorMap *map, const float *base, int64_t rows, int64_t cols, int64_t ld,
              int box_cols, int box_rows, bool swizzle128) {
    auto fn = gemv_encode_fn();
    if (!fn || (reinterpret_cast<uintptr_t>(base) & 15) != 0 || ld % 4 != 0 || rows < 1 || cols < 1 ||
        rows > (int64_t{1} << 31) || cols > (int64_t{1} << 31))
        return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int round_up_pow2(int64_t v) {
    int r = 1;
    while (r < v) r *= 2;
    return r;
}

template <int MODE, int R, bool ROWS, bool TMA>
cudaError_t launch_one(const CUtensorMap &map, const GemvProblem &g, int64_t blocks, int64_t groups,
                       cudaStream_t s) {
    auto kernel = gemv_kernel<MODE, R, ROWS, TMA>;
    const int smem = static_cast<int>(GemvSmem<R>::kBytes);
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kernel<<<dim3(static_cast<unsigned>(blocks), static_cast<unsigned>(groups * g.col_groups),
                  static_cast<unsigned>(g.images)),
             kGemvThreads, smem, s>>>(map, g);
    return cudaGetLastError();
}

template <int MODE, bool ROWS, bool TMA>
cudaError_t launch_r(const CUtensorMap &map, const GemvProblem &g, int r, int64_t blocks, int64_t groups,
                     cudaStream_t s) {
    switch (r) {
        case 1: return launch_one<MODE, 1, ROWS, TMA>(map, g, blocks, groups, s);
        case 2: return launch_one<MODE, 2, ROWS, TMA>(map, g, blocks, groups, s);
        case 4: return launch_one<MODE, 4, ROWS, TMA>(map, g, blocks, groups, s);
        case 8: return launch_one<MODE, 8, ROWS, TMA>(map, g, blocks, groups, s);
        default: return cudaErrorNotSupported;
    }
}

template <int MODE>
cudaError_t launch_mode(const CUtensorMap &map, const GemvProblem &g, bool rows, bool tma, int r,
                        int64_t blocks, int64_t groups, cudaStream_t s) {
    if (rows)
        return tma ? launch_r<MODE, true, true>(map, g, r, blocks, groups, s)
                   : launch_r<MODE, true, false>(map, g, r, blocks, groups, s);
    return tma ? launch_r<MODE, false, true>(map, g, r, blocks, groups, s)
               : launch_r<MODE, false, false>(map, g, r, blocks, groups, s);
}

// map_rows: rows of the large operand's tensor map (!rows: all groups' A
// rows); the map is built here when the operand allows it.
cudaError_t launch_gemv(GemvProblem g, int mode, bool rows, int64_t groups, int64_t map_rows,
                        int64_t map_ld, cudaStream_t s) {
    if (g.col_groups < 1) g.col_groups = 1;
    if (g.images < 1) g.images = 1;
    if (g.b_jw < 1) g.b_jw = int64_t{1} << 62;  // one row: j / b_jw == 0
    // with column groups each block takes col_width columns
    if (g.col_width < 1) g.col_width = kGemvMaxSmall;
    const int64_t small = rows ? g.m : (g.col_groups > 1 ? g.col_width : g.n);
    const int64_t big = rows ? g.n : g.m;
    if (small < 1 || small > kGemvMaxSmall || g.k < 1 || groups < 1 ||
        groups * g.col_groups > 65535 || g.images > 65535 || g.k > 0x7FFFFFFF - kGemvRS ||
        (rows && (g.col_groups != 1 || g.images != 1)))
        return cudaErrorNotSupported;
    const int64_t blocks = (big + kGemvOut - 1) / kGemvOut;
    if (blocks > 0x7FFFFFFF) return cudaErrorNotSupported;
    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    bool tma;
    if (rows)
        tma = g.b_sj == 1 && gemv_map(&map, g.B, g.k, g.n, g.b_sp, kGemvOut, kGemvRS, false);
    else
        tma = g.a_sp == 1 && map_rows <= 0x7FFFFFFF - kGemvOut &&
              gemv_map(&map, g.A, map_rows, g.k, map_ld, kGemvBox, kGemvOut, true);
    const int r = round_up_pow2(small);
    return mode == kFast ? launch_mode<kFast>(map, g, rows, tma, r, blocks, groups, s)
                         : launch_mode<kExact>(map, g, rows, tma, r, blocks, groups, s);
}

}  // namespace

cudaError_t launch_gemm_gemv(const GemmProblem &p, int mode, cudaStream_t s) {
    GemvProblem g{};
    g.m = p.m; g.n = p.n; g.k = p.k;
    g.A = p.A; g.a_si = p.lda; g.a_sp = 1;
    g.B = p.B; g.b_sp = p.ldb; g.b_sj = 1;
    g.C = p.C; g.c_si = p.ldc; g.c_sj = 1;
    g.bias = p.ep.bias; g.bias_si = 0; g.bias_sj = 1;
    g.res = p.ep.res; g.res_si = p.ep.ldr; g.res_sj = 1;
    g.act = p.ep.act;
    g.status = p.status;
    if (p.m <= kGemvMaxSmall) return launch_gemv(g, mode, true, 1, 0, 0, s);
    if (p.n <= kGemvMaxSmall) return launch_gemv(g, mode, false, 1, p.m, p.lda, s);
    return cudaErrorNotSupported;
}

cudaError_t launch_conv_gemv(const ConvProblem &p, int mode, cudaStream_t s) {
    // a 1x1 kernel over a 1x1 input with no padding: per group, output
    // channel oc of image n is the product of weight row oc with the image's
    // input channels
    if (p.KH != 1 || p.KW != 1 || p.H != 1 || p.W != 1 || p.pT != 0 || p.pL != 0 || p.OH != 1 ||
        p.OW != 1 || p.N > kGemvMaxSmall || p.N < 1)
        return cudaErrorNotSupported;
    const int64_t M = p.Cout / p.G, cin_g = p.Cin / p.G;
    GemvProblem g{};
    g.m = M; g.n = p.N; g.k = cin_g;
    g.A = p.w; g.a_si = p.w_ld; g.a_sp = 1;
    g.B = p.x; g.b_sp = 1; g.b_sj = p.Cin;
    g.C = p.y; g.c_si = 1; g.c_sj = p.Cout;
    g.bias = p.ep.bias; g.bias_si = 1; g.bias_sj = 0;
    g.res = p.ep.res; g.res_si = 1; g.res_sj = p.Cout;
    g.act = p.ep.act;
    g.status = p.status;
    g.grp_a = M * p.w_ld; g.grp_b = cin_g; g.grp_c = M; g.grp_bias = M; g.grp_res = M;
    g.grp_map_rows = M;
    return launch_gemv(g, mode, false, p.G, p.Cout, p.w_ld, s);
}

cudaError_t launch_conv_columns(const ConvProblem &p, int mode, bool choose, cudaStream_t s) {
    // per image and group, the product of the group's weights (Cout/G x K)
    // with the patch matrix (K x OH*OW) in blocks of 32 output channels by 8
    // pixels: a 1x1 unpadded kernel reads the input pixels directly (rows
    // H*W apart, stride sH, sW); any other kernel of up to 64 taps gathers
    // its patches during the copy (im2col, zero border included)
    if (p.N < 1) return cudaErrorNotSupported;
    const int64_t M = p.Cout / p.G, cin_g = p.Cin / p.G, P = p.OH * p.OW, HW = p.H * p.W;
    const int64_t taps = p.KH * p.KW;
    const bool direct = p.KH == 1 && p.KW == 1 && p.pT == 0 && p.pL == 0;
    if (!direct && (taps > 64 || p.K >= (int64_t{1} << 24) || p.H > (1 << 24) || p.W > (1 << 24) ||
                    p.OW > (1 << 24) || p.pT > (1 << 24) || p.pL > (1 << 24) || p.sH > (1 << 24) ||
                    p.sW > (1 << 24) || p.dH * p.KH > (1 << 24) || p.dW * p.KW > (1 << 24) ||
                    P > (int64_t{1} << 30)))
        return cudaErrorNotSupported;
    if (P < 1) return cudaSuccess;
    // columns per block: 8, halved while there are fewer than two blocks per
    // SM (measured on ResNet-50 at batch 1: fewer outputs per consumer warp
    // beat the extra weight re-reads from L2 down to two blocks per SM, not to
    // four)
    int width = kGemvMaxSmall;
    auto blocks = [&](int w) { return (M + kGemvOut - 1) / kGemvOut * ((P + w - 1) / w) * p.N * p.G; };
    while (width > 1 && blocks(width) < 2 * static_cast<int64_t>(num_sms())) width /= 2;
    // when choosing: gathered patches pay off with a long k loop and a block
    // for every SM, and in-place columns with k of 128 or more (measured on
    // ResNet-50 at batch 1: the 7x7 stem and the 64-channel 1x1 layers at
    // 56 x 56 ran faster in the few-pixel kernel)
    if (choose && !direct && (p.K < 256 || blocks(width) < num_sms())) return cudaErrorNotSupported;
    if (choose && direct && p.K < 128) return cudaErrorNotSupported;
    GemvProblem g{};
    g.m = M; g.n = P; g.k = p.K;
    g.A = p.w; g.a_si = p.w_ld; g.a_sp = 1;
    // direct: output pixel (oy, ox) reads input (oy * sH, ox * sW)
    g.B = p.x; g.b_sp = HW; g.b_sj = p.sW; g.b_jw = p.OW; g.b_sjy = p.sH * p.W;
    g.C = p.y; g.c_si = P; g.c_sj = 1;
    g.bias = p.ep.bias; g.bias_si = 1; g.bias_sj = 0;
    g.res = p.ep.res; g.res_si = P; g.res_sj = 1;
    g.act = p.ep.act;
    g.status = p.status;
    g.grp_a = M * p.w_ld; g.grp_b = cin_g * HW; g.grp_c = M * P; g.grp_bias = M; g.grp_res = M * P;
    g.grp_map_rows = M;
    g.col_width = width;
    g.col_groups = static_cast<int>(std::min<int64_t>((P + width - 1) / width, 65536));
    g.images = static_cast<int>(std::min<int64_t>(p.N, 65536));
    g.img_b = p.Cin * HW; g.img_c = p.Cout * P; g.img_res = p.Cout * P;
    if (!direct) {
        g.im2col = 1;
        g.H = static_cast<int>(p.H); g.W = static_cast<int>(p.W); g.OW = static_cast<int>(p.OW);
        g.KW = static_cast<int>(p.KW); g.taps = static_cast<int>(taps);
        g.sH = static_cast<int>(p.sH); g.sW = static_cast<int>(p.sW);
        g.pT = static_cast<int>(p.pT); g.pL = static_cast<int>(p.pL);
        g.dH = static_cast<int>(p.dH); g.dW = static_cast<int>(p.dW);
        g.HW = HW;
        // ceil(2^32 / d): exact quotients for numerators below 2^24 and d <= 64
        g.magic_kw = p.KW > 1 ? static_cast<uint32_t>(((uint64_t{1} << 32) + p.KW - 1) / p.KW) : 0u;
    }
    return launch_gemv(g, mode, false, p.G, p.Cout, p.w_ld, s);
}

cudaError_t read_clear_status_gemv(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status_gemv, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*out) e = cudaMemcpyToSymbol(g_status_gemv, &zero, sizeof(unsigned));
    return e;
}

}  // namespace om
