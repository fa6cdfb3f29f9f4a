// conv_rows.cu -- stride-1 NCHW convolution in which each warp owns whole
// output-row segments for 64 output channels, on the CUDA cores of sm_103a,
// bit-exact in both modes.
//
// What each output is ("Exact mode" page, section "Convolution"; "Convolution
// (fast mode)" page, section "What each output is"): output (n, oc, oy, ox)
// of group g sums, for taps in (c, ky, kx) order from +0, the term
// w[oc][c][ky][kx] * v with v = x[n][g*Cin/G + c][oy - pad + ky][ox - pad + kx]
// inside the plane and +0 outside; padding taps are real products (an
// infinite or NaN weight meeting padding gives NaN); NaN is stored as
// 0x7FC00000. k is never split: every output is one thread's register over
// all of its taps.
//
// Layout of the work (the pages' "runs": consecutive output columns of one
// output row read consecutive input columns, so one copy of the input rows
// serves every tap of a kernel row):
//   * A warp task is four segments of 14 consecutive output pixels (one
//     56-pixel row, two 28-pixel rows, ...) of one image, for a block of 64
//     output channels of one group. Thread (tr, tc) of the warp owns output
//     channels 8*tr .. 8*tr+7 of the block and segment tc: 8 x 14 outputs.
//   * The warp streams its own input window through a ring of shared-memory
//     stages by TMA (4-D box: columns, rows, CC channels, image). The box
//     starts left of the plane and above it as the padding needs; TMA fills
//     every element outside the plane with +0, which writes the zero border
//     at copy time -- padding is never materialised in HBM.
//   * The block's weights stay in shared memory for the whole block,
//     transposed to [tap][channel] so that two channels' weights of one tap
//     are one register pair. Each term is one paired-lane instruction over two
//     output channels (two outputs per instruction, each lane rounded on its
//     own), with the input value broadcast: a kernel row's input values are
//     loaded once per channel and serve all KW taps from registers.
//   * Tasks are handed out so that a launch over the 56 x 56 ResNet-50
//     stage-1 shapes at batch 32 is one round of 12 warps per SM.
#include <cudaTypedefs.h>

#include <cstring>

#include "om_internal.h"
#include "om_device.cuh"

namespace om {

__device__ unsigned g_status_rows;

namespace {

constexpr int kRowsWarps = 12;  // warps per CTA: three per scheduler
constexpr int kRowsThreads = kRowsWarps * 32;
constexpr int kRowsMB = 64;     // output channels per weight block
constexpr int kRowsTN = 14;     // output pixels per thread (one row segment)
constexpr int kRowsStagePitch = 60;  // floats per row of the epilogue staging area

struct RowsGeom {
    float *y;
    const float *w;
    int Cin, Cout, cin_g, M, KH, OH, OW;
    int K, w_ld;
    int SR;        // segments of kRowsTN pixels per output row
    int Q;         // warp tasks (four consecutive segments) per image
    int NQ;        // images * Q
    int mblocks;   // M / 64
    int nblocks;   // G * mblocks
    int CC, nch;   // input channels per stage, stages per task
    int BW, BH;    // window box: columns, rows
    int x0;        // first window column (a multiple of 4, <= -pad)
    int box_floats, box_stride;  // floats copied per stage, floats between stages
    int stages;
    int w_vec;     // weight rows 16-byte aligned: 16-byte loads
    Epilogue ep;
    unsigned *status;  // the call's status word in a caller workspace, or NULL
};

// Shared memory: the transposed weight block, kRowsWarps rings of window
// stages, one mbarrier per stage, an abort word.
struct RowsSmem {
    float *wT;
    float *win;
    uint64_t *full;
    int *abort_flag;
    int *rec;  // per warp: [0] first chunk of the current task, [1] chunks issued, [2] chunks awaited
};

__device__ __forceinline__ RowsSmem rows_smem(uint8_t *raw, const RowsGeom &g) {
    RowsSmem s;
    uint8_t *base = raw + ((128u - (smem_u32(raw) & 127u)) & 127u);
    s.wT = reinterpret_cast<float *>(base);
    s.win = s.wT + g.K * kRowsMB;
    s.full = reinterpret_cast<uint64_t *>(s.win + kRowsWarps * g.stages * g.box_stride);
    s.abort_flag = reinterpret_cast<int *>(s.full + kRowsWarps * g.stages);
    s.rec = s.abort_flag + 4;
    return s;
}

// Position of block channel ch (0..63) in a transposed weight row: channel
// ch belongs to thread row tr = ch / 8 and half h = (ch % 8) / 4; the 16-byte
// chunk 8h + tr holds channels 8tr + 4h .. +3, so the eight thread rows of
// one 16-byte load read 128 contiguous bytes.
__device__ __forceinline__ int wt_pos(int ch) { return ((((ch & 4) << 1) | (ch >> 3)) << 2) | (ch & 3); }

// One term on two outputs with the compiler's paired-lane builtins, which
// keep each float2 in a register pair the paired instructions read and write
// in place: fast mode one paired fused multiply-add; exact mode two scalar
// rounded multiplies and one paired rounded add (the form the library's
// bit-exact tests pin; the multiplies are never contracted into the add).
template <int MODE>
__device__ __forceinline__ float2 pterm(float2 acc, float2 a, float2 b) {
    if constexpr (MODE == kFast) {
        return __ffma2_rn(a, b, acc);
    } else {
        return __fadd2_rn(acc, make_float2(mul_rn_scalar(a.x, b.x), mul_rn_scalar(a.y, b.y)));
    }
}

__device__ __forceinline__ void rows_record_timeout(unsigned *status, int *abort_flag) {
    report_timeout(status, &g_status_rows);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
}

// The window chunk of chunk sequence index i of warp gw: task (image n,
// segment quad q) of weight block b, input channels ch*CC .. of the group.
struct ChunkPos {
    int b, r, ch;
};

__device__ __forceinline__ ChunkPos chunk_pos(const RowsGeom &g, int i, int per_block) {
    ChunkPos c;
    c.b = i / per_block;
    const int rem = i - c.b * per_block;
    c.r = rem / g.nch;
    c.ch = rem - c.r * g.nch;
    return c;
}

template <int PAD>
__device__ __forceinline__ void issue_chunk(const RowsGeom &g, const CUtensorMap *map, float *dst,
                                            uint64_t *bar, int i, int per_block, int gw, int WT) {
    const ChunkPos c = chunk_pos(g, i, per_block);
    const int t = gw + c.r * WT;
    const int n = t / g.Q, q = t - n * g.Q;
    const int grp = c.b / g.mblocks;
    const int oyq = (4 * q) / g.SR;  // first output row of the quad
    mbar_arrive_expect_tx(bar, static_cast<uint32_t>(g.box_floats) * 4u);
    tma_load_4d(dst, map, bar, g.x0, oyq - PAD, grp * g.cin_g + c.ch * g.CC, n);
}

// Stores one staged slice: eight rows (thread rows rr, output channel
// ch0 + 8*rr) of the warp's four segments, 8 bytes per lane per step, with
// the output epilogue and canonical NaN. seg_off[sg] is the offset of
// segment sg's first output pixel in an output plane.
template <bool HAS_EP>
__device__ __forceinline__ void store_slice(const RowsGeom &g, const float *stg, int lane, int64_t ybase,
                                         int so0, int so1, int so2, int so3, int ch0) {
    constexpr int kPairs = 8 * 4 * kRowsTN / 2;  // 224 value pairs in the slice
    const int64_t plane = static_cast<int64_t>(g.OH) * g.OW;
#pragma unroll 1
    for (int u = 0; u < (kPairs + 31) / 32; ++u) {
        const int idx = lane + 32 * u;
        if (idx < kPairs) {
            const int rr = idx / (2 * kRowsTN);  // thread row 0..7
            const int p2 = idx - rr * (2 * kRowsTN);
            const int sg = p2 / (kRowsTN / 2);  // segment 0..3
            const int off = 2 * (p2 - sg * (kRowsTN / 2));
            const float2 val = *reinterpret_cast<const float2 *>(stg + rr * kRowsStagePitch + sg * kRowsTN + off);
            const int och = ch0 + 8 * rr;
            const int so = sg == 0 ? so0 : sg == 1 ? so1 : sg == 2 ? so2 : so3;
            const int64_t o = ybase + och * plane + so + off;
            float e0 = val.x, e1 = val.y;
            if constexpr (HAS_EP) {
                const float *bp = g.ep.bias ? g.ep.bias + och : nullptr;
                e0 = epilogue_value(e0, bp, g.ep.res ? g.ep.res + o : nullptr, g.ep.act);
                e1 = epilogue_value(e1, bp, g.ep.res ? g.ep.res + o + 1 : nullptr, g.ep.act);
            }
            *reinterpret_cast<float2 *>(g.y + o) = make_float2(canonical_nan(e0), canonical_nan(e1));
        }
    }
}

// Weight block b (64 output channels of one group) into shared memory,
// transposed to [tap][channel] at the positions wt_pos gives. Consecutive
// threads take consecutive channels, so a warp's stores of one tap row hit
// distinct banks; with 16-byte aligned rows each thread loads four taps at
// once, kLoadBatch loads in flight before their values are stored.
__device__ __noinline__ void load_weight_block(const RowsGeom &g, float *wT, int b) {
    const int grp = b / g.mblocks, mb = b - grp * g.mblocks;
    const float *wb = g.w + static_cast<int64_t>(grp * g.M + mb * kRowsMB) * g.w_ld;
    if (g.w_vec) {
        const int items = kRowsMB * (g.K / 4);
        constexpr int kLoadBatch = 8;
        for (int e0 = threadIdx.x; e0 < items; e0 += kRowsThreads * kLoadBatch) {
            float4 vals[kLoadBatch];
#pragma unroll
            for (int u = 0; u < kLoadBatch; ++u) {
                const int e = e0 + u * kRowsThreads;
                if (e < items)
                    vals[u] = __ldg(reinterpret_cast<const float4 *>(
                        wb + static_cast<int64_t>(e & (kRowsMB - 1)) * g.w_ld + 4 * (e / kRowsMB)));
            }
#pragma unroll
            for (int u = 0; u < kLoadBatch; ++u) {
                const int e = e0 + u * kRowsThreads;
                if (e < items) {
                    float *d = wT + (4 * (e / kRowsMB)) * kRowsMB + wt_pos(e & (kRowsMB - 1));
                    d[0] = vals[u].x;
                    d[kRowsMB] = vals[u].y;
                    d[2 * kRowsMB] = vals[u].z;
                    d[3 * kRowsMB] = vals[u].w;
                }
            }
        }
    } else {
        const int count = kRowsMB * g.K;
        for (int e = threadIdx.x; e < count; e += kRowsThreads) {
            const int ch = e & (kRowsMB - 1), k = e / kRowsMB;
            wT[k * kRowsMB + wt_pos(ch)] = __ldg(wb + static_cast<int64_t>(ch) * g.w_ld + k);
        }
    }
}

}  // namespace

template <int MODE, int KS, int PAD, bool HAS_EP>
__global__ void __launch_bounds__(kRowsThreads, 1)
    conv_rows_kernel(const __grid_constant__ CUtensorMap mapX, RowsGeom g) {
    extern __shared__ uint8_t smem_raw[];
    const RowsSmem sm = rows_smem(smem_raw, g);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int tr = lane >> 2, tc = lane & 3;
    // Per-warp task bookkeeping lives in shared memory (sm.rec) or is
    // recomputed from the launch indices where it is needed, so that the
    // accumulators and the operands of the inner loop own the registers.
    const int gw = blockIdx.x * kRowsWarps + warp;
    const int cnt = gw < g.NQ ? (g.NQ - 1 - gw) / (gridDim.x * kRowsWarps) + 1 : 0;  // tasks per block
    volatile int *rec = sm.rec + 4 * warp;
    uint64_t *full = sm.full + warp * g.stages;
    float *ring = sm.win + warp * g.stages * g.box_stride;

    if (lane == 0) {
        for (int st = 0; st < g.stages; ++st) mbar_init(&full[st], 1);
        if (warp == 0) *sm.abort_flag = 0;
        fence_mbar_init();
        if (warp == 0) prefetch_tensormap(&mapX);
    }
    __syncthreads();
    // Start the window stream before the weights: the copies overlap the
    // weight transpose.
    if (lane == 0) {
        const int total = cnt * g.nch * g.nblocks;
        int issued = 0;
        for (; issued < g.stages && issued < total; ++issued)
            issue_chunk<PAD>(g, &mapX, ring + issued * g.box_stride, &full[issued], issued, cnt * g.nch,
                             gw, gridDim.x * kRowsWarps);
        rec[1] = issued;
        rec[2] = 0;
    }
    __syncwarp();

    // The thread's input window in a stage: the box column of its first
    // tap, rounded down to an 8-byte boundary (POFF = the remainder).
    constexpr int POFF = (PAD + 4 * ((PAD + 3) / 4)) & 1;
    constexpr int NV = (kRowsTN + KS - 1 + POFF + 1) / 2 * 2;  // window values loaded per row

    bool aborted = false;
    for (int b = 0; b < g.nblocks; ++b) {
        // ---- weight block b, transposed into shared memory by every thread
        __syncthreads();
        load_weight_block(g, sm.wT, b);
        __syncthreads();
        if (*reinterpret_cast<volatile int *>(sm.abort_flag)) aborted = true;

        for (int r = 0; r < cnt; ++r) {
            int toff;  // this thread's window offset in a stage: row row0, column wcol
            {
                const int t = gw + r * gridDim.x * kRowsWarps;
                const int n = t / g.Q, q = t - n * g.Q;
                const int seg = 4 * q + tc;
                const int oy = seg / g.SR;
                const int ox0 = (seg - oy * g.SR) * kRowsTN;
                toff = (oy - (4 * q) / g.SR) * g.BW + ox0 - PAD - g.x0 - POFF;
            }
            if (lane == 0) rec[0] = (b * cnt + r) * g.nch;
            __syncwarp();

            float2 acc[4][kRowsTN];
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int j = 0; j < kRowsTN; ++j) acc[p][j] = make_float2(0.0f, 0.0f);

            // One loop over the task's input channels (the accumulators stay
            // in one loop nest); at each stage boundary the finished stage is
            // handed back to the copy engine and the next one awaited.
            int left = 0;                            // channels left in the stage
            const float *cwin = ring;                // this thread's window rows of channel c
            const float *wk = sm.wT + 4 * tr;        // weight rows of channel c's taps
            for (int c = 0; c < g.cin_g && !aborted; ++c) {
                if (left == 0) {
                    const int ci = rec[0] + c / g.CC;  // chunk index of channel c
                    if (c != 0) {
                        __syncwarp();
                        if (lane == 0) {
                            const int issued = rec[1];
                            const int per_block = cnt * g.nch;
                            if (issued < per_block * g.nblocks) {
                                // every lane's reads of the finished stage are done
                                // (syncwarp); order them before the async proxy
                                // overwrites it
                                const int sp = (ci - 1) % g.stages;
                                fence_proxy_async_smem();
                                issue_chunk<PAD>(g, &mapX, ring + sp * g.box_stride, &full[sp], issued,
                                                 per_block, gw, gridDim.x * kRowsWarps);
                                rec[1] = issued + 1;
                            }
                        }
                    }
                    const int sl = ci % g.stages;
                    if (!mbar_wait(&full[sl], static_cast<uint32_t>((ci / g.stages) & 1))) {
                        rows_record_timeout(g.status, sm.abort_flag);
                        aborted = true;
                        break;
                    }
                    if (lane == 0) rec[2] = ci + 1;
                    cwin = ring + sl * g.box_stride + toff;
                    left = min(g.CC, g.cin_g - c);
                }
                --left;
                if constexpr (KS == 1) {
                    // 1x1: channel pairs with the input value broadcast
                    float2 bp[kRowsTN / 2];
#pragma unroll
                    for (int u = 0; u < kRowsTN / 2; ++u) bp[u] = *reinterpret_cast<const float2 *>(cwin + 2 * u);
                    const float4 a0 = *reinterpret_cast<const float4 *>(wk);
                    const float4 a1 = *reinterpret_cast<const float4 *>(wk + 32);
                    const float2 ap[4] = {make_float2(a0.x, a0.y), make_float2(a0.z, a0.w),
                                          make_float2(a1.x, a1.y), make_float2(a1.z, a1.w)};
#pragma unroll
                    for (int u = 0; u < kRowsTN / 2; ++u) {
                        const float2 bx = make_float2(bp[u].x, bp[u].x);
                        const float2 by = make_float2(bp[u].y, bp[u].y);
#pragma unroll
                        for (int p = 0; p < 4; ++p) {
                            acc[p][2 * u] = pterm<MODE>(acc[p][2 * u], bx, ap[p]);
                            acc[p][2 * u + 1] = pterm<MODE>(acc[p][2 * u + 1], by, ap[p]);
                        }
                    }
                    wk += kRowsMB;
                } else {
#pragma unroll 1
                    for (int ky = 0; ky < KS; ++ky) {
                        // window row row0 + ky of channel c in the stage
                        const float *wr0 = cwin + ky * g.BW;
                        float v[NV];
#pragma unroll
                        for (int u = 0; u < NV / 2; ++u) {
                            const float2 t2 = *reinterpret_cast<const float2 *>(wr0 + 2 * u);
                            v[2 * u] = t2.x;
                            v[2 * u + 1] = t2.y;
                        }
                        // the two channel pairs of each half of the thread's
                        // eight channels, per kernel column
                        float2 ap[KS][4];
#pragma unroll
                        for (int kx = 0; kx < KS; ++kx) {
                            const float *wr = wk + (ky * KS + kx) * kRowsMB;
                            const float4 a0 = *reinterpret_cast<const float4 *>(wr);
                            const float4 a1 = *reinterpret_cast<const float4 *>(wr + 32);
                            ap[kx][0] = make_float2(a0.x, a0.y);
                            ap[kx][1] = make_float2(a0.z, a0.w);
                            ap[kx][2] = make_float2(a1.x, a1.y);
                            ap[kx][3] = make_float2(a1.z, a1.w);
                        }
                        // per output the kernel columns go in order: output j
                        // of column kx reads window value j + kx
#pragma unroll
                        for (int j = 0; j < kRowsTN; ++j) {
#pragma unroll
                            for (int kx = 0; kx < KS; ++kx) {
                                const float bv = v[j + kx + POFF];
                                const float2 b2 = make_float2(bv, bv);
#pragma unroll
                                for (int p = 0; p < 4; ++p) acc[p][j] = pterm<MODE>(acc[p][j], b2, ap[kx][p]);
                            }
                        }
                    }
                    wk += KS * KS * kRowsMB;
                }
                cwin += g.BH * g.BW;
            }
            __syncwarp();
            if (aborted) continue;
            // ---- epilogue through the last stage (the next copy into it is
            // issued afterwards): per channel slot cs, the eight thread rows'
            // channels 8*tr + cs as eight rows of the warp's four segments,
            // then 8-byte stores along output rows.
            {
                const int last = rec[0] + g.nch - 1;
                const int sl = last % g.stages;
                float *stg = ring + sl * g.box_stride;
                const int t = gw + r * gridDim.x * kRowsWarps;
                const int n = t / g.Q, q = t - n * g.Q;
                const int grp = b / g.mblocks, mb = b - grp * g.mblocks;
                const int ch_base = grp * g.M + mb * kRowsMB;
                const int64_t ybase = static_cast<int64_t>(n) * g.Cout * g.OH * g.OW;
                int seg_off[4];
#pragma unroll
                for (int sg = 0; sg < 4; ++sg) {
                    const int gs = 4 * q + sg;
                    const int ory = gs / g.SR;
                    seg_off[sg] = ory * g.OW + (gs - ory * g.SR) * kRowsTN;
                }
#pragma unroll
                for (int cs = 0; cs < 8; ++cs) {
#pragma unroll
                    for (int j = 0; j < kRowsTN; j += 2) {
                        const float2 o = (cs & 1) ? make_float2(acc[cs >> 1][j].y, acc[cs >> 1][j + 1].y)
                                                  : make_float2(acc[cs >> 1][j].x, acc[cs >> 1][j + 1].x);
                        *reinterpret_cast<float2 *>(stg + tr * kRowsStagePitch + tc * kRowsTN + j) = o;
                    }
                    __syncwarp();
                    store_slice<HAS_EP>(g, stg, lane, ybase, seg_off[0], seg_off[1], seg_off[2], seg_off[3],
                                        ch_base + cs);
                    __syncwarp();
                }
                if (lane == 0) {
                    const int issued = rec[1];
                    const int per_block = cnt * g.nch;
                    if (issued < per_block * g.nblocks) {
                        fence_proxy_async_smem();
                        issue_chunk<PAD>(g, &mapX, ring + sl * g.box_stride, &full[sl], issued, per_block, gw,
                                         gridDim.x * kRowsWarps);
                        rec[1] = issued + 1;
                    }
                }
            }
        }
    }
    // Copies still in flight (only after a timeout) must land before the
    // CTA's shared memory is released.
    __syncwarp();
    if (lane == 0) {
        for (int j = rec[2]; j < rec[1]; ++j)
            (void)mbar_wait(&full[j % g.stages], static_cast<uint32_t>((j / g.stages) & 1));
    }
}

// -------------------------------------------------------------- host side
namespace {

PFN_cuTensorMapEncodeTiled_v12000 rows_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                             &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        }
    }
    return fn;
}

// x as a 4-D tensor (W, H, Cin, N), box (BW, BH, CC, 1), zero fill outside.
bool make_input_map(CUtensorMap *map, const ConvProblem &p, const RowsGeom &g) {
    auto fn = rows_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[4] = {static_cast<cuuint64_t>(p.W), static_cast<cuuint64_t>(p.H),
                          static_cast<cuuint64_t>(p.Cin), static_cast<cuuint64_t>(p.N)};
    cuuint64_t strides[3] = {static_cast<cuuint64_t>(p.W) * 4, static_cast<cuuint64_t>(p.H * p.W) * 4,
                             static_cast<cuuint64_t>(p.Cin * p.H * p.W) * 4};
    cuuint32_t box[4] = {static_cast<cuuint32_t>(g.BW), static_cast<cuuint32_t>(g.BH),
                         static_cast<cuuint32_t>(g.CC), 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, const_cast<float *>(p.x), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int MODE, int KS, int PAD>
cudaError_t launch_rows(const ConvProblem &p, const RowsGeom &g, int grid, int smem, cudaStream_t s) {
    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    if (!make_input_map(&map, p, g)) return cudaErrorNotSupported;
    const bool has_ep = p.ep.bias || p.ep.res || p.ep.act;
    void (*kernel)(const CUtensorMap, RowsGeom) =
        has_ep ? conv_rows_kernel<MODE, KS, PAD, true> : conv_rows_kernel<MODE, KS, PAD, false>;
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return e;
    kernel<<<static_cast<unsigned>(grid), kRowsThreads, static_cast<size_t>(smem), s>>>(map, g);
    return cudaGetLastError();
}

}  // namespace

// Output pixels per warp task row segment, and the geometry checks of the
// row kernel; false when the problem is not its shape.
bool conv_rows_geometry(const ConvProblem &p, int *tasks) {
    const bool k3 = p.KW == 3 && p.pL == 1 && p.pT == 1;
    const bool k1 = p.KW == 1 && p.pL == 0 && p.pT == 0;
    if (!(k3 || k1) || p.KH != p.KW) return false;
    if (p.sH != 1 || p.sW != 1 || p.dH != 1 || p.dW != 1) return false;
    const int64_t M = p.Cout / p.G;
    if (M % kRowsMB != 0) return false;
    if (p.OW % kRowsTN != 0) return false;
    const int64_t SR = p.OW / kRowsTN;
    if (!(SR == 1 || SR == 2 || SR == 4 || SR % 4 == 0)) return false;
    if ((p.OH * SR) % 4 != 0) return false;
    if (p.W % 4 != 0 || (reinterpret_cast<uintptr_t>(p.x) & 15) != 0) return false;
    if ((reinterpret_cast<uintptr_t>(p.y) & 7) != 0) return false;
    if (p.ep.res && (reinterpret_cast<uintptr_t>(p.ep.res) & 7) != 0) return false;
    if (p.W > 248 || p.N > 0x7FFFFFFF) return false;
    const int64_t nq = p.N * (p.OH * SR / 4);
    const int64_t t = nq * p.G * (M / kRowsMB);
    if (nq > 0x3FFFFFFF || t > 0x3FFFFFFF) return false;
    if (tasks) *tasks = static_cast<int>(t);
    return true;
}

cudaError_t launch_conv_rows(const ConvProblem &p, int mode, bool choose, cudaStream_t s) {
    int tasks = 0;
    if (!conv_rows_geometry(p, &tasks)) return cudaErrorNotSupported;
    const int sms = num_sms();
    // By itself the dispatcher takes this kernel for 3x3 kernels whose warp
    // tasks fill most of one round of kRowsWarps warps on every SM, or
    // several (1x1 kernels measured faster in the implicit GEMM: 81 against
    // 90 us on the ResNet-50 stage-1 1x1 layer at batch 32).
    if (choose && p.KW == 1) return cudaErrorNotSupported;
    if (choose) {
        const int64_t slots = static_cast<int64_t>(sms) * kRowsWarps;
        const int64_t rounds = (tasks + slots - 1) / slots;
        if (static_cast<double>(tasks) / static_cast<double>(rounds * slots) < 0.8) return cudaErrorNotSupported;
    }
    RowsGeom g;
    memset(&g, 0, sizeof(g));
    g.y = p.y;
    g.w = p.w;
    g.Cin = static_cast<int>(p.Cin);
    g.Cout = static_cast<int>(p.Cout);
    g.cin_g = static_cast<int>(p.Cin / p.G);
    g.M = static_cast<int>(p.Cout / p.G);
    g.KH = static_cast<int>(p.KH);
    g.OH = static_cast<int>(p.OH);
    g.OW = static_cast<int>(p.OW);
    g.K = static_cast<int>(p.K);
    g.w_ld = static_cast<int>(p.w_ld);
    g.SR = static_cast<int>(p.OW / kRowsTN);
    g.Q = static_cast<int>(p.OH * g.SR / 4);
    g.NQ = static_cast<int>(p.N) * g.Q;
    g.mblocks = g.M / kRowsMB;
    g.nblocks = static_cast<int>(p.G) * g.mblocks;
    const int KW = static_cast<int>(p.KW), PAD = static_cast<int>(p.pL);
    g.w_vec = (g.K % 4 == 0) && (g.w_ld % 4 == 0) && ((reinterpret_cast<uintptr_t>(p.w) & 15) == 0);
    const int RQ = g.SR >= 4 ? 1 : 4 / g.SR;  // output rows per task
    g.BH = RQ - 1 + g.KH;
    g.x0 = -4 * ((PAD + 3) / 4);
    const int poff = (PAD - g.x0) & 1;
    const int nv = (kRowsTN + KW - 1 + poff + 1) / 2 * 2;
    const int max_col = (g.SR - 1) * kRowsTN + (-PAD - g.x0 - poff) + nv - 1;
    g.BW = (max_col + 1 + 3) / 4 * 4;
    if (g.BW > 256 || g.BH > 256) return cudaErrorNotSupported;
    g.ep = p.ep;
    g.status = p.status;
    // Stage size: as many input channels as fit with two or three stages per
    // warp beside the weight block (at most 32; a stage also holds the
    // epilogue's 8 x 60-float staging rows).
    const int64_t wt_bytes = static_cast<int64_t>(g.K) * kRowsMB * 4;
    const int64_t budget = static_cast<int64_t>(max_smem_optin()) - wt_bytes - 128 - 16 - kRowsWarps * 16 -
                           static_cast<int64_t>(kRowsWarps) * 3 * 8;
    const int64_t row_floats = static_cast<int64_t>(g.BW) * g.BH;
    int best_cc = 0, best_st = 0;
    for (int st = 3; st >= 2 && best_cc == 0; --st) {
        for (int cc = (g.cin_g < 32 ? g.cin_g : 32); cc >= 1; --cc) {
            const int64_t stride = (row_floats * cc + 31) / 32 * 32;  // 128-byte aligned stages
            if (stride < 8 * kRowsStagePitch) continue;
            if (static_cast<int64_t>(kRowsWarps) * st * stride * 4 <= budget) {
                // three stages only when they keep at least 8 channels each
                if (st == 3 && cc < 8 && cc < g.cin_g) break;
                best_cc = cc;
                best_st = st;
                break;
            }
        }
    }
    if (best_cc == 0) return cudaErrorNotSupported;
    g.CC = best_cc;
    g.stages = best_st;
    g.nch = (g.cin_g + g.CC - 1) / g.CC;
    g.box_floats = g.BW * g.BH * g.CC;
    g.box_stride = (g.box_floats + 31) / 32 * 32;
    const int64_t smem = wt_bytes + static_cast<int64_t>(kRowsWarps) * g.stages * g.box_stride * 4 +
                         static_cast<int64_t>(kRowsWarps) * g.stages * 8 + 16 + kRowsWarps * 16 + 128;
    if (smem > max_smem_optin()) return cudaErrorNotSupported;
    const int64_t nwarps_needed = (static_cast<int64_t>(g.NQ) + 0);
    int64_t grid = (nwarps_needed + kRowsWarps - 1) / kRowsWarps;
    if (grid > sms) grid = sms;
    if (grid < 1) grid = 1;
    const int sm = static_cast<int>(smem);
    if (KW == 3 && PAD == 1)
        return mode == kFast ? launch_rows<kFast, 3, 1>(p, g, static_cast<int>(grid), sm, s)
                             : launch_rows<kExact, 3, 1>(p, g, static_cast<int>(grid), sm, s);
    if (KW == 1 && PAD == 0)
        return mode == kFast ? launch_rows<kFast, 1, 0>(p, g, static_cast<int>(grid), sm, s)
                             : launch_rows<kExact, 1, 0>(p, g, static_cast<int>(grid), sm, s);
    return cudaErrorNotSupported;
}

cudaError_t read_clear_status_rows(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status_rows, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*out) e = cudaMemcpyToSymbol(g_status_rows, &zero, sizeof(unsigned));
    return e;
}

}  // namespace om
