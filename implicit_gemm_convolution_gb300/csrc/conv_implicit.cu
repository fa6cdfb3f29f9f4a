// conv_implicit.cu -- NCHW 2-D convolution as an implicit matrix product on
// the CUDA cores of sm_103a, bit-exact in both modes.
//
// What each output is ("Exact mode" page, section "Convolution"; "Convolution
// (fast mode)" page, section "What each output is"): output (n, oc, oy, ox)
// of group g sums, for taps p = (c*KH + ky)*KW + kx in increasing order, the
// term w[oc][c][ky][kx] * v with
//   v = x[n][g*Cin/G + c][oy*s - pad + ky*d][ox*s - pad + kx*d]
// inside the plane and +0 outside; padding taps are real products, so an
// infinite or NaN weight meeting padding gives NaN. NaN is stored as
// 0x7FC00000.
//
// The product per group g ("Convolution (fast mode)", section "Layout of the
// work"): A = the group's weights, Cout/G rows by K = Cin/G*KH*KW taps; B = the
// patches, K rows by N*OutH*OutW columns (all images of the call side by side:
// every output is independent, so merging images changes no bit); C = the
// group's output planes. B is never built: the producer warpgroup gathers each
// 32-tap x BN-column strip straight from the input planes into shared memory
// with 4-byte cp.async, writing +0 (src-size 0) for taps outside the plane --
// the zero border is written during the gather, never materialised. Weight
// tiles come by TMA when the weight rows are 16-byte aligned (always for the
// packed layout), else by 4-byte cp.async. The consumer warpgroups run the
// same register-tile loop as the matrix product (simt_tile.cuh), so every
// output accumulates its taps in order from +0 in one thread's registers.
#include <cudaTypedefs.h>

#include <cstring>

#include "om_internal.h"
#include "schedule_host.h"
#include "simt_tile.cuh"

namespace om {

__device__ unsigned g_status_conv;

// The gather runs on one producer warpgroup, each thread keeping its
// columns' state in registers; copying A with cp.async as well needs more.
constexpr int kConvProducers = 128;
template <bool A_TMA>
constexpr int kConvProducerRegs = A_TMA ? 72 : 88;

// Geometry the kernel reads (all per-image quantities fit in 32 bits; the
// host validated Cin*H*W, Cout*OH*OW and K below 2^31).
struct ConvGeom {
    const float *x;
    const float *w;
    float *y;
    int64_t ncols;  // N * OH * OW
    int H, W, HW, OH, OW, P;  // P = OH*OW
    int Cin, Cout, cin_g, M;  // M = Cout/G
    int KH, KW, sH, sW, pT, pL, dH, dW;
    int K, w_ld;
    int tiles_m, tiles_n, G;
    Epilogue ep;
    unsigned *status;  // the call's status word in a caller workspace, or NULL
};

__device__ __forceinline__ void conv_record_timeout(unsigned *status, int *abort_flag) {
    report_timeout(status, &g_status_conv);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
}

// Tile t -> (m tile, column tile, group); the m tiles of one column strip are
// adjacent so they run together and share the gathered input through L2.
__device__ __forceinline__ void conv_tile(const ConvGeom &g, int t, int &tm, int64_t &tn,
                                          int &grp) {
    tm = t % g.tiles_m;
    const int r = t / g.tiles_m;
    tn = r % g.tiles_n;
    grp = r / g.tiles_n;
}

// Gather kinds: the general per-element gather; the masked gather (kernels
// of up to 32 taps per channel, input below 2^31 elements, tap table in
// shared memory); and the in-place copy of a 1x1, stride-1, unpadded
// convolution (B is the input planes themselves; four consecutive pixels of
// one channel per 16-byte copy).
enum GatherKind : int { kGatherGeneral = 0, kGatherMasked = 1, kGather1x1 = 2 };

// Shared-memory bytes of the masked gather's tap table: per tap p (padded
// to whole k blocks) its input offset c*H*W + ky*dH*W + kx*dW and the bit
// 1 << (ky*KW + kx), or 0 past K.
template <class Cfg>
inline int64_t conv_tap_table_bytes(int64_t K) {
    return (K + Cfg::BK - 1) / Cfg::BK * Cfg::BK * 8;
}

template <class Cfg, bool A_TMA, int GATHER>
__device__ __forceinline__ void conv_produce(const ConvGeom &g, const CUtensorMap *mapW,
                                             uint8_t *smem, uint64_t *full, uint64_t *empty,
                                             int *abort_flag, const Schedule &sched, int pt,
                                             uint8_t *tap_table) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK;
    constexpr int CPT = BN / kConvProducers;  // gathered columns per producer thread
    static_assert(BN % kConvProducers == 0, "columns split evenly over the producers");
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    const int taps_per_channel = g.KH * g.KW;
    constexpr bool MASKED = GATHER == kGatherMasked;
    const uint32_t tab32 = smem_u32(tap_table);
    if constexpr (MASKED) {
        const int kpad = (g.K + BK - 1) / BK * BK;
        for (int p = pt; p < kpad; p += kConvProducers) {
            const int c = p / taps_per_channel;
            const int t = p - c * taps_per_channel;
            const int ky = t / g.KW, kx = t - (t / g.KW) * g.KW;
            const int off = c * g.HW + ky * g.dH * g.W + kx * g.dW;
            reinterpret_cast<int2 *>(tap_table)[p] = make_int2(off, p < g.K ? static_cast<int>(1u << t) : 0);
        }
        asm volatile("bar.sync 2, %0;" ::"n"(kConvProducers) : "memory");
    }
    const Schedule::Local L = sched.local();
    for (int si = 0; si < L.count; ++si) {
        const Segment sg = sched.at(L, si);
        int tm, grp;
        int64_t tn;
        conv_tile(g, sg.tile, tm, tn, grp);
        // Per gathered column: the group's first input plane of its image and
        // the input coordinates of tap (0, 0).
        const float *base[CPT];
        int iy0[CPT], ix0[CPT];
        bool cvalid[CPT];
#pragma unroll
        for (int j = 0; j < CPT; ++j) {
            const int64_t col = tn * BN + pt + kConvProducers * j;
            cvalid[j] = col < g.ncols;
            const int64_t img = cvalid[j] ? col / g.P : 0;
            const int pix = cvalid[j] ? static_cast<int>(col - img * g.P) : 0;
            const int oy = pix / g.OW, ox = pix - (pix / g.OW) * g.OW;
            base[j] = g.x + (img * g.Cin + static_cast<int64_t>(grp) * g.cin_g) * g.HW;
            iy0[j] = oy * g.sH - g.pT;
            ix0[j] = ox * g.sW - g.pL;
        }
        const int row0 = grp * g.M + tm * BM;  // first weight row of the tile
        // tap state of the segment's first tap p = (c*KH + ky)*KW + kx
        const int p0 = sg.kb * BK;
        int c = p0 / taps_per_channel;
        int ky = (p0 - c * taps_per_channel) / g.KW;
        int kx = p0 - c * taps_per_channel - ky * g.KW;
        // Masked gather: per column the offset of its tap-(0,0) position (an
        // int: the input has fewer than 2^31 elements) and which taps lie in
        // the plane.
        uint32_t mask[CPT];
        int coloff[CPT];
        if constexpr (MASKED) {
#pragma unroll
            for (int j = 0; j < CPT; ++j) {
                coloff[j] = static_cast<int>((base[j] - g.x) + static_cast<int64_t>(iy0[j]) * g.W + ix0[j]);
                uint32_t mk = 0;
                if (cvalid[j]) {
                    for (int y = 0; y < g.KH; ++y) {
                        const bool yok = static_cast<unsigned>(iy0[j] + y * g.dH) < static_cast<unsigned>(g.H);
                        for (int x = 0; x < g.KW; ++x) {
                            const bool xok = static_cast<unsigned>(ix0[j] + x * g.dW) < static_cast<unsigned>(g.W);
                            if (yok && xok) mk |= 1u << (y * g.KW + x);
                        }
                    }
                }
                mask[j] = mk;
            }
        }
        for (int kt = sg.kb; kt < sg.ke; ++kt) {
            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                conv_record_timeout(g.status, abort_flag);
                cp_async_wait_all();
                if (A_TMA && pt == 0) {
                    // let the weight tiles already requested land first
                    for (int s2 = 0; s2 < Cfg::STAGES; ++s2) {
                        if (issued > s2) {
                            const int64_t last = s2 + ((issued - 1 - s2) / Cfg::STAGES) * Cfg::STAGES;
                            (void)mbar_wait(&full[s2], static_cast<uint32_t>((last / Cfg::STAGES) & 1));
                        }
                    }
                }
                return;
            }
            ++issued;
            uint8_t *sa = smem + stage * Cfg::STAGE_BYTES;
            const uint32_t sa32 = smem_u32(sa);
            const uint32_t sb32 = sa32 + Cfg::A_BYTES;
            if constexpr (A_TMA) {
                if (pt == 0) {
                    mbar_arrive_expect_tx(&full[stage], Cfg::A_BYTES);
                    tma_load_2d(sa, mapW, &full[stage], kt * BK, row0);
                }
            } else {
                // rows of this group only; +0 past the group's rows and past K
                const int kk = pt % 32;
                const int p = kt * BK + kk;
                for (int r = pt / 32; r < BM; r += kConvProducers / 32) {
                    const int mrow = tm * BM + r;
                    const bool ok = (mrow < g.M) && (p < g.K);
                    const float *src = ok ? g.w + static_cast<int64_t>(row0 + r) * g.w_ld + p : g.w;
                    cp_async_4(sa32 + a_tile_offset(r, kk), src, ok ? 4u : 0u);
                }
            }
            // Gather the 32 taps of this stage for the thread's columns.
            if constexpr (GATHER == kGather1x1) {
                // thread pt copies pixels 4*(pt % 64) .. +3 of the tile for the
                // channels of parity pt / 64; each group of four is one image
                // (OH*OW is a multiple of 4) and 16-byte aligned
                const int q = pt % (BN / 4);
                const int64_t col = tn * BN + 4 * q;
                const bool col_ok = col < g.ncols;
                const int64_t img = col_ok ? col / g.P : 0;
                const int64_t pix = col - img * g.P;
                const float *cbase = g.x + (img * g.Cin + static_cast<int64_t>(grp) * g.cin_g) * g.HW + pix;
                constexpr int kRowsPerPass = kConvProducers / (BN / 4);
#pragma unroll 4
                for (int kk = pt / (BN / 4); kk < BK; kk += kRowsPerPass) {
                    const int ch = kt * BK + kk;
                    const bool ok = col_ok && ch < g.K;
                    const float *src = ok ? cbase + static_cast<int64_t>(ch) * g.HW : g.x;
                    cp_async_16(sb32 + (kk * BN + 4 * q) * 4, src, ok ? 16u : 0u);
                }
            } else if constexpr (MASKED) {
                // tap p is in the plane for column j iff mask[j] has the tap's
                // bit; its input element is then coloff[j] + the tap's offset
                const uint32_t trow = tab32 + kt * BK * 8;
#pragma unroll 8
                for (int kk = 0; kk < BK; ++kk) {
                    const int2 e = lds_int2(trow + kk * 8);
#pragma unroll
                    for (int j = 0; j < CPT; ++j) {
                        const bool ok = (mask[j] & static_cast<uint32_t>(e.y)) != 0u;
                        const int off = ok ? coloff[j] + e.x : 0;
                        cp_async_4_if(sb32 + (kk * BN + pt + kConvProducers * j) * 4, g.x + off, ok);
                    }
                }
            } else {
#pragma unroll 4
                for (int kk = 0; kk < BK; ++kk) {
                    const int p = kt * BK + kk;
                    const bool tap_ok = p < g.K;
                    const int dy = ky * g.dH, dx = kx * g.dW;
                    const int plane = tap_ok ? c * g.HW : 0;
#pragma unroll
                    for (int j = 0; j < CPT; ++j) {
                        const int iy = iy0[j] + dy, ix = ix0[j] + dx;
                        const bool ok = tap_ok && cvalid[j] && static_cast<unsigned>(iy) < static_cast<unsigned>(g.H) &&
                                        static_cast<unsigned>(ix) < static_cast<unsigned>(g.W);
                        const float *src = ok ? base[j] + (plane + iy * g.W + ix) : g.x;
                        cp_async_4(sb32 + (kk * BN + pt + kConvProducers * j) * 4, src, ok ? 4u : 0u);
                    }
                    if (++kx == g.KW) {
                        kx = 0;
                        if (++ky == g.KH) {
                            ky = 0;
                            ++c;
                        }
                    }
                }
            }
            cp_async_arrive_noinc(&full[stage]);
            if (++stage == Cfg::STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
    }
    cp_async_wait_all();
}

// Moves this thread's outputs of a tile between registers and y. Row i of
// the tile is output channel grp*M + tm*BM + i; column j is (image, pixel) =
// divmod(j, OH*OW). OP 0: final store (canonical NaN); 1: raw store of an
// early part's accumulators; 2: load of the accumulators an earlier CTA stored.
template <class Cfg, int OP, bool HAS_EP>
__device__ __forceinline__ void conv_tile_io(const ConvGeom &g, Accum<Cfg> &acc, int tm,
                                             int64_t tn, int grp, int arow0, int bcol0) {
    const bool vec_ok = (g.P % 4 == 0) && ((reinterpret_cast<uintptr_t>(g.y) & 15) == 0);
#pragma unroll
    for (int q = 0; q < Cfg::TN / 4; ++q) {
        const int64_t col = tn * Cfg::BN + bcol0 + 16 * q;
        if (col >= g.ncols) continue;
        const int64_t img = col / g.P;
        const int pix = static_cast<int>(col - img * g.P);
        const bool vec = vec_ok && (col + 3 < g.ncols);
#pragma unroll
        for (int i = 0; i < Cfg::TM; ++i) {
            const int mrow = tm * Cfg::BM + arow0 + 8 * i;
            if (mrow >= g.M) continue;
            const int oc = grp * g.M + mrow;
            float *dst = g.y + (img * g.Cout + oc) * static_cast<int64_t>(g.P) + pix;
            if constexpr (OP == 2) {
                float e[4] = {0.0f, 0.0f, 0.0f, 0.0f};
                if (vec) {
                    const float4 v = __ldcg(reinterpret_cast<const float4 *>(dst));
                    e[0] = v.x; e[1] = v.y; e[2] = v.z; e[3] = v.w;
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int64_t cu = col + u;
                        if (cu >= g.ncols) break;
                        const int64_t iu = cu / g.P;
                        e[u] = __ldcg(g.y + (iu * g.Cout + oc) * static_cast<int64_t>(g.P) + (cu - iu * g.P));
                    }
                }
                acc.v[i][2 * q] = make_float2(e[0], e[1]);
                acc.v[i][2 * q + 1] = make_float2(e[2], e[3]);
            } else {
                float e[4] = {acc.v[i][2 * q].x, acc.v[i][2 * q].y, acc.v[i][2 * q + 1].x,
                              acc.v[i][2 * q + 1].y};
                if (vec) {
                    // four columns of one image: consecutive outputs from dst
                    if constexpr (OP == 0) {
                        const int64_t o = dst - g.y;
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (HAS_EP)
                                e[u] = epilogue_value(e[u], g.ep.bias ? g.ep.bias + oc : nullptr,
                                                      g.ep.res ? g.ep.res + o + u : nullptr, g.ep.act);
                            e[u] = canonical_nan(e[u]);
                        }
                    }
                    *reinterpret_cast<float4 *>(dst) = make_float4(e[0], e[1], e[2], e[3]);
                } else {
#pragma unroll
                    for (int u = 0; u < 4; ++u) {
                        const int64_t cu = col + u;
                        if (cu >= g.ncols) break;
                        const int64_t iu = cu / g.P;
                        const int64_t o = (iu * g.Cout + oc) * static_cast<int64_t>(g.P) + (cu - iu * g.P);
                        float v = e[u];
                        if constexpr (OP == 0) {
                            if (HAS_EP)
                                v = epilogue_value(v, g.ep.bias ? g.ep.bias + oc : nullptr,
                                                   g.ep.res ? g.ep.res + o : nullptr, g.ep.act);
                            v = canonical_nan(v);
                        }
                        g.y[o] = v;
                    }
                }
            }
        }
    }
}

template <int MODE, class Cfg, bool A_TMA, bool HAS_EP, int GATHER>
__global__ void __launch_bounds__(Cfg::CONSUMERS + kConvProducers, 1)
    conv_implicit_kernel(const __grid_constant__ CUtensorMap mapW, ConvGeom g, Schedule sched) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem<Cfg>(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::STAGES * Cfg::STAGE_BYTES);
    uint64_t *empty = full + Cfg::STAGES;
    int *abort_flag = reinterpret_cast<int *>(empty + Cfg::STAGES);
    uint8_t *tap_table = smem + Cfg::STAGES * Cfg::STAGE_BYTES + 256;
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            // every producer thread arrives after its copies land; with TMA
            // weights, producer thread 0 also arrives with the byte count
            mbar_init(&full[s], kConvProducers + (A_TMA ? 1 : 0));
            mbar_init(&empty[s], Cfg::CONSUMER_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    if (warp >= Cfg::CONSUMER_WARPS) {
        RegSplit<kConvProducerRegs<A_TMA>, kConvProducers, Cfg::CONSUMERS>::producer();
        if constexpr (A_TMA) {
            if (threadIdx.x == Cfg::CONSUMERS) prefetch_tensormap(&mapW);
        }
        conv_produce<Cfg, A_TMA, GATHER>(g, &mapW, smem, full, empty, abort_flag, sched,
                                         threadIdx.x - Cfg::CONSUMERS, tap_table);
        return;
    }

    RegSplit<kConvProducerRegs<A_TMA>, kConvProducers, Cfg::CONSUMERS>::consumer();
    const int ty = lane / 4, tx = lane % 4;
    const int arow0 = (warp / Cfg::WARPS_N) * Cfg::WM + ty;
    const int bcol0 = (warp % Cfg::WARPS_N) * Cfg::WN + tx * 4;
    int stage = 0;
    uint32_t phase = 0;
    const Schedule::Local L = sched.local();
    for (int si = 0; si < L.count; ++si) {
        const Segment sg = sched.at(L, si);
        int tm, grp;
        int64_t tn;
        conv_tile(g, sg.tile, tm, tn, grp);
        Accum<Cfg> acc;
        acc.zero();
        if (sg.kind == kSegLate) {
            if (!wait_previous_part(sched.flags, Cfg::CONSUMERS, abort_flag)) {
                report_timeout(g.status, &g_status_conv);
                return;
            }
            conv_tile_io<Cfg, 2, false>(g, acc, tm, tn, grp, arow0, bcol0);
        }
        for (int kt = sg.kb; kt < sg.ke; ++kt) {
            if (!mbar_wait(&full[stage], phase)) {
                conv_record_timeout(g.status, abort_flag);
                return;
            }
            const float *As = reinterpret_cast<const float *>(smem + stage * Cfg::STAGE_BYTES);
            const float *Bs = reinterpret_cast<const float *>(smem + stage * Cfg::STAGE_BYTES + Cfg::A_BYTES);
            mma_stage<MODE, Cfg>(acc, As, Bs, arow0, bcol0, ty);
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[stage]);
            if (++stage == Cfg::STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
        if (sg.kind == kSegEarly) {
            conv_tile_io<Cfg, 1, false>(g, acc, tm, tn, grp, arow0, bcol0);
            signal_early_part(sched.flags, Cfg::CONSUMERS);
        } else {
            conv_tile_io<Cfg, 0, HAS_EP>(g, acc, tm, tn, grp, arow0, bcol0);
        }
    }
}

// -------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 conv_encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess) {
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
        }
    }
    return fn;
}

// Weight matrix Cout x K (row stride w_ld), box 32 taps x BM rows, 128B
// swizzle; taps >= K and rows >= Cout read as +0.
static bool make_weight_map(CUtensorMap *map, const ConvProblem &p, int box_rows) {
    auto fn = conv_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(p.Cout)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.w_ld) * 4};
    cuuint32_t box[2] = {32, static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(p.w), dims, strides, box,
              estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

using ConvCfg64x256 = TileCfg<64, 256, 8, 8, 1, 8, 4, true>;

template <int MODE, class Cfg>
static cudaError_t launch_conv_cfg(const ConvProblem &p, unsigned *flags, cudaStream_t s) {
    ConvGeom g;
    g.x = p.x; g.w = p.w; g.y = p.y;
    g.ncols = p.N * p.OH * p.OW;
    g.H = static_cast<int>(p.H); g.W = static_cast<int>(p.W); g.HW = static_cast<int>(p.H * p.W);
    g.OH = static_cast<int>(p.OH); g.OW = static_cast<int>(p.OW); g.P = static_cast<int>(p.OH * p.OW);
    g.Cin = static_cast<int>(p.Cin); g.Cout = static_cast<int>(p.Cout);
    g.cin_g = static_cast<int>(p.Cin / p.G); g.M = static_cast<int>(p.Cout / p.G);
    g.KH = static_cast<int>(p.KH); g.KW = static_cast<int>(p.KW);
    g.sH = static_cast<int>(p.sH); g.sW = static_cast<int>(p.sW);
    g.pT = static_cast<int>(p.pT); g.pL = static_cast<int>(p.pL);
    g.dH = static_cast<int>(p.dH); g.dW = static_cast<int>(p.dW);
    g.K = static_cast<int>(p.K); g.w_ld = static_cast<int>(p.w_ld);
    g.G = static_cast<int>(p.G);
    g.ep = p.ep;
    g.status = p.status;
    const int64_t tiles_m = (g.M + Cfg::BM - 1) / Cfg::BM;
    const int64_t tiles_n = (g.ncols + Cfg::BN - 1) / Cfg::BN;
    if (tiles_m * tiles_n * p.G > 0x7FFFFFFF || p.w_ld > 0x7FFFFFFF) return cudaErrorNotSupported;
    g.tiles_m = static_cast<int>(tiles_m);
    g.tiles_n = static_cast<int>(tiles_n);
    Schedule sched;
    make_schedule(static_cast<int>(tiles_m * tiles_n * p.G), (g.K + Cfg::BK - 1) / Cfg::BK, flags,
                  &sched);

    CUtensorMap map;
    memset(&map, 0, sizeof(map));
    const bool a_tma = ((reinterpret_cast<uintptr_t>(p.w) & 15) == 0) && (p.w_ld % 4 == 0) &&
                       make_weight_map(&map, p, Cfg::BM);
    const bool has_ep = p.ep.bias || p.ep.res || p.ep.act;
    // 1x1, stride 1, no padding, pixel counts multiples of 4, 16-byte aligned
    // input: B is the input planes, copied 16 bytes at a time
    const bool in_place = p.KH == 1 && p.KW == 1 && p.sH == 1 && p.sW == 1 && p.pT == 0 &&
                          p.pL == 0 && (p.OH * p.OW) % 4 == 0 && (p.H * p.W) % 4 == 0 &&
                          (reinterpret_cast<uintptr_t>(p.x) & 15) == 0;
    const int64_t table_bytes = conv_tap_table_bytes<Cfg>(p.K);
    const bool masked = p.KH * p.KW <= 32 && p.N * p.Cin * p.H * p.W <= 0x7FFFFFFF &&
                        Cfg::SMEM_BYTES + table_bytes <= max_smem_optin();
    const int gather = in_place ? kGather1x1 : (masked ? kGatherMasked : kGatherGeneral);
    const int smem_bytes = Cfg::SMEM_BYTES + (gather == kGatherMasked ? static_cast<int>(table_bytes) : 0);
    void (*kernel)(const CUtensorMap, ConvGeom, Schedule) = nullptr;
#define OM_CONV_PICK(T, E, G) \
    if (a_tma == T && has_ep == E && gather == G) kernel = conv_implicit_kernel<MODE, Cfg, T, E, G>;
#define OM_CONV_PICK_G(T, E)             \
    OM_CONV_PICK(T, E, kGatherGeneral)   \
    OM_CONV_PICK(T, E, kGatherMasked)    \
    OM_CONV_PICK(T, E, kGather1x1)
    OM_CONV_PICK_G(true, false)
    OM_CONV_PICK_G(true, true)
    OM_CONV_PICK_G(false, false)
    OM_CONV_PICK_G(false, true)
#undef OM_CONV_PICK_G
#undef OM_CONV_PICK
    const cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               smem_bytes);
    if (e != cudaSuccess) return e;
    cudaError_t el = launch_scheduled(kernel, sched, Cfg::CONSUMERS + kConvProducers, smem_bytes, s, map, g,
                                      sched);
    if (el == cudaErrorCooperativeLaunchTooLarge) {
        const Schedule whole = whole_tiles(sched);
        el = launch_scheduled(kernel, whole, Cfg::CONSUMERS + kConvProducers, smem_bytes, s, map, g, whole);
    }
    return el;
}

cudaError_t launch_conv_implicit(const ConvProblem &p, int mode, int cfg, unsigned *flags,
                                 cudaStream_t s) {
    if (p.K == 0) return cudaErrorNotSupported;
    if (cfg == kConvAuto) cfg = kConvImplicit;
    switch (cfg) {
        case kConvImplicit:
            return mode == kFast ? launch_conv_cfg<kFast, ConvCfg64x256>(p, flags, s)
                                 : launch_conv_cfg<kExact, ConvCfg64x256>(p, flags, s);
        default:
            return cudaErrorNotSupported;
    }
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
