// sgemm_tiled.cu -- tiled fp32 matrix product on the CUDA cores of sm_103a,
// bit-exact in both modes.
//
// What each output is: the OneModel "Exact mode" page, section "Matrix
// product": acc = +0, then for p = 0 .. k-1 in increasing order one term
// (exact: round(acc + round(a*b)); fast: fma(a, b, acc), "Matrix product and
// convolution kernels" page, section "Fast mode"), then NaN -> 0x7FC00000.
// k is never split: each output lives in one thread's registers for the
// whole of k, so grid, tile shape and stream cannot change a bit.
//
// Design (the pages' CPU blocking -- packed B strips, MR x NR register
// microkernel, KC blocks -- recast for one GB300 SM):
//   * Persistent CTAs, one per SM, walking output tiles in a grouped raster.
//   * Warp specialisation: a producer warpgroup fills a STAGES-deep ring of
//     shared-memory stages (A tile BM x 32, B tile 32 x BN): one thread with
//     TMA (cp.async.bulk.tensor, zero fill outside the matrix) or, for
//     operands that are not 16-byte aligned, all 128 threads with 4-byte
//     cp.async (zero fill by src-size 0). Full/empty mbarriers hand stages
//     over; every wait is bounded.
//   * A lands 128-byte swizzled, so the A transpose of the pages' packing is
//     absorbed by the swizzle (simt_tile.cuh); B lands row-major.
//   * Each consumer thread owns TM x TN outputs and runs the rank-1 update per
//     k with paired-lane fp32 instructions (two outputs per instruction, each
//     lane rounded on its own).
//   * Zero fill past k is bit-neutral: both operands are +0 there, the
//     product is +0, and acc + (+0) == acc because acc is never -0 (it starts
//     at +0 and a round-to-nearest sum is -0 only when both addends are -0).
#include <cudaTypedefs.h>

#include <cstring>

#include "om_internal.h"
#include "schedule_host.h"
#include "simt_tile.cuh"

namespace om {

__device__ unsigned g_status_gemm;

// kProdMixed: A by TMA, B by 4-byte cp.async (B rows not 16-byte aligned).
enum Producer : int { kProdTma = 0, kProdAsync = 1, kProdMixed = 2 };

__device__ __forceinline__ void record_timeout(unsigned *status, int *abort_flag) {
    report_timeout(status, &g_status_gemm);
    *reinterpret_cast<volatile int *>(abort_flag) = 1;
}

// -------------------------------------------------------------- producers
template <class Cfg>
__device__ __forceinline__ void produce_tma(const CUtensorMap *mapA, const CUtensorMap *mapB,
                                            uint8_t *smem, uint64_t *full, uint64_t *empty,
                                            int *abort_flag, const TileRaster &rs,
                                            const Schedule &sched, unsigned *status) {
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    const Schedule::Local L = sched.local();
    for (int i = 0; i < L.count; ++i) {
        const Segment sg = sched.at(L, i);
        int tm, tn;
        rs.at(sg.tile, tm, tn);
        for (int kt = sg.kb; kt < sg.ke; ++kt) {
            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                record_timeout(status, abort_flag);
                // Let the copies already issued land before shared memory goes away.
                for (int s = 0; s < Cfg::STAGES; ++s) {
                    if (issued > s) {
                        const int64_t last = s + ((issued - 1 - s) / Cfg::STAGES) * Cfg::STAGES;
                        (void)mbar_wait(&full[s], static_cast<uint32_t>((last / Cfg::STAGES) & 1));
                    }
                }
                return;
            }
            ++issued;
            uint8_t *sa = smem + stage * Cfg::STAGE_BYTES;
            uint8_t *sb = sa + Cfg::A_BYTES;
            mbar_arrive_expect_tx(&full[stage], Cfg::STAGE_BYTES);
            tma_load_2d(sa, mapA, &full[stage], kt * Cfg::BK, tm * Cfg::BM);
            tma_load_2d(sb, mapB, &full[stage], tn * Cfg::BN, kt * Cfg::BK);
            if (++stage == Cfg::STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
    }
}

// 4-byte cp.async producer for operands of any alignment. Producer thread pt
// copies A elements (r, kk) with kk = pt % 32 and B elements (kk, c) with
// c = pt + 128j, so every warp reads 128 contiguous bytes of one row.
template <class Cfg>
__device__ __forceinline__ void produce_async(const GemmProblem &p, uint8_t *smem,
                                              uint64_t *full, uint64_t *empty, int *abort_flag,
                                              const TileRaster &rs, const Schedule &sched, int pt) {
    constexpr int BM = Cfg::BM, BN = Cfg::BN, BK = Cfg::BK;
    int stage = 0;
    uint32_t phase = 0;
    const int kk_a = pt % 32;
    const int r_a0 = pt / 32;  // 0..3
    const Schedule::Local L = sched.local();
    for (int i = 0; i < L.count; ++i) {
        const Segment sg = sched.at(L, i);
        int tm, tn;
        rs.at(sg.tile, tm, tn);
        const int64_t m0 = static_cast<int64_t>(tm) * BM, n0 = static_cast<int64_t>(tn) * BN;
        for (int kt = sg.kb; kt < sg.ke; ++kt) {
            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                record_timeout(p.status, abort_flag);
                cp_async_wait_all();
                return;
            }
            const uint32_t sa = smem_u32(smem + stage * Cfg::STAGE_BYTES);
            const uint32_t sb = sa + Cfg::A_BYTES;
            const int64_t kg = static_cast<int64_t>(kt) * BK + kk_a;
#pragma unroll 4
            for (int r = r_a0; r < BM; r += 4) {
                const int64_t row = m0 + r;
                const bool ok = (row < p.m) && (kg < p.k);
                const float *src = ok ? p.A + row * p.lda + kg : p.A;
                cp_async_4(sa + a_tile_offset(r, kk_a), src, ok ? 4u : 0u);
            }
#pragma unroll 4
            for (int kk = 0; kk < BK; ++kk) {
                const int64_t krow = static_cast<int64_t>(kt) * BK + kk;
                for (int c = pt; c < BN; c += 128) {
                    const int64_t col = n0 + c;
                    const bool ok = (krow < p.k) && (col < p.n);
                    const float *src = ok ? p.B + krow * p.ldb + col : p.B;
                    cp_async_4(sb + (kk * BN + c) * 4, src, ok ? 4u : 0u);
                }
            }
            cp_async_arrive_noinc(&full[stage]);
            if (++stage == Cfg::STAGES) {
                stage = 0;
                phase ^= 1;
            }
        }
    }
    // Keep shared memory alive until this thread's copies have landed.
    cp_async_wait_all();
}

// A by TMA (producer thread 0, with the A tile's byte count), B by 4-byte
// cp.async from every producer thread as in produce_async; each thread's
// copies arrive on the stage's full barrier as they land.
template <class Cfg>
__device__ __forceinline__ void produce_mixed(const GemmProblem &p, const CUtensorMap *mapA,
                                              uint8_t *smem, uint64_t *full, uint64_t *empty,
                                              int *abort_flag, const TileRaster &rs,
                                              const Schedule &sched, int pt) {
    constexpr int BN = Cfg::BN, BK = Cfg::BK;
    int stage = 0;
    uint32_t phase = 0;
    int64_t issued = 0;
    const Schedule::Local L = sched.local();
    for (int i = 0; i < L.count; ++i) {
        const Segment sg = sched.at(L, i);
        int tm, tn;
        rs.at(sg.tile, tm, tn);
        const int64_t n0 = static_cast<int64_t>(tn) * BN;
        for (int kt = sg.kb; kt < sg.ke; ++kt) {
            if (!mbar_wait(&empty[stage], phase ^ 1)) {
                record_timeout(p.status, abort_flag);
                cp_async_wait_all();
                if (pt == 0) {
                    // let the A tiles already requested land first
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
            const uint32_t sb = smem_u32(sa) + Cfg::A_BYTES;
            if (pt == 0) {
                mbar_arrive_expect_tx(&full[stage], Cfg::A_BYTES);
                tma_load_2d(sa, mapA, &full[stage], kt * BK, tm * Cfg::BM);
            }
#pragma unroll 4
            for (int kk = 0; kk < BK; ++kk) {
                const int64_t krow = static_cast<int64_t>(kt) * BK + kk;
#pragma unroll
                for (int c = pt; c < BN; c += kProducerThreads) {
                    const int64_t col = n0 + c;
                    const bool ok = (krow < p.k) && (col < p.n);
                    cp_async_4_if(sb + (kk * BN + c) * 4, ok ? p.B + krow * p.ldb + col : p.B, ok);
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

// Moves this thread's outputs of a tile between registers and C.
// OP 0: final store (canonical NaN); 1: raw store of an early part's
// accumulators; 2: load of the accumulators an earlier CTA stored.
template <class Cfg, int OP>
__device__ __forceinline__ void tile_io(const GemmProblem &p, Accum<Cfg> &acc, int64_t row0,
                                        int64_t col0, int vec_store) {
#pragma unroll
    for (int i = 0; i < Cfg::TM; ++i) {
        const int64_t row = row0 + 8 * i;
        if (row >= p.m) continue;
        float *crow = p.C + row * p.ldc;
#pragma unroll
        for (int q = 0; q < Cfg::TN / 4; ++q) {
            const int64_t col = col0 + 16 * q;
            const bool vec = vec_store && col + 3 < p.n;
            if constexpr (OP == 2) {
                float4 v = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
                if (vec) {
                    v = __ldcg(reinterpret_cast<const float4 *>(crow + col));
                } else {
                    if (col < p.n) v.x = __ldcg(crow + col);
                    if (col + 1 < p.n) v.y = __ldcg(crow + col + 1);
                    if (col + 2 < p.n) v.z = __ldcg(crow + col + 2);
                    if (col + 3 < p.n) v.w = __ldcg(crow + col + 3);
                }
                acc.v[i][2 * q] = make_float2(v.x, v.y);
                acc.v[i][2 * q + 1] = make_float2(v.z, v.w);
            } else {
                float4 v = make_float4(acc.v[i][2 * q].x, acc.v[i][2 * q].y, acc.v[i][2 * q + 1].x,
                                       acc.v[i][2 * q + 1].y);
                if constexpr (OP == 0) {
                    if (p.ep.bias || p.ep.res || p.ep.act) {
                        float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if (col + u < p.n)
                                e[u] = epilogue_value(e[u], p.ep.bias ? p.ep.bias + col + u : nullptr,
                                                      p.ep.res ? p.ep.res + row * p.ep.ldr + col + u : nullptr,
                                                      p.ep.act);
                        }
                        v = make_float4(e[0], e[1], e[2], e[3]);
                    }
                    v.x = canonical_nan(v.x);
                    v.y = canonical_nan(v.y);
                    v.z = canonical_nan(v.z);
                    v.w = canonical_nan(v.w);
                }
                if (vec) {
                    *reinterpret_cast<float4 *>(crow + col) = v;
                } else {
                    if (col < p.n) crow[col] = v.x;
                    if (col + 1 < p.n) crow[col + 1] = v.y;
                    if (col + 2 < p.n) crow[col + 2] = v.z;
                    if (col + 3 < p.n) crow[col + 3] = v.w;
                }
            }
        }
    }
}

// -------------------------------------------------------------- kernel
template <int MODE, class Cfg, int PROD>
__global__ void __launch_bounds__(Cfg::CONSUMERS + kProducerThreads, 1)
    sgemm_tiled_kernel(const __grid_constant__ CUtensorMap mapA,
                       const __grid_constant__ CUtensorMap mapB, GemmProblem p, TileRaster rs,
                       Schedule sched, int vec_store) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = aligned_smem<Cfg>(smem_raw);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Cfg::STAGES * Cfg::STAGE_BYTES);
    uint64_t *empty = full + Cfg::STAGES;
    int *abort_flag = reinterpret_cast<int *>(empty + Cfg::STAGES);

    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    if (threadIdx.x == 0) {
        for (int s = 0; s < Cfg::STAGES; ++s) {
            mbar_init(&full[s], PROD == kProdTma ? 1 : kProducerThreads + (PROD == kProdMixed ? 1 : 0));
            mbar_init(&empty[s], Cfg::CONSUMER_WARPS);
        }
        *abort_flag = 0;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    __syncthreads();

    if (warp >= Cfg::CONSUMER_WARPS) {
        RegSplit<(PROD == kProdTma ? 24 : 56)>::producer();
        if constexpr (PROD == kProdTma) {
            if (warp == Cfg::CONSUMER_WARPS && lane == 0) {
                prefetch_tensormap(&mapA);
                prefetch_tensormap(&mapB);
                produce_tma<Cfg>(&mapA, &mapB, smem, full, empty, abort_flag, rs, sched, p.status);
            }
        } else if constexpr (PROD == kProdMixed) {
            if (threadIdx.x == Cfg::CONSUMERS) prefetch_tensormap(&mapA);
            produce_mixed<Cfg>(p, &mapA, smem, full, empty, abort_flag, rs, sched,
                               threadIdx.x - Cfg::CONSUMERS);
        } else {
            produce_async<Cfg>(p, smem, full, empty, abort_flag, rs, sched,
                               threadIdx.x - Cfg::CONSUMERS);
        }
        return;
    }

    // Consumer warps.
    RegSplit<(PROD == kProdTma ? 24 : 56)>::consumer();
    const int ty = lane / 4, tx = lane % 4;
    const int arow0 = (warp / Cfg::WARPS_N) * Cfg::WM + ty;
    const int bcol0 = (warp % Cfg::WARPS_N) * Cfg::WN + tx * 4;
    int stage = 0;
    uint32_t phase = 0;
    const Schedule::Local L = sched.local();
    for (int si = 0; si < L.count; ++si) {
        const Segment sg = sched.at(L, si);
        int tm, tn;
        rs.at(sg.tile, tm, tn);
        const int64_t row0 = static_cast<int64_t>(tm) * Cfg::BM + arow0;
        const int64_t col0 = static_cast<int64_t>(tn) * Cfg::BN + bcol0;
        Accum<Cfg> acc;
        acc.zero();
        if (sg.kind == kSegLate) {
            if (!wait_previous_part(sched.flags, Cfg::CONSUMERS, abort_flag)) {
                report_timeout(p.status, &g_status_gemm);
                return;
            }
            tile_io<Cfg, 2>(p, acc, row0, col0, vec_store);
        }
        for (int kt = sg.kb; kt < sg.ke; ++kt) {
            if (!mbar_wait(&full[stage], phase)) {
                record_timeout(p.status, abort_flag);
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
            tile_io<Cfg, 1>(p, acc, row0, col0, vec_store);
            signal_early_part(sched.flags, Cfg::CONSUMERS);
        } else {
            // canonical NaN, predicated stores; columns >= n untouched
            tile_io<Cfg, 0>(p, acc, row0, col0, vec_store);
        }
    }
}

// -------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
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

// 2-D fp32 tensor map over a row-major matrix rows x cols with row stride ld
// (elements), box box_cols x box_rows; reads outside the matrix give +0.
static bool make_map_2d(CUtensorMap *map, const float *base, int64_t rows, int64_t cols,
                        int64_t ld, int box_cols, int box_rows, bool swizzle128) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims,
                    strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

static bool tma_eligible(const GemmProblem &p) {
    const auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    if (!al16(p.A) || !al16(p.B)) return false;
    if ((p.lda % 4) != 0 || (p.ldb % 4) != 0) return false;
    if (p.m > 0x7FFFFFFF || p.n > 0x7FFFFFFF || p.k > 0x7FFFFFFF) return false;
    if (p.lda * 4 >= (int64_t(1) << 40) || p.ldb * 4 >= (int64_t(1) << 40)) return false;
    return true;
}

// A alone can come by TMA (the mixed producer).
static bool tma_eligible_a(const GemmProblem &p) {
    if ((reinterpret_cast<uintptr_t>(p.A) & 15) != 0 || (p.lda % 4) != 0) return false;
    if (p.m > 0x7FFFFFFF || p.n > 0x7FFFFFFF || p.k > 0x7FFFFFFF) return false;
    return p.lda * 4 < (int64_t(1) << 40);
}

template <int MODE, class Cfg, int PROD>
static cudaError_t launch_cfg(const GemmProblem &p, unsigned *flags, cudaStream_t s) {
    auto kernel = sgemm_tiled_kernel<MODE, Cfg, PROD>;
    CUtensorMap mapA, mapB;
    memset(&mapA, 0, sizeof(mapA));
    memset(&mapB, 0, sizeof(mapB));
    if constexpr (PROD == kProdTma) {
        if (!tma_eligible(p)) return cudaErrorNotSupported;
        if (!make_map_2d(&mapA, p.A, p.m, p.k, p.lda, Cfg::BK, Cfg::BM, true)) return cudaErrorNotSupported;
        if (!make_map_2d(&mapB, p.B, p.k, p.n, p.ldb, Cfg::BN, Cfg::BK, false)) return cudaErrorNotSupported;
    } else if constexpr (PROD == kProdMixed) {
        if (!tma_eligible_a(p)) return cudaErrorNotSupported;
        if (!make_map_2d(&mapA, p.A, p.m, p.k, p.lda, Cfg::BK, Cfg::BM, true)) return cudaErrorNotSupported;
    }
    const int64_t tm = (p.m + Cfg::BM - 1) / Cfg::BM, tn = (p.n + Cfg::BN - 1) / Cfg::BN;
    if (tm * tn > 0x7FFFFFFF || p.k > 0x7FFFFFFF) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         Cfg::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    TileRaster rs;
    rs.tiles_m = static_cast<int>(tm);
    rs.tiles_n = static_cast<int>(tn);
    Schedule sched;
    make_schedule(static_cast<int>(tm * tn), static_cast<int>((p.k + Cfg::BK - 1) / Cfg::BK),
                  flags, &sched);
    const int vec = ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0) && (p.ldc % 4 == 0);
    cudaError_t el = launch_scheduled(kernel, sched, Cfg::CONSUMERS + kProducerThreads, Cfg::SMEM_BYTES, s,
                                      mapA, mapB, p, rs, sched, vec);
    if (el == cudaErrorCooperativeLaunchTooLarge) {
        const Schedule whole = whole_tiles(sched);
        el = launch_scheduled(kernel, whole, Cfg::CONSUMERS + kProducerThreads, Cfg::SMEM_BYTES, s, mapA,
                              mapB, p, rs, whole, vec);
    }
    return el;
}

using Cfg128x256 = TileCfg<128, 256, 8, 16, 2, 4, 4, true>;
using Cfg128x128 = TileCfg<128, 128, 8, 8, 2, 4, 4, true>;
using Cfg128x256Scalar = TileCfg<128, 256, 8, 16, 2, 4, 4, false>;

template <int MODE>
static cudaError_t launch_mode(const GemmProblem &p, int cfg, unsigned *flags, cudaStream_t s) {
    switch (cfg) {
        case kCfgTma128x256: return launch_cfg<MODE, Cfg128x256, kProdTma>(p, flags, s);
        case kCfgTma128x128: return launch_cfg<MODE, Cfg128x128, kProdTma>(p, flags, s);
        case kCfgAsync128x128: return launch_cfg<MODE, Cfg128x128, kProdAsync>(p, flags, s);
        case kCfgTmaScalar128x256: return launch_cfg<MODE, Cfg128x256Scalar, kProdTma>(p, flags, s);
        case kCfgMixed128x256: return launch_cfg<MODE, Cfg128x256, kProdMixed>(p, flags, s);
        case kCfgMixed128x128: return launch_cfg<MODE, Cfg128x128, kProdMixed>(p, flags, s);
        default: return cudaErrorNotSupported;
    }
}

cudaError_t launch_gemm_tiled(const GemmProblem &p, int mode, int cfg, unsigned *flags,
                              cudaStream_t s) {
    return mode == kFast ? launch_mode<kFast>(p, cfg, flags, s)
                         : launch_mode<kExact>(p, cfg, flags, s);
}

cudaError_t read_clear_status_gemm(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status_gemm, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*out) e = cudaMemcpyToSymbol(g_status_gemm, &zero, sizeof(unsigned));
    return e;
}

}  // namespace om
