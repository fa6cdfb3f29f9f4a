// gemm_tf32x3.cu -- the tolerance mode OM_MODE_TF32X3: C = A*B on the 5th
// generation tensor cores (tcgen05) with a three-product TF32 split.
//
// This mode is not one of the pages' bit-exact modes; it is an optional,
// separate tolerance mode with a stated bound:
//   |C - C_exact| <= 1e-5 * sqrt(k) * sum_p |A[i][p]| * |B[p][j]|
// for outputs whose exact-mode result is finite. Each operand value x is
// split into x_hi = x truncated to TF32 and x_lo = x - x_hi (exact in fp32,
// of which the tensor core reads the TF32 part); the product a*b is taken as
// a_lo*b_hi + a_hi*b_lo + a_hi*b_hi (a_lo*b_lo, below 2^-20 |ab|, is
// dropped), accumulated in fp32 in tensor memory in the tensor core's own
// order. NaN results are stored as 0x7FC00000 like the exact modes.
//
// CTA (one per SM, persistent over 128 x 128 output tiles), 22 warps:
//   warp 0      TMA producer: fp32 A tile 128 x 32 (128B swizzle, k
//               innermost) and fp32 B tile 32 x 128 into a 3-stage ring.
//   warp 1      allocates 256 tensor-memory columns (two 128-column fp32
//               accumulators), then one thread issues tcgen05.mma.
//   warps 2-17  converters: split each fp32 stage into hi/lo tiles in the
//               tensor cores' K-major 128B-swizzled layout (A keeps its
//               layout, B is transposed), then fence to the async proxy.
//   warps 18-21 epilogue: tcgen05.ld the finished accumulator (each warp
//               owns the 32 tensor-memory lanes of its warp index mod 4),
//               canonical NaN, predicated stores to C.
// Every mbarrier wait is bounded; on a timeout the CTA records the error,
// stops, still meets the final barrier and frees its tensor memory.
#include <cudaTypedefs.h>

#include <cstring>

#include "om_internal.h"
#include "om_device.cuh"

namespace om {

__device__ unsigned g_status_tc;

namespace tc {

constexpr int BM = 128, BN = 128, BK = 32;  // BK fp32 = one 128-byte row
constexpr int S_F32 = 3;                     // fp32 stages
constexpr int S_OPS = 2;                     // converted operand stages
constexpr int TILE_BYTES = 128 * 32 * 4;     // 16 KB: any 128 x 32 fp32 tile
constexpr int F32_STAGE = 2 * TILE_BYTES;    // A, B
constexpr int OPS_STAGE = 4 * TILE_BYTES;    // A_hi, A_lo, B_hi, B_lo
// measured: 8 -> 12 -> 16 warps gave 126 -> 141 -> 147 TFLOP/s with the
// rounding split; with the truncating split 12, 16, 20 and 24 warps give
// 200, 202, 198 and 189 TFLOP/s
constexpr int kConvWarps = 16;
constexpr int kConvThreads = kConvWarps * 32;
constexpr int kFirstConvWarp = 2;
constexpr int kFirstEpiWarp = kFirstConvWarp + kConvWarps;  // 18
constexpr int kThreads = (kFirstEpiWarp + 4) * 32;          // 704
constexpr int kTmemCols = 256;                               // 2 accumulators
constexpr int SMEM_BYTES = S_F32 * F32_STAGE + S_OPS * OPS_STAGE + 1024 + 256;

// Instruction descriptor of tcgen05.mma kind::tf32: D fp32 (bits 4-5 = 1),
// A and B TF32 (bits 7-9, 10-12 = 2), both K-major (bits 15, 16 = 0),
// N >> 3 in bits 17-22, M >> 4 in bits 24-28.
constexpr uint32_t kIdesc = (1u << 4) | (2u << 7) | (2u << 10) |
                            (static_cast<uint32_t>(BN >> 3) << 17) |
                            (static_cast<uint32_t>(BM >> 4) << 24);

// Shared-memory matrix descriptor: K-major, 128-byte swizzle (layout 2),
// 8-row groups 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr) {
    return (static_cast<uint64_t>((addr & 0x3FFFFu) >> 4)) | (static_cast<uint64_t>(1) << 16) |
           (static_cast<uint64_t>(1024 >> 4) << 32) | (static_cast<uint64_t>(1) << 46) |
           (static_cast<uint64_t>(2) << 61);
}

__device__ __forceinline__ void mma_tf32(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.u32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::tf32 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(kIdesc), "r"(acc)
        : "memory");
}

__device__ __forceinline__ void commit(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
            smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// TF32 split of one value: hi = a truncated to TF32 (its 13 low mantissa bits
// cleared: round toward zero, so a finite value never overflows), lo = a - hi
// (exact in fp32; the tensor core reads its TF32 part); lo = 0 when hi is not
// finite. Two instructions and a select per value (measured: 202 -> 209
// TFLOP/s on 4096^3 against converting lo with cvt.rna.tf32 and hi with
// cvt.rz.tf32).
__device__ __forceinline__ void split(float a, float &hi, float &lo) {
    const float fh = __uint_as_float(__float_as_uint(a) & 0xFFFFE000u);
    hi = fh;
    const float r = __fsub_rn(a, fh);
    lo = fabsf(fh) < INFINITY ? r : 0.0f;
}

// Explicit shared-memory accesses on 32-bit shared addresses.
__device__ __forceinline__ float4 lds128(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(a));
    return v;
}
__device__ __forceinline__ float lds32(uint32_t a) {
    float v;
    asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a));
    return v;
}
__device__ __forceinline__ void sts128(uint32_t a, float4 v) {
    asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(a), "f"(v.x), "f"(v.y), "f"(v.z),
                 "f"(v.w)
                 : "memory");
}

struct Smem {
    uint8_t *base;
    __device__ uint8_t *a32(int s) const { return base + s * F32_STAGE; }
    __device__ uint8_t *b32(int s) const { return base + s * F32_STAGE + TILE_BYTES; }
    __device__ uint8_t *ops(int s, int which) const {
        return base + S_F32 * F32_STAGE + s * OPS_STAGE + which * TILE_BYTES;
    }
};

struct Bars {
    uint64_t full_f[S_F32], empty_f[S_F32], full_o[S_OPS], empty_o[S_OPS];
    uint64_t tmem_full[2], tmem_empty[2];
    uint64_t drained;  // one commit after the last MMA: every MMA has finished
    uint32_t tmem_base;
    int abort;
    unsigned *status;  // the call's status word in a caller workspace, or NULL
};
static_assert(sizeof(Bars) <= 256, "the barriers fit the 256 bytes reserved after the stages");

__device__ __forceinline__ bool aborted(Bars *b) {
    return *reinterpret_cast<volatile int *>(&b->abort) != 0;
}
__device__ __forceinline__ void fail(Bars *b) {
    report_timeout(b->status, &g_status_tc);
    *reinterpret_cast<volatile int *>(&b->abort) = 1;
}
// Bounded wait that also gives up once another role has failed.
__device__ __forceinline__ bool wait(Bars *b, uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    while (!mbar_try_wait(bar, parity)) {
        if (aborted(b)) return false;
        if (global_ns() - t0 > kWaitLimitNs) {
            fail(b);
            return false;
        }
    }
    return true;
}

}  // namespace tc

__global__ void __launch_bounds__(tc::kThreads, 1)
    gemm_tf32x3_kernel(const __grid_constant__ CUtensorMap mapA,
                       const __grid_constant__ CUtensorMap mapB, GemmProblem p, int tiles_m,
                       int tiles_n, int vec_store) {
    using namespace tc;
    extern __shared__ uint8_t smem_raw[];
    Smem sm{smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u)};
    Bars *bars = reinterpret_cast<Bars *>(sm.base + S_F32 * F32_STAGE + S_OPS * OPS_STAGE);
    const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
    const int total = tiles_m * tiles_n;
    const int nk = static_cast<int>((p.k + BK - 1) / BK);

    if (threadIdx.x == 0) {
        for (int s = 0; s < S_F32; ++s) {
            mbar_init(&bars->full_f[s], 1);
            mbar_init(&bars->empty_f[s], kConvWarps);
        }
        for (int s = 0; s < S_OPS; ++s) {
            mbar_init(&bars->full_o[s], kConvWarps);
            mbar_init(&bars->empty_o[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&bars->tmem_full[b], 1);
            mbar_init(&bars->tmem_empty[b], 4);
        }
        mbar_init(&bars->drained, 1);
        bars->abort = 0;
        bars->status = p.status;
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 1) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(
                         smem_u32(&bars->tmem_base)),
                     "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
    }
    fence_before();
    __syncthreads();
    fence_after();
    const uint32_t tmem = bars->tmem_base;

    if (warp == 0) {
        // ---------------------------------------------------------- TMA
        if (lane == 0) {
            prefetch_tensormap(&mapA);
            prefetch_tensormap(&mapB);
            int s = 0;
            uint32_t ph = 0;
            int64_t issued = 0;
            for (int t = blockIdx.x; t < total && !aborted(bars); t += gridDim.x) {
                const int tm = t % tiles_m, tn = t / tiles_m;
                for (int kt = 0; kt < nk; ++kt) {
                    if (!wait(bars, &bars->empty_f[s], ph ^ 1)) break;
                    ++issued;
                    mbar_arrive_expect_tx(&bars->full_f[s], F32_STAGE);
                    tma_load_2d(sm.a32(s), &mapA, &bars->full_f[s], kt * BK, tm * BM);
                    tma_load_2d(sm.b32(s), &mapB, &bars->full_f[s], tn * BN, kt * BK);
                    if (++s == S_F32) {
                        s = 0;
                        ph ^= 1;
                    }
                }
            }
            // Every issued copy lands before shared memory can go away (on
            // the normal path the converters already waited for all of them).
            for (int i = 0; i < S_F32; ++i) {
                if (issued > i) {
                    const int64_t last = i + ((issued - 1 - i) / S_F32) * S_F32;
                    (void)mbar_wait(&bars->full_f[i], static_cast<uint32_t>((last / S_F32) & 1));
                }
            }
        }
    } else if (warp == 1) {
        // ---------------------------------------------------------- MMA
        if (lane == 0) {
            int s = 0, acc_i = 0;
            uint32_t ph = 0, acc_ph = 0;
            for (int t = blockIdx.x; t < total && !aborted(bars); t += gridDim.x) {
                if (!wait(bars, &bars->tmem_empty[acc_i], acc_ph ^ 1)) break;
                fence_after();
                const uint32_t d = tmem + static_cast<uint32_t>(acc_i * BN);
                for (int kt = 0; kt < nk; ++kt) {
                    if (!wait(bars, &bars->full_o[s], ph)) break;
                    fence_after();
                    const uint32_t ahi = smem_u32(sm.ops(s, 0)), alo = smem_u32(sm.ops(s, 1));
                    const uint32_t bhi = smem_u32(sm.ops(s, 2)), blo = smem_u32(sm.ops(s, 3));
#pragma unroll
                    for (int j = 0; j < BK / 8; ++j) {  // 8 tf32 (32 bytes) per instruction
                        const uint32_t off = static_cast<uint32_t>(j * 32);
                        const uint32_t first = (kt == 0 && j == 0) ? 0u : 1u;
                        mma_tf32(d, smem_desc(alo + off), smem_desc(bhi + off), first);
                        mma_tf32(d, smem_desc(ahi + off), smem_desc(blo + off), 1u);
                        mma_tf32(d, smem_desc(ahi + off), smem_desc(bhi + off), 1u);
                    }
                    commit(&bars->empty_o[s]);  // frees the operand stage once read
                    if (++s == S_OPS) {
                        s = 0;
                        ph ^= 1;
                    }
                }
                commit(&bars->tmem_full[acc_i]);  // accumulator complete
                if (++acc_i == 2) {
                    acc_i = 0;
                    acc_ph ^= 1;
                }
            }
            // No MMA may still read shared memory or write tensor memory when
            // the CTA frees them: one more commit arrives once all are done.
            commit(&bars->drained);
            (void)mbar_wait(&bars->drained, 0);
        }
    } else if (warp < kFirstEpiWarp) {
        // ---------------------------------------------------------- converters
        const int ct = threadIdx.x - kFirstConvWarp * 32;  // 0..255
        int sf = 0, so = 0;
        uint32_t phf = 0, pho = 0;
        for (int t = blockIdx.x; t < total && !aborted(bars); t += gridDim.x) {
            for (int kt = 0; kt < nk; ++kt) {
                if (!wait(bars, &bars->full_f[sf], phf)) break;
                if (!wait(bars, &bars->empty_o[so], pho ^ 1)) break;
                const uint32_t a32 = smem_u32(sm.a32(sf)), b32 = smem_u32(sm.b32(sf));
                const uint32_t ahi = smem_u32(sm.ops(so, 0)), alo = smem_u32(sm.ops(so, 1));
                const uint32_t bhi = smem_u32(sm.ops(so, 2)), blo = smem_u32(sm.ops(so, 3));
                // A: same 128B-swizzled K-major layout, 16-byte chunks
#pragma unroll
                for (int idx = ct; idx < BM * BK / 4; idx += kConvThreads) {
                    const uint32_t off = static_cast<uint32_t>(idx * 16);
                    const float4 v = lds128(a32 + off);
                    float4 h, l;
                    split(v.x, h.x, l.x);
                    split(v.y, h.y, l.y);
                    split(v.z, h.z, l.z);
                    split(v.w, h.w, l.w);
                    sts128(ahi + off, h);
                    sts128(alo + off, l);
                }
                // B: [32 k][128 n] row-major -> [128 n][32 k] 128B-swizzled;
                // (n, 4-k chunk kc) pairs, n fastest across threads
#pragma unroll
                for (int idx = ct; idx < BN * BK / 4; idx += kConvThreads) {
                    const int n = idx % BN, kc = idx / BN;
                    float4 h, l;
                    split(lds32(b32 + ((4 * kc + 0) * BN + n) * 4), h.x, l.x);
                    split(lds32(b32 + ((4 * kc + 1) * BN + n) * 4), h.y, l.y);
                    split(lds32(b32 + ((4 * kc + 2) * BN + n) * 4), h.z, l.z);
                    split(lds32(b32 + ((4 * kc + 3) * BN + n) * 4), h.w, l.w);
                    const uint32_t off = static_cast<uint32_t>(n * 128 + ((kc ^ (n & 7)) << 4));
                    sts128(bhi + off, h);
                    sts128(blo + off, l);
                }
                fence_proxy_async_smem();  // generic writes -> tensor-core reads
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&bars->empty_f[sf]);
                    mbar_arrive(&bars->full_o[so]);
                }
                if (++sf == S_F32) {
                    sf = 0;
                    phf ^= 1;
                }
                if (++so == S_OPS) {
                    so = 0;
                    pho ^= 1;
                }
            }
        }
    } else {
        // ---------------------------------------------------------- epilogue
        const int q = warp % 4;  // tensor-memory lanes 32q .. 32q+31
        int acc_i = 0;
        uint32_t acc_ph = 0;
        for (int t = blockIdx.x; t < total && !aborted(bars); t += gridDim.x) {
            const int tm = t % tiles_m, tn = t / tiles_m;
            if (!wait(bars, &bars->tmem_full[acc_i], acc_ph)) break;
            fence_after();
            const int64_t row = static_cast<int64_t>(tm) * BM + q * 32 + lane;
            float *crow = p.C + row * p.ldc;
#pragma unroll 1
            for (int cc = 0; cc < BN / 32; ++cc) {
                uint32_t r[32];
                const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) +
                                       static_cast<uint32_t>(acc_i * BN + cc * 32);
                asm volatile(
                    "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,"
                    "%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,"
                    "%30,%31}, [%32];"
                    : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                      "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]),
                      "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),
                      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                      "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]),
                      "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                    : "r"(taddr));
                asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
                if (row < p.m) {
                    const int64_t col0 = static_cast<int64_t>(tn) * BN + cc * 32;
#pragma unroll
                    for (int v = 0; v < 8; ++v) {
                        const int64_t col = col0 + 4 * v;
                        float e[4] = {__uint_as_float(r[4 * v + 0]), __uint_as_float(r[4 * v + 1]),
                                      __uint_as_float(r[4 * v + 2]), __uint_as_float(r[4 * v + 3])};
#pragma unroll
                        for (int u = 0; u < 4; ++u) {
                            if ((p.ep.bias || p.ep.res || p.ep.act) && col + u < p.n)
                                e[u] = epilogue_value(e[u], p.ep.bias ? p.ep.bias + col + u : nullptr,
                                                      p.ep.res ? p.ep.res + row * p.ep.ldr + col + u : nullptr,
                                                      p.ep.act);
                            e[u] = canonical_nan(e[u]);
                        }
                        const float4 o = make_float4(e[0], e[1], e[2], e[3]);
                        if (vec_store && col + 3 < p.n) {
                            *reinterpret_cast<float4 *>(crow + col) = o;
                        } else {
                            if (col < p.n) crow[col] = o.x;
                            if (col + 1 < p.n) crow[col + 1] = o.y;
                            if (col + 2 < p.n) crow[col + 2] = o.z;
                            if (col + 3 < p.n) crow[col + 3] = o.w;
                        }
                    }
                }
            }
            fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&bars->tmem_empty[acc_i]);
            if (++acc_i == 2) {
                acc_i = 0;
                acc_ph ^= 1;
            }
        }
    }

    // Every role meets here before the tensor memory is freed.
    fence_before();
    __syncthreads();
    fence_after();
    if (warp == 1) {
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem),
                     "n"(kTmemCols)
                     : "memory");
    }
}

// -------------------------------------------------------------- host side
static PFN_cuTensorMapEncodeTiled_v12000 tc_encode_fn() {
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

static bool tc_map(CUtensorMap *map, const float *base, int64_t rows, int64_t cols, int64_t ld,
                   int box_cols, int box_rows, bool swizzle128) {
    auto fn = tc_encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(cols), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 4};
    cuuint32_t box[2] = {static_cast<cuuint32_t>(box_cols), static_cast<cuuint32_t>(box_rows)};
    cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<float *>(base), dims, strides,
              box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

cudaError_t launch_gemm_tf32x3(const GemmProblem &p, cudaStream_t s) {
    using namespace tc;
    const auto al16 = [](const void *q) { return (reinterpret_cast<uintptr_t>(q) & 15) == 0; };
    if (!al16(p.A) || !al16(p.B) || (p.lda % 4) != 0 || (p.ldb % 4) != 0) return cudaErrorNotSupported;
    if (p.m > 0x7FFFFFFF || p.n > 0x7FFFFFFF || p.k > 0x7FFFFFFF) return cudaErrorNotSupported;
    if (p.lda * 4 >= (int64_t(1) << 40) || p.ldb * 4 >= (int64_t(1) << 40)) return cudaErrorNotSupported;
    const int64_t tm = (p.m + BM - 1) / BM, tn = (p.n + BN - 1) / BN;
    if (tm * tn > 0x7FFFFFFF) return cudaErrorNotSupported;
    CUtensorMap mapA, mapB;
    memset(&mapA, 0, sizeof(mapA));
    memset(&mapB, 0, sizeof(mapB));
    if (!tc_map(&mapA, p.A, p.m, p.k, p.lda, BK, BM, true)) return cudaErrorNotSupported;
    if (!tc_map(&mapB, p.B, p.k, p.n, p.ldb, BN, BK, false)) return cudaErrorNotSupported;
    cudaError_t e = cudaFuncSetAttribute(gemm_tf32x3_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    if (e != cudaSuccess) return e;
    const int64_t total = tm * tn;
    const int64_t grid = total < num_sms() ? total : num_sms();
    const int vec = ((reinterpret_cast<uintptr_t>(p.C) & 15) == 0) && (p.ldc % 4 == 0);
    gemm_tf32x3_kernel<<<static_cast<unsigned>(grid), kThreads, SMEM_BYTES, s>>>(
        mapA, mapB, p, static_cast<int>(tm), static_cast<int>(tn), vec);
    return cudaGetLastError();
}

cudaError_t read_clear_status_tc(unsigned *out, cudaStream_t s) {
    unsigned zero = 0;
    cudaError_t e = cudaMemcpyFromSymbolAsync(out, g_status_tc, sizeof(unsigned), 0,
                                              cudaMemcpyDeviceToHost, s);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return e;
    if (*out) e = cudaMemcpyToSymbol(g_status_tc, &zero, sizeof(unsigned));
    return e;
}

}  // namespace om
