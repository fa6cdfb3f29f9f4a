// simt_tile.cuh -- the shared-memory tile layout and the register-tile inner
// loop used by the tiled matrix product and the implicit-GEMM convolution.
//
// Per output the loop adds one term per k in increasing k, from the
// accumulator the previous stage left ("Exact mode" page, section "Matrix
// product"; the k-block continuation of the "Matrix product and convolution
// kernels" page, item 3 "Microkernel"). The accumulators stay in registers
// for the whole of k, so a stage boundary adds no rounding.
//
// Shared-memory stage: A tile BM x 32 (k innermost), 128-byte swizzled: row r,
// 16-byte chunk c is stored at chunk c ^ (r % 8) of the row's 128 bytes (the
// pattern TMA's 128B swizzle writes). B tile 32 x BN, row-major. Thread
// (ty, tx) of a warp owns rows arow0 + 8i (i < TM) and columns
// bcol0 + 16q + e (q < TN/4, e < 4) of its warp tile. One 128-bit load gives
// four consecutive k of one A row (the swizzle keeps the eight rows of a
// load instruction on distinct banks) or four consecutive B columns.
#pragma once

#include "om_device.cuh"

// 4-k chunks of a 32-k stage per unrolled loop body, per mode (tuning knobs;
// measured on the 4096^3 product and the 3x3 / 1x1 convolutions: 2 is as
// fast as 4 or 8 in fast mode and faster for the 1x1 convolution, 1 is
// slower in exact mode).
#ifndef OM_KC_UNROLL_EXACT
#define OM_KC_UNROLL_EXACT 2
#endif
#ifndef OM_KC_UNROLL_FAST
#define OM_KC_UNROLL_FAST 2
#endif


namespace om {

constexpr int kKcUnrollExact = OM_KC_UNROLL_EXACT;
constexpr int kKcUnrollFast = OM_KC_UNROLL_FAST;

template <int BM_, int BN_, int TM_, int TN_, int WARPS_M_, int WARPS_N_, int STAGES_, bool X2_>
struct TileCfg {
    static constexpr int BM = BM_, BN = BN_, BK = 32, TM = TM_, TN = TN_;
    static constexpr int WARPS_M = WARPS_M_, WARPS_N = WARPS_N_;
    static constexpr int CONSUMER_WARPS = WARPS_M * WARPS_N;
    static constexpr int CONSUMERS = CONSUMER_WARPS * 32;
    static constexpr int STAGES = STAGES_;
    static constexpr bool X2 = X2_;
    static constexpr int WM = BM / WARPS_M, WN = BN / WARPS_N;
    static_assert(WM == 8 * TM, "a warp tile is 8 thread rows of TM rows");
    static_assert(WN == 4 * TN, "a warp tile is 4 thread columns of TN columns");
    static_assert(TN % 4 == 0, "columns come in groups of four");
    static constexpr int A_BYTES = BM * BK * 4;
    static constexpr int B_BYTES = BK * BN * 4;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static_assert(A_BYTES % 1024 == 0 && B_BYTES % 1024 == 0, "swizzled tiles need 1 KB alignment");
    static constexpr int SMEM_BYTES = STAGES * STAGE_BYTES + 1024 + 256;
    static_assert(CONSUMERS % 128 == 0, "consumers come in whole warpgroups");
};

// Producer warpgroup(s) and two consumer warpgroups. At launch every thread
// gets the same registers (65536 / threads, rounded down to 8); the
// producers give registers back (setmaxnreg.dec) and the consumers take them
// (setmaxnreg.inc): a TMA producer needs almost none, a gathering producer
// keeps per-column state.
constexpr int kProducerThreads = 128;  // one producer warpgroup (the GEMM kernels)
constexpr int kLaunchRegs = 168;       // 384 threads

template <int PRODUCER_REGS, int PRODUCERS = 128, int CONSUMERS = 256>
struct RegSplit {
    static constexpr int kThreads = PRODUCERS + CONSUMERS;
    static constexpr int kLaunch = (65536 / kThreads) / 8 * 8;
    static constexpr int kProducer = PRODUCER_REGS;
    static constexpr int kConsumer =
        ((kThreads * kLaunch - PRODUCERS * PRODUCER_REGS) / CONSUMERS) / 8 * 8 > 256
            ? 256
            : ((kThreads * kLaunch - PRODUCERS * PRODUCER_REGS) / CONSUMERS) / 8 * 8;
    static_assert(PRODUCERS % 128 == 0 && CONSUMERS % 128 == 0, "whole warpgroups");
    static_assert(PRODUCER_REGS >= 24 && PRODUCER_REGS % 8 == 0 && PRODUCER_REGS <= kLaunch,
                  "setmaxnreg range");
    static_assert(PRODUCERS * kProducer + CONSUMERS * kConsumer <= kThreads * kLaunch,
                  "register split exceeds the launch allocation");
    __device__ __forceinline__ static void producer() {
        asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;" ::"n"(kProducer));
    }
    __device__ __forceinline__ static void consumer() {
        asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;" ::"n"(kConsumer));
    }
};

// Byte offset of A element (r, kk) inside a stage's A tile.
__device__ __forceinline__ uint32_t a_tile_offset(int r, int kk) {
    return static_cast<uint32_t>(r * 128 + ((((kk >> 2) ^ (r & 7)) << 4) | ((kk & 3) << 2)));
}

template <class Cfg>
struct Accum {
    float2 v[Cfg::TM][Cfg::TN / 2];
    __device__ __forceinline__ void zero() {
#pragma unroll
        for (int i = 0; i < Cfg::TM; ++i)
#pragma unroll
            for (int j = 0; j < Cfg::TN / 2; ++j) v[i][j] = make_float2(0.0f, 0.0f);
    }
    // The four outputs of row i, column group q, NaN canonicalised.
    __device__ __forceinline__ float4 out4(int i, int q) const {
        float4 r;
        r.x = canonical_nan(v[i][2 * q].x);
        r.y = canonical_nan(v[i][2 * q].y);
        r.z = canonical_nan(v[i][2 * q + 1].x);
        r.w = canonical_nan(v[i][2 * q + 1].y);
        return r;
    }
};

// All 32 k of one stage, in increasing k, for this thread's TM x TN outputs.
template <int MODE, class Cfg>
__device__ __forceinline__ void mma_stage(Accum<Cfg> &acc, const float *As, const float *Bs,
                                          int arow0, int bcol0, int ty) {
    constexpr int TM = Cfg::TM, TN = Cfg::TN, BN = Cfg::BN;
    // A few of the eight 4-k chunks per loop body: enough independent work to
    // hide shared-memory latency while keeping the loop in the instruction cache.
#pragma unroll(MODE == kFast ? kKcUnrollFast : kKcUnrollExact)
    for (int kc = 0; kc < Cfg::BK / 4; ++kc) {
        float4 a[TM];
#pragma unroll
        for (int i = 0; i < TM; ++i) {
            // row arow0 + 8i has (row % 8) == ty, so its chunk kc sits at kc ^ ty
            a[i] = *reinterpret_cast<const float4 *>(As + (arow0 + 8 * i) * 32 + ((kc ^ ty) << 2));
        }
#pragma unroll
        for (int kk = 0; kk < 4; ++kk) {
            float4 b[TN / 4];
#pragma unroll
            for (int q = 0; q < TN / 4; ++q) {
                b[q] = *reinterpret_cast<const float4 *>(Bs + (kc * 4 + kk) * BN + bcol0 + 16 * q);
            }
#pragma unroll
            for (int i = 0; i < TM; ++i) {
                const float av = (kk == 0) ? a[i].x : (kk == 1) ? a[i].y : (kk == 2) ? a[i].z : a[i].w;
                if constexpr (Cfg::X2) {
                    const float2 a2 = make_float2(av, av);
#pragma unroll
                    for (int q = 0; q < TN / 4; ++q) {
                        acc.v[i][2 * q] = term2<MODE>(acc.v[i][2 * q], a2, make_float2(b[q].x, b[q].y));
                        acc.v[i][2 * q + 1] =
                            term2<MODE>(acc.v[i][2 * q + 1], a2, make_float2(b[q].z, b[q].w));
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < TN / 4; ++q) {
                        float2 &u = acc.v[i][2 * q];
                        float2 &w = acc.v[i][2 * q + 1];
                        u.x = term<MODE>(u.x, av, b[q].x);
                        u.y = term<MODE>(u.y, av, b[q].y);
                        w.x = term<MODE>(w.x, av, b[q].z);
                        w.y = term<MODE>(w.y, av, b[q].w);
                    }
                }
            }
        }
    }
}

// Output tiles in a grouped raster: kGroupM tile rows at a time, so the
// tiles running together share A row panels and B column panels in L2.
struct TileRaster {
    int tiles_m, tiles_n;
    static constexpr int kGroupM = 8;
    __device__ __forceinline__ void at(int t, int &tm, int &tn) const {
        const int per_group = kGroupM * tiles_n;
        const int group = t / per_group;
        const int first_m = group * kGroupM;
        const int gsize = min(tiles_m - first_m, kGroupM);
        const int r = t - group * per_group;
        tm = first_m + r % gsize;
        tn = r / gsize;
    }
};

// ----------------------------------------------------------------- schedule
// A CTA's work is a list of segments (tile, first k-stage, end k-stage, kind).
//
// Tiles [0, dp_tiles) are handed out round-robin, whole (data-parallel, in
// the raster order that keeps concurrently running tiles close in L2).
// The remaining tiles -- between one and two per CTA -- are balanced: their
// units (tile, k-stage), tile-major, are cut into gridDim.x equal contiguous
// ranges. A range can end inside a tile (its "early part": stages [0, e))
// and start inside the tile the previous CTA ended in (its "late part":
// stages [s, nk)). After its whole tiles a CTA runs its early part (from +0;
// the raw accumulators are stored to the output and a flag is raised), then
// the whole tiles of its range, then its late part, which waits for the
// previous CTA's flag, loads the stored accumulators and continues from
// them. This is the pages' k-block continuation: a later k-block starts from
// the values the earlier blocks stored, and the stored value is the
// accumulator itself, so every output still sees one sequential loop over k
// from +0 and the bits equal the data-parallel schedule's. The previous CTA
// stores its early part long before this CTA reaches its late part.
enum SegKind : int { kSegFull = 0, kSegEarly = 1, kSegLate = 2 };

struct Segment {
    int tile, kb, ke, kind;
};

struct Schedule {
    int tiles;         // output tiles (< 2^31)
    int nk;            // k-stages per tile
    int dp_tiles;      // tiles handed out whole; the rest are balanced
    unsigned *flags;   // balanced part: flags[c] raised once CTA c's early part is stored

    struct Local {
        int count, dp_count, has_early, has_late;
        int early_tile, late_tile, full0, early_ke, late_kb;
    };

    __device__ __forceinline__ Local local() const {
        Local L{};
        const int c = blockIdx.x, P = gridDim.x;
        L.dp_count = (dp_tiles > c) ? (dp_tiles - 1 - c) / P + 1 : 0;
        L.count = L.dp_count;
        if (dp_tiles >= tiles) return L;
        const int64_t U = static_cast<int64_t>(tiles - dp_tiles) * nk;
        const int64_t lo = c * U / P, hi = (c + 1) * U / P;
        L.has_late = (lo % nk) != 0;
        L.late_tile = dp_tiles + static_cast<int>(lo / nk);
        L.late_kb = static_cast<int>(lo % nk);
        L.has_early = (hi % nk) != 0;
        L.early_tile = dp_tiles + static_cast<int>(hi / nk);
        L.early_ke = static_cast<int>(hi % nk);
        L.full0 = dp_tiles + static_cast<int>((lo + nk - 1) / nk);
        const int full1 = dp_tiles + static_cast<int>(hi / nk);
        L.count += L.has_early + L.has_late + (full1 > L.full0 ? full1 - L.full0 : 0);
        return L;
    }

    __device__ __forceinline__ Segment at(const Local &L, int i) const {
        Segment s;
        s.kb = 0;
        s.ke = nk;
        s.kind = kSegFull;
        if (i < L.dp_count) {
            s.tile = static_cast<int>(blockIdx.x) + i * static_cast<int>(gridDim.x);
            return s;
        }
        i -= L.dp_count;
        if (L.has_early && i == 0) {
            s.tile = L.early_tile;
            s.ke = L.early_ke;
            s.kind = kSegEarly;
        } else if (L.has_late && i == L.count - L.dp_count - 1) {
            s.tile = L.late_tile;
            s.kb = L.late_kb;
            s.kind = kSegLate;
        } else {
            s.tile = L.full0 + (i - L.has_early);
        }
        return s;
    }
};

// Raise CTA blockIdx.x's flag after every consumer thread stored its part
// (called by all consumer threads; named barrier 1 spans the consumers).
__device__ __forceinline__ void signal_early_part(unsigned *flags, int consumers) {
    asm volatile("bar.sync 1, %0;" ::"r"(consumers) : "memory");
    if (threadIdx.x == 0) {
        __threadfence();
        atomicExch(&flags[blockIdx.x], 1u);
    }
}

// Wait (bounded) for the previous CTA's early part; false on timeout.
__device__ __forceinline__ bool wait_previous_part(unsigned *flags, int consumers, int *abort_flag) {
    if (threadIdx.x == 0) {
        if (!acquire_flag(flags + blockIdx.x - 1, kWaitLimitNs))
            *reinterpret_cast<volatile int *>(abort_flag) = 2;
    }
    asm volatile("bar.sync 1, %0;" ::"r"(consumers) : "memory");
    return *reinterpret_cast<volatile int *>(abort_flag) != 2;
}

// The dynamic shared-memory base advanced to a 1024-byte boundary (what the
// 128B swizzle pattern repeats on). The offset is added to the shared pointer
// itself, so the compiler keeps knowing the address is shared memory and
// emits shared loads (an integer round trip would turn them into generic
// loads through the L1 path).
template <class Cfg>
__device__ __forceinline__ uint8_t *aligned_smem(uint8_t *raw) {
    const uint32_t base = smem_u32(raw);
    return raw + ((1024u - (base & 1023u)) & 1023u);
}

}  // namespace om
