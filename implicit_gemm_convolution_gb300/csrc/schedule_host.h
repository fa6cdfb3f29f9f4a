// schedule_host.h -- host side of the tile schedule (simt_tile.cuh): how many
// tiles go out whole, and the launch (cooperative when CTAs hand partial
// tiles to one another, which needs every CTA resident at once).
#pragma once

#include <cuda_runtime.h>

#include "om_internal.h"
#include "simt_tile.cuh"

namespace om {

// Without flags, or when the tiles already fill whole rounds of the SMs, every
// tile goes out whole. Otherwise all but the last one-to-two rounds go out
// whole and the rest are balanced with k-block continuation.
inline void make_schedule(int tiles, int nk, unsigned *flags, Schedule *sched) {
    const int sms = num_sms();
    sched->tiles = tiles;
    sched->nk = nk;
    sched->dp_tiles = tiles;
    sched->flags = nullptr;
    if (flags != nullptr && tiles > sms && (tiles % sms) != 0 && sms <= kMaxScheduleCtas && nk > 1) {
        sched->dp_tiles = (tiles / sms - 1) * sms;
        sched->flags = flags;
    }
}

template <class Kernel, class... Args>
cudaError_t launch_scheduled(Kernel kernel, const Schedule &sched, int threads, int smem,
                             cudaStream_t s, Args... args) {
    const int sms = num_sms();
    if (sched.flags == nullptr) {
        const int grid = sched.tiles < sms ? sched.tiles : sms;
        kernel<<<static_cast<unsigned>(grid), threads, smem, s>>>(args...);
        return cudaGetLastError();
    }
    cudaError_t e = cudaMemsetAsync(sched.flags, 0, static_cast<size_t>(sms) * sizeof(unsigned), s);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sms));
    cfg.blockDim = dim3(static_cast<unsigned>(threads));
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t el = cudaLaunchKernelEx(&cfg, kernel, args...);
    // Fewer SMs than the device has can be available to this context (MPS
    // limits, partitioned contexts): the cooperative launch is then refused.
    // The caller reruns the problem with the whole-tile schedule, which gives
    // the same bits and needs no co-residency.
    if (el == cudaErrorCooperativeLaunchTooLarge) (void)cudaGetLastError();
    return el;
}

// Whole tiles only: the schedule to fall back to when a balanced launch is
// refused for lack of co-resident CTAs.
inline Schedule whole_tiles(const Schedule &balanced) {
    Schedule s = balanced;
    s.dp_tiles = s.tiles;
    s.flags = nullptr;
    return s;
}

}  // namespace om
