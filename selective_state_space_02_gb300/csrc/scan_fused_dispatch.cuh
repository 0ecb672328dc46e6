// Instantiation dispatch of the fused scan kernel for one I/O type.  Included
// by scan_fused_f32.cu and scan_fused_bf16.cu, which compile in parallel.
#pragma once

#include "scan_fused_impl.cuh"

namespace ssm {
namespace fused {

template <typename T, int NP, int S, int NW, bool TMA>
cudaError_t by_mode(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps, unsigned int *status,
                    int mode, cudaStream_t st) {
    const bool gate = a.z != nullptr;
    switch (mode) {
        case kWhole:
            return gate ? launch_one<T, NP, S, NW, true, kWhole, TMA>(a, sg, maps, status, st)
                        : launch_one<T, NP, S, NW, false, kWhole, TMA>(a, sg, maps, status, st);
        case kTotals:
            return launch_one<T, NP, S, NW, false, kTotals, TMA>(a, sg, maps, status, st);
        default:
            return gate ? launch_one<T, NP, S, NW, true, kSeeded, TMA>(a, sg, maps, status, st)
                        : launch_one<T, NP, S, NW, false, kSeeded, TMA>(a, sg, maps, status, st);
    }
}

// Tile configurations (states per lane S, consumer warps NW) per padded state
// count.  cfg 0: more states per lane (fewer threads, cheaper per step);
// cfg 1: fewer states per lane (twice the threads for narrow problems).  The
// element-load path (rows not 16-byte aligned) always uses cfg 1.
template <typename T>
cudaError_t launch_typed_impl(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps,
                              unsigned int *status, int mode, bool tma, int cfg, cudaStream_t st) {
    const int N = a.dstate;
    if (N <= 8) {
        return tma ? by_mode<T, 8, 2, 4, true>(a, sg, maps, status, mode, st)
                   : by_mode<T, 8, 2, 4, false>(a, sg, maps, status, mode, st);
    }
    if (N <= 16) {
        if (!tma) return by_mode<T, 16, 2, 4, false>(a, sg, maps, status, mode, st);
        return cfg == 0 ? by_mode<T, 16, 4, 4, true>(a, sg, maps, status, mode, st)
                        : by_mode<T, 16, 2, 4, true>(a, sg, maps, status, mode, st);
    }
    if (N <= 32) {
        return tma ? by_mode<T, 32, 4, 4, true>(a, sg, maps, status, mode, st)
                   : by_mode<T, 32, 4, 4, false>(a, sg, maps, status, mode, st);
    }
    if (!tma) return by_mode<T, 64, 4, 4, false>(a, sg, maps, status, mode, st);
    return cfg == 0 ? by_mode<T, 64, 8, 4, true>(a, sg, maps, status, mode, st)
                    : by_mode<T, 64, 4, 4, true>(a, sg, maps, status, mode, st);
}

}  // namespace fused
}  // namespace ssm
