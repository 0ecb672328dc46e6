// Instantiation dispatch of the fused scan kernel for one I/O type.  Included
// by scan_fused_f32.cu and scan_fused_bf16.cu, which compile in parallel.
#pragma once

#include "scan_fused_impl.cuh"

namespace ssm {
namespace fused {

template <typename T, int NP, int S, bool TMA, bool CKPT>
cudaError_t by_mode(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps, unsigned int *status,
                    int mode, bool prepare, cudaStream_t st) {
    constexpr int NW = consumer_warps(S);
    if constexpr (CKPT)   // the forward's y passes with checkpoints
        if (a.conv_k > 0 || (mode != kWhole && mode != kSeeded)) return cudaErrorInvalidValue;
    if (prepare) {
        const cudaError_t e = launch_prepare<T, NP, S>(a, const_cast<float *>(sg.bc), st);
        if (e != cudaSuccess) return e;
    }
    const bool gate = a.z != nullptr;
    if constexpr (CKPT) {
        if (mode == kWhole)
            return gate ? launch_one<T, NP, S, NW, true, kWhole, TMA, 0, true>(a, sg, maps, status, st)
                        : launch_one<T, NP, S, NW, false, kWhole, TMA, 0, true>(a, sg, maps, status, st);
        return gate ? launch_one<T, NP, S, NW, true, kSeeded, TMA, 0, true>(a, sg, maps, status, st)
                    : launch_one<T, NP, S, NW, false, kSeeded, TMA, 0, true>(a, sg, maps, status, st);
    } else {
        switch (mode) {
            case kWhole:
                if (a.conv_k > 0)   // causal convolution (up to 4 taps) fused in front of the scan
                    return gate ? launch_one<T, NP, S, NW, true, kWhole, TMA, 4>(a, sg, maps, status, st)
                                : launch_one<T, NP, S, NW, false, kWhole, TMA, 4>(a, sg, maps, status, st);
                return gate ? launch_one<T, NP, S, NW, true, kWhole, TMA>(a, sg, maps, status, st)
                            : launch_one<T, NP, S, NW, false, kWhole, TMA>(a, sg, maps, status, st);
            case kTotals:
                return launch_one<T, NP, S, NW, false, kTotals, TMA>(a, sg, maps, status, st);
            case kStates:
                return launch_one<T, NP, S, NW, false, kStates, TMA>(a, sg, maps, status, st);
            default:
                return gate ? launch_one<T, NP, S, NW, true, kSeeded, TMA>(a, sg, maps, status, st)
                            : launch_one<T, NP, S, NW, false, kSeeded, TMA>(a, sg, maps, status, st);
        }
    }
}

// States per lane for a padded state count and configuration index; the
// configurations trade states per lane (fewer shuffles per update) against
// lanes per channel (more warps for problems with few channels).  Keep in
// step with fused_states() in scan_fused.cu.
template <typename T, bool CKPT>
cudaError_t launch_typed_impl(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps,
                              unsigned int *status, int mode, bool tma, int cfg, bool prep, cudaStream_t st) {
    const int N = a.dstate;
    if (N <= 8) {
        if (tma) return cfg == 0 ? by_mode<T, 8, 8, true, CKPT>(a, sg, maps, status, mode, prep, st)
                                 : by_mode<T, 8, 4, true, CKPT>(a, sg, maps, status, mode, prep, st);
        return by_mode<T, 8, 4, false, CKPT>(a, sg, maps, status, mode, prep, st);
    }
    if (N <= 16) {
        if (tma) return cfg == 0 ? by_mode<T, 16, 16, true, CKPT>(a, sg, maps, status, mode, prep, st)
                      : cfg == 1 ? by_mode<T, 16, 8, true, CKPT>(a, sg, maps, status, mode, prep, st)
                      : cfg == 2 ? by_mode<T, 16, 4, true, CKPT>(a, sg, maps, status, mode, prep, st)
                                 : by_mode<T, 16, 2, true, CKPT>(a, sg, maps, status, mode, prep, st);
        return by_mode<T, 16, 8, false, CKPT>(a, sg, maps, status, mode, prep, st);
    }
    if (N <= 32) {
        if (tma) return cfg == 0 ? by_mode<T, 32, 16, true, CKPT>(a, sg, maps, status, mode, prep, st)
                                 : by_mode<T, 32, 8, true, CKPT>(a, sg, maps, status, mode, prep, st);
        return by_mode<T, 32, 8, false, CKPT>(a, sg, maps, status, mode, prep, st);
    }
    return tma ? by_mode<T, 64, 16, true, CKPT>(a, sg, maps, status, mode, prep, st)
               : by_mode<T, 64, 16, false, CKPT>(a, sg, maps, status, mode, prep, st);
}

}  // namespace fused
}  // namespace ssm
