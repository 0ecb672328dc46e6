// f32 instantiations of the fused scan kernel that also stores the
// forward's checkpoints (a translation unit of its own, compiled in parallel).
#include "scan_fused_dispatch.cuh"

namespace ssm {
namespace fused {
template <>
cudaError_t launch_typed_ckpt<float>(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps, unsigned int *status,
                                  int mode, bool tma, int cfg, bool prepare, cudaStream_t st) {
    return launch_typed_impl<float, true>(a, sg, maps, status, mode, tma, cfg, prepare, st);
}
}  // namespace fused
}  // namespace ssm
