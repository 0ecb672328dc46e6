// f32 instantiations of the fused scan kernel.
#include "scan_fused_dispatch.cuh"

namespace ssm {
namespace fused {
template <>
cudaError_t launch_typed<float>(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps, unsigned int *status,
                             int mode, bool tma, int cfg, bool prepare, cudaStream_t st) {
    return launch_typed_impl<float, false>(a, sg, maps, status, mode, tma, cfg, prepare, st);
}
}  // namespace fused
}  // namespace ssm
