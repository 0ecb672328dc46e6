// Allocation-free entry point: the FUSED scan with its scratch in a fixed
// device array that ships inside the library.
//
// Some callers cannot call cudaMalloc at the point where they run the scan:
// cudaMalloc may synchronise the device and can fail under memory pressure,
// so latency-critical serving loops, code that runs inside a host callback,
// and hosts that hand a library nothing but their input and output buffers
// need a call that touches no allocator at all.  ssm_scan_fwd_noalloc serves
// them: it takes the same inputs and outputs as ssm_scan_fwd and keeps the
// fused kernel's only scratch -- B and C re-laid out as float32 rows -- in
// g_noalloc_scratch below, a file-scope __device__ array of
// kNoAllocScratchBytes (16 MiB) that every GPU loading this library holds
// until the process exits.
#include <cstdint>

#include "../../include/ssm_scan.h"
#include "scan_internal.h"

namespace {

constexpr size_t kNoAllocScratchBytes = (size_t)16 << 20;   // 16 MiB

// The scratch itself.  Host code must not use this name as a device address:
// on the host it is only a stand-in, so the kernel receives the address that
// cudaGetSymbolAddress returns for the current device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

// Device address of g_noalloc_scratch on the current device, or nullptr if
// the lookup fails.  It is looked up on every call rather than cached: after
// a cudaDeviceReset the library's module is loaded again and the array may sit
// at a new address.  Once the module is loaded on a device the lookup
// allocates nothing.
void *scratch_address() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    return p;
}

// Whether the fused kernel's scratch for these sizes fits the array.  The
// first test divides instead of multiplying, so that no product of the sizes
// can wrap around: every prepared row holds at least 128 bytes per (batch,
// step).  Past it batch * seqlen is at most 2^17 and the exact size below
// cannot overflow.
bool scratch_fits(int batch, int dim, int dstate, int64_t seqlen) {
    constexpr uint64_t kMinRowBytes = 128;
    if ((uint64_t)seqlen > kNoAllocScratchBytes / ((uint64_t)batch * kMinRowBytes)) return false;
    return ssm::fused_workspace_bytes(batch, dim, dstate, seqlen) <= kNoAllocScratchBytes;
}

}  // namespace

extern "C" int ssm_scan_fwd_noalloc(const void *x, const void *delta, const float *A, const void *B,
                                    const void *C, const float *D, const void *z, const float *dt_bias,
                                    int delta_softplus, void *y, float *final_state, int batch, int dim,
                                    int dstate, int64_t seqlen, int io_dtype, void *stream) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (batch < 0 || dim < 0 || dstate < 1 || dstate > 64 || seqlen < 0) return SSM_ERR_DIMS;
    // The scratch must hold the fused kernel's B/C rows; reject larger
    // problems before anything touches the GPU.
    if (batch > 0 && dim > 0 && seqlen > 0 && !scratch_fits(batch, dim, dstate, seqlen))
        return SSM_ERR_TOO_LARGE;
    void *scratch = nullptr;
    if (batch > 0 && dim > 0 && seqlen > 0) {
        scratch = scratch_address();
        if (!scratch) return SSM_ERR_LAUNCH;
    }
    // Validation, the empty cases and the launch are those of the device entry
    // point; the fused kernel fully rewrites the scratch before reading it, so
    // nothing in it needs clearing between calls.
    return ssm_scan_fwd_variant(x, delta, A, B, C, D, z, dt_bias, delta_softplus, y, final_state, batch, dim,
                                dstate, seqlen, io_dtype, scratch, kNoAllocScratchBytes, stream,
                                SSM_VARIANT_FUSED);
}
