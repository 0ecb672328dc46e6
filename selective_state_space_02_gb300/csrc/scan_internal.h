// Internal interface between the C ABI (ssm_scan_api.cu) and the kernel
// translation units.  Not installed; the public interface is include/ssm_scan.h.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>

namespace ssm {

// One validated forward problem (all pointers are device pointers).
struct FwdArgs {
    const void *x;
    const void *delta;
    const float *A;
    const void *B;
    const void *C;
    const float *D;        // nullable
    const void *z;         // nullable
    const float *dt_bias;  // nullable
    int softplus;
    void *y;
    float *final_state;    // nullable
    int batch;
    int dim;
    int dstate;
    int64_t L;
    int bf16;              // 1: io elements are bf16, 0: float32
    int vec16;             // 1: every io row starts 16-byte aligned
    const float *h0 = nullptr;   // nullable start state [batch, dim, dstate]; zeros if null
    // causal depthwise convolution + SiLU fused in front of the scan (FUSED
    // variant, whole sequences): x is then the raw input, conv_k taps (1..4)
    int conv_k = 0;
    const float *conv_w = nullptr;       // [dim, conv_k]
    const float *conv_b = nullptr;       // nullable [dim]
    const void *conv_state = nullptr;    // nullable [batch, dim, conv_k - 1], io dtype: inputs before t = 0
    // nullable: checkpoints for the backward, the state at the start of every
    // kCkptSteps-step chunk, [nchunk][batch*dim][dstate] float32 (FUSED and
    // TWOPASS variants)
    float *ckpt = nullptr;
};

// Steps per checkpointed chunk: the chunk length of the backward's recomputation.
constexpr int kCkptSteps = 32;

// Each launcher returns cudaSuccess or the launch error.
cudaError_t launch_fused(const FwdArgs &a, void *workspace, cudaStream_t s);
cudaError_t launch_chunked(const FwdArgs &a, void *workspace, cudaStream_t s);
cudaError_t launch_twopass(const FwdArgs &a, void *workspace, cudaStream_t s);

// States at the start of every segment of seg_len steps (segment 0 starts
// from a.h0, or zero), as [nseg][batch*dim][dstate] float32 at the start of
// `workspace`.  With channels for one consumer warp per SM sub-partition one
// whole-sequence pass of the fused kernel writes them as it goes; otherwise
// the two-pass forward's totals pass and carry scan compute them.  The
// workspace also holds that pass's segment sums and prepared B/C rows.
size_t chunk_states_workspace_bytes(int batch, int dim, int dstate, int64_t L, int64_t seg_len);
cudaError_t chunk_start_states(const FwdArgs &a, int64_t seg_len, void *workspace, cudaStream_t st);
// Kernels chunk_start_states launches for these sizes.
int chunk_start_states_kernels(int batch, int dim, int dstate, int64_t L, int64_t seg_len);

// Device address of the status word of the bounded waits on the current
// device (nullptr if the lookup fails); kernels OR bit 0 into it.
unsigned int *device_status_word();

// Launch the self-test kernel whose bounded wait runs out after `limit` SM
// cycles and flags the status word.
cudaError_t selftest_wait_timeout(long long limit, cudaStream_t st);

// Device status word of the bounded waits (bit 0: a wait gave up).  Reads it
// through `st` (synchronising the stream), optionally clearing it.
int read_device_status(cudaStream_t st, bool clear, unsigned int *out);

// Workspace bytes of the fused variant (B/C prepared as float32 rows).
size_t fused_workspace_bytes(int batch, int dim, int dstate, int64_t L);

// Workspace bytes of the chunked variant (B/C prepared per chunk).
size_t chunked_workspace_bytes(int batch, int dim, int dstate, int64_t L);

// Chunk length and workspace bytes of the two-pass variant.
int64_t twopass_chunk_len(int batch, int dim, int dstate, int64_t L);
size_t twopass_workspace_bytes(int batch, int dim, int dstate, int64_t L);

}  // namespace ssm
