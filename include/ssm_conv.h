/*
 * ssm_conv.h -- C ABI of the causal depthwise convolution that runs in front
 * of the selective scan, in libssmscan.so (sm_103a).
 *
 * Operation.  "Mamba (part 2): parallel scan and hardware-aware optimisation"
 * (scwacadex.pages.dev) sect. 4.1 lists a 1-D convolution and SiLU among the
 * operators fused ahead of the scan.  For every channel (b, d), with K taps
 * weight[d, 0..K-1]:
 *
 *     v_t = bias[d] + sum_{k=0}^{K-1} weight[d,k] * x[b,d,t-K+1+k]
 *     y_t = silu(v_t)              (or v_t when silu is 0)
 *
 * where the inputs before t = 0 are state_in[b,d,0..K-2] (the K-1 inputs that
 * preceded the sequence, oldest first), or zeros.  state_out receives the last
 * K-1 inputs of that history followed by the sequence, so that the next
 * segment of a stream continues the convolution exactly.
 *
 * Layouts (row-major, contiguous): x, y [batch, dim, seqlen] and state_in,
 * state_out [batch, dim, K-1] in io_dtype; weight [dim, K] and bias [dim]
 * float32.  Arithmetic is float32; bf16 outputs are rounded to nearest even.
 *
 * Ownership and errors as in ssm_scan.h: device pointers owned by the caller,
 * nothing allocated or retained, asynchronous on `stream`; host-side
 * validation returns a negative ssm_status_t (SSM_ERR_NULL, _DIMS, _ALIGN,
 * _DTYPE, _ALIAS) before anything is launched.  y and state_out must not
 * overlap any input or each other.
 */
#ifndef SSM_CONV_H_
#define SSM_CONV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 *   x          required.  [batch, dim, seqlen], io_dtype.
 *   weight     required.  [dim, width] float32.
 *   bias       optional (NULL: none).  [dim] float32.
 *   state_in   optional (NULL: zero history).  [batch, dim, width-1], io_dtype.
 *   y          required output.  [batch, dim, seqlen], io_dtype.
 *   state_out  optional output (NULL: not written).  [batch, dim, width-1], io_dtype.
 *   silu       nonzero: apply SiLU to the convolution.
 *   batch, dim >= 0; seqlen >= 0; width 1 .. 8; io_dtype SSM_F32 or SSM_BF16.
 * Returns SSM_OK or a negative ssm_status_t.
 */
int ssm_conv1d_fwd(const void *x, const float *weight, const float *bias, const void *state_in, void *y,
                   void *state_out, int silu, int batch, int dim, int64_t seqlen, int width, int io_dtype,
                   void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_CONV_H_ */
