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

/*
 * Convolution and scan in one call.  "Mamba (part 2)" sect. 4.1 describes the
 * fused block: the 1-D convolution and its SiLU feed the selective scan
 * without the convolution's output going through global memory.  This call
 * computes, for every channel,
 *
 *     xc = ssm_conv1d_fwd(x, conv_weight, conv_bias, conv_state, silu = 1)
 *     y  = the selective scan of ssm_scan_fwd with xc as its input x
 *
 * (the D skip uses xc).  Scan arguments, layouts and errors as in
 * ssm_scan_fwd (ssm_scan.h), x being the convolution's raw input; conv_weight
 * [dim, conv_width] float32 (required), conv_bias [dim] float32 and
 * conv_state [batch, dim, conv_width - 1] io_dtype (optional) as in
 * ssm_conv1d_fwd; conv_width 1 .. 8.  The final state is the scan's.
 *   mode SSM_CONV_FUSED   : the convolution runs inside the FUSED scan
 *                           kernel; its output stays in float32 registers
 *                           (never rounded to io_dtype).  conv_width <= 4,
 *                           else SSM_ERR_UNSUPPORTED.
 *   mode SSM_CONV_SEPARATE: ssm_conv1d_fwd writes xc (io_dtype) to the start
 *                           of the workspace, then the AUTO scan reads it.
 *   mode SSM_CONV_AUTO    : FUSED when conv_width <= 4 and the scan's AUTO
 *                           variant for the shape is FUSED, else SEPARATE.
 * The workspace must hold ssm_scan_fwd_conv_workspace_size(...) bytes
 * (256-byte aligned; NULL allowed when that is 0).  Asynchronous on `stream`.
 */
enum { SSM_CONV_AUTO = -1, SSM_CONV_SEPARATE = 0, SSM_CONV_FUSED = 1 };

size_t ssm_scan_fwd_conv_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int conv_width,
                                        int io_dtype, int mode);

int ssm_scan_fwd_conv(const void *x, const float *conv_weight, const float *conv_bias, const void *conv_state,
                      int conv_width, const void *delta, const float *A, const void *B, const void *C,
                      const float *D, const void *z, const float *dt_bias, int delta_softplus, void *y,
                      float *final_state, int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                      void *workspace, size_t workspace_bytes, void *stream, int mode);

#ifdef __cplusplus
}
#endif

#endif /* SSM_CONV_H_ */
