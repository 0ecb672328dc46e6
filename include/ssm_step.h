/*
 * ssm_step.h -- C ABI of the single-token (decode) step of the selective
 * state-space recurrence in libssmscan.so (sm_103a).
 *
 * Operation.  Inference advances the recurrence one token at a time with
 * constant work and memory per token ("Mamba (part 2): parallel scan and
 * hardware-aware optimisation", scwacadex.pages.dev, sect. 6 and 7): for every
 * channel (b, d) and state n,
 *
 *     Delta       = softplus(delta[b,d] + dt_bias[d])        (or without softplus)
 *     state[b,d,n] <- exp(Delta * A[d,n]) * state[b,d,n] + Delta * B[b,n] * x[b,d]
 *     y[b,d]      = (sum_n C[b,n] * state[b,d,n] + D[d] * x[b,d]) * silu(z[b,d])
 *
 * which is one step t of the forward in ssm_scan.h, so that seqlen calls
 * reproduce ssm_scan_fwd_from_state over seqlen steps up to float32 rounding.
 *
 * Layouts (row-major, contiguous; element type io_dtype unless stated):
 *   state          : [batch, dim, dstate]  float32, read and updated in place
 *   x, delta, z, y : [batch, dim]
 *   B, C           : [batch, dstate]
 *   A              : [dim, dstate]         float32
 *   D, dt_bias     : [dim]                 float32
 *
 * Ownership.  Device pointers owned by the caller; nothing is allocated or
 * retained.  Asynchronous on `stream`.  Inputs are only read; `y` must not
 * overlap any input or the state, and the state must not overlap an input.
 *
 * Errors.  Host-side validation returns a negative ssm_status_t from
 * ssm_scan.h (SSM_ERR_NULL, _DIMS, _ALIGN, _DTYPE, _ALIAS) and launches
 * nothing; a launch rejected by the CUDA runtime returns SSM_ERR_LAUNCH.
 * The kernel has no waits.
 *
 * Precision.  float32 arithmetic and state for both I/O types; bf16 y is
 * rounded to nearest even.
 */
#ifndef SSM_STEP_H_
#define SSM_STEP_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/*
 *   state         required, in/out.  [batch, dim, dstate] float32, 4-byte aligned.
 *   x, delta      required.  [batch, dim], io_dtype.
 *   A             required.  [dim, dstate] float32.
 *   B, C          required.  [batch, dstate], io_dtype.
 *   D, z, dt_bias optional (NULL: no skip / no gate / zero bias).
 *   delta_softplus  nonzero: Delta = softplus(delta + dt_bias).
 *   y             required output.  [batch, dim], io_dtype.
 *   batch, dim    >= 0 (0: nothing is launched).   dstate 1 .. 64.
 *   io_dtype      SSM_F32 or SSM_BF16.
 * Returns SSM_OK or a negative ssm_status_t.
 */
int ssm_scan_step(float *state, const void *x, const void *delta, const float *A, const void *B,
                  const void *C, const float *D, const void *z, const float *dt_bias,
                  int delta_softplus, void *y, int batch, int dim, int dstate, int io_dtype,
                  void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_STEP_H_ */
