/*
 * ssm_bwd.h -- C ABI of the backward of the forward selective scan in
 * libssmscan.so (sm_103a).
 *
 * Operation.  For the forward of ssm_scan.h (started from initial_state, or
 * zero) and a scalar loss with dL/dy = dy and dL/dfinal_state = dfinal, the
 * call writes the gradients of every input.  With u_t = Delta_t x_t,
 * q_t = sum_n C h_t + D x_t, g_t = silu(z_t) and dq_t = dy_t g_t, the adjoint
 * of the state runs backwards,
 *
 *     lambda_t[n] = dq_t C[b,n,t] + exp(Delta_{t+1} A[d,n]) lambda_{t+1}[n],
 *     lambda_{L-1} starts from dfinal,
 *
 * and gives
 *     dC[b,n,t] = sum_d dq_t h_t[n]            dB[b,n,t] = sum_d lambda_t[n] u_t
 *     dA[d,n]   = sum_{b,t} lambda_t[n] h_{t-1}[n] a_t[n] Delta_t
 *     ddelta_t  = (sum_n lambda_t[n] h_{t-1}[n] a_t[n] A[d,n] + x_t sum_n lambda_t[n] B[b,n,t]) softplus'(v_t)
 *     dx_t      = Delta_t sum_n lambda_t[n] B[b,n,t] + dq_t D[d]
 *     dD[d]     = sum_{b,t} dq_t x_t           dz_t = dy_t q_t silu'(z_t)
 *     ddt_bias[d] = sum_{b,t} ddelta_t         dinitial_state[b,d,n] = a_0[n] lambda_0[n]
 *
 * evaluated the way "Mamba (part 2): parallel scan and hardware-aware
 * optimisation" (scwacadex.pages.dev) sect. 4.2-4.3 describes: the states are
 * never stored for the whole sequence; only the states at the start of every
 * 32-step chunk are kept -- computed by ssm_scan_bwd (one whole-sequence
 * forward pass that stores them where the channels fill the GPU, else the
 * two-pass forward's totals pass and carry scan), or taken from the
 * checkpoints of the training forward by ssm_scan_bwd_ckpt -- and each
 * chunk's states are recomputed from its start state while the chunks are
 * walked in reverse.
 *
 * Layouts as in ssm_scan.h.  dy, dx, ddelta and dz have the forward's I/O
 * dtype and shape [batch, dim, seqlen]; dA [dim, dstate], dB and dC
 * [batch, dstate, seqlen], dD and ddt_bias [dim], dinitial_state and
 * dfinal_state [batch, dim, dstate] are float32.
 *
 * Ownership and errors as in ssm_scan.h: device pointers owned by the caller,
 * nothing retained, asynchronous on `stream`, host-side validation returning
 * a negative ssm_status_t before anything is launched.  Outputs must not
 * overlap inputs or each other.  dA, dB, dC, dD and ddt_bias are sums formed
 * with float32 atomic additions: their last bits depend on the order in which
 * the additions land.
 */
#ifndef SSM_BWD_H_
#define SSM_BWD_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Device workspace, in bytes, of ssm_scan_bwd (chunk-start states, segment
 * sums and B/C rows prepared as float32); (size_t)-1 for invalid sizes. */
size_t ssm_scan_bwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype);

/* Kernels one ssm_scan_bwd call with these sizes launches on the GPU: the
 * B/C re-layout and the chunk-start states (one whole-sequence pass of the
 * fused forward where the channels give at least one consumer warp per SM
 * sub-partition, else a totals pass and a carry scan over the chunks), the
 * reverse walk, and for walks split into segments the adjoint totals and
 * their carry.  0 for an empty problem, -1 for invalid sizes.  Host only. */
int ssm_scan_bwd_kernel_count(int batch, int dim, int dstate, int64_t seqlen);

/*
 *   x, delta, A, B, C, D, z, dt_bias, delta_softplus, initial_state
 *                  the forward's inputs (as ssm_scan_fwd_from_state; D, z,
 *                  dt_bias and initial_state may be NULL).
 *   dy             required.  [batch, dim, seqlen], io_dtype.
 *   dfinal_state   optional (NULL: zero).  [batch, dim, dstate] float32.
 *   dx, ddelta     required outputs.  [batch, dim, seqlen], io_dtype.
 *   dA             required output.  [dim, dstate] float32.
 *   dB, dC         required outputs.  [batch, dstate, seqlen] float32.
 *   dD             required output iff D is given.  [dim] float32.
 *   dz             required output iff z is given.  [batch, dim, seqlen], io_dtype.
 *   ddt_bias       optional output (NULL: not written).  [dim] float32.
 *   dinitial_state optional output (NULL: not written).  [batch, dim, dstate] float32.
 *   batch, dim >= 0, dstate 1 .. 64, seqlen >= 0, io_dtype SSM_F32 or SSM_BF16.
 *   workspace      at least ssm_scan_bwd_workspace_size() bytes, 256-byte
 *                  aligned (NULL when that size is 0).
 * Returns SSM_OK or a negative ssm_status_t.
 */
int ssm_scan_bwd(const void *x, const void *delta, const float *A, const void *B, const void *C,
                 const float *D, const void *z, const float *dt_bias, int delta_softplus,
                 const float *initial_state, const void *dy, const float *dfinal_state,
                 void *dx, void *ddelta, float *dA, float *dB, float *dC, float *dD, void *dz,
                 float *ddt_bias, float *dinitial_state,
                 int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Device workspace, in bytes, of ssm_scan_bwd_ckpt (segment sums of walks
 * split into segments; often 0); (size_t)-1 for invalid sizes. */
size_t ssm_scan_bwd_ckpt_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype);

/* Kernels one ssm_scan_bwd_ckpt call launches: the reverse walk, plus the
 * adjoint totals and their carry for walks split into segments.  0 for an
 * empty problem, -1 for invalid sizes.  Host only. */
int ssm_scan_bwd_ckpt_kernel_count(int batch, int dim, int dstate, int64_t seqlen);

/*
 * The backward from the checkpoints a forward wrote (ssm_scan_fwd_ckpt,
 * ssm_scan.h): ssm_scan_bwd without the chunk-start states pass.
 *   ckpt          required input.  The checkpoints of ssm_scan_fwd_ckpt over
 *                 the same inputs and start state, ssm_scan_ckpt_size() bytes;
 *                 the start state enters only through them.
 * Every other argument as ssm_scan_bwd (which takes initial_state where this
 * takes ckpt); the workspace is ssm_scan_bwd_ckpt_workspace_size() bytes.
 */
int ssm_scan_bwd_ckpt(const void *x, const void *delta, const float *A, const void *B, const void *C,
                      const float *D, const void *z, const float *dt_bias, int delta_softplus,
                      const float *ckpt, const void *dy, const float *dfinal_state,
                      void *dx, void *ddelta, float *dA, float *dB, float *dC, float *dD, void *dz,
                      float *ddt_bias, float *dinitial_state,
                      int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                      void *workspace, size_t workspace_bytes, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_BWD_H_ */
