/*
 * ssm_scan.h -- C ABI of the GB300 forward selective-scan library
 * (libssmscan.so, sm_103a).
 *
 * Operation.  For every channel (b, d) of a Mamba-style selective state-space
 * layer with diagonal A, the library evaluates
 *
 *     Delta_t = softplus(delta[b,d,t] + dt_bias[d])          (or without softplus)
 *     a_t[n]  = exp(Delta_t * A[d,n]),   b_t[n] = Delta_t * B[b,n,t] * x[b,d,t]
 *     h_t[n]  = a_t[n] * h_{t-1}[n] + b_t[n],  h_{-1} = 0
 *     y[b,d,t] = (sum_n C[b,n,t] * h_t[n] + D[d] * x[b,d,t]) * silu(z[b,d,t])
 *
 * as an associative scan over the affine pairs (a, b) under
 * (a2,b2) o (a1,b1) = (a2*a1, a2*b1 + b2), identity (1, 0).
 * Sources: "Mamba hardware-aware parallel associative scan"
 * (pwwt.cn/news/6375169) sect. 1.2 (pairs, composition, discretisation),
 * sect. 2.1-2.2 (prefix scan, chunked two-pass), sect. 3.3 (chunk carry),
 * sect. 4.1 (fusion); "Mamba (part 2): parallel scan and hardware-aware
 * optimisation" (scwacadex.pages.dev) sect. 2.2-2.4 (operator, tree),
 * sect. 4.1-4.2 (fusion, intermediate states never written to HBM).
 *
 * Layouts (all row-major and contiguous, element type `io_dtype` unless
 * stated):
 *   x, delta, z, y : [batch, dim, seqlen]
 *   B, C           : [batch, dstate, seqlen]
 *   A              : [dim, dstate]            float32
 *   D, dt_bias     : [dim]                    float32
 *   final_state    : [batch, dim, dstate]     float32  (h after the last step)
 *
 * Ownership.  Every pointer of the device entry points is a device pointer
 * owned by the caller.  The library allocates no memory and keeps no
 * pointer after a call returns.  Inputs are only read.  `y` and
 * `final_state` must not overlap any input.  Calls are asynchronous on
 * `stream` (a cudaStream_t; NULL means the legacy default stream).
 *
 * Errors.  Arguments are validated on the host before anything is launched;
 * a failed check returns a negative ssm_status_t and launches nothing.  A
 * launch failure reported by the CUDA runtime returns SSM_ERR_LAUNCH.
 * Device-side faults are not expected for validated arguments; none of the
 * kernels waits on another block.
 *
 * Precision.  All arithmetic (discretisation, exp, scan, contraction, gate)
 * is float32 for both I/O types; the state is float32.  bf16 outputs are
 * rounded to nearest even.  Results differ from an exact evaluation only by
 * float32 rounding (the scan order changes the rounding, not the result).
 */
#ifndef SSM_SCAN_H_
#define SSM_SCAN_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Element type of x, delta, z, B, C and y. */
typedef enum { SSM_F32 = 0, SSM_BF16 = 1 } ssm_dtype_t;

typedef enum {
    SSM_OK = 0,
    SSM_ERR_NULL = -1,        /* a required pointer is NULL                       */
    SSM_ERR_DIMS = -2,        /* a size is out of range (see each entry point)    */
    SSM_ERR_ALIGN = -3,       /* a pointer is not aligned to its element size     */
    SSM_ERR_DTYPE = -4,       /* io_dtype is not an ssm_dtype_t                   */
    SSM_ERR_WORKSPACE = -5,   /* workspace missing, too small or misaligned       */
    SSM_ERR_LAUNCH = -6,      /* the CUDA runtime rejected a launch or a copy     */
    SSM_ERR_UNSUPPORTED = -8, /* the variant cannot run this shape                */
    SSM_ERR_ALIAS = -9,       /* an output overlaps an input                      */
    SSM_ERR_VARIANT = -10,    /* unknown variant number                           */
    SSM_ERR_TOO_LARGE = -11   /* problem exceeds the built-in scratch of
                                 ssm_scan_fwd_noalloc                             */
} ssm_status_t;

/* Evaluation strategies; all compute the same function.
 *  FUSED   : channel-parallel, time-serial.  Each thread keeps a few states of
 *            one channel in registers and walks the sequence in staged tiles
 *            ("Mamba hardware-aware parallel associative scan", sect. 2.2,
 *            third approach).  Workspace: B and C re-laid out once per call
 *            as float32 rows (batch * seqlen * (2 * padded dstate + 16) * 4
 *            bytes, padded dstate = 8, 16, 32 or 64).
 *  CHUNKED : time-parallel.  One warp per channel scans chunks of 32*k
 *            steps: every lane folds its k steps, a warp-shuffle
 *            Hillis-Steele scan per state pair combines the lanes' (a, b)
 *            totals, and the state is carried from chunk to chunk (sect. 2.1
 *            hybrid, sect. 3.2 warp shuffle).  Workspace: B and C re-laid out
 *            per chunk, batch * ceil(seqlen / 32k) * ceil(dstate / 2) * 32k
 *            * 16 bytes (k = 8, or 4 above 32 states).
 *  TWOPASS : the sequence is cut into chunks processed in parallel; pass 1
 *            writes every chunk's total (A_k, B_k), a small scan over the
 *            chunk totals gives each chunk's start state, and pass 2 re-runs
 *            the fused scan from that state (sect. 2.2, 3.3).  Workspace:
 *            the chunk totals plus the fused variant's B/C rows.
 *  AUTO    : the library picks one from the shape (ssm_scan_select_variant). */
typedef enum {
    SSM_VARIANT_AUTO = 0,
    SSM_VARIANT_FUSED = 1,
    SSM_VARIANT_CHUNKED = 2,
    SSM_VARIANT_TWOPASS = 3
} ssm_variant_t;

/* Library version, (major << 16) | minor. */
int ssm_scan_version(void);

/* Static description of a status code (never NULL). */
const char *ssm_scan_status_string(int status);

/* The variant AUTO resolves to for this shape (host only, no GPU needed).
 * Returns an ssm_variant_t > 0, or a negative status for invalid sizes. */
int ssm_scan_select_variant(int batch, int dim, int dstate, int64_t seqlen, int io_dtype);

/* Device workspace, in bytes, that ssm_scan_fwd needs for `variant` (AUTO
 * resolves first).  0 means the workspace pointer may be NULL.  Returns
 * (size_t)-1 for invalid sizes. */
size_t ssm_scan_fwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen,
                                   int io_dtype, int variant);

/*
 * Forward selective scan on device buffers (the hot path).
 *
 *   x, delta      required.  [batch, dim, seqlen], io_dtype.
 *   A             required.  [dim, dstate] float32 (normally negative).
 *   B, C          required.  [batch, dstate, seqlen], io_dtype.
 *   D             optional (NULL: no skip term).  [dim] float32.
 *   z             optional (NULL: no gate).  [batch, dim, seqlen], io_dtype.
 *   dt_bias       optional (NULL: zero bias).  [dim] float32.
 *   delta_softplus  nonzero: Delta = softplus(delta + dt_bias); zero: Delta = delta + dt_bias.
 *   y             required output.  [batch, dim, seqlen], io_dtype.
 *   final_state   optional output (NULL: not written).  [batch, dim, dstate] float32.
 *   batch, dim    >= 0 (0 is an empty problem: nothing is launched).
 *   dstate        1 .. 64.
 *   seqlen        >= 0 (0: y is empty and final_state, if given, is set to 0).
 *   io_dtype      SSM_F32 or SSM_BF16.
 *   workspace     device scratch of at least ssm_scan_fwd_workspace_size()
 *                 bytes, 256-byte aligned; may be NULL when that size is 0.
 *   stream        cudaStream_t to launch on.
 * Alignment: io_dtype pointers must be aligned to the element size, float32
 * pointers to 4 bytes.  16-byte aligned rows (seqlen * element size a
 * multiple of 16 and 16-byte aligned bases) take the vectorised path;
 * anything else runs the element-wise load path on the GPU.
 * Returns SSM_OK or a negative ssm_status_t.
 */
int ssm_scan_fwd(const void *x, const void *delta, const float *A, const void *B,
                 const void *C, const float *D, const void *z, const float *dt_bias,
                 int delta_softplus, void *y, float *final_state,
                 int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                 void *workspace, size_t workspace_bytes, void *stream);

/* Same as ssm_scan_fwd with an explicit ssm_variant_t. */
int ssm_scan_fwd_variant(const void *x, const void *delta, const float *A, const void *B,
                         const void *C, const float *D, const void *z, const float *dt_bias,
                         int delta_softplus, void *y, float *final_state,
                         int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                         void *workspace, size_t workspace_bytes, void *stream, int variant);

/*
 * Forward selective scan from a given start state: h_{-1} = initial_state
 * instead of 0, everything else as ssm_scan_fwd_variant.  A long sequence cut
 * into segments is scanned one segment per call, each call starting from the
 * state the previous one ended in -- the boundary state a segment restarts
 * from in "Mamba (part 2)" sect. 4.3 -- so that the concatenated y equals one
 * call over the whole sequence up to float32 rounding.
 *   initial_state  optional input (NULL: zero state, identical to
 *                  ssm_scan_fwd_variant).  [batch, dim, dstate] float32,
 *                  4-byte aligned.  It must not overlap y.  final_state may be
 *                  the same array (the state is then advanced in place) but
 *                  must not overlap it otherwise (SSM_ERR_ALIAS).
 *   seqlen == 0    final_state, if given, receives initial_state (or 0).
 * The workspace size is that of ssm_scan_fwd_workspace_size for the variant.
 */
int ssm_scan_fwd_from_state(const void *x, const void *delta, const float *A, const void *B,
                            const void *C, const float *D, const void *z, const float *dt_bias,
                            int delta_softplus, const float *initial_state, void *y, float *final_state,
                            int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                            void *workspace, size_t workspace_bytes, void *stream, int variant);

/* Bytes of the checkpoints of ssm_scan_fwd_ckpt: ceil(seqlen / 32) chunk
 * states of [batch, dim, dstate] float32.  (size_t)-1 for invalid sizes. */
size_t ssm_scan_ckpt_size(int batch, int dim, int dstate, int64_t seqlen);

/* Device workspace, in bytes, of ssm_scan_fwd_ckpt for `variant`; (size_t)-1
 * for invalid sizes or a variant that cannot write checkpoints. */
size_t ssm_scan_fwd_ckpt_workspace_size(int batch, int dim, int dstate, int64_t seqlen,
                                        int io_dtype, int variant);

/*
 * Forward for training: ssm_scan_fwd_from_state that also stores the state
 * at the start of every 32-step chunk, the boundary states the backward
 * recomputes each chunk from ("Mamba (part 2)" sect. 4.3: store the states
 * at chunk boundaries, recompute inside the chunk).  ssm_scan_bwd_ckpt
 * (ssm_bwd.h) then starts from them instead of computing them again.
 *   ckpt          required output.  [ceil(seqlen / 32)][batch * dim][dstate]
 *                 float32, 4-byte aligned, ssm_scan_ckpt_size() bytes; entry
 *                 k is h before step 32 k (entry 0: initial_state, or 0).  It
 *                 must not overlap any input or output.
 *   variant       FUSED or TWOPASS store the checkpoints as they go; AUTO
 *                 resolves as for ssm_scan_fwd but takes TWOPASS where that
 *                 would pick CHUNKED; CHUNKED returns SSM_ERR_UNSUPPORTED.
 *   workspace     at least ssm_scan_fwd_ckpt_workspace_size() bytes.
 * y and final_state are those of ssm_scan_fwd_from_state with the same
 * variant (the same kernels, with the extra stores).
 */
int ssm_scan_fwd_ckpt(const void *x, const void *delta, const float *A, const void *B,
                      const void *C, const float *D, const void *z, const float *dt_bias,
                      int delta_softplus, const float *initial_state, void *y, float *final_state,
                      float *ckpt, int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                      void *workspace, size_t workspace_bytes, void *stream, int variant);

/* Device status of earlier launches on the current device: bit 0 is set when
 * a kernel's bounded wait on its own TMA copies gave up (the output of that
 * call is then invalid).  The word is one per device and process, shared by
 * every call on that device: a set bit says that some call since the last
 * clear gave up, not which one, so callers that share a device clear and read
 * it at points where they know which calls ran in between.  Synchronises
 * `stream`; `clear` nonzero resets the word.  Returns the status (>= 0) or
 * SSM_ERR_LAUNCH. */
int ssm_scan_device_status(void *stream, int clear);

/* Self-test of the bounded waits (the failure detection behind
 * ssm_scan_device_status).  Launches one small kernel on `stream` whose
 * thread waits, with the same bounded wait the scan kernels use, on a
 * shared-memory mbarrier that nothing ever arrives on and that no copy
 * targets.  After `limit_cycles` SM cycles (1 .. 2^31) the wait gives up, sets
 * bit 0 of the device status word and the kernel returns normally, so the
 * context stays usable.  The caller then reads (and clears) the word with
 * ssm_scan_device_status.  Returns SSM_OK, SSM_ERR_DIMS for a limit out of
 * range or SSM_ERR_LAUNCH.  Sets the status word shared by every call on the
 * device: run it only while no scan is in flight. */
int ssm_scan_selftest_wait_timeout(long long limit_cycles, void *stream);

/* Device bytes that ssm_scan_fwd_host needs as `device_buffer`: room for the
 * device copies of every input and output, the state carried between time
 * chunks and the largest workspace a chunk needs, each 256-byte aligned.
 * Returns (size_t)-1 for invalid sizes. */
size_t ssm_scan_fwd_host_buffer_size(int batch, int dim, int dstate, int64_t seqlen,
                                     int io_dtype, int has_D, int has_z, int has_dt_bias,
                                     int has_final_state, int variant);

/*
 * Forward selective scan on HOST buffers: the end-to-end call.  Same
 * arguments and layouts as ssm_scan_fwd, but every tensor pointer is a host
 * pointer (page-locked memory gives the fastest copies); `device_buffer` is
 * caller-owned device memory of at least ssm_scan_fwd_host_buffer_size()
 * bytes, 256-byte aligned.
 *
 * Problems of 16 MiB or more (x, delta, z and y together) are cut along the
 * sequence into two time chunks, from 48 MiB into three.  Chunk j's columns of
 * x, delta, z, B and C are copied in on an internal stream, scanned on
 * `stream` starting from the state chunk j-1 ended in (ssm_scan_fwd_from_state
 * semantics, the state kept in float32 on the device), and y's columns are
 * copied back on a second internal stream, so the copies of neighbouring
 * chunks overlap the scans; `variant` applies to every chunk (AUTO picks per
 * chunk shape).  The internal streams and events are created by the first
 * call on a device and kept until the process exits; calls on one device
 * are serialised.  Work already queued on `stream` runs first, and the call
 * returns after every copy has finished, also on error.
 */
int ssm_scan_fwd_host(const void *x, const void *delta, const float *A, const void *B,
                      const void *C, const float *D, const void *z, const float *dt_bias,
                      int delta_softplus, void *y, float *final_state,
                      int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                      void *device_buffer, size_t device_buffer_bytes, void *stream,
                      int variant);

/*
 * Forward selective scan that allocates nothing (no counterpart in the source
 * pages; it exists for callers that cannot allocate).
 *
 * For callers that cannot call cudaMalloc where they run the scan --
 * cudaMalloc may synchronise the device and can fail under memory pressure,
 * which latency-critical serving loops, host callbacks and hosts that hand
 * over only their input and output buffers cannot afford.  Same arguments,
 * layouts, validation and result as ssm_scan_fwd_variant(..., FUSED) without
 * the workspace: the fused kernel's scratch (B and C re-laid out as float32
 * rows) lives in a 16 MiB device array inside the library, which every GPU
 * that loads the library holds until the process exits.
 *   Limit: batch * seqlen * (2 * padded dstate + 16) * 4 bytes (rounded up to
 *   256) must not exceed 16 MiB, padded dstate = 8, 16, 32 or 64; larger
 *   problems return SSM_ERR_TOO_LARGE before anything is launched.
 *   Set-up: every call looks up the array's device address on the current
 *   device (cudaGetSymbolAddress).  With CUDA's lazy module loading the first
 *   call on a device may be the one that loads the library's module there,
 *   which reserves the 16 MiB array at that moment (and can fail or
 *   synchronise like any module load); later calls allocate nothing.  Make
 *   that first call before any stream capture, for example once at start-up.
 *   After cudaDeviceReset the next call finds the array at its new address.
 *   Sharing: all calls on a device use the same array.  Each call rewrites
 *   the part it reads, so no clearing is needed between calls, but calls that
 *   overlap on the GPU (different streams, no ordering) race on it and must
 *   be serialised by the caller.
 * Beyond the first call's module load described above, allocates no memory,
 * host or device, and calls no allocating CUDA routine.
 */
int ssm_scan_fwd_noalloc(const void *x, const void *delta, const float *A, const void *B,
                         const void *C, const float *D, const void *z, const float *dt_bias,
                         int delta_softplus, void *y, float *final_state,
                         int batch, int dim, int dstate, int64_t seqlen, int io_dtype, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* SSM_SCAN_H_ */
