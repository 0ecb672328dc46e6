/*
 * ssm_oracle.c -- serial fp64 reference for the forward selective scan.
 *
 * TEST INFRASTRUCTURE ONLY.  Only tests, the package smoke check and the
 * benchmark's CPU-baseline leg may load this code.  It shares no source,
 * header, table or helper with the CUDA library; the two are independent
 * statements of the same mathematics so that one can check the other.
 *
 * Sources (cited below by tag and section):
 *   [P1] "Mamba hardware-aware parallel associative scan" (pwwt.cn/news/6375169)
 *        sect. 1.2 (affine pair, composition, identity, discretisation),
 *        sect. 2.1 (prefix result, Hillis-Steele, Blelloch, identity padding),
 *        sect. 2.2 + 3.3 (chunked two-pass scan, boundary-state formula),
 *        sect. 4.3 (numerics).
 *   [P3] "Mamba (part 2): parallel scan and hardware-aware optimisation"
 *        (scwacadex.pages.dev, blog8_mamba_parallel_scan)
 *        sect. 2.1-2.3 (operator (x), associativity proof),
 *        sect. 2.4 (tree reduction), sect. 4.3 (chunk-boundary states),
 *        sect. 6-7 (inference runs the recurrence one token at a time).
 *
 * Everything is computed in IEEE double with the plain definitions; nothing
 * is blocked, fused or reordered beyond what the cited definition states.
 * Inputs are read as float (the exact values the GPU receives: bf16 inputs
 * are widened exactly to float by the caller) and widened to double here.
 */
#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------ */
/* Algebra of affine steps h -> a*h + b                                */
/* ------------------------------------------------------------------ */

/* [P1 sect. 1.2], [P3 sect. 2.2]: (a2,b2) o (a1,b1) = (a2*a1, a2*b1 + b2);
 * the step on the left is applied after the step on the right. */
void ssm_oracle_compose(double a2, double b2, double a1, double b1,
                        double *a_out, double *b_out)
{
    *a_out = a2 * a1;
    *b_out = a2 * b1 + b2;
}

/* [P1 sect. 2.1]: inclusive prefix (A_t, B_t) = (a_t,b_t) o ... o (a_1,b_1),
 * so that h_t = A_t*h_0 + B_t.  Serial left-to-right evaluation. */
void ssm_oracle_scan_serial(const double *a, const double *b, long L,
                            double *A_out, double *B_out)
{
    double A = 1.0, B = 0.0;            /* identity (1,0) */
    for (long t = 0; t < L; ++t) {
        double nA, nB;
        ssm_oracle_compose(a[t], b[t], A, B, &nA, &nB);
        A = nA; B = nB;
        A_out[t] = A; B_out[t] = B;
    }
}

/* [P1 sect. 2.1] Hillis-Steele inclusive scan: ceil(log2 L) rounds; in round
 * with distance d every i >= d takes (x[i]) o (x[i-d]).  Double buffered. */
int ssm_oracle_scan_hillis_steele(const double *a, const double *b, long L,
                                  double *A_out, double *B_out)
{
    if (L <= 0) return 0;
    double *ta = (double *)malloc(sizeof(double) * (size_t)L);
    double *tb = (double *)malloc(sizeof(double) * (size_t)L);
    if (!ta || !tb) { free(ta); free(tb); return -1; }
    memcpy(A_out, a, sizeof(double) * (size_t)L);
    memcpy(B_out, b, sizeof(double) * (size_t)L);
    double *ca = A_out, *cb = B_out, *na = ta, *nb = tb;
    for (long d = 1; d < L; d <<= 1) {
        for (long i = 0; i < L; ++i) {
            if (i >= d)
                ssm_oracle_compose(ca[i], cb[i], ca[i - d], cb[i - d], &na[i], &nb[i]);
            else { na[i] = ca[i]; nb[i] = cb[i]; }
        }
        double *s;
        s = ca; ca = na; na = s;
        s = cb; cb = nb; nb = s;
    }
    if (ca != A_out) {
        memcpy(A_out, ca, sizeof(double) * (size_t)L);
        memcpy(B_out, cb, sizeof(double) * (size_t)L);
    }
    free(ta); free(tb);
    return 0;
}

/* [P1 sect. 2.1] Blelloch work-efficient scan.  The sequence is padded with
 * the identity (1,0) up to a power of two, an up-sweep builds the reduction
 * tree [P3 sect. 2.4], a down-sweep distributes exclusive prefixes, and the
 * inclusive result is each element composed after its exclusive prefix. */
int ssm_oracle_scan_blelloch(const double *a, const double *b, long L,
                             double *A_out, double *B_out)
{
    if (L <= 0) return 0;
    long P = 1;
    while (P < L) P <<= 1;
    double *ta = (double *)malloc(sizeof(double) * (size_t)P);
    double *tb = (double *)malloc(sizeof(double) * (size_t)P);
    if (!ta || !tb) { free(ta); free(tb); return -1; }
    for (long i = 0; i < P; ++i) {
        ta[i] = (i < L) ? a[i] : 1.0;
        tb[i] = (i < L) ? b[i] : 0.0;
    }
    /* up-sweep: node at i+2d-1 becomes (right) o (left) */
    for (long d = 1; d < P; d <<= 1) {
        for (long i = 0; i < P; i += 2 * d) {
            long l = i + d - 1, r = i + 2 * d - 1;
            double na, nb;
            ssm_oracle_compose(ta[r], tb[r], ta[l], tb[l], &na, &nb);
            ta[r] = na; tb[r] = nb;
        }
    }
    /* down-sweep: root gets the identity; each node passes its prefix to its
     * left child, and (own left subtree total) o (prefix) to its right child */
    ta[P - 1] = 1.0; tb[P - 1] = 0.0;
    for (long d = P >> 1; d >= 1; d >>= 1) {
        for (long i = 0; i < P; i += 2 * d) {
            long l = i + d - 1, r = i + 2 * d - 1;
            double la = ta[l], lb = tb[l];   /* left subtree total */
            double pa = ta[r], pb = tb[r];   /* prefix arriving at this node */
            ta[l] = pa; tb[l] = pb;
            double na, nb;
            ssm_oracle_compose(la, lb, pa, pb, &na, &nb);
            ta[r] = na; tb[r] = nb;
        }
    }
    for (long i = 0; i < L; ++i)
        ssm_oracle_compose(a[i], b[i], ta[i], tb[i], &A_out[i], &B_out[i]);
    free(ta); free(tb);
    return 0;
}

/* [P1 sect. 2.2, 3.3] chunked two-pass scan.  The sequence is cut into chunks
 * of length `chunk`; each chunk is scanned locally from the identity, giving
 * its total (A_tot^(k), B_tot^(k)); the chunk start states follow
 *     h_init^(0) = h0,  h_init^(k) = A_tot^(k-1) * h_init^(k-1) + B_tot^(k-1),
 * and the fix-up gives h_t = A_loc_t * h_init^(k) + B_loc_t.
 * Writes h_t for every t (h_out[t] is the state after step t), and the state
 * at the end of every chunk into boundary[k] (k = 0 .. ceil(L/chunk)-1).  */
int ssm_oracle_scan_chunked(const double *a, const double *b, long L, long chunk,
                            double h0, double *h_out, double *boundary)
{
    if (L <= 0) return 0;
    if (chunk <= 0) return -1;
    long K = (L + chunk - 1) / chunk;
    double *Atot = (double *)malloc(sizeof(double) * (size_t)K);
    double *Btot = (double *)malloc(sizeof(double) * (size_t)K);
    double *Aloc = (double *)malloc(sizeof(double) * (size_t)L);
    double *Bloc = (double *)malloc(sizeof(double) * (size_t)L);
    if (!Atot || !Btot || !Aloc || !Bloc) {
        free(Atot); free(Btot); free(Aloc); free(Bloc); return -1;
    }
    /* pass 1: independent local scans, one per chunk */
    for (long k = 0; k < K; ++k) {
        long s = k * chunk, e = s + chunk < L ? s + chunk : L;
        ssm_oracle_scan_serial(a + s, b + s, e - s, Aloc + s, Bloc + s);
        Atot[k] = Aloc[e - 1];
        Btot[k] = Bloc[e - 1];
    }
    /* carry across chunks, then fix-up */
    double hinit = h0;
    for (long k = 0; k < K; ++k) {
        long s = k * chunk, e = s + chunk < L ? s + chunk : L;
        for (long t = s; t < e; ++t)
            h_out[t] = Aloc[t] * hinit + Bloc[t];
        if (boundary) boundary[k] = h_out[e - 1];
        hinit = Atot[k] * hinit + Btot[k];
    }
    free(Atot); free(Btot); free(Aloc); free(Bloc);
    return 0;
}

/* ------------------------------------------------------------------ */
/* Discretisation and gate                                             */
/* ------------------------------------------------------------------ */

/* softplus(v) = log(1 + e^v) ([P1 sect. 1.2]: the step is made positive by a
 * softplus).  For v > 0 the same value is written v + log(1 + e^-v) so that
 * e^v cannot overflow; both forms are the same real function. */
double ssm_oracle_softplus(double v)
{
    if (v > 0.0) return v + log1p(exp(-v));
    return log1p(exp(v));
}

/* silu(z) = z * sigmoid(z) = z / (1 + e^-z) */
double ssm_oracle_silu(double z)
{
    return z / (1.0 + exp(-z));
}

/* ------------------------------------------------------------------ */
/* Forward selective scan, the plain definition                        */
/* ------------------------------------------------------------------ */

/*
 * For every channel (b, d), with h[n] = h0[b,d,n] at the start (0 when h0 is
 * NULL; a given start state is how a sequence resumes from the boundary state
 * of the segment before it, [P3 sect. 4.3]):
 *   v      = delta[b,d,t] + dt_bias[d]                  (dt_bias optional)
 *   Delta  = softplus(v) if `softplus` else v
 *   a_n    = exp(Delta * A[d,n]),  b_n = Delta * B[b,n,t] * x[b,d,t]
 *                                                       ([P1 sect. 1.2])
 *   h[n]   = a_n * h[n] + b_n                           ([P1 sect. 1], [P3 sect. 1])
 *   y      = sum_n C[b,n,t] * h[n]  + D[d] * x[b,d,t]   (D optional)
 *   y     *= silu(z[b,d,t])                             (z optional)
 * and final_state[b,d,n] = h[n] after the last step.
 *
 * Layouts (row-major): x, delta, z: [batch, dim, L]; B, C: [batch, dstate, L];
 * A: [dim, dstate]; D, dt_bias: [dim]; h0: [batch, dim, dstate] (double).
 *
 * `chan` selects which channels (index b*dim + d) to evaluate; NULL means all
 * channels in order.  y is written as [nchan, L] and final_state as
 * [nchan, dstate] in the order of `chan`.  `nthreads` > 1 evaluates
 * independent channels on that many OpenMP threads (each channel is still
 * the same serial loop); 0 leaves the OpenMP default.
 * Returns 0, or -1 on bad arguments.
 */
int ssm_oracle_fwd_from(const float *x, const float *delta, const float *A,
                        const float *Bm, const float *Cm, const float *Dskip,
                        const float *z, const float *dt_bias, int softplus,
                        const double *h0, double *y, double *final_state,
                        long batch, long dim, long dstate, long L,
                        const long *chan, long nchan, int nthreads)
{
    if (!x || !delta || !A || !Bm || !Cm || !y) return -1;
    if (batch <= 0 || dim <= 0 || dstate <= 0 || L < 0) return -1;
    long nall = batch * dim;
    if (!chan) nchan = nall;
    if (nchan < 0) return -1;
    for (long i = 0; chan && i < nchan; ++i)
        if (chan[i] < 0 || chan[i] >= nall) return -1;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (long i = 0; i < nchan; ++i) {
        long c = chan ? chan[i] : i;
        long bb = c / dim, d = c % dim;
        double *h = (double *)calloc((size_t)dstate, sizeof(double));
        if (!h) {
#pragma omp atomic write
            err = 1;
            continue;
        }
        if (h0)
            for (long n = 0; n < dstate; ++n) h[n] = h0[(size_t)c * (size_t)dstate + (size_t)n];
        const float *xr = x + (size_t)c * (size_t)L;
        const float *dr = delta + (size_t)c * (size_t)L;
        const float *zr = z ? z + (size_t)c * (size_t)L : NULL;
        const float *Br = Bm + (size_t)bb * (size_t)dstate * (size_t)L;
        const float *Cr = Cm + (size_t)bb * (size_t)dstate * (size_t)L;
        const float *Ar = A + (size_t)d * (size_t)dstate;
        double bias = dt_bias ? (double)dt_bias[d] : 0.0;
        double Dd = Dskip ? (double)Dskip[d] : 0.0;
        double *yr = y + (size_t)i * (size_t)L;
        for (long t = 0; t < L; ++t) {
            double xt = (double)xr[t];
            double v = (double)dr[t] + bias;
            double Delta = softplus ? ssm_oracle_softplus(v) : v;
            double acc = 0.0;
            for (long n = 0; n < dstate; ++n) {
                double an = exp(Delta * (double)Ar[n]);
                double bn = Delta * (double)Br[(size_t)n * (size_t)L + (size_t)t] * xt;
                h[n] = an * h[n] + bn;
                acc += (double)Cr[(size_t)n * (size_t)L + (size_t)t] * h[n];
            }
            double yv = acc + Dd * xt;
            if (zr) yv *= ssm_oracle_silu((double)zr[t]);
            yr[t] = yv;
        }
        if (final_state)
            for (long n = 0; n < dstate; ++n)
                final_state[(size_t)i * (size_t)dstate + (size_t)n] = h[n];
        free(h);
    }
    return err ? -1 : 0;
}

/* The forward from the zero state. */
int ssm_oracle_fwd(const float *x, const float *delta, const float *A,
                   const float *Bm, const float *Cm, const float *Dskip,
                   const float *z, const float *dt_bias, int softplus,
                   double *y, double *final_state,
                   long batch, long dim, long dstate, long L,
                   const long *chan, long nchan, int nthreads)
{
    return ssm_oracle_fwd_from(x, delta, A, Bm, Cm, Dskip, z, dt_bias, softplus, NULL, y,
                               final_state, batch, dim, dstate, L, chan, nchan, nthreads);
}

/*
 * One token of the recurrence for every channel: the recurrent (decode) mode
 * in which inference advances the state one step at a time with constant
 * work and memory per token ([P3 sect. 6-7]).  With s = state[b,d,:]:
 *   Delta     = softplus(delta[b,d] + dt_bias[d])   (or without softplus)
 *   s[k]     <- exp(Delta * A[d,k]) * s[k] + Delta * B[b,k] * x[b,d]
 *   y[b,d]    = (sum_k C[b,k] * s[k] + D[d] * x[b,d]) * silu(z[b,d])
 * D, z and dt_bias are optional.  The arithmetic is that of one iteration of
 * the forward above, in the same order, so L calls reproduce a forward over L
 * steps exactly.
 * Layouts: state [batch, dim, dstate] (double, updated in place);
 * x, delta, z [batch, dim]; B, C [batch, dstate]; A [dim, dstate];
 * D, dt_bias [dim]; y [batch, dim].  Returns 0, or -1 on bad arguments.
 */
int ssm_oracle_step(double *state, const float *x, const float *delta, const float *A,
                    const float *Bv, const float *Cv, const float *Dskip, const float *z,
                    const float *dt_bias, int softplus, double *y,
                    long batch, long dim, long dstate)
{
    if (!state || !x || !delta || !A || !Bv || !Cv || !y) return -1;
    if (batch < 0 || dim < 0 || dstate <= 0) return -1;
    for (long c = 0; c < batch * dim; ++c) {
        long bb = c / dim, d = c % dim;
        double xin = (double)x[c];
        double arg = (double)delta[c] + (dt_bias ? (double)dt_bias[d] : 0.0);
        double step = softplus ? ssm_oracle_softplus(arg) : arg;
        double skip = Dskip ? (double)Dskip[d] : 0.0;
        double *s = state + (size_t)c * (size_t)dstate;
        double out = 0.0;
        for (long k = 0; k < dstate; ++k) {
            double decay = exp(step * (double)A[(size_t)d * (size_t)dstate + (size_t)k]);
            double inject = step * (double)Bv[(size_t)bb * (size_t)dstate + (size_t)k] * xin;
            s[k] = decay * s[k] + inject;
            out += (double)Cv[(size_t)bb * (size_t)dstate + (size_t)k] * s[k];
        }
        out = out + skip * xin;
        if (z) out *= ssm_oracle_silu((double)z[c]);
        y[c] = out;
    }
    return 0;
}

/*
 * Gradients of the forward above (reverse mode, written out from its
 * definition) for a scalar loss whose derivatives with respect to y and to the
 * final state are dy [batch, dim, L] and dfinal [batch, dim, dstate] (NULL:
 * zero).  This is the backward that the recomputation strategy of [P3]
 * sect. 4.2-4.3 evaluates: the forward states h_t are recomputed (here all of
 * them, serially, per channel) and the adjoint of the state runs backwards,
 *   lambda_t[n] = dq_t * C[b,n,t] + a_{t+1}[n] * lambda_{t+1}[n],
 * with q_t = sum_n C h_t + D x_t, g_t = silu(z_t), y_t = q_t g_t and
 * dq_t = dy_t g_t.  From lambda:
 *   dC[b,n,t] += dq_t h_t[n]               dB[b,n,t] += lambda_t[n] u_t
 *   du_t = sum_n lambda_t[n] B[b,n,t]      da_t[n] = lambda_t[n] h_{t-1}[n]
 *   dA[d,n] += da_t[n] a_t[n] Delta_t      dDelta_t = sum_n da_t[n] a_t[n] A[d,n] + du_t x_t
 *   dx_t = du_t Delta_t + dq_t D[d]        dD[d] += dq_t x_t
 *   dz_t = dy_t q_t silu'(z_t)             ddelta_t = dDelta_t softplus'(v_t) (or dDelta_t)
 *   ddt_bias[d] += ddelta_t                dh0[b,d,n] = a_0[n] lambda_0[n]
 * with u_t = Delta_t x_t, v_t = delta_t + dt_bias[d], softplus' = sigmoid.
 * B and C are shared by the channels of a batch and A, D, dt_bias by the
 * batches, so dB, dC, dA, dD and ddt_bias are sums over channels or batches.
 *
 * Outputs (double, overwritten; NULL skips one): dx, ddelta, dz [batch, dim, L];
 * dA [dim, dstate]; dB, dC [batch, dstate, L]; dD, ddt_bias [dim];
 * dh0 [batch, dim, dstate].  Runs serially (the sums above are shared).
 * Returns 0, or -1 on bad arguments or allocation failure.
 */
int ssm_oracle_bwd(const float *x, const float *delta, const float *A,
                   const float *Bm, const float *Cm, const float *Dskip,
                   const float *z, const float *dt_bias, int softplus,
                   const double *h0, const double *dy, const double *dfinal,
                   double *dx, double *ddelta, double *dA, double *dBm, double *dCm,
                   double *dD, double *dz, double *ddt_bias, double *dh0,
                   long batch, long dim, long dstate, long L)
{
    if (!x || !delta || !A || !Bm || !Cm || !dy) return -1;
    if (batch <= 0 || dim <= 0 || dstate <= 0 || L < 0) return -1;
    size_t nx = (size_t)batch * (size_t)dim * (size_t)L;
    size_t nb = (size_t)batch * (size_t)dstate * (size_t)L;
    if (dx) memset(dx, 0, nx * sizeof(double));
    if (ddelta) memset(ddelta, 0, nx * sizeof(double));
    if (dz) memset(dz, 0, nx * sizeof(double));
    if (dA) memset(dA, 0, (size_t)dim * (size_t)dstate * sizeof(double));
    if (dBm) memset(dBm, 0, nb * sizeof(double));
    if (dCm) memset(dCm, 0, nb * sizeof(double));
    if (dD) memset(dD, 0, (size_t)dim * sizeof(double));
    if (ddt_bias) memset(ddt_bias, 0, (size_t)dim * sizeof(double));
    size_t Lz = L > 0 ? (size_t)L : 1;
    double *hs = (double *)malloc((Lz + 1) * (size_t)dstate * sizeof(double));   /* h_{-1} .. h_{L-1} */
    double *Dl = (double *)malloc(Lz * sizeof(double));
    double *vv = (double *)malloc(Lz * sizeof(double));
    double *qq = (double *)malloc(Lz * sizeof(double));
    double *lam = (double *)malloc((size_t)dstate * sizeof(double));
    if (!hs || !Dl || !vv || !qq || !lam) {
        free(hs); free(Dl); free(vv); free(qq); free(lam);
        return -1;
    }
    for (long c = 0; c < batch * dim; ++c) {
        long bb = c / dim, d = c % dim;
        const float *xr = x + (size_t)c * (size_t)L;
        const float *dr = delta + (size_t)c * (size_t)L;
        const float *zr = z ? z + (size_t)c * (size_t)L : NULL;
        const float *Br = Bm + (size_t)bb * (size_t)dstate * (size_t)L;
        const float *Cr = Cm + (size_t)bb * (size_t)dstate * (size_t)L;
        const float *Ar = A + (size_t)d * (size_t)dstate;
        const double *dyr = dy + (size_t)c * (size_t)L;
        double bias = dt_bias ? (double)dt_bias[d] : 0.0;
        double Dd = Dskip ? (double)Dskip[d] : 0.0;
        /* forward, keeping every state: row t+1 of hs holds h_t */
        for (long n = 0; n < dstate; ++n) hs[n] = h0 ? h0[(size_t)c * (size_t)dstate + (size_t)n] : 0.0;
        for (long t = 0; t < L; ++t) {
            double xt = (double)xr[t];
            vv[t] = (double)dr[t] + bias;
            Dl[t] = softplus ? ssm_oracle_softplus(vv[t]) : vv[t];
            double p = 0.0;
            for (long n = 0; n < dstate; ++n) {
                double at = exp(Dl[t] * (double)Ar[n]);
                double prev = hs[(size_t)t * (size_t)dstate + (size_t)n];
                double cur = at * prev + Dl[t] * xt * (double)Br[(size_t)n * (size_t)L + (size_t)t];
                hs[(size_t)(t + 1) * (size_t)dstate + (size_t)n] = cur;
                p += (double)Cr[(size_t)n * (size_t)L + (size_t)t] * cur;
            }
            qq[t] = p + Dd * xt;
        }
        /* reverse */
        for (long n = 0; n < dstate; ++n) lam[n] = dfinal ? dfinal[(size_t)c * (size_t)dstate + (size_t)n] : 0.0;
        for (long t = L - 1; t >= 0; --t) {
            double xt = (double)xr[t];
            double dq = dyr[t];
            if (zr) {
                double zt = (double)zr[t];
                double sg = 1.0 / (1.0 + exp(-zt));
                if (dz) dz[(size_t)c * (size_t)L + (size_t)t] = dyr[t] * qq[t] * (sg + zt * sg * (1.0 - sg));
                dq = dyr[t] * zt * sg;
            }
            if (dD) dD[d] += dq * xt;
            double du = 0.0, dDl = 0.0;
            for (long n = 0; n < dstate; ++n) {
                size_t bi = (size_t)bb * (size_t)dstate * (size_t)L + (size_t)n * (size_t)L + (size_t)t;
                double ht = hs[(size_t)(t + 1) * (size_t)dstate + (size_t)n];
                double hp = hs[(size_t)t * (size_t)dstate + (size_t)n];
                lam[n] += dq * (double)Cr[(size_t)n * (size_t)L + (size_t)t];
                if (dCm) dCm[bi] += dq * ht;
                if (dBm) dBm[bi] += lam[n] * Dl[t] * xt;
                du += lam[n] * (double)Br[(size_t)n * (size_t)L + (size_t)t];
                double at = exp(Dl[t] * (double)Ar[n]);
                double da = lam[n] * hp;
                if (dA) dA[(size_t)d * (size_t)dstate + (size_t)n] += da * at * Dl[t];
                dDl += da * at * (double)Ar[n];
                lam[n] *= at;
            }
            dDl += du * xt;
            if (dx) dx[(size_t)c * (size_t)L + (size_t)t] = du * Dl[t] + dq * Dd;
            double dv = softplus ? dDl / (1.0 + exp(-vv[t])) : dDl;
            if (ddelta) ddelta[(size_t)c * (size_t)L + (size_t)t] = dv;
            if (ddt_bias) ddt_bias[d] += dv;
        }
        if (dh0)
            for (long n = 0; n < dstate; ++n) dh0[(size_t)c * (size_t)dstate + (size_t)n] = lam[n];
    }
    free(hs); free(Dl); free(vv); free(qq); free(lam);
    return 0;
}

/*
 * Causal depthwise convolution in front of the scan ([P3] sect. 4.1 lists it
 * among the operators the fused kernel runs before the scan): for every
 * channel (b, d), with K taps w[d, 0..K-1],
 *   v_t = bias[d] + sum_{k=0}^{K-1} w[d,k] * x[b,d,t-K+1+k]
 *   y_t = silu(v_t) if `silu` else v_t
 * where inputs before t = 0 come from state_in[b,d,0..K-2] (the K-1 inputs
 * that preceded the sequence, oldest first; zeros if state_in is NULL).
 * state_out[b,d,0..K-2] receives the last K-1 inputs of the history followed
 * by the sequence, so that a following segment continues the convolution.
 * Layouts: x [batch, dim, L] (float), w [dim, K], bias [dim] (optional),
 * state_in [batch, dim, K-1] (float, optional), y [batch, dim, L] (double),
 * state_out [batch, dim, K-1] (double, optional).  Returns 0, or -1 on bad
 * arguments.
 */
int ssm_oracle_conv1d(const float *x, const float *w, const float *bias, const float *state_in, int silu,
                      double *y, double *state_out, long batch, long dim, long L, long K)
{
    if (!x || !w || !y || batch < 0 || dim < 0 || L < 0 || K < 1 || K > 64) return -1;
    double hist[64 + 1];
    for (long c = 0; c < batch * dim; ++c) {
        long d = c % dim;
        const float *xr = x + (size_t)c * (size_t)L;
        for (long k = 0; k < K - 1; ++k)
            hist[k] = state_in ? (double)state_in[(size_t)c * (size_t)(K - 1) + (size_t)k] : 0.0;
        for (long t = 0; t < L; ++t) {
            double acc = bias ? (double)bias[d] : 0.0;
            for (long k = 0; k < K; ++k) {
                long src = t - (K - 1) + k;                      /* index into the sequence */
                double xv = src >= 0 ? (double)xr[src] : hist[K - 1 + src];
                acc += (double)w[(size_t)d * (size_t)K + (size_t)k] * xv;
            }
            y[(size_t)c * (size_t)L + (size_t)t] = silu ? ssm_oracle_silu(acc) : acc;
        }
        if (state_out)
            for (long k = 0; k < K - 1; ++k) {
                long src = L - (K - 1) + k;
                state_out[(size_t)c * (size_t)(K - 1) + (size_t)k] = src >= 0 ? (double)xr[src] : hist[K - 1 + src];
            }
    }
    return 0;
}

/* The per-step pairs (a_t, b_t) of one recurrence (b, d, n), t = 0..L-1, as
 * defined in [P1 sect. 1.2]; used to feed the scan orderings above with the
 * exact pairs the forward recurrence consumes. */
int ssm_oracle_pairs(const float *x, const float *delta, const float *A,
                     const float *Bm, const float *dt_bias, int softplus,
                     long batch, long dim, long dstate, long L,
                     long b, long d, long n, double *a_out, double *b_out)
{
    if (b < 0 || b >= batch || d < 0 || d >= dim || n < 0 || n >= dstate) return -1;
    long c = b * dim + d;
    for (long t = 0; t < L; ++t) {
        double xt = (double)x[(size_t)c * (size_t)L + (size_t)t];
        double v = (double)delta[(size_t)c * (size_t)L + (size_t)t] + (dt_bias ? (double)dt_bias[d] : 0.0);
        double Delta = softplus ? ssm_oracle_softplus(v) : v;
        a_out[t] = exp(Delta * (double)A[(size_t)d * (size_t)dstate + (size_t)n]);
        b_out[t] = Delta * (double)Bm[((size_t)b * (size_t)dstate + (size_t)n) * (size_t)L + (size_t)t] * xt;
    }
    return 0;
}

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
int ssm_oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
