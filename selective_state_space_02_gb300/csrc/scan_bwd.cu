// Backward of the forward selective scan (include/ssm_bwd.h), by chunked
// recomputation: "Mamba (part 2): parallel scan and hardware-aware
// optimisation" (scwacadex.pages.dev) sect. 4.2-4.3 -- the forward keeps no
// state sequence; the backward reads the state at the start of each chunk and
// recomputes the chunk's states from it while walking the chunks in reverse.
//
// 1. Chunk-start states: the two-pass forward's totals pass and carry scan
//    with segments of kChunk steps (chunk_start_states in scan_fused.cu) give
//    h at the start of every chunk, seeded with the start state.
// 2. bwd_kernel: a CTA owns CPC channels of one batch (LPC lanes per channel,
//    S2 states per lane) and walks their chunks from the last to the first.
//    The two serial chains are kept minimal and everything else is done by
//    all threads in parallel afterwards:
//      a. the chunk's x, delta, z, dy (per step and channel) and B, C (per
//         step and state), prefetched into registers while the previous chunk
//         was processed, go to shared memory as Delta, u = Delta x,
//         softplus'(v), dq = dy silu(z) and dy silu'(z);
//      b. (serial, per lane) the chunk's states h_t = a_t h_{t-1} + u_t B_t,
//         recomputed from its start state into shared memory;
//      c. (serial, per lane) the state's adjoint backwards over the chunk,
//         lambda <- lambda + dq C, stored, then lambda <- a lambda;
//      d. (parallel) per lane, dA += sum_t lambda_t h_{t-1} a_t Delta_t; per
//         (step, channel), the sums over the states of lambda B, of
//         lambda h_{t-1} a A and of C h, which finish dx, ddelta and dz; per
//         (step, state), dB and dC summed over the CTA's channels and added
//         to global memory (one atomic addition per element per CTA);
//    and at the end adds dA, dD and ddt_bias (shared by batches) and writes
//    the start state's gradient.
#include "../../include/ssm_bwd.h"
#include "../../include/ssm_scan.h"
#include "scan_device.cuh"
#include "scan_internal.h"

namespace ssm {
namespace {

constexpr int kChunk = 32;     // steps per recomputed chunk
constexpr int kWarps = 4;      // warps per CTA

struct BwdArgs {
    const void *x;
    const void *delta;
    const float *A;
    const void *B;
    const void *C;
    const float *D;          // nullable
    const void *z;           // nullable
    const float *dt_bias;    // nullable
    int softplus;
    const float *ws_h;       // [nchunk][batch*dim][N] chunk-start states
    const void *dy;
    const float *dfinal;     // nullable
    void *dx;
    void *ddelta;
    float *dA;
    float *dB;
    float *dC;
    float *dD;               // nullable
    void *dz;                // nullable
    float *ddt_bias;         // nullable
    float *dh0;              // nullable
    int batch;
    int dim;
    int N;
    int64_t L;
};

template <int NP>
struct Shape {
    static constexpr int LPC = NP < 32 ? NP : 32;   // lanes per channel
    static constexpr int S2 = NP / LPC;             // states per lane
    static constexpr int CPW = 32 / LPC;            // channels per warp
    static constexpr int CPC = kWarps * CPW;        // channels per CTA
    static constexpr int NT = kWarps * 32;
    static constexpr int RW = NP + 1;               // padded row of a (step, channel) state vector
    // shared memory layout, in floats
    static constexpr int per = CPC * kChunk;        // one value per (step, channel): index j * CPC + c
    static constexpr int o_dl = 0, o_u = per, o_x = 2 * per, o_dq = 3 * per, o_sg = 4 * per, o_zp = 5 * per;
    static constexpr int o_B = 6 * per;                       // [kChunk][NP]
    static constexpr int o_C = o_B + kChunk * NP;
    static constexpr int o_A = o_C + kChunk * NP;             // [CPC][NP]
    static constexpr int o_H = o_A + CPC * NP;                // [kChunk + 1][CPC][RW]: row 0 = chunk start
    static constexpr int o_G = o_H + (kChunk + 1) * CPC * RW; // [kChunk][CPC][RW]: the adjoint lambda_t
    static constexpr size_t bytes = (size_t)(o_G + kChunk * CPC * RW) * 4;
    // per-thread shares of the cooperative loops
    static constexpr int PER_T = per / NT;          // (step, channel) items per thread
    static constexpr int BC_T = kChunk * NP / NT;   // (step, state) items per thread
    static_assert(per % NT == 0 && (kChunk * NP) % NT == 0 && NT % CPC == 0, "thread split");
};

__device__ __forceinline__ float sigmoid_f(float v) { return 1.0f / (1.0f + ex2(-v * kLog2e)); }

// The raw inputs of one chunk, as each thread loads them (prefetched one
// chunk ahead into registers).
template <int NP>
struct Raw {
    float x[Shape<NP>::PER_T], v[Shape<NP>::PER_T], dy[Shape<NP>::PER_T], z[Shape<NP>::PER_T];
    float B[Shape<NP>::BC_T], C[Shape<NP>::BC_T];
};

template <typename T, int NP>
__device__ __forceinline__ void load_raw(const BwdArgs &p, int b, int d0, int k, Raw<NP> &r) {
    using Sh = Shape<NP>;
    const int64_t t0 = (int64_t)k * kChunk;
    const int jn = (p.L - t0) < kChunk ? (int)(p.L - t0) : kChunk;
#pragma unroll
    for (int i = 0; i < Sh::PER_T; ++i) {
        const int e = threadIdx.x + i * Sh::NT;
        const int c = e % Sh::CPC, j = e / Sh::CPC;
        const int dd = d0 + c;
        r.x[i] = r.v[i] = r.dy[i] = r.z[i] = 0.0f;
        if (dd < p.dim && j < jn) {
            const int64_t idx = ((int64_t)b * p.dim + dd) * p.L + t0 + j;
            r.x[i] = Io<T>::ld(p.x, idx);
            r.v[i] = Io<T>::ld(p.delta, idx) + (p.dt_bias ? __ldg(p.dt_bias + dd) : 0.0f);
            r.dy[i] = Io<T>::ld(p.dy, idx);
            if (p.z) r.z[i] = Io<T>::ld(p.z, idx);
        }
    }
#pragma unroll
    for (int i = 0; i < Sh::BC_T; ++i) {
        const int e = threadIdx.x + i * Sh::NT;
        const int n = e % NP, j = e / NP;
        r.B[i] = r.C[i] = 0.0f;
        if (n < p.N && j < jn) {
            const int64_t idx = ((int64_t)b * p.N + n) * p.L + t0 + j;
            r.B[i] = Io<T>::ld(p.B, idx);
            r.C[i] = Io<T>::ld(p.C, idx);
        }
    }
}

template <typename T, int NP>
__global__ void __launch_bounds__(kWarps * 32, 1) bwd_kernel(const BwdArgs p) {
    using Sh = Shape<NP>;
    constexpr int LPC = Sh::LPC, S2 = Sh::S2, CPW = Sh::CPW, CPC = Sh::CPC, RW = Sh::RW, NT = Sh::NT;
    extern __shared__ __align__(16) float sm[];
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int li = lane % LPC;
    const int c = warp * CPW + lane / LPC;          // the lane's channel within the CTA (lane phases)
    const int b = blockIdx.y;
    const int d0 = blockIdx.x * CPC;
    const int d = d0 + c;
    const int dim = p.dim, N = p.N;
    const bool dok = d < dim;
    const int64_t L = p.L;
    const int64_t nchan = (int64_t)p.batch * dim;
    const int64_t chn = (int64_t)b * dim + d;
    const bool has_z = p.z != nullptr;
    const int nchunk = (int)((L + kChunk - 1) / kChunk);
    const int tc = tid % CPC;                        // the thread's channel in the (step, channel) phases
    const int td = d0 + tc;
    const float tD = (td < dim && p.D) ? __ldg(p.D + td) : 0.0f;

    float A2[S2], lam[S2], dAacc[S2];
#pragma unroll
    for (int s = 0; s < S2; ++s) {
        const int n = li + LPC * s;
        const bool ok = dok && n < N;
        const float Av = ok ? __ldg(p.A + (int64_t)d * N + n) : 0.0f;
        A2[s] = Av * kLog2e;
        lam[s] = (ok && p.dfinal) ? p.dfinal[chn * N + n] : 0.0f;
        dAacc[s] = 0.0f;
    }
    for (int e = tid; e < CPC * NP; e += NT) {
        const int cc = e / NP, n = e % NP;
        sm[Sh::o_A + e] = (d0 + cc < dim && n < N) ? __ldg(p.A + (int64_t)(d0 + cc) * N + n) : 0.0f;
    }
    float sum_dD = 0.0f, sum_db = 0.0f;              // this thread's share of dD, ddt_bias (channel tc)

    Raw<NP> raw;
    if (nchunk > 0) load_raw<T, NP>(p, b, d0, nchunk - 1, raw);
    for (int k = nchunk - 1; k >= 0; --k) {
        const int64_t t0 = (int64_t)k * kChunk;
        const int jn = (L - t0) < kChunk ? (int)(L - t0) : kChunk;
        // ---- a. the chunk's inputs into shared memory ------------------------
#pragma unroll
        for (int i = 0; i < Sh::PER_T; ++i) {
            const int e = tid + i * NT;                     // = j * CPC + tc
            const float v = raw.v[i], xx = raw.x[i], g = raw.dy[i];
            const float dl = p.softplus ? softplus2(make_float2(v, v)).x : v;
            sm[Sh::o_dl + e] = dl;
            sm[Sh::o_u + e] = dl * xx;
            sm[Sh::o_x + e] = xx;
            sm[Sh::o_sg + e] = p.softplus ? sigmoid_f(v) : 1.0f;
            if (has_z) {
                const float zz = raw.z[i];
                const float s = sigmoid_f(zz);
                sm[Sh::o_dq + e] = g * zz * s;
                sm[Sh::o_zp + e] = g * (s + zz * s * (1.0f - s));
            } else {
                sm[Sh::o_dq + e] = g;
            }
        }
#pragma unroll
        for (int i = 0; i < Sh::BC_T; ++i) {
            const int e = tid + i * NT;                     // = j * NP + n
            sm[Sh::o_B + e] = raw.B[i];
            sm[Sh::o_C + e] = raw.C[i];
        }
#pragma unroll
        for (int s = 0; s < S2; ++s) {                      // the chunk's start state is row 0 of H
            const int n = li + LPC * s;
            sm[Sh::o_H + c * RW + n] = (dok && n < N) ? p.ws_h[((int64_t)k * nchan + chn) * N + n] : 0.0f;
        }
        __syncthreads();
        if (k > 0) load_raw<T, NP>(p, b, d0, k - 1, raw);   // next chunk's inputs, in flight meanwhile
        // ---- b. recompute the chunk's states (row j + 1 of H holds h_j) -----------
        {
            float h[S2];
#pragma unroll
            for (int s = 0; s < S2; ++s) h[s] = sm[Sh::o_H + c * RW + li + LPC * s];
            for (int j = 0; j < jn; ++j) {
                const float dl = sm[Sh::o_dl + j * CPC + c], u = sm[Sh::o_u + j * CPC + c];
#pragma unroll
                for (int s = 0; s < S2; ++s) {
                    const int n = li + LPC * s;
                    h[s] = fmaf(ex2(dl * A2[s]), h[s], u * sm[Sh::o_B + j * NP + n]);
                    sm[Sh::o_H + ((j + 1) * CPC + c) * RW + n] = h[s];
                }
            }
        }
        // ---- c. the adjoint, backwards over the chunk: lambda_t into G ---------
        for (int j = jn - 1; j >= 0; --j) {
            const float dq = sm[Sh::o_dq + j * CPC + c], dl = sm[Sh::o_dl + j * CPC + c];
#pragma unroll
            for (int s = 0; s < S2; ++s) {
                const int n = li + LPC * s;
                lam[s] = fmaf(dq, sm[Sh::o_C + j * NP + n], lam[s]);
                sm[Sh::o_G + (j * CPC + c) * RW + n] = lam[s];
                lam[s] *= ex2(dl * A2[s]);
            }
        }
        // ---- dA: sum over the chunk of lambda_t h_{t-1} a_t Delta_t ------------------
        for (int j = 0; j < jn; ++j) {
            const float dl = sm[Sh::o_dl + j * CPC + c];
#pragma unroll
            for (int s = 0; s < S2; ++s) {
                const int n = li + LPC * s;
                const float a = ex2(dl * A2[s]);
                dAacc[s] = fmaf(sm[Sh::o_G + (j * CPC + c) * RW + n] * sm[Sh::o_H + (j * CPC + c) * RW + n] * a, dl,
                                dAacc[s]);
            }
        }
        __syncthreads();
        // ---- d. per (step, channel): sums over the states; dx, ddelta, dz ---------
#pragma unroll
        for (int i = 0; i < Sh::PER_T; ++i) {
            const int e = tid + i * NT;
            const int j = e / CPC;
            if (td < dim && j < jn) {
                const float dl = sm[Sh::o_dl + e];
                const float *g = sm + Sh::o_G + (j * CPC + tc) * RW;
                const float *hp = sm + Sh::o_H + (j * CPC + tc) * RW;          // h_{t-1}
                const float *hc = sm + Sh::o_H + ((j + 1) * CPC + tc) * RW;    // h_t
                const float *Bj = sm + Sh::o_B + j * NP, *Cj = sm + Sh::o_C + j * NP, *Ac = sm + Sh::o_A + tc * NP;
                float du = 0.0f, ds = 0.0f, pp = 0.0f;
                for (int n = 0; n < N; ++n) {
                    const float a = ex2(dl * Ac[n] * kLog2e);
                    du = fmaf(g[n], Bj[n], du);
                    ds = fmaf(g[n] * hp[n] * a, Ac[n], ds);
                    pp = fmaf(Cj[n], hc[n], pp);
                }
                const float xx = sm[Sh::o_x + e], dq = sm[Sh::o_dq + e];
                const float dv = (ds + du * xx) * sm[Sh::o_sg + e];
                const int64_t idx = ((int64_t)b * dim + td) * L + t0 + j;
                Io<T>::st(p.dx, idx, fmaf(du, dl, dq * tD));
                Io<T>::st(p.ddelta, idx, dv);
                if (has_z) Io<T>::st(p.dz, idx, sm[Sh::o_zp + e] * fmaf(tD, xx, pp));
                sum_dD = fmaf(dq, xx, sum_dD);
                sum_db += dv;
            }
        }
        // ---- per (step, state): dB and dC summed over the CTA's channels ----------
#pragma unroll
        for (int i = 0; i < Sh::BC_T; ++i) {
            const int e = tid + i * NT;
            const int n = e % NP, j = e / NP;
            if (n < N && j < jn) {
                float db = 0.0f, dc = 0.0f;
#pragma unroll 4
                for (int cc = 0; cc < CPC; ++cc) {
                    db = fmaf(sm[Sh::o_G + (j * CPC + cc) * RW + n], sm[Sh::o_u + j * CPC + cc], db);
                    dc = fmaf(sm[Sh::o_dq + j * CPC + cc], sm[Sh::o_H + ((j + 1) * CPC + cc) * RW + n], dc);
                }
                const int64_t idx = ((int64_t)b * N + n) * L + t0 + j;
                atomicAdd(p.dB + idx, db);
                atomicAdd(p.dC + idx, dc);
            }
        }
        __syncthreads();   // shared memory is refilled by the next chunk
    }
#pragma unroll
    for (int s = 0; s < S2; ++s) {
        const int n = li + LPC * s;
        if (dok && n < N) {
            atomicAdd(p.dA + (int64_t)d * N + n, dAacc[s]);
            if (p.dh0) p.dh0[chn * N + n] = lam[s];
        }
    }
    if (td < dim) {
        if (p.dD) atomicAdd(p.dD + td, sum_dD);
        if (p.ddt_bias) atomicAdd(p.ddt_bias + td, sum_db);
    }
}

template <typename T, int NP>
cudaError_t launch_np(const BwdArgs &a, cudaStream_t st) {
    using Sh = Shape<NP>;
    auto kern = bwd_kernel<T, NP>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sh::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.dim + Sh::CPC - 1) / Sh::CPC), (unsigned)a.batch);
    kern<<<grid, kWarps * 32, Sh::bytes, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const BwdArgs &a, cudaStream_t st) {
    if (a.N <= 8) return launch_np<T, 8>(a, st);
    if (a.N <= 16) return launch_np<T, 16>(a, st);
    if (a.N <= 32) return launch_np<T, 32>(a, st);
    return launch_np<T, 64>(a, st);
}

bool aligned(const void *q, size_t n) { return (reinterpret_cast<uintptr_t>(q) % n) == 0; }

struct Span {
    uintptr_t lo, hi;
};
Span span(const void *q, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(q);
    return Span{a, a + (q ? bytes : 0)};
}
bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

}  // namespace
}  // namespace ssm

extern "C" size_t ssm_scan_bwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return (size_t)-1;
    if (batch < 0 || dim < 0 || dstate < 1 || dstate > 64 || seqlen < 0) return (size_t)-1;
    if (batch == 0 || dim == 0 || seqlen == 0) return 0;
    return ssm::chunk_states_workspace_bytes(batch, dim, dstate, seqlen, ssm::kChunk);
}

extern "C" int ssm_scan_bwd(const void *x, const void *delta, const float *A, const void *B, const void *C,
                            const float *D, const void *z, const float *dt_bias, int delta_softplus,
                            const float *initial_state, const void *dy, const float *dfinal_state, void *dx,
                            void *ddelta, float *dA, float *dB, float *dC, float *dD, void *dz, float *ddt_bias,
                            float *dinitial_state, int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                            void *workspace, size_t workspace_bytes, void *stream) {
    using namespace ssm;
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (batch < 0 || dim < 0 || dstate < 1 || dstate > 64 || seqlen < 0) return SSM_ERR_DIMS;
    if (seqlen > ((int64_t)1 << 40) || (int64_t)batch * dim > ((int64_t)1 << 31)) return SSM_ERR_DIMS;
    if (batch == 0 || dim == 0) return SSM_OK;
    if (!A || !dA) return SSM_ERR_NULL;
    if (seqlen > 0 && (!x || !delta || !B || !C || !dy || !dx || !ddelta || !dB || !dC)) return SSM_ERR_NULL;
    if ((D && !dD) || (z && !dz)) return SSM_ERR_NULL;
    const size_t es = io_dtype == SSM_BF16 ? 2 : 4;
    const void *iop[] = {x, delta, B, C, z, dy, dx, ddelta, dz};
    for (const void *q : iop)
        if (q && !aligned(q, es)) return SSM_ERR_ALIGN;
    const void *fp[] = {A, D, dt_bias, initial_state, dfinal_state, dA, dB, dC, dD, ddt_bias, dinitial_state};
    for (const void *q : fp)
        if (q && !aligned(q, 4)) return SSM_ERR_ALIGN;
    const size_t nx = (size_t)batch * dim * (size_t)seqlen * es;
    const size_t nb = (size_t)batch * dstate * (size_t)seqlen;
    const size_t ns = (size_t)batch * dim * dstate * 4;
    const Span ins[] = {span(x, nx), span(delta, nx), span(z, nx), span(B, nb * es), span(C, nb * es),
                        span(A, (size_t)dim * dstate * 4), span(D, (size_t)dim * 4), span(dt_bias, (size_t)dim * 4),
                        span(initial_state, ns), span(dy, nx), span(dfinal_state, ns)};
    const Span outs[] = {span(dx, nx), span(ddelta, nx), span(z ? dz : nullptr, nx), span(dA, (size_t)dim * dstate * 4),
                         span(dB, nb * 4), span(dC, nb * 4), span(D ? dD : nullptr, (size_t)dim * 4),
                         span(ddt_bias, (size_t)dim * 4), span(dinitial_state, ns)};
    for (const Span &o : outs) {
        for (const Span &i : ins)
            if (overlap(o, i)) return SSM_ERR_ALIAS;
        for (const Span &o2 : outs)
            if (&o != &o2 && overlap(o, o2)) return SSM_ERR_ALIAS;
    }
    const size_t need = ssm_scan_bwd_workspace_size(batch, dim, dstate, seqlen, io_dtype);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256))) return SSM_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    // the accumulated gradients start from zero
    if (cudaMemsetAsync(dA, 0, (size_t)dim * dstate * 4, st) != cudaSuccess) return SSM_ERR_LAUNCH;
    if (D && cudaMemsetAsync(dD, 0, (size_t)dim * 4, st) != cudaSuccess) return SSM_ERR_LAUNCH;
    if (ddt_bias && cudaMemsetAsync(ddt_bias, 0, (size_t)dim * 4, st) != cudaSuccess) return SSM_ERR_LAUNCH;
    if (seqlen == 0) {   // no step: the start state's gradient is the final state's
        if (dinitial_state) {
            const cudaError_t e = dfinal_state ? cudaMemcpyAsync(dinitial_state, dfinal_state, ns,
                                                                 cudaMemcpyDeviceToDevice, st)
                                               : cudaMemsetAsync(dinitial_state, 0, ns, st);
            if (e != cudaSuccess) return SSM_ERR_LAUNCH;
        }
        return SSM_OK;
    }
    if (cudaMemsetAsync(dB, 0, nb * 4, st) != cudaSuccess || cudaMemsetAsync(dC, 0, nb * 4, st) != cudaSuccess)
        return SSM_ERR_LAUNCH;
    FwdArgs f;
    f.x = x; f.delta = delta; f.A = A; f.B = B; f.C = C; f.D = nullptr; f.z = nullptr; f.dt_bias = dt_bias;
    f.softplus = delta_softplus ? 1 : 0;
    f.y = nullptr; f.final_state = nullptr; f.h0 = initial_state;
    f.batch = batch; f.dim = dim; f.dstate = dstate; f.L = seqlen;
    f.bf16 = io_dtype == SSM_BF16;
    bool v16 = ((size_t)seqlen * es) % 16 == 0;
    const void *rows[] = {x, delta, B, C};
    for (const void *q : rows)
        if (!aligned(q, 16)) v16 = false;
    f.vec16 = v16 ? 1 : 0;
    if (chunk_start_states(f, kChunk, workspace, st) != cudaSuccess) return SSM_ERR_LAUNCH;
    BwdArgs a{x, delta, A, B, C, D, z, dt_bias, delta_softplus ? 1 : 0, static_cast<const float *>(workspace),
              dy, dfinal_state, dx, ddelta, dA, dB, dC, D ? dD : nullptr, z ? dz : nullptr, ddt_bias,
              dinitial_state, batch, dim, dstate, seqlen};
    const cudaError_t e = io_dtype == SSM_BF16 ? launch_t<__nv_bfloat16>(a, st) : launch_t<float>(a, st);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}
