// Backward of the forward selective scan (include/ssm_bwd.h), by chunked
// recomputation: "Mamba (part 2): parallel scan and hardware-aware
// optimisation" (scwacadex.pages.dev) sect. 4.2-4.3 -- the forward keeps no
// state sequence; the backward reads the state at the start of each chunk and
// recomputes the chunk's states from it while walking the chunks in reverse.
//
// 1. Chunk-start states: h at the start of every chunk.  The training
//    forward (ssm_scan_fwd_ckpt) stores them as it runs, and
//    ssm_scan_bwd_ckpt starts from those; otherwise chunk_start_states
//    (scan_fused.cu) computes them from the start state -- by one
//    whole-sequence pass of the fused forward where the channels fill the
//    GPU, else by the two-pass forward's totals pass and carry scan with
//    segments of kChunk steps.
// 2. bwd_kernel: a CTA owns CPC channels of one batch (LPC lanes per channel,
//    S2 states per lane) and walks their chunks from the last to the first.
//    The two serial chains are kept minimal and everything else is done by
//    all threads in parallel afterwards:
//      a. the chunk's x, delta, z, dy (per step and channel) and B, C (per
//         step and state), prefetched into registers while the previous chunk
//         was processed, go to shared memory as Delta, u = Delta x,
//         softplus'(v), dq = dy silu(z) and dy silu'(z);
//      b. (serial, per lane) the chunk's states h_t = a_t h_{t-1} + u_t B_t,
//         recomputed from its start state into registers, SC steps at a time
//         (the last SC steps first; a sub-chunk's start state is advanced from
//         the chunk's start again);
//      c. (serial, per lane) the state's adjoint backwards over those steps,
//         lambda <- lambda + dq C, then lambda <- a lambda, with per step the
//         lane's terms lambda B, lambda h_{t-1} a A and C h summed over its
//         states (reduce-scattered over the channel's lanes by shuffles, so
//         that after F steps each of F lanes holds one step's sums and
//         finishes its dx, ddelta and dz), and lambda u and dq h per state
//         written to shared memory;
//      d. (parallel, every F steps) per (step, state), dB and dC summed over
//         the CTA's channels are added to global memory (one atomic addition
//         per element per CTA); dA accumulates per lane;
//    and at the end adds dA, dD and ddt_bias (shared by batches) and writes
//    the start state's gradient.
#include "../../include/ssm_bwd.h"
#include "../../include/ssm_scan.h"
#include "scan_device.cuh"
#include "scan_internal.h"

namespace ssm {
namespace {

constexpr int kChunk = kCkptSteps;   // steps per recomputed chunk (the forward's checkpoint chunks)
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
    const float *lam_in;     // nullable: [nseg][batch*dim][N] adjoint entering each segment from its right
    int seg_chunks;          // chunks per segment (a CTA walks one segment)
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
    static constexpr int LPC = NP == 16 ? 8 : NP < 32 ? NP : 32;   // lanes per channel (2 states each at N = 16)
    static constexpr int S2 = NP / LPC;             // states per lane
    static constexpr int CPW = 32 / LPC;            // channels per warp
    static constexpr int CPC = kWarps * CPW;        // channels per CTA
    static constexpr int NT = kWarps * 32;
    static constexpr int SC = 16;                   // steps whose states a lane keeps in registers
    static constexpr int F = 8;                     // steps between reductions of the adjoint's terms
    // shared memory layout, in floats
    static constexpr int IR = kChunk + 1;           // padded per-channel row of the step inputs
    static constexpr int BR = LPC + 1;              // padded row of B/C records (one per lane of a channel)
    static constexpr int CR = NP + 1;               // padded C row of the adjoint totals pass
    // dB/dC term rows: channel stride CS and step stride TR (float2) chosen so
    // that a warp's term stores (CPW channels x LPC lanes) and the reduction's
    // reads (8 steps x 4 states per warp) each take the minimum two wavefronts.
    // A 64-bit access is served a half-warp at a time: the reduction's half-warp
    // reads 8 steps x 2 states, which a step stride of 2 (mod 16 float2) spreads
    // over all 16 bank pairs; a stride of 4 put steps j and j + 4 on one pair.
    static constexpr int CS = NP == 16 ? NP + 8 : NP;
    static constexpr int TR = CPC * CS + 2;
    static_assert(TR % 16 == 2, "term row stride");
    static constexpr int o_in = 0;                           // float4 [CPC][IR]: Delta, u, dq, x
    static constexpr int o_sz = o_in + 4 * IR * CPC;         // float2 [CPC][IR]: softplus'(v), dy silu'(z)
    // B and C of a lane's states per step: interleaved records of 2 S2 floats
    // (the B, then the C) for 8 lanes a channel, where a warp reads 8 distinct
    // records; separate B and C rows for 32 lanes a channel, where the B-only
    // reads of the recomputation would otherwise find the B halves of the
    // records on half the banks (a 4-way conflict)
    static constexpr bool kSplit = LPC == 32;
    static constexpr int o_bc = o_sz + 2 * IR * CPC;         // [kChunk][BR] records, or [kChunk][BR] B then C
    static constexpr int o_tb = o_bc + 2 * S2 * kChunk * BR; // float2 [F][TR]: per-(channel, state) dB, dC terms
    static constexpr int o_bias = o_tb + 2 * F * TR;         // float [CPC]: dt_bias of the CTA's channels
    static constexpr size_t bytes = (size_t)(o_bias + CPC) * 4;
    // per-thread shares of the cooperative loops
    static constexpr int PER_T = CPC * kChunk / NT;           // (step, channel) items per thread
    static constexpr int BC_T = kChunk * LPC / NT;            // (step, lane) B/C records per thread
    static constexpr int TB_T = (F * NP + NT - 1) / NT;       // reduction over the channels: (step, state) items
    static_assert((CPC * kChunk) % NT == 0 && (kChunk * LPC) % NT == 0 && NT % CPC == 0, "thread split");
    static_assert(o_bc % 4 == 0 && o_tb % 2 == 0 && CPC % 2 == 0, "16-byte records, channel pairs");
    static_assert(kChunk % SC == 0 && SC % F == 0 && F == 8 && LPC >= F, "sub-chunks; F steps over a channel's lanes");
};

__device__ __forceinline__ float sigmoid_f(float v) { return 1.0f / (1.0f + ex2(-v * kLog2e)); }

// One round of a reduce-scatter over the lane pairs (lane, lane ^ m): of the
// two triples a lane holds it keeps the one its bit m selects (hi where set)
// and adds its partner's copy of that one.
__device__ __forceinline__ float3 rs_round(const float3 &hi, const float3 &lo, int m) {
    const bool up = (threadIdx.x & m) != 0;
    const float3 keep = up ? hi : lo, send = up ? lo : hi;
    return make_float3(keep.x + __shfl_xor_sync(0xffffffffu, send.x, m),
                       keep.y + __shfl_xor_sync(0xffffffffu, send.y, m),
                       keep.z + __shfl_xor_sync(0xffffffffu, send.z, m));
}

// A lane's S2 states (li and li + LPC) as one value: a float, or a packed pair
// whose arithmetic is one f32x2 instruction for both states.  Rec is the
// lane's shared-memory record of one step: its states' B, then their C.
template <int S2> struct Lane;
template <> struct Lane<1> {
    using V = float;
    using Rec = float2;
    static __device__ __forceinline__ V splat(float v) { return v; }
    static __device__ __forceinline__ V make(const float (&v)[1]) { return v[0]; }
    static __device__ __forceinline__ float at(V a, int) { return a; }
    static __device__ __forceinline__ float sum(V a) { return a; }
    static __device__ __forceinline__ V fma(V a, V b, V c) { return fmaf(a, b, c); }
    static __device__ __forceinline__ V mul(V a, V b) { return a * b; }
    static __device__ __forceinline__ V exp2(V a) { return ex2(a); }
    static __device__ __forceinline__ Rec rec(const float (&b)[1], const float (&c)[1]) { return make_float2(b[0], c[0]); }
    static __device__ __forceinline__ V B(Rec r) { return r.x; }
    static __device__ __forceinline__ V C(Rec r) { return r.y; }
    static __device__ __forceinline__ V load_B(const Rec *r) { return *reinterpret_cast<const float *>(r); }
};
template <> struct Lane<2> {
    using V = float2;
    using Rec = float4;
    static __device__ __forceinline__ V splat(float v) { return make_float2(v, v); }
    static __device__ __forceinline__ V make(const float (&v)[2]) { return make_float2(v[0], v[1]); }
    static __device__ __forceinline__ float at(V a, int s) { return s ? a.y : a.x; }
    static __device__ __forceinline__ float sum(V a) { return a.x + a.y; }
    static __device__ __forceinline__ V fma(V a, V b, V c) { return __ffma2_rn(a, b, c); }
    static __device__ __forceinline__ V mul(V a, V b) { return __fmul2_rn(a, b); }
    static __device__ __forceinline__ V exp2(V a) { return make_float2(ex2(a.x), ex2(a.y)); }
    static __device__ __forceinline__ Rec rec(const float (&b)[2], const float (&c)[2]) {
        return make_float4(b[0], b[1], c[0], c[1]);
    }
    static __device__ __forceinline__ V B(Rec r) { return make_float2(r.x, r.y); }
    static __device__ __forceinline__ V C(Rec r) { return make_float2(r.z, r.w); }
    static __device__ __forceinline__ V load_B(const Rec *r) { return *reinterpret_cast<const float2 *>(r); }
};

// The raw inputs of one chunk, as each thread loads them (prefetched one
// chunk ahead into registers) and unconverted: a float's bits, or a bf16 in
// the low half.  Nothing in the block that issues the loads uses a loaded
// value -- addresses outside the problem are clamped to element 0 instead of
// predicating the load, and the conversion, the zero outside the problem and
// dt_bias are applied when the chunk is processed -- so the warp never waits
// for the prefetch where it issues it.
template <int NP>
struct Raw {
    uint32_t x[Shape<NP>::PER_T], v[Shape<NP>::PER_T], dy[Shape<NP>::PER_T], z[Shape<NP>::PER_T];
    uint32_t B[Shape<NP>::BC_T * Shape<NP>::S2], C[Shape<NP>::BC_T * Shape<NP>::S2];   // [record][state of the lane]
};

template <typename T> __device__ __forceinline__ uint32_t ld_bits(const void *p, int64_t i);
template <> __device__ __forceinline__ uint32_t ld_bits<float>(const void *p, int64_t i) {
    return __float_as_uint(__ldg(static_cast<const float *>(p) + i));
}
template <> __device__ __forceinline__ uint32_t ld_bits<__nv_bfloat16>(const void *p, int64_t i) {
    return (uint32_t)__ldg(static_cast<const unsigned short *>(p) + i);
}
template <typename T> __device__ __forceinline__ float of_bits(uint32_t b) {
    return sizeof(T) == 4 ? __uint_as_float(b) : __uint_as_float(b << 16);
}

template <typename T, int NP>
__device__ __forceinline__ void load_raw(const BwdArgs &p, int b, int d0, int k, Raw<NP> &r) {
    using Sh = Shape<NP>;
    const int64_t t0 = (int64_t)k * kChunk;
    const int jn = (p.L - t0) < kChunk ? (int)(p.L - t0) : kChunk;
#pragma unroll
    for (int i = 0; i < Sh::PER_T; ++i) {
        const int e = threadIdx.x + i * Sh::NT;          // consecutive threads: consecutive steps
        const int c = e / kChunk, j = e % kChunk;
        const int dd = d0 + c;
        const int64_t idx = (dd < p.dim && j < jn) ? ((int64_t)b * p.dim + dd) * p.L + t0 + j : 0;
        r.x[i] = ld_bits<T>(p.x, idx);
        r.v[i] = ld_bits<T>(p.delta, idx);
        r.dy[i] = ld_bits<T>(p.dy, idx);
        r.z[i] = p.z ? ld_bits<T>(p.z, idx) : 0u;
    }
#pragma unroll
    for (int i = 0; i < Sh::BC_T; ++i) {
        const int e = threadIdx.x + i * Sh::NT;          // = li * kChunk + j: a warp loads 32 steps of one row
        const int li = e / kChunk, j = e % kChunk;
#pragma unroll
        for (int s = 0; s < Sh::S2; ++s) {
            const int n = li + Sh::LPC * s;
            const int64_t idx = (n < p.N && j < jn) ? ((int64_t)b * p.N + n) * p.L + t0 + j : 0;
            r.B[i * Sh::S2 + s] = ld_bits<T>(p.B, idx);
            r.C[i * Sh::S2 + s] = ld_bits<T>(p.C, idx);
        }
    }
}

// The start state of chunk k for the lane's states (zero outside the problem).
template <int NP>
__device__ __forceinline__ void load_start(const BwdArgs &p, int k, int64_t chn, int li, bool dok,
                                           float (&h)[Shape<NP>::S2]) {
    constexpr int LPC = Shape<NP>::LPC;
    const int64_t nchan = (int64_t)p.batch * p.dim;
#pragma unroll
    for (int s = 0; s < Shape<NP>::S2; ++s) {
        const int n = li + LPC * s;
        h[s] = (dok && n < p.N) ? p.ws_h[((int64_t)k * nchan + chn) * p.N + n] : 0.0f;
    }
}

// MINB CTAs per SM: 3 (at most 168 registers, no spills) or 4 (at most 128,
// a few spilled bytes); the launch picks by grid size (launch_np).
template <typename T, int NP, int MINB>
__global__ void __launch_bounds__(kWarps * 32, MINB) bwd_kernel(const BwdArgs p) {
    using Sh = Shape<NP>;
    constexpr int LPC = Sh::LPC, S2 = Sh::S2, CPW = Sh::CPW, CPC = Sh::CPC, NT = Sh::NT, F = Sh::F, SC = Sh::SC;
    extern __shared__ __align__(16) float sm[];
    constexpr int IR = Sh::IR, BR = Sh::BR, TR = Sh::TR;
    float4 *in = reinterpret_cast<float4 *>(sm + Sh::o_in);   // [CPC][IR]
    float2 *sz = reinterpret_cast<float2 *>(sm + Sh::o_sz);   // [CPC][IR]
    using Ln = Lane<S2>;
    using V = typename Ln::V;
    using Rec = typename Ln::Rec;
    Rec *bc = reinterpret_cast<Rec *>(sm + Sh::o_bc);         // [kChunk][BR] records (not kSplit)
    V *bsp = reinterpret_cast<V *>(sm + Sh::o_bc);             // kSplit: [kChunk][BR] B, then
    V *csp = bsp + kChunk * BR;                                //         [kChunk][BR] C
    float2 *tb = reinterpret_cast<float2 *>(sm + Sh::o_tb);   // [F][TR]
    float *sbias = sm + Sh::o_bias;                            // [CPC]
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int li = lane % LPC;
    const int c = warp * CPW + lane / LPC;          // the lane's channel within the CTA
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
    const float Dd = (dok && p.D) ? __ldg(p.D + d) : 0.0f;

    V Av, A2, lam, dAacc = Ln::splat(0.0f);
    {
        float av_[S2], a2_[S2], lam_[S2];
#pragma unroll
        for (int s = 0; s < S2; ++s) {
            const int n = li + LPC * s;
            const bool ok = dok && n < N;
            av_[s] = ok ? __ldg(p.A + (int64_t)d * N + n) : 0.0f;
            a2_[s] = av_[s] * kLog2e;
            lam_[s] = (ok && p.lam_in) ? p.lam_in[((int64_t)blockIdx.z * nchan + chn) * N + n] : 0.0f;
        }
        Av = Ln::make(av_);
        A2 = Ln::make(a2_);
        lam = Ln::make(lam_);
    }
    float sum_dD = 0.0f, sum_db = 0.0f;              // this lane's share of dD, ddt_bias (its channel)
    if (tid < CPC) sbias[tid] = (p.dt_bias && d0 + tid < dim) ? __ldg(p.dt_bias + d0 + tid) : 0.0f;
    __syncthreads();

    // this CTA's segment: chunks k_lo .. k_hi - 1
    const int k_lo = blockIdx.z * p.seg_chunks;
    const int k_hi = k_lo + p.seg_chunks < nchunk ? k_lo + p.seg_chunks : nchunk;
    Raw<NP> raw;
    float hnext[S2];                                    // the next chunk's start state, in flight like raw
    if (k_hi > k_lo) {
        load_raw<T, NP>(p, b, d0, k_hi - 1, raw);
        load_start<NP>(p, k_hi - 1, chn, li, dok, hnext);
    }
    for (int k = k_hi - 1; k >= k_lo; --k) {
        const int64_t t0 = (int64_t)k * kChunk;
        const int jn = (L - t0) < kChunk ? (int)(L - t0) : kChunk;
        // ---- a. the chunk's inputs (zero past the sequence and the channels) ----
#pragma unroll
        for (int i = 0; i < Sh::PER_T; ++i) {
            const int e = tid + i * NT;                     // = channel * kChunk + j
            // past the sequence or the channels every input is zero and the
            // step is the identity: Delta = 0 (softplus(0) would be ln 2)
            const bool valid = d0 + e / kChunk < dim && e % kChunk < jn;
            const float v = valid ? of_bits<T>(raw.v[i]) + sbias[e / kChunk] : 0.0f;
            const float xx = valid ? of_bits<T>(raw.x[i]) : 0.0f, g = valid ? of_bits<T>(raw.dy[i]) : 0.0f;
            const float dl = !valid ? 0.0f : p.softplus ? softplus2(make_float2(v, v)).x : v;
            float dq = g, zp = 0.0f;
            if (has_z) {
                const float zz = valid ? of_bits<T>(raw.z[i]) : 0.0f;
                const float sg = sigmoid_f(zz);
                dq = g * zz * sg;
                zp = g * (sg + zz * sg * (1.0f - sg));
            }
            in[(e / kChunk) * IR + e % kChunk] = make_float4(dl, dl * xx, dq, xx);
            sz[(e / kChunk) * IR + e % kChunk] = make_float2(p.softplus ? sigmoid_f(v) : 1.0f, zp);
        }
#pragma unroll
        for (int i = 0; i < Sh::BC_T; ++i) {
            const int e = tid + i * NT;                     // = lane-of-channel * kChunk + j
            const int l = e / kChunk, j = e % kChunk;
            float bv[S2], cv[S2];
#pragma unroll
            for (int s = 0; s < S2; ++s) {
                const bool ok = l + LPC * s < N && j < jn;
                bv[s] = ok ? of_bits<T>(raw.B[i * S2 + s]) : 0.0f;
                cv[s] = ok ? of_bits<T>(raw.C[i * S2 + s]) : 0.0f;
            }
            if constexpr (Sh::kSplit) {
                bsp[j * BR + l] = Ln::make(bv);
                csp[j * BR + l] = Ln::make(cv);
            } else {
                bc[j * BR + l] = Ln::rec(bv, cv);
            }
        }
        const V hst = Ln::make(hnext);                      // the chunk's start state
        __syncthreads();
        if (k > k_lo) {                                     // next chunk's inputs, in flight meanwhile
            load_raw<T, NP>(p, b, d0, k - 1, raw);
            load_start<NP>(p, k - 1, chn, li, dok, hnext);
        }
        // the chunk in sub-chunks of SC steps, last first: SC + 1 states per
        // state fit in registers; a sub-chunk's start state is advanced from
        // the chunk's start again
        for (int sub = kChunk / SC - 1; sub >= 0; --sub) {
            const int j0 = sub * SC;
            const Rec *bcl = bc + li;                       // the lane's records, row stride BR
            const V *bsl = bsp + li, *csl = csp + li;       // kSplit: the lane's B and C, row stride BR
            V h[SC + 1];                                    // h[j + 1] = state after step j0 + j
            V av[SC];                                       // av[j] = a of step j0 + j (for the adjoint)
            h[0] = hst;
#pragma unroll 4
            for (int j = 0; j < j0; ++j) {
                const float4 q = in[c * IR + j];
                h[0] = Ln::fma(Ln::exp2(Ln::mul(Ln::splat(q.x), A2)), h[0],
                               Ln::mul(Ln::splat(q.y), Sh::kSplit ? bsl[j * BR] : Ln::load_B(bcl + j * BR)));
            }
            // ---- b. recompute the sub-chunk's states into registers ----------
#pragma unroll
            for (int j = 0; j < SC; ++j) {
                const float4 q = in[c * IR + j0 + j];
                av[j] = Ln::exp2(Ln::mul(Ln::splat(q.x), A2));
                const V bj = Sh::kSplit ? bsl[(j0 + j) * BR] : Ln::load_B(bcl + (j0 + j) * BR);
                h[j + 1] = Ln::fma(av[j], h[j], Ln::mul(Ln::splat(q.y), bj));
            }
            // ---- c. the adjoint backwards, F steps between reductions ----------
#pragma unroll
            for (int f = SC / F - 1; f >= 0; --f) {
                // the lane's sums over its states (du, ds, pp) of the F steps,
                // reduce-scattered over the channel's lanes as they come: pairs
                // of steps over lane bit 0, pairs of pairs over bit 1, the two
                // halves over bit 2, so lane li ends with step li's sums over
                // 8 lanes
                float3 tv[F], wa[F / 2], wb[F / 4];
#pragma unroll
                for (int jj = F - 1; jj >= 0; --jj) {
                    const int jl = f * F + jj;                  // step within the sub-chunk
                    const int j = j0 + jl;
                    const float4 q = in[c * IR + j];
                    V Bv, Cv;
                    if constexpr (Sh::kSplit) {
                        Bv = bsl[j * BR];
                        Cv = csl[j * BR];
                    } else {
                        const Rec r = bcl[j * BR];
                        Bv = Ln::B(r);
                        Cv = Ln::C(r);
                    }
                    const V a = av[jl], hn = h[jl + 1];
                    lam = Ln::fma(Ln::splat(q.z), Cv, lam);
                    const V daa = Ln::mul(Ln::mul(lam, h[jl]), a);  // (dL/da_t) a_t
                    dAacc = Ln::fma(daa, Ln::splat(q.x), dAacc);
                    const V du = Ln::mul(lam, Bv), ds = Ln::mul(daa, Av), pp = Ln::mul(Cv, hn);
#pragma unroll
                    for (int s = 0; s < S2; ++s)
                        tb[jj * TR + c * Sh::CS + li + LPC * s] = make_float2(Ln::at(lam, s) * q.y, q.z * Ln::at(hn, s));
                    tv[jj] = make_float3(Ln::sum(du), Ln::sum(ds), Ln::sum(pp));
                    if (jj % 2 == 0) wa[jj / 2] = rs_round(tv[jj + 1], tv[jj], 1);
                    if (jj % 4 == 0) wb[jj / 4] = rs_round(wa[jj / 2 + 1], wa[jj / 2], 2);
                    lam = Ln::mul(lam, a);
                }
                float3 w = rs_round(wb[1], wb[0], 4);
#pragma unroll
                for (int m = F; m < LPC; m <<= 1) {         // wider channels: the 8-lane groups' sums added
                    w.x += __shfl_xor_sync(0xffffffffu, w.x, m);
                    w.y += __shfl_xor_sync(0xffffffffu, w.y, m);
                    w.z += __shfl_xor_sync(0xffffffffu, w.z, m);
                }
                // dx, ddelta, dz of the lane's step (one lane per step and channel)
                {
                    const int j = j0 + f * F + (li & (F - 1));
                    if (li < F && dok && j < jn) {
                        const float4 q = in[c * IR + j];
                        const float2 g = sz[c * IR + j];
                        const float dv = fmaf(w.x, q.w, w.y) * g.x;
                        const int64_t idx = chn * L + t0 + j;
                        Io<T>::st(p.dx, idx, fmaf(w.x, q.x, q.z * Dd));
                        Io<T>::st(p.ddelta, idx, dv);
                        if (has_z) Io<T>::st(p.dz, idx, g.y * fmaf(Dd, q.w, w.z));
                        sum_dD = fmaf(q.z, q.w, sum_dD);
                        sum_db += dv;
                    }
                }
                __syncthreads();
                // sums over the CTA's channels: dB, dC of (step, state)
#pragma unroll
                for (int i = 0; i < Sh::TB_T; ++i) {
                    const int e = tid + i * NT;          // consecutive threads: consecutive steps
                    const int jj = e % F, n = e / F;
                    const int j = j0 + f * F + jj;
                    if (e < F * NP && n < N && j < jn) {
                        // (dB, dC) pairs summed packed, two chains over the channels
                        float2 s0 = make_float2(0.0f, 0.0f), s1 = make_float2(0.0f, 0.0f);
#pragma unroll
                        for (int cc = 0; cc < CPC; cc += 2) {
                            s0 = __fadd2_rn(s0, tb[jj * TR + cc * Sh::CS + n]);
                            s1 = __fadd2_rn(s1, tb[jj * TR + (cc + 1) * Sh::CS + n]);
                        }
                        const float2 g = __fadd2_rn(s0, s1);
                        const int64_t idx = ((int64_t)b * N + n) * L + t0 + j;
                        atomicAdd(p.dB + idx, g.x);
                        atomicAdd(p.dC + idx, g.y);
                    }
                }
                __syncthreads();   // the term buffers are refilled by the next group
            }
        }
    }
#pragma unroll
    for (int s = 0; s < S2; ++s) {
        const int n = li + LPC * s;
        if (dok && n < N) {
            atomicAdd(p.dA + (int64_t)d * N + n, Ln::at(dAacc, s));
            if (p.dh0 && blockIdx.z == 0) p.dh0[chn * N + n] = Ln::at(lam, s);   // the adjoint of the start state
        }
    }
#pragma unroll
    for (int m = 1; m < LPC; m <<= 1) {
        sum_dD += __shfl_xor_sync(0xffffffffu, sum_dD, m);
        sum_db += __shfl_xor_sync(0xffffffffu, sum_db, m);
    }
    if (dok && li == 0) {
        if (p.dD) atomicAdd(p.dD + d, sum_dD);
        if (p.ddt_bias) atomicAdd(p.ddt_bias + d, sum_db);
    }
}

// The adjoint's affine map over one segment of chunks: walking the segment's
// steps backwards from lambda = 0 gives Q (lambda <- (lambda + dq C) a per
// step), and the segment's sum of Delta gives P = exp(A sum Delta), so that
// the adjoint leaving the segment on its left is P lambda_in + Q.  Same
// lanes, chunk loads and Delta as bwd_kernel; no state is needed.
template <typename T, int NP>
__global__ void __launch_bounds__(kWarps * 32, 1) adj_totals_kernel(const BwdArgs p, float *q_out, float *s_out) {
    using Sh = Shape<NP>;
    constexpr int LPC = Sh::LPC, S2 = Sh::S2, CPW = Sh::CPW, CPC = Sh::CPC, NT = Sh::NT, IR = Sh::IR, CR = Sh::CR;
    extern __shared__ __align__(16) float sm[];
    float2 *dd = reinterpret_cast<float2 *>(sm);            // [CPC][IR]: Delta, dq
    float *cs = sm + 2 * CPC * IR;                          // [kChunk][CR]: C
    float *sbias = cs + kChunk * CR;                        // [CPC]: dt_bias of the CTA's channels
    const int tid = threadIdx.x;
    const int lane = tid & 31, warp = tid >> 5;
    const int li = lane % LPC;
    const int c = warp * CPW + lane / LPC;
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
    const int k_lo = blockIdx.z * p.seg_chunks;
    const int k_hi = k_lo + p.seg_chunks < nchunk ? k_lo + p.seg_chunks : nchunk;
    float A2[S2], lam[S2];
#pragma unroll
    for (int s = 0; s < S2; ++s) {
        const int n = li + LPC * s;
        A2[s] = (dok && n < N) ? __ldg(p.A + (int64_t)d * N + n) * kLog2e : 0.0f;
        lam[s] = 0.0f;
    }
    float ssum = 0.0f;
    if (tid < CPC) sbias[tid] = (p.dt_bias && d0 + tid < dim) ? __ldg(p.dt_bias + d0 + tid) : 0.0f;
    __syncthreads();
    Raw<NP> raw;
    if (k_hi > k_lo) load_raw<T, NP>(p, b, d0, k_hi - 1, raw);
    for (int k = k_hi - 1; k >= k_lo; --k) {
        const int jn = (L - (int64_t)k * kChunk) < kChunk ? (int)(L - (int64_t)k * kChunk) : kChunk;
#pragma unroll
        for (int i = 0; i < Sh::PER_T; ++i) {
            const int e = tid + i * NT;                     // = channel * kChunk + j
            const bool valid = d0 + e / kChunk < dim && e % kChunk < jn;
            const float v = valid ? of_bits<T>(raw.v[i]) + sbias[e / kChunk] : 0.0f;
            const float g = valid ? of_bits<T>(raw.dy[i]) : 0.0f;
            const float dl = !valid ? 0.0f : p.softplus ? softplus2(make_float2(v, v)).x : v;
            float dq = g;
            if (has_z) {
                const float zz = valid ? of_bits<T>(raw.z[i]) : 0.0f;
                dq = g * zz * sigmoid_f(zz);
            }
            dd[(e / kChunk) * IR + e % kChunk] = make_float2(dl, dq);
        }
#pragma unroll
        for (int i = 0; i < Sh::BC_T; ++i) {
            const int e = tid + i * NT;                     // = lane-of-channel * kChunk + j
            const int l = e / kChunk, j = e % kChunk;
#pragma unroll
            for (int s = 0; s < S2; ++s) {
                const int n = l + LPC * s;
                cs[j * CR + n] = (n < N && j < jn) ? of_bits<T>(raw.C[i * S2 + s]) : 0.0f;
            }
        }
        __syncthreads();
        if (k > k_lo) load_raw<T, NP>(p, b, d0, k - 1, raw);
#pragma unroll 4
        for (int j = kChunk - 1; j >= 0; --j) {
            const float2 q = dd[c * IR + j];
#pragma unroll
            for (int s = 0; s < S2; ++s)
                lam[s] = fmaf(q.y, cs[j * CR + li + LPC * s], lam[s]) * ex2(q.x * A2[s]);
            ssum += q.x;
        }
        __syncthreads();
    }
#pragma unroll
    for (int s = 0; s < S2; ++s) {
        const int n = li + LPC * s;
        if (dok && n < N) q_out[((int64_t)blockIdx.z * nchan + chn) * N + n] = lam[s];
    }
    if (dok && li == 0) s_out[(int64_t)blockIdx.z * nchan + chn] = ssum;
}

// The adjoint entering every segment from its right: starting from dfinal at
// the end of the sequence, lambda <- exp(A sum Delta_s) lambda + Q_s from the
// last segment to the first (the sum of Delta is the log-domain decay of the
// segment).  ws_q holds Q_s on entry and the entering adjoint on return.
__global__ void adj_carry_kernel(const float *__restrict__ A, const float *__restrict__ dfinal, float *ws_q,
                                 const float *__restrict__ ws_s, int64_t nchan, int dim, int N, int nseg) {
    const int64_t pair = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (pair >= nchan * N) return;
    const int64_t ch = pair / N;
    const int n = (int)(pair % N);
    const float a2 = A[(ch % dim) * N + n] * kLog2e;
    float lam = dfinal ? dfinal[ch * N + n] : 0.0f;
    for (int z = nseg - 1; z >= 0; --z) {
        const int64_t i = ((int64_t)z * nchan + ch) * N + n;
        const float q = ws_q[i];
        ws_q[i] = lam;
        lam = fmaf(ex2(a2 * ws_s[(int64_t)z * nchan + ch]), lam, q);
    }
}

// Segments of chunks: one CTA walks one segment.  Problems whose channels
// fill at least half a wave (3 CTAs per SM fit at once) keep one segment --
// the totals pass costs more than the extra parallelism gives there (the
// mid-size shape's 384 CTAs: 0.87 ms unsegmented, 0.99 ms in 5 segments).
// Fewer channels get segments enough for about four waves (measured best on
// the long-sequence shape: shorter serial walks, and the totals pass walks
// shorter segments too); the adjoint entering each segment then comes from the
// segment totals and the reverse carry.
constexpr int64_t kWaveCtas = 152 * 3;
constexpr int64_t kTargetCtas = 4 * kWaveCtas;

int padded_np(int dstate) { return dstate <= 8 ? 8 : dstate <= 16 ? 16 : dstate <= 32 ? 32 : 64; }
// Channels per CTA of the reverse walk for a padded state count (the
// kernel's own Shape, so the segment plan and the launch agree).
int cta_channels(int np) {
    return np == 8 ? Shape<8>::CPC : np == 16 ? Shape<16>::CPC : np == 32 ? Shape<32>::CPC : Shape<64>::CPC;
}

struct Plan {
    int seg_chunks;   // chunks per segment
    int nseg;         // segments
};

Plan plan_for(int batch, int dim, int dstate, int64_t L) {
    const int nchunk = (int)((L + kChunk - 1) / kChunk);
    const int cpc = cta_channels(padded_np(dstate));
    const int64_t ncta = (int64_t)batch * ((dim + cpc - 1) / cpc);
    if (nchunk <= 1 || 2 * ncta >= kWaveCtas) return Plan{nchunk > 0 ? nchunk : 1, 1};
    const int64_t want = (kTargetCtas + ncta - 1) / ncta;
    const int seg = (int)((nchunk + want - 1) / want);
    return Plan{seg, (nchunk + seg - 1) / seg};
}

size_t r256(size_t n) { return (n + 255) / 256 * 256; }

// Bytes of the segment totals (adjoint Q, then the entering adjoint; sum of Delta).
size_t seg_bytes(const Plan &pl, int64_t nchan, int dstate) {
    if (pl.nseg <= 1) return 0;
    return r256((size_t)pl.nseg * nchan * dstate * 4) + r256((size_t)pl.nseg * nchan * 4);
}

template <typename T, int NP>
cudaError_t launch_np(BwdArgs a, const Plan &pl, const float *dfinal, char *seg_ws, cudaStream_t st) {
    using Sh = Shape<NP>;
    const unsigned gx = (unsigned)((a.dim + Sh::CPC - 1) / Sh::CPC);
    a.seg_chunks = pl.seg_chunks;
    a.lam_in = dfinal;
    cudaError_t e;
    if (pl.nseg > 1) {
        const int64_t nchan = (int64_t)a.batch * a.dim;
        float *q = reinterpret_cast<float *>(seg_ws);
        float *ssum = reinterpret_cast<float *>(seg_ws + r256((size_t)pl.nseg * nchan * a.N * 4));
        const size_t tb = (size_t)(2 * Sh::CPC * Sh::IR + kChunk * Sh::CR + Sh::CPC) * 4;
        adj_totals_kernel<T, NP><<<dim3(gx, (unsigned)a.batch, (unsigned)pl.nseg), kWarps * 32, tb, st>>>(a, q, ssum);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        const int64_t pairs = nchan * a.N;
        adj_carry_kernel<<<(unsigned)((pairs + 255) / 256), 256, 0, st>>>(a.A, dfinal, q, ssum, nchan, a.dim, a.N,
                                                                          pl.nseg);
        if ((e = cudaGetLastError()) != cudaSuccess) return e;
        a.lam_in = q;
    }
    // The walk is latency-bound: a grid that fits one wave of 3 CTAs per SM
    // runs them without spills (mid, 384 CTAs, 2.5 per SM either way: 0.523
    // against 0.539 ms with 4); larger grids take 4 CTAs per SM, whose extra
    // warps outweigh the spilled bytes and whose waves are fewer (large
    // 2.42 -> 2.19 ms, wide 12.41 -> 12.19 ms).
    const int64_t ctas = (int64_t)gx * a.batch * pl.nseg;
    auto kern = ctas > kWaveCtas ? bwd_kernel<T, NP, 4> : bwd_kernel<T, NP, 3>;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Sh::bytes);
    if (e != cudaSuccess) return e;
    kern<<<dim3(gx, (unsigned)a.batch, (unsigned)pl.nseg), kWarps * 32, Sh::bytes, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const BwdArgs &a, const Plan &pl, const float *dfinal, char *seg_ws, cudaStream_t st) {
    if (a.N <= 8) return launch_np<T, 8>(a, pl, dfinal, seg_ws, st);
    if (a.N <= 16) return launch_np<T, 16>(a, pl, dfinal, seg_ws, st);
    if (a.N <= 32) return launch_np<T, 32>(a, pl, dfinal, seg_ws, st);
    return launch_np<T, 64>(a, pl, dfinal, seg_ws, st);
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

bool valid_bwd_sizes(int batch, int dim, int dstate, int64_t seqlen) {
    return batch >= 0 && dim >= 0 && dstate >= 1 && dstate <= 64 && seqlen >= 0;
}

// Bytes of the checkpoints: the state at the start of every kChunk-step chunk.
size_t ckpt_bytes(int batch, int dim, int dstate, int64_t seqlen) {
    return (size_t)((seqlen + kChunk - 1) / kChunk) * (size_t)batch * dim * dstate * sizeof(float);
}

int bwd_impl(const void *x, const void *delta, const float *A, const void *B, const void *C, const float *D,
             const void *z, const float *dt_bias, int delta_softplus, const float *initial_state,
             const float *ckpt, const void *dy, const float *dfinal_state, void *dx, void *ddelta, float *dA,
             float *dB, float *dC, float *dD, void *dz, float *ddt_bias, float *dinitial_state, int batch, int dim,
             int dstate, int64_t seqlen, int io_dtype, void *workspace, size_t workspace_bytes, void *stream);

}  // namespace
}  // namespace ssm

extern "C" size_t ssm_scan_bwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return (size_t)-1;
    if (!ssm::valid_bwd_sizes(batch, dim, dstate, seqlen)) return (size_t)-1;
    if (batch == 0 || dim == 0 || seqlen == 0) return 0;
    const ssm::Plan pl = ssm::plan_for(batch, dim, dstate, seqlen);
    return ssm::r256(ssm::chunk_states_workspace_bytes(batch, dim, dstate, seqlen, ssm::kChunk)) +
           ssm::seg_bytes(pl, (int64_t)batch * dim, dstate);
}

extern "C" size_t ssm_scan_bwd_ckpt_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return (size_t)-1;
    if (!ssm::valid_bwd_sizes(batch, dim, dstate, seqlen)) return (size_t)-1;
    if (batch == 0 || dim == 0 || seqlen == 0) return 0;
    return ssm::seg_bytes(ssm::plan_for(batch, dim, dstate, seqlen), (int64_t)batch * dim, dstate);
}

extern "C" size_t ssm_scan_ckpt_size(int batch, int dim, int dstate, int64_t seqlen) {
    if (!ssm::valid_bwd_sizes(batch, dim, dstate, seqlen)) return (size_t)-1;
    return ssm::ckpt_bytes(batch, dim, dstate, seqlen);
}

extern "C" int ssm_scan_bwd_kernel_count(int batch, int dim, int dstate, int64_t seqlen) {
    if (!ssm::valid_bwd_sizes(batch, dim, dstate, seqlen)) return -1;
    if (batch == 0 || dim == 0 || seqlen == 0) return 0;
    const ssm::Plan pl = ssm::plan_for(batch, dim, dstate, seqlen);
    return ssm::chunk_start_states_kernels(batch, dim, dstate, seqlen, ssm::kChunk) + (pl.nseg > 1 ? 3 : 1);
}

extern "C" int ssm_scan_bwd_ckpt_kernel_count(int batch, int dim, int dstate, int64_t seqlen) {
    if (!ssm::valid_bwd_sizes(batch, dim, dstate, seqlen)) return -1;
    if (batch == 0 || dim == 0 || seqlen == 0) return 0;
    return ssm::plan_for(batch, dim, dstate, seqlen).nseg > 1 ? 3 : 1;
}

extern "C" int ssm_scan_bwd(const void *x, const void *delta, const float *A, const void *B, const void *C,
                            const float *D, const void *z, const float *dt_bias, int delta_softplus,
                            const float *initial_state, const void *dy, const float *dfinal_state, void *dx,
                            void *ddelta, float *dA, float *dB, float *dC, float *dD, void *dz, float *ddt_bias,
                            float *dinitial_state, int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                            void *workspace, size_t workspace_bytes, void *stream) {
    return ssm::bwd_impl(x, delta, A, B, C, D, z, dt_bias, delta_softplus, initial_state, nullptr, dy,
                         dfinal_state, dx, ddelta, dA, dB, dC, dD, dz, ddt_bias, dinitial_state, batch, dim,
                         dstate, seqlen, io_dtype, workspace, workspace_bytes, stream);
}

extern "C" int ssm_scan_bwd_ckpt(const void *x, const void *delta, const float *A, const void *B, const void *C,
                                 const float *D, const void *z, const float *dt_bias, int delta_softplus,
                                 const float *ckpt, const void *dy, const float *dfinal_state, void *dx,
                                 void *ddelta, float *dA, float *dB, float *dC, float *dD, void *dz,
                                 float *ddt_bias, float *dinitial_state, int batch, int dim, int dstate,
                                 int64_t seqlen, int io_dtype, void *workspace, size_t workspace_bytes,
                                 void *stream) {
    if (!ckpt && seqlen > 0) return SSM_ERR_NULL;
    return ssm::bwd_impl(x, delta, A, B, C, D, z, dt_bias, delta_softplus, nullptr, ckpt, dy, dfinal_state, dx,
                         ddelta, dA, dB, dC, dD, dz, ddt_bias, dinitial_state, batch, dim, dstate, seqlen,
                         io_dtype, workspace, workspace_bytes, stream);
}

namespace ssm {
namespace {

// The backward: chunk-start states from `ckpt` when given (the checkpoints of
// the forward), else computed here from the start state into the workspace.
int bwd_impl(const void *x, const void *delta, const float *A, const void *B, const void *C, const float *D,
                  const void *z, const float *dt_bias, int delta_softplus, const float *initial_state,
                  const float *ckpt, const void *dy, const float *dfinal_state, void *dx, void *ddelta, float *dA,
                  float *dB, float *dC, float *dD, void *dz, float *ddt_bias, float *dinitial_state, int batch,
                  int dim, int dstate, int64_t seqlen, int io_dtype, void *workspace, size_t workspace_bytes,
                  void *stream) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (!valid_bwd_sizes(batch, dim, dstate, seqlen)) return SSM_ERR_DIMS;
    if (seqlen > ((int64_t)1 << 40) || (int64_t)batch * dim > ((int64_t)1 << 31)) return SSM_ERR_DIMS;
    if (batch == 0 || dim == 0) return SSM_OK;
    if (!A || !dA) return SSM_ERR_NULL;
    if (seqlen > 0 && (!x || !delta || !B || !C || !dy || !dx || !ddelta || !dB || !dC)) return SSM_ERR_NULL;
    if ((D && !dD) || (z && !dz)) return SSM_ERR_NULL;
    const size_t es = io_dtype == SSM_BF16 ? 2 : 4;
    const void *iop[] = {x, delta, B, C, z, dy, dx, ddelta, dz};
    for (const void *q : iop)
        if (q && !aligned(q, es)) return SSM_ERR_ALIGN;
    const void *fp[] = {A, D, dt_bias, initial_state, ckpt, dfinal_state, dA, dB, dC, dD, ddt_bias, dinitial_state};
    for (const void *q : fp)
        if (q && !aligned(q, 4)) return SSM_ERR_ALIGN;
    const size_t nx = (size_t)batch * dim * (size_t)seqlen * es;
    const size_t nb = (size_t)batch * dstate * (size_t)seqlen;
    const size_t ns = (size_t)batch * dim * dstate * 4;
    const Span ins[] = {span(x, nx), span(delta, nx), span(z, nx), span(B, nb * es), span(C, nb * es),
                        span(A, (size_t)dim * dstate * 4), span(D, (size_t)dim * 4), span(dt_bias, (size_t)dim * 4),
                        span(initial_state, ns), span(dy, nx), span(dfinal_state, ns),
                        span(ckpt, ckpt_bytes(batch, dim, dstate, seqlen))};
    const Span outs[] = {span(dx, nx), span(ddelta, nx), span(z ? dz : nullptr, nx), span(dA, (size_t)dim * dstate * 4),
                         span(dB, nb * 4), span(dC, nb * 4), span(D ? dD : nullptr, (size_t)dim * 4),
                         span(ddt_bias, (size_t)dim * 4), span(dinitial_state, ns)};
    for (const Span &o : outs) {
        for (const Span &i : ins)
            if (overlap(o, i)) return SSM_ERR_ALIAS;
        for (const Span &o2 : outs)
            if (&o != &o2 && overlap(o, o2)) return SSM_ERR_ALIAS;
    }
    const size_t need = ckpt ? ssm_scan_bwd_ckpt_workspace_size(batch, dim, dstate, seqlen, io_dtype)
                             : ssm_scan_bwd_workspace_size(batch, dim, dstate, seqlen, io_dtype);
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
    const Plan pl = plan_for(batch, dim, dstate, seqlen);
    char *seg_ws = static_cast<char *>(workspace);
    const float *states = ckpt;
    if (!ckpt) {
        if (chunk_start_states(f, kChunk, workspace, st) != cudaSuccess) return SSM_ERR_LAUNCH;
        states = static_cast<const float *>(workspace);
        seg_ws += r256(chunk_states_workspace_bytes(batch, dim, dstate, seqlen, kChunk));
    }
    BwdArgs a{x, delta, A, B, C, D, z, dt_bias, delta_softplus ? 1 : 0, states,
              dy, nullptr, 1, dx, ddelta, dA, dB, dC, D ? dD : nullptr, z ? dz : nullptr, ddt_bias,
              dinitial_state, batch, dim, dstate, seqlen};
    const cudaError_t e = io_dtype == SSM_BF16 ? launch_t<__nv_bfloat16>(a, pl, dfinal_state, seg_ws, st)
                                               : launch_t<float>(a, pl, dfinal_state, seg_ws, st);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

}  // namespace
}  // namespace ssm
