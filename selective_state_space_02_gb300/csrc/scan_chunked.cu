// CHUNKED variant: time-parallel forward selective scan, one warp per channel.
//
// "Mamba hardware-aware parallel associative scan" (pwwt.cn/news/6375169):
//   sect. 2.1 -- hybrid scan: serial accumulation inside a block of steps,
//     a Hillis-Steele scan across blocks, identity (1, 0) for padding;
//   sect. 3.2 -- for up to 32 parts a warp scan with shuffles;
//   sect. 3.3 -- the state at the end of one chunk starts the next.
// "Mamba (part 2)" (scwacadex.pages.dev) sect. 2.2-2.4 -- the operator and
// its tree evaluation.
//
// A warp owns one channel (b, d) and walks the sequence in chunks of
// CH = 32 K steps; lane i owns steps [t0 + i K, t0 + i K + K).  Per chunk:
//   * the lane forms Delta = softplus(delta + dt_bias) and u = Delta x for
//     its K steps;
//   * for each pair of states (packed f32x2 arithmetic) the lane forms its
//     pairs a_k = 2^(Delta_k A log2 e), b_k = u_k B_k and folds them into the
//     lane total (A_i, B_i), with A_i = 2^(A log2 e sum_k Delta_k) (one
//     exponential); a 5-round warp-shuffle Hillis-Steele scan turns the lane
//     totals into inclusive prefixes, and the prefix of the lanes before it,
//     applied to the state carried from the previous chunk, is the lane's
//     start state; the lane re-walks its K steps from there with the pairs
//     kept in registers, accumulating C.h per step; lane 31's final state is
//     the next chunk's carry;
//   * y = (C.h + D x) silu(z) is stored.
// Parallelism is over channels and over time inside a chunk, so every
// channel is a warp of work whatever the number of states, at the price of
// the scan (10 shuffles per state pair and round, amortised over K steps).
//
// Data movement.  A pre-pass (bc_chunk_prepare) lays B and C out once per
// call as float4 (B_2q, B_2q+1, C_2q, C_2q+1) per (chunk, state pair q, step
// k of a lane, lane), zero past the sequence and the states, so that one
// bulk copy brings a chunk's B and C for all states into shared memory for
// the CTA's W warps (W channels of one batch) and every read of a lane is a
// conflict-free 16-byte load.  Full chunks of x, delta and z of each warp's
// channel arrive by bulk copies too; the last chunk, when partial or when
// rows are not 16-byte aligned, is read element by element from global
// memory.  Two buffers: the copies of chunk c+2 are issued as soon as every
// warp has finished chunk c.  Every wait on a copy is bounded.
#include "scan_internal.h"
#include "scan_device.cuh"
#include "scan_tma.cuh"

namespace ssm {

size_t chunked_workspace_bytes(int batch, int dim, int dstate, int64_t L);

namespace {

// Steps per lane: 8, or 4 when a chunk's B and C for 64 states would not fit
// twice in shared memory.
int chunk_k(int N) { return N > 32 ? 4 : 8; }
int pairs_of(int N) { return (N + 1) / 2; }

struct ChunkArgs {
    const float4 *bcp;   // prepared B/C: [batch][nchunk][nq][K][32]
    int nq;              // state pairs
    int nchunk;
    unsigned int *status;
};

// B and C of one batch, [N][L] in the I/O type, re-laid out per chunk as
// float4 (B_2q, B_2q+1, C_2q, C_2q+1) at [q][k][lane] for step
// chunk * 32K + lane * K + k; zeros past the sequence and for n >= N.
// One CTA of CH threads per (chunk, batch, state pair).
template <typename T, int K>
__global__ void __launch_bounds__(32 * K) bc_chunk_prepare(const void *Bm, const void *Cm, float4 *out, int N, int nq,
                                                           int64_t L, int nchunk) {
    constexpr int CH = 32 * K;
    const int b = blockIdx.y, c = blockIdx.x, q = blockIdx.z;
    float4 *dst = out + ((int64_t)b * nchunk + c) * nq * CH + (int64_t)q * CH;
    const int64_t t0 = (int64_t)c * CH;
    {
        const int e = threadIdx.x;
        const int lane = e % 32, k = e / 32;
        const int64_t t = t0 + lane * K + k;
        float v[4] = {0.0f, 0.0f, 0.0f, 0.0f};
        if (t < L) {
#pragma unroll
            for (int h = 0; h < 2; ++h) {
                const int n = 2 * q + h;
                if (n < N) {
                    v[h] = Io<T>::ld(Bm, ((int64_t)b * N + n) * L + t);
                    v[2 + h] = Io<T>::ld(Cm, ((int64_t)b * N + n) * L + t);
                }
            }
        }
        dst[e] = make_float4(v[0], v[1], v[2], v[3]);
    }
}

// K consecutive elements from shared memory (16-byte aligned) or, past the
// end or for unaligned rows, element by element from global memory.
template <typename T, int K>
__device__ __forceinline__ void unpack_smem(const unsigned char *src, float (&v)[K]) {
    if constexpr (sizeof(T) == 4) {
        const float4 *q = reinterpret_cast<const float4 *>(src);
#pragma unroll
        for (int i = 0; i < K / 4; ++i) {
            const float4 w = q[i];
            v[4 * i] = w.x; v[4 * i + 1] = w.y; v[4 * i + 2] = w.z; v[4 * i + 3] = w.w;
        }
    } else {
        uint32_t w[K / 2];
        if constexpr (K == 8) {
            const uint4 q = *reinterpret_cast<const uint4 *>(src);
            w[0] = q.x; w[1] = q.y; w[2] = q.z; w[3] = q.w;
        } else {
            const uint2 q = *reinterpret_cast<const uint2 *>(src);
            w[0] = q.x; w[1] = q.y;
        }
#pragma unroll
        for (int i = 0; i < K / 2; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
}

template <typename T, int K>
__device__ __forceinline__ void load_direct(const void *base, int64_t row, int64_t L, int64_t t, float (&v)[K]) {
#pragma unroll
    for (int k = 0; k < K; ++k) v[k] = (t + k < L) ? Io<T>::ld(base, row * L + t + k) : 0.0f;
}

template <typename T, int K>
__device__ __forceinline__ void store_out(void *y, int64_t row, int64_t L, int64_t t, bool vec, const float (&v)[K]) {
    const int64_t idx = row * L + t;
    if (vec && t + K <= L) {
        if constexpr (sizeof(T) == 4) {
            float *p = static_cast<float *>(y) + idx;
#pragma unroll
            for (int i = 0; i < K / 4; ++i)
                *reinterpret_cast<float4 *>(p + 4 * i) = make_float4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
        } else {
            uint32_t w[K / 2];
#pragma unroll
            for (int i = 0; i < K / 2; ++i) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
                w[i] = *reinterpret_cast<const uint32_t *>(&pr);
            }
            __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(y) + idx;
            if constexpr (K == 8) *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
            else *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
        }
    } else {
#pragma unroll
        for (int k = 0; k < K; ++k)
            if (t + k < L) Io<T>::st(y, idx + k, v[k]);
    }
}

__device__ __forceinline__ float2 shfl_up2(float2 v, int off) {
    return make_float2(__shfl_up_sync(0xffffffffu, v.x, off), __shfl_up_sync(0xffffffffu, v.y, off));
}

// Shared memory of one CTA.
template <typename T, int K, int W>
struct ChLayout {
    static constexpr int CH = 32 * K;
    static constexpr size_t row_bytes = (size_t)CH * sizeof(T);            // one channel's chunk of x, delta or z
    __host__ __device__ static size_t bc_bytes(int nq) { return (size_t)nq * CH * 16; }
    __host__ __device__ static size_t io_bytes() { return (size_t)W * 3 * row_bytes; }        // x, delta, z of the W channels
    __host__ __device__ static size_t off_io(int nq) { return 2 * bc_bytes(nq); }
    __host__ __device__ static size_t off_a(int nq) { return off_io(nq) + 2 * io_bytes(); }   // A log2 e, [W][64]
    __host__ __device__ static size_t off_carry(int nq) { return off_a(nq) + (size_t)W * 64 * 4; }
    __host__ __device__ static size_t off_bar(int nq) { return off_carry(nq) + (size_t)W * 64 * 4; }
    __host__ __device__ static size_t bytes(int nq) { return off_bar(nq) + 2 * 8 + 16; }
};

template <typename T, int K, int W, bool GATE>
__global__ void __launch_bounds__(W * 32, 2) chunked_scan_kernel(const FwdArgs p, const ChunkArgs ca) {
    using Ly = ChLayout<T, K, W>;
    constexpr int CH = Ly::CH;
    constexpr unsigned FULL = 0xffffffffu;
    extern __shared__ __align__(128) unsigned char smem[];
    const int nq = ca.nq;
    // buffer s: B/C at smem + s * bc_bytes, x/delta/z at smem + off_io + s * io_bytes
    float *A2s = reinterpret_cast<float *>(smem + Ly::off_a(nq));
    float *carry_all = reinterpret_cast<float *>(smem + Ly::off_carry(nq));
    uint64_t *bar = reinterpret_cast<uint64_t *>(smem + Ly::off_bar(nq));

    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int b = blockIdx.y;
    const int d = blockIdx.x * W + w;
    const bool live = d < p.dim;                      // warps past the channels idle but join every barrier
    const int N = p.dstate;
    const int64_t L = p.L;
    const int64_t ch = (int64_t)b * p.dim + d;
    const int nchunk = ca.nchunk;
    const bool gate = GATE;
    float *A2 = A2s + w * 64;
    float *carry = carry_all + w * 64;
    for (int n = lane; n < 64; n += 32) {
        const bool ok = live && n < N;
        A2[n] = ok ? __ldg(p.A + (int64_t)d * N + n) * kLog2e : 0.0f;
        carry[n] = (ok && p.h0) ? p.h0[ch * N + n] : 0.0f;
    }
    const float bias = (live && p.dt_bias) ? __ldg(p.dt_bias + d) : 0.0f;
    const float Dd = (live && p.D) ? __ldg(p.D + d) : 0.0f;
    const bool vec16 = p.vec16 != 0;
    const bool sp = p.softplus != 0;
    const int dlast = p.dim - 1 - blockIdx.x * W < W - 1 ? p.dim - 1 - blockIdx.x * W : W - 1;   // last live warp
    const size_t bcb = Ly::bc_bytes(nq);

    // Copies of chunk c into buffer s (thread 0).  Only full chunks of
    // 16-byte aligned rows get x/delta/z by copy.
    auto issue = [&](int c, int s) {
        const int64_t t0 = (int64_t)c * CH;
        const bool io_copy = vec16 && t0 + CH <= L;
        const uint32_t tx = (uint32_t)(bcb + (io_copy ? (size_t)(dlast + 1) * (GATE ? 3 : 2) * Ly::row_bytes : 0));
        fence_proxy_async();
        mbar_arrive_expect_tx(&bar[s], tx);
        bulk_load(smem + s * bcb, ca.bcp + ((int64_t)b * nchunk + c) * nq * CH, (uint32_t)bcb, &bar[s]);
        if (io_copy) {
            for (int ww = 0; ww <= dlast; ++ww) {
                const int64_t row = (int64_t)b * p.dim + blockIdx.x * W + ww;
                unsigned char *dst = smem + Ly::off_io(nq) + s * Ly::io_bytes() + (size_t)ww * 3 * Ly::row_bytes;
                const size_t off = ((size_t)row * L + t0) * sizeof(T);
                bulk_load(dst, static_cast<const unsigned char *>(p.x) + off, (uint32_t)Ly::row_bytes, &bar[s]);
                bulk_load(dst + Ly::row_bytes, static_cast<const unsigned char *>(p.delta) + off, (uint32_t)Ly::row_bytes, &bar[s]);
                if (GATE) bulk_load(dst + 2 * Ly::row_bytes, static_cast<const unsigned char *>(p.z) + off, (uint32_t)Ly::row_bytes, &bar[s]);
            }
        }
    };

    if (threadIdx.x == 0) {
        mbar_init(&bar[0], 1);
        mbar_init(&bar[1], 1);
        fence_mbar_init();
    }
    __syncthreads();
    int issued = 0;
    if (threadIdx.x == 0) {
        for (; issued < 2 && issued < nchunk; ++issued) issue(issued, issued);
    }

    bool aborted = false;
    for (int c = 0; c < nchunk; ++c) {
        const int s = c & 1;
        const bool ok = wait_parity(&bar[s], (uint32_t)((c >> 1) & 1), ca.status);
        if (__syncthreads_or(!ok)) { aborted = true; break; }
        const int64_t t0 = (int64_t)c * CH;
        const int64_t tl = t0 + (int64_t)lane * K;   // this lane's first step
        const bool io_copy = vec16 && t0 + CH <= L;
        // this lane's K steps of x, delta, z: from the copied chunk, or from
        // global memory for a partial or unaligned chunk (zeros past the end)
        const unsigned char *src = smem + Ly::off_io(nq) + s * Ly::io_bytes() + (size_t)w * 3 * Ly::row_bytes +
                                   (size_t)lane * K * sizeof(T);
        auto load_in = [&](int which, const void *g, float (&v)[K]) {
            if (!live) {
#pragma unroll
                for (int k = 0; k < K; ++k) v[k] = 0.0f;
            } else if (io_copy) {
                unpack_smem<T, K>(src + which * Ly::row_bytes, v);
            } else {
                load_direct<T, K>(g, ch, L, tl, v);
            }
        };
        float Dl[K], ul[K];
        {
            float xv[K], dv[K];
            load_in(0, p.x, xv);
            load_in(1, p.delta, dv);
#pragma unroll
            for (int k = 0; k < K; k += 2) {
                const float2 v = __fadd2_rn(make_float2(dv[k], dv[k + 1]), make_float2(bias, bias));
                float2 Dv = sp ? softplus2(v) : v;
                Dv = make_float2((live && tl + k < L) ? Dv.x : 0.0f, (live && tl + k + 1 < L) ? Dv.y : 0.0f);
                const float2 Uv = __fmul2_rn(Dv, make_float2(xv[k], xv[k + 1]));
                Dl[k] = Dv.x; Dl[k + 1] = Dv.y;
                ul[k] = Uv.x; ul[k + 1] = Uv.y;
            }
        }
        float sd = 0.0f;
#pragma unroll
        for (int k = 0; k < K; ++k) sd += Dl[k];
        float2 yacc[K];
#pragma unroll
        for (int k = 0; k < K; ++k) yacc[k] = make_float2(0.0f, 0.0f);

        const float4 *bq = reinterpret_cast<const float4 *>(smem + s * bcb) + lane;
#pragma unroll 1
        for (int q = 0; q < nq; ++q, bq += CH) {
            const float2 a2 = make_float2(A2[2 * q], A2[2 * q + 1]);
            float2 av[K], bv[K];
            float2 Bt = make_float2(0.0f, 0.0f);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const float2 Bk = *reinterpret_cast<const float2 *>(bq + k * 32);
                const float2 arg = __fmul2_rn(make_float2(Dl[k], Dl[k]), a2);
                av[k] = make_float2(ex2(arg.x), ex2(arg.y));
                bv[k] = __fmul2_rn(make_float2(ul[k], ul[k]), Bk);
                Bt = __ffma2_rn(av[k], Bt, bv[k]);
            }
            const float2 sa = __fmul2_rn(make_float2(sd, sd), a2);
            float2 At = make_float2(ex2(sa.x), ex2(sa.y));
            // inclusive Hillis-Steele scan of the lane totals: x_i <- x_i o x_{i-off}
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float2 Ap = shfl_up2(At, off);
                const float2 Bp = shfl_up2(Bt, off);
                if (lane >= off) {
                    Bt = __ffma2_rn(At, Bp, Bt);
                    At = __fmul2_rn(At, Ap);
                }
            }
            // the lanes before this one, applied to the carried state
            float2 Ae = shfl_up2(At, 1), Be = shfl_up2(Bt, 1);
            if (lane == 0) { Ae = make_float2(1.0f, 1.0f); Be = make_float2(0.0f, 0.0f); }
            float2 h = __ffma2_rn(Ae, make_float2(carry[2 * q], carry[2 * q + 1]), Be);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                const float2 Ck = *(reinterpret_cast<const float2 *>(bq + k * 32) + 1);
                h = __ffma2_rn(av[k], h, bv[k]);
                yacc[k] = __ffma2_rn(Ck, h, yacc[k]);
            }
            const float hx = __shfl_sync(FULL, h.x, 31), hy = __shfl_sync(FULL, h.y, 31);
            __syncwarp();
            if (lane == 0) { carry[2 * q] = hx; carry[2 * q + 1] = hy; }
        }

        if (live) {
            float xv[K], zv[K], yv[K];
            load_in(0, p.x, xv);
            if (GATE) load_in(2, p.z, zv);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                float v = fmaf(Dd, xv[k], yacc[k].x + yacc[k].y);
                if (gate) v *= silu_f(zv[k]);
                yv[k] = v;
            }
            store_out<T, K>(p.y, ch, L, tl, vec16, yv);
        }
        // every warp is done with buffer s: refill it with chunk c + 2
        __syncthreads();
        if (threadIdx.x == 0 && c + 2 < nchunk) {
            issue(c + 2, s);
            issued = c + 3;
        }
    }
    if (aborted) {
        // no CTA exits with copies in flight: wait (bounded) for the ones issued
        if (threadIdx.x == 0) {
            for (int c = issued > 2 ? issued - 2 : 0; c < issued; ++c)
                wait_parity(&bar[c & 1], (uint32_t)((c >> 1) & 1), ca.status, 1ll << 28);
        }
        return;
    }
    __syncwarp();
    if (live && p.final_state)
        for (int n = lane; n < N; n += 32) p.final_state[ch * N + n] = carry[n];
}

template <typename T, int K, int W, bool GATE>
cudaError_t launch_kw(const FwdArgs &a, const ChunkArgs &ca, cudaStream_t st) {
    using Ly = ChLayout<T, K, W>;
    auto kern = chunked_scan_kernel<T, K, W, GATE>;
    const size_t bytes = Ly::bytes(ca.nq);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.dim + W - 1) / W), (unsigned)a.batch);
    kern<<<grid, W * 32, bytes, st>>>(a, ca);
    return cudaGetLastError();
}

template <typename T, int K>
cudaError_t launch_t(const FwdArgs &a, const ChunkArgs &ca, float4 *bcp, cudaStream_t st) {
    dim3 pg((unsigned)ca.nchunk, (unsigned)a.batch, (unsigned)ca.nq);
    bc_chunk_prepare<T, K><<<pg, 32 * K, 0, st>>>(a.B, a.C, bcp, a.dstate, ca.nq, a.L, ca.nchunk);
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    constexpr int W = 8;
    return a.z ? launch_kw<T, K, W, true>(a, ca, st) : launch_kw<T, K, W, false>(a, ca, st);
}

}  // namespace

size_t chunked_workspace_bytes(int batch, int dim, int dstate, int64_t L) {
    (void)dim;
    const int K = chunk_k(dstate);
    const int64_t CH = 32 * K;
    const int64_t nchunk = (L + CH - 1) / CH;
    const size_t n = (size_t)batch * nchunk * pairs_of(dstate) * CH * 16;
    return (n + 255) / 256 * 256;
}

cudaError_t launch_chunked(const FwdArgs &a, void *workspace, cudaStream_t st) {
    unsigned int *status = device_status_word();
    if (!status) return cudaErrorInvalidSymbol;
    const int K = chunk_k(a.dstate);
    const int64_t CH = 32 * K;
    ChunkArgs ca;
    ca.bcp = static_cast<const float4 *>(workspace);
    ca.nq = pairs_of(a.dstate);
    ca.nchunk = (int)((a.L + CH - 1) / CH);
    ca.status = status;
    float4 *bcp = static_cast<float4 *>(workspace);
    if (a.bf16) return K == 8 ? launch_t<__nv_bfloat16, 8>(a, ca, bcp, st) : launch_t<__nv_bfloat16, 4>(a, ca, bcp, st);
    return K == 8 ? launch_t<float, 8>(a, ca, bcp, st) : launch_t<float, 4>(a, ca, bcp, st);
}

}  // namespace ssm
