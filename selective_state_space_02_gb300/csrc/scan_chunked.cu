// CHUNKED variant: time-parallel forward selective scan inside a warp.
//
// "Mamba hardware-aware parallel associative scan" (pwwt.cn/news/6375169):
//   sect. 2.1 -- hybrid scan: serial accumulation inside a block of steps,
//     a Hillis-Steele scan across blocks, identity (1, 0) for padding;
//   sect. 3.2 -- for chunks of up to 32 parts a warp scan with shuffles and
//     no shared memory;
//   sect. 3.3 -- the state at the end of one chunk starts the next.
// "Mamba (part 2)" (scwacadex.pages.dev) sect. 2.2-2.4 -- the operator and
// its tree evaluation.
//
// One warp owns one channel (b, d).  The warp walks the sequence in chunks of
// 32*K steps; lane i owns steps [t0 + i*K, t0 + i*K + K).  Per chunk:
//   * x, delta (and z) of the lane's K steps are loaded (one 16-byte load per
//     tensor when the rows are 16-byte aligned), Delta = softplus(delta +
//     dt_bias) and u = Delta * x are formed once per element;
//   * for every state n: the lane forms its pairs a_k = exp(Delta_k A[d,n]),
//     b_k = u_k B[n,t_k] and composes them serially into the lane total
//     (A_i, B_i); a 5-round warp-shuffle Hillis-Steele scan turns the lane
//     totals into inclusive prefixes; shifting by one lane gives each lane's
//     exclusive prefix, applied to the state carried in from the previous
//     chunk to give the lane's start state; the lane then re-walks its K
//     steps from that start state, h = a_k h + b_k, accumulating
//     y_k += C[n,t_k] h.  Lane 31's final h is the carry for the next chunk;
//   * y = (y + D x) silu(z) is stored.
// Steps beyond L are the identity pair (Delta = u = 0).
#include "scan_internal.h"
#include "scan_device.cuh"

namespace ssm {
namespace {

constexpr int kWarps = 4;   // warps (channels) per CTA

template <typename T> struct Vec;
// K consecutive elements in one 16-byte vector: 4 float32 or 8 bf16.
template <> struct Vec<float> {
    static constexpr int K = 4;
    static __device__ __forceinline__ void load(const void *base, int64_t idx, float (&v)[K]) {
        const float4 q = __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(base) + idx));
        v[0] = q.x; v[1] = q.y; v[2] = q.z; v[3] = q.w;
    }
    static __device__ __forceinline__ void store(void *base, int64_t idx, const float (&v)[K]) {
        *reinterpret_cast<float4 *>(static_cast<float *>(base) + idx) = make_float4(v[0], v[1], v[2], v[3]);
    }
};
template <> struct Vec<__nv_bfloat16> {
    static constexpr int K = 8;
    static __device__ __forceinline__ void load(const void *base, int64_t idx, float (&v)[K]) {
        const uint4 q = __ldg(reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(base) + idx));
        const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            v[2 * i] = __uint_as_float(w[i] << 16);
            v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ void store(void *base, int64_t idx, const float (&v)[K]) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * i], v[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t *>(&pr);
        }
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(base) + idx) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// Load the K steps [t, t+K) of row `row` (row length L): vectorised when the
// whole vector is in range and rows are 16-byte aligned, else element-wise
// with zeros past the end.
template <typename T, int K>
__device__ __forceinline__ void load_steps(const void *base, int64_t row, int64_t L, int64_t t,
                                           bool vec16, float (&v)[K]) {
    const int64_t idx = row * L + t;
    if (vec16 && t + K <= L) {
        Vec<T>::load(base, idx, v);
    } else {
#pragma unroll
        for (int k = 0; k < K; ++k) v[k] = (t + k < L) ? Io<T>::ld(base, idx + k) : 0.0f;
    }
}

template <typename T, bool GATE>
__global__ void __launch_bounds__(kWarps * 32)
chunked_scan_kernel(FwdArgs p) {
    constexpr int K = Vec<T>::K;
    constexpr int CH = 32 * K;                       // steps per chunk
    __shared__ float carry_sm[kWarps][64];           // state at the chunk start

    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int64_t nchan = (int64_t)p.batch * p.dim;
    const int64_t ch = (int64_t)blockIdx.x * kWarps + w;
    if (ch >= nchan) return;                          // whole warp leaves; no CTA barrier below
    const int b = (int)(ch / p.dim);
    const int d = (int)(ch % p.dim);
    const int N = p.dstate;
    const int64_t L = p.L;
    const bool vec16 = p.vec16 != 0;
    float *carry = carry_sm[w];
    for (int n = lane; n < N; n += 32) carry[n] = p.h0 ? p.h0[ch * N + n] : 0.0f;
    __syncwarp();

    const float bias = p.dt_bias ? __ldg(p.dt_bias + d) : 0.0f;
    const float Dd = p.D ? __ldg(p.D + d) : 0.0f;
    const int64_t brow0 = (int64_t)b * N;

    for (int64_t t0 = 0; t0 < L; t0 += CH) {
        const int64_t tl = t0 + (int64_t)lane * K;   // first step of this lane
        float xv[K], Delta[K], u[K], y[K];
        load_steps<T, K>(p.x, ch, L, tl, vec16, xv);
        load_steps<T, K>(p.delta, ch, L, tl, vec16, Delta);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            const bool in = tl + k < L;
            Delta[k] = in ? step_delta(Delta[k], bias, p.softplus) : 0.0f;
            u[k] = Delta[k] * xv[k];
            y[k] = 0.0f;
        }

        for (int n = 0; n < N; ++n) {
            const float a2 = __ldg(p.A + (int64_t)d * N + n) * kLog2e;
            float Bv[K], Cv[K], av[K], bv[K];
            load_steps<T, K>(p.B, brow0 + n, L, tl, vec16, Bv);
            load_steps<T, K>(p.C, brow0 + n, L, tl, vec16, Cv);
            // serial composition of the lane's K pairs
            float At = 1.0f, Bt = 0.0f;
#pragma unroll
            for (int k = 0; k < K; ++k) {
                av[k] = ex2(Delta[k] * a2);
                bv[k] = u[k] * Bv[k];
                Bt = fmaf(av[k], Bt, bv[k]);
                At *= av[k];
            }
            // warp-shuffle Hillis-Steele inclusive scan over the 32 lane totals
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const float Ap = __shfl_up_sync(0xffffffffu, At, off);
                const float Bp = __shfl_up_sync(0xffffffffu, Bt, off);
                if (lane >= off) {
                    Bt = fmaf(At, Bp, Bt);
                    At = At * Ap;
                }
            }
            // exclusive prefix of this lane applied to the carried state
            float Ae = __shfl_up_sync(0xffffffffu, At, 1);
            float Be = __shfl_up_sync(0xffffffffu, Bt, 1);
            if (lane == 0) { Ae = 1.0f; Be = 0.0f; }
            const float hc = carry[n];
            float hs = fmaf(Ae, hc, Be);
#pragma unroll
            for (int k = 0; k < K; ++k) {
                hs = fmaf(av[k], hs, bv[k]);
                y[k] = fmaf(Cv[k], hs, y[k]);
            }
            const float hend = __shfl_sync(0xffffffffu, hs, 31);
            __syncwarp();
            if (lane == 0) carry[n] = hend;
            __syncwarp();
        }

        // skip, gate, store
        float zv[K];
        if (GATE) load_steps<T, K>(p.z, ch, L, tl, vec16, zv);
#pragma unroll
        for (int k = 0; k < K; ++k) {
            float v = fmaf(Dd, xv[k], y[k]);
            if (GATE) v *= silu_f(zv[k]);
            y[k] = v;
        }
        const int64_t idx = ch * L + tl;
        if (vec16 && tl + K <= L) {
            Vec<T>::store(p.y, idx, y);
        } else {
#pragma unroll
            for (int k = 0; k < K; ++k)
                if (tl + k < L) Io<T>::st(p.y, idx + k, y[k]);
        }
    }

    if (p.final_state) {
        for (int n = lane; n < N; n += 32) p.final_state[ch * N + n] = carry[n];
    }
}

template <typename T, bool GATE>
cudaError_t launch_t(const FwdArgs &a, cudaStream_t st) {
    const int64_t nchan = (int64_t)a.batch * a.dim;
    const unsigned grid = (unsigned)((nchan + kWarps - 1) / kWarps);
    chunked_scan_kernel<T, GATE><<<grid, kWarps * 32, 0, st>>>(a);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_chunked(const FwdArgs &a, cudaStream_t st) {
    const bool gate = a.z != nullptr;
    if (a.bf16) return gate ? launch_t<__nv_bfloat16, true>(a, st) : launch_t<__nv_bfloat16, false>(a, st);
    return gate ? launch_t<float, true>(a, st) : launch_t<float, false>(a, st);
}

}  // namespace ssm
