// Causal depthwise convolution (+ SiLU) in front of the scan: "Mamba (part 2):
// parallel scan and hardware-aware optimisation" (scwacadex.pages.dev)
// sect. 4.1.  Declared in include/ssm_conv.h.
//
// The operation reads x once and writes y once, so it is bound by HBM
// bandwidth.  A thread produces U x G consecutive outputs of one channel: U
// vector loads bring its inputs (16 bytes of bf16, 32 of float32, each) and
// are all issued before the first is used; one more brings the neighbouring
// run's last group, whose last K-1 inputs precede them (an L1/L2 hit: its
// owner loads the same bytes), or the start history for the first run; U
// vector stores write the outputs.  The loaded vectors stay packed until
// their turn, so that bf16 runs hold twice the vectors (U = 4: 64 bytes in
// flight per thread, like float32's U = 2) in about as many registers.  The
// tap count K is a template parameter so that the input window and the taps
// stay in registers.
#include "../../include/ssm_conv.h"
#include "../../include/ssm_scan.h"
#include "scan_device.cuh"

namespace ssm {
namespace {

constexpr int kThreads = 256;
constexpr int G = 8;   // outputs per vector
// vectors per thread: 64 bytes of input in flight for either type
template <typename T> constexpr int runs_of() { return sizeof(T) == 2 ? 4 : 2; }

struct ConvArgs {
    const void *x;
    const float *w;
    const float *bias;   // nullable
    const void *sin;     // nullable: [batch, dim, K-1]
    void *y;
    void *sout;          // nullable: [batch, dim, K-1]
    int silu;
    int dim;
    int64_t nchan;
    int64_t L;
    int64_t ngroups;     // groups of G steps per channel
};

// 8 consecutive I/O elements (the caller guarantees 16-byte alignment).
template <typename T> struct Vec8;
template <> struct Vec8<float> {
    static __device__ __forceinline__ void ld(const void *p, int64_t i, float *v) {
        const float4 a = *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
        const float4 b = *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i + 4);
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
    static __device__ __forceinline__ void st(void *p, int64_t i, const float *v) {
        *reinterpret_cast<float4 *>(static_cast<float *>(p) + i) = make_float4(v[0], v[1], v[2], v[3]);
        *reinterpret_cast<float4 *>(static_cast<float *>(p) + i + 4) = make_float4(v[4], v[5], v[6], v[7]);
    }
};
template <> struct Vec8<__nv_bfloat16> {
    static __device__ __forceinline__ void ld(const void *p, int64_t i, float *v) {
        const uint4 w = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p) + i);
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(ws[k] << 16);
            v[2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
        }
    }
    static __device__ __forceinline__ void st(void *p, int64_t i, const float *v) {
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const __nv_bfloat162 pr = __floats2bfloat162_rn(v[2 * k], v[2 * k + 1]);
            w[k] = *reinterpret_cast<const uint32_t *>(&pr);
        }
        *reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(p) + i) = make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// 8 consecutive I/O elements as loaded (16-byte aligned), expanded to float32
// only when they are used.
template <typename T> struct Raw8;
template <> struct Raw8<float> {
    float4 a, b;
    __device__ __forceinline__ void ld(const void *p, int64_t i) {
        a = *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i);
        b = *reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i + 4);
    }
    __device__ __forceinline__ void get(float *v) const {
        v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w; v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
    }
};
template <> struct Raw8<__nv_bfloat16> {
    uint4 w;
    __device__ __forceinline__ void ld(const void *p, int64_t i) {
        w = *reinterpret_cast<const uint4 *>(static_cast<const __nv_bfloat16 *>(p) + i);
    }
    __device__ __forceinline__ void get(float *v) const {
        const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            v[2 * k] = __uint_as_float(ws[k] << 16);
            v[2 * k + 1] = __uint_as_float(ws[k] & 0xffff0000u);
        }
    }
};

// SiLU of an output stored in I/O type T: the accurate form for float32; for
// bf16 outputs the one-instruction form z/2 (1 + tanh(z/2)), whose ~2^-11
// relative error is far below bf16 rounding (one special-function operation
// instead of an exponential and a reciprocal).
template <typename T>
__device__ __forceinline__ float silu_out(float z) {
    if constexpr (sizeof(T) == 4) {
        return silu_f(z);
    } else {
        const float hz = 0.5f * z;
        float t;
        asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hz));
        return fmaf(hz, t, hz);
    }
}

// Input t of channel ch's stream: the sequence for t >= 0, the start history
// for -(K-1) <= t < 0, zero before that (or without a history).
template <typename T, int K>
__device__ __forceinline__ float stream_at(const ConvArgs &p, int64_t ch, int64_t t) {
    if (t >= 0) return Io<T>::ld(p.x, ch * p.L + t);
    if (K > 1 && t >= -(K - 1) && p.sin) return Io<T>::ld(p.sin, ch * (K - 1) + (K - 1) + t);
    return 0.0f;
}

// Block: threadIdx.x over runs of U groups of G steps, threadIdx.y over
// channels (blockDim.x is the run count rounded up to a warp, at most
// kThreads), grid y over blocks of channels with a stride loop, so no thread
// divides an index.  A thread issues its U vector loads before it needs them.
// The K-1 history, G inputs and G outputs of one vector of steps.
template <typename T, int K>
__device__ __forceinline__ void conv_vector(const float (&win)[K - 1 + G], const float (&wk)[K], float bias,
                                            int silu, float (&out)[G]) {
#pragma unroll
    for (int j = 0; j < G; ++j) {
        float acc = bias;
#pragma unroll
        for (int k = 0; k < K; ++k) acc = fmaf(wk[k], win[j + k], acc);
        out[j] = silu ? silu_out<T>(acc) : acc;
    }
}

// bf16 threads take two channels and issue the next channel's loads before
// they compute the current one (each thread computes twice the outputs of a
// float32 thread between its loads); float32 threads take one.
template <typename T> constexpr int chans_per_thread() { return sizeof(T) == 2 ? 2 : 1; }
// CTAs per SM the register budget is set for: 4 for the bf16 loop (the
// current and the next channel's vectors in flight), 5 for float32.
template <typename T> constexpr int conv_min_blocks() { return sizeof(T) == 2 ? 4 : 5; }

// One run of U vectors of channel ch whose loads are `raw`: the history
// before it, then window, outputs and store one vector at a time.
template <typename T, int K>
__device__ __forceinline__ void conv_whole_run(const ConvArgs &p, int64_t ch, int d, int64_t g0,
                                               const Raw8<T> (&raw)[runs_of<T>()]) {
    constexpr int U = runs_of<T>();
    constexpr int KH = K > 1 ? K - 1 : 1;
    const int64_t L = p.L, t0 = g0 * G;
    float hist[KH];                                      // the K-1 inputs before the vector in turn
    if (K > 1) {
        if (g0 > 0) {
            Raw8<T> pv;
            pv.ld(p.x, ch * L + t0 - G);                 // the neighbouring run's last group: an L1/L2 hit
            float prev[G];
            pv.get(prev);
#pragma unroll
            for (int k = 0; k < K - 1; ++k) hist[k] = prev[G - (K - 1) + k];
        } else {
#pragma unroll
            for (int k = 0; k < K - 1; ++k) hist[k] = stream_at<T, K>(p, ch, t0 - (K - 1) + k);
        }
    }
    float wk[K];
#pragma unroll
    for (int k = 0; k < K; ++k) wk[k] = __ldg(p.w + (int64_t)d * K + k);
    const float bias = p.bias ? __ldg(p.bias + d) : 0.0f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
        float win[K - 1 + G], out[G];
#pragma unroll
        for (int k = 0; k < K - 1; ++k) win[k] = hist[k];
        raw[u].get(win + K - 1);
        conv_vector<T, K>(win, wk, bias, p.silu, out);
        Vec8<T>::st(p.y, ch * L + t0 + u * G, out);
#pragma unroll
        for (int k = 0; k < K - 1; ++k) hist[k] = win[G + k];
    }
}

// One run of channel ch vector by vector: the row's last run, or rows not
// 16-byte aligned.
template <typename T, int K, bool VEC>
__device__ __forceinline__ void conv_general_run(const ConvArgs &p, int64_t ch, int d, int64_t g0) {
    constexpr int U = runs_of<T>();
    constexpr int KH = K > 1 ? K - 1 : 1;
    const int64_t L = p.L, t0 = g0 * G;
    float hist[KH];
#pragma unroll
    for (int k = 0; k < K - 1; ++k) hist[k] = stream_at<T, K>(p, ch, t0 - (K - 1) + k);
    float wk[K];
#pragma unroll
    for (int k = 0; k < K; ++k) wk[k] = __ldg(p.w + (int64_t)d * K + k);
    const float bias = p.bias ? __ldg(p.bias + d) : 0.0f;
#pragma unroll 1
    for (int u = 0; u < U; ++u) {
        const int64_t t = t0 + u * G;
        if (t >= L) break;
        float win[K - 1 + G], out[G];
#pragma unroll
        for (int k = 0; k < K - 1; ++k) win[k] = hist[k];
        if (VEC && t + G <= L) {
            Raw8<T> one;
            one.ld(p.x, ch * L + t);
            one.get(win + K - 1);
        } else {
#pragma unroll
            for (int j = 0; j < G; ++j) win[K - 1 + j] = t + j < L ? Io<T>::ld(p.x, ch * L + t + j) : 0.0f;
        }
        conv_vector<T, K>(win, wk, bias, p.silu, out);
        if (VEC && t + G <= L) {
            Vec8<T>::st(p.y, ch * L + t, out);
        } else {
#pragma unroll
            for (int j = 0; j < G; ++j)
                if (t + j < L) Io<T>::st(p.y, ch * L + t + j, out[j]);
        }
#pragma unroll
        for (int k = 0; k < K - 1; ++k) hist[k] = win[G + k];
    }
}

template <typename T, int K, bool VEC>
__global__ void __launch_bounds__(kThreads, conv_min_blocks<T>()) conv_kernel(const ConvArgs p) {
    constexpr int U = runs_of<T>();
    const int64_t r = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;   // run of U groups
    const int64_t g0 = r * U;
    if (g0 >= p.ngroups) return;                         // no block-wide synchronisation below
    const int64_t L = p.L;
    const int64_t t0 = g0 * G;
    const bool whole = VEC && t0 + U * G <= L;           // the whole run inside the row
    const int64_t stride = (int64_t)gridDim.y * blockDim.y;
    int64_t ch = (int64_t)blockIdx.y * blockDim.y + threadIdx.y;
    if constexpr (chans_per_thread<T>() > 1) {
        // the next channel's vectors are in flight while the current one is computed
        Raw8<T> raw[U];
        if (whole && ch < p.nchan) {
#pragma unroll
            for (int u = 0; u < U; ++u) raw[u].ld(p.x, ch * L + t0 + u * G);
        }
        for (; ch < p.nchan; ch += stride) {
            const int d = (int)(ch % p.dim);
            if (whole) {
                Raw8<T> cur[U];
#pragma unroll
                for (int u = 0; u < U; ++u) cur[u] = raw[u];
                if (ch + stride < p.nchan) {
#pragma unroll
                    for (int u = 0; u < U; ++u) raw[u].ld(p.x, (ch + stride) * L + t0 + u * G);
                }
                conv_whole_run<T, K>(p, ch, d, g0, cur);
            } else {
                conv_general_run<T, K, VEC>(p, ch, d, g0);
            }
            if (K > 1 && p.sout && g0 + U >= p.ngroups) {   // the last run: the next segment's history
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
                    Io<T>::st(p.sout, ch * (K - 1) + k, stream_at<T, K>(p, ch, L - (K - 1) + k));
            }
        }
    } else {
        for (; ch < p.nchan; ch += stride) {
            const int d = (int)(ch % p.dim);
            if (whole) {
                Raw8<T> raw[U];                          // the run's U loads first
#pragma unroll
                for (int u = 0; u < U; ++u) raw[u].ld(p.x, ch * L + t0 + u * G);
                conv_whole_run<T, K>(p, ch, d, g0, raw);
            } else {
                conv_general_run<T, K, VEC>(p, ch, d, g0);
            }
            if (K > 1 && p.sout && g0 + U >= p.ngroups) {   // the last run: the next segment's history
#pragma unroll
                for (int k = 0; k < K - 1; ++k)
                    Io<T>::st(p.sout, ch * (K - 1) + k, stream_at<T, K>(p, ch, L - (K - 1) + k));
            }
        }
    }
}

template <typename T, int K>
cudaError_t launch_k(const ConvArgs &a, bool vec, cudaStream_t st) {
    constexpr int U = runs_of<T>();
    const int64_t runs = (a.ngroups + U - 1) / U;
    const unsigned bx = (unsigned)(runs >= kThreads ? kThreads : (runs + 31) / 32 * 32);
    const unsigned by = kThreads / bx;
    const unsigned gx = (unsigned)((runs + bx - 1) / bx);
    const int64_t per = (int64_t)by * chans_per_thread<T>();
    const int64_t cb = (a.nchan + per - 1) / per;
    const unsigned gy = (unsigned)(cb < 65535 ? cb : 65535);
    dim3 grid(gx, gy), block(bx, by);
    if (vec) conv_kernel<T, K, true><<<grid, block, 0, st>>>(a);
    else conv_kernel<T, K, false><<<grid, block, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const ConvArgs &a, int K, bool vec, cudaStream_t st) {
    switch (K) {
        case 1: return launch_k<T, 1>(a, vec, st);
        case 2: return launch_k<T, 2>(a, vec, st);
        case 3: return launch_k<T, 3>(a, vec, st);
        case 4: return launch_k<T, 4>(a, vec, st);
        case 5: return launch_k<T, 5>(a, vec, st);
        case 6: return launch_k<T, 6>(a, vec, st);
        case 7: return launch_k<T, 7>(a, vec, st);
        default: return launch_k<T, 8>(a, vec, st);
    }
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

extern "C" int ssm_conv1d_fwd(const void *x, const float *weight, const float *bias, const void *state_in,
                              void *y, void *state_out, int silu, int batch, int dim, int64_t seqlen, int width,
                              int io_dtype, void *stream) {
    using namespace ssm;
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (batch < 0 || dim < 0 || seqlen < 0 || width < 1 || width > 8) return SSM_ERR_DIMS;
    if (seqlen > ((int64_t)1 << 40) || (int64_t)batch * dim > ((int64_t)1 << 31)) return SSM_ERR_DIMS;
    if (batch == 0 || dim == 0) return SSM_OK;
    if (!weight || (seqlen > 0 && (!x || !y))) return SSM_ERR_NULL;
    const size_t es = io_dtype == SSM_BF16 ? 2 : 4;
    const void *iop[] = {x, y, state_in, state_out};
    for (const void *q : iop)
        if (q && !aligned(q, es)) return SSM_ERR_ALIGN;
    if (!aligned(weight, 4) || (bias && !aligned(bias, 4))) return SSM_ERR_ALIGN;
    const size_t nc = (size_t)batch * dim;
    const size_t nx = nc * (size_t)seqlen * es, ns = nc * (size_t)(width - 1) * es;
    const Span ins[] = {span(x, nx), span(weight, (size_t)dim * width * 4), span(bias, (size_t)dim * 4),
                        span(state_in, ns)};
    const Span outs[] = {span(y, nx), span(state_out, ns)};
    for (const Span &o : outs)
        for (const Span &i : ins)
            if (overlap(o, i)) return SSM_ERR_ALIAS;
    if (overlap(outs[0], outs[1])) return SSM_ERR_ALIAS;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (seqlen == 0) {   // the history passes through unchanged
        if (state_out && ns) {
            const cudaError_t e = state_in ? cudaMemcpyAsync(state_out, state_in, ns, cudaMemcpyDeviceToDevice, st)
                                           : cudaMemsetAsync(state_out, 0, ns, st);
            if (e != cudaSuccess) return SSM_ERR_LAUNCH;
        }
        return SSM_OK;
    }
    ConvArgs a{x, weight, bias, state_in, y, state_out, silu ? 1 : 0, dim, (int64_t)nc, seqlen,
               (seqlen + G - 1) / G};
    const bool vec = ((size_t)seqlen * es) % 16 == 0 && aligned(x, 16) && aligned(y, 16);
    const cudaError_t e = io_dtype == SSM_BF16 ? launch_t<__nv_bfloat16>(a, width, vec, st)
                                               : launch_t<float>(a, width, vec, st);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}
