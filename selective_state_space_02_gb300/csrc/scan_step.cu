// Single-token (decode) step of the selective state-space recurrence:
// "Mamba (part 2): parallel scan and hardware-aware optimisation"
// (scwacadex.pages.dev), sect. 6-7 -- at inference the state advances one
// token at a time, O(1) work and memory per token.  Declared in
// include/ssm_step.h.
//
// The step streams the state once (read, update, write back) and is bound by
// HBM bandwidth: per channel 8 * dstate bytes of state plus x, delta, (z) and
// y.  One lane owns up to 16 states of a channel (G = 1, 2 or 4 lanes per
// channel for dstate <= 16, 32, 64) and issues all of its 16-byte state loads
// before the arithmetic, so each thread keeps up to 64 bytes in flight; the
// index division, Delta and the epilogue are paid once per lane.  With G > 1
// the contraction sum_n C h is reduced over the G lanes with xor shuffles and
// the channel's first lane finishes the skip, the gate and the store.
#include <mutex>

#include "../../include/ssm_scan.h"
#include "../../include/ssm_step.h"
#include "scan_device.cuh"
#include "scan_internal.h"
#include "scan_tma.cuh"

namespace ssm {
namespace {

struct StepArgs {
    float *state;
    const void *x;
    const void *delta;
    const float *A;
    const void *B;
    const void *C;
    const float *D;        // nullable
    const void *z;         // nullable
    const float *dt_bias;  // nullable
    int softplus;
    void *y;
    int batch;
    int dim;
    int N;
};

constexpr int kThreads = 256;

// Four consecutive I/O elements as float4 (16-byte loads for float32, 8-byte
// for bf16; the caller guarantees the alignment).
template <typename T> struct Quad;
template <> struct Quad<float> {
    static __device__ __forceinline__ float4 ld(const void *p, int64_t i) {
        return __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i));
    }
};
template <> struct Quad<__nv_bfloat16> {
    static __device__ __forceinline__ float4 ld(const void *p, int64_t i) {
        const uint2 w = __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p) + i));
        return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    }
};

// Four consecutive I/O elements as loaded, before conversion (float4, or four
// bf16 in a uint2), and their conversion: the TMA kernel loads ahead of use
// and converts only where the values are needed, so that no instruction next
// to the load waits for it.
template <typename T> struct QuadRaw;
template <> struct QuadRaw<float> {
    using type = float4;
    static __device__ __forceinline__ float4 ld(const void *p, int64_t i) {
        return __ldg(reinterpret_cast<const float4 *>(static_cast<const float *>(p) + i));
    }
    static __device__ __forceinline__ float4 cvt(float4 v) { return v; }
};
template <> struct QuadRaw<__nv_bfloat16> {
    using type = uint2;
    static __device__ __forceinline__ uint2 ld(const void *p, int64_t i) {
        return __ldg(reinterpret_cast<const uint2 *>(static_cast<const __nv_bfloat16 *>(p) + i));
    }
    static __device__ __forceinline__ float4 cvt(uint2 w) {
        return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
    }
};

// One I/O element as loaded (a float's bits, or a bf16 in the low half) and
// its conversion.
template <typename T> __device__ __forceinline__ uint32_t ld_bits(const void *p, int64_t i) {
    if constexpr (sizeof(T) == 4) return __float_as_uint(__ldg(static_cast<const float *>(p) + i));
    else return (uint32_t)__ldg(static_cast<const unsigned short *>(p) + i);
}
template <typename T> __device__ __forceinline__ float of_bits(uint32_t b) {
    return sizeof(T) == 4 ? __uint_as_float(b) : __uint_as_float(b << 16);
}

// Elements n .. n+3 of an [rows][N] array at row `row`, zeros past N.
template <typename T, bool VEC>
__device__ __forceinline__ float4 quad(const void *base, int64_t row, int N, int n) {
    if (VEC) return Quad<T>::ld(base, row * N + n);
    float v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = n + k < N ? Io<T>::ld(base, row * N + n + k) : 0.0f;
    return make_float4(v[0], v[1], v[2], v[3]);
}

// G lanes per channel, S states per lane (S a multiple of 4; G = 1 up to 16
// states).  A lane issues all S/4 state loads before it needs them, forms
// Delta once, and updates its states with packed f32x2 arithmetic.
template <typename T, int S, int G, bool VEC>
__global__ void __launch_bounds__(kThreads, 1) step_kernel(const StepArgs p) {
    constexpr int NQ = S / 4;
    const uint64_t gid = (uint64_t)blockIdx.x * kThreads + threadIdx.x;
    const uint64_t c = gid / G;
    const int gl = (int)(gid % G);
    const uint32_t nchan = (uint32_t)((int64_t)p.batch * p.dim);
    const bool live = c < nchan;
    const uint32_t ch = live ? (uint32_t)c : 0u;
    const uint32_t dim = (uint32_t)p.dim;
    const uint32_t b = ch / dim;
    const uint32_t d = ch - b * dim;
    const int N = p.N;
    const int n0 = gl * S;
    float *srow = p.state + (int64_t)ch * N;
    float4 h[NQ];
    float xv = 0.0f, v = 0.0f;
    if (live) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int n = n0 + 4 * q;
            h[q] = make_float4(0.0f, 0.0f, 0.0f, 0.0f);
            if (n < N) {
                if (VEC) h[q] = *reinterpret_cast<const float4 *>(srow + n);
                else h[q] = make_float4(srow[n], n + 1 < N ? srow[n + 1] : 0.0f, n + 2 < N ? srow[n + 2] : 0.0f,
                                        n + 3 < N ? srow[n + 3] : 0.0f);
            }
        }
        xv = Io<T>::ld(p.x, ch);
        v = Io<T>::ld(p.delta, ch) + (p.dt_bias ? __ldg(p.dt_bias + d) : 0.0f);
    }
    const float Delta = p.softplus ? softplus2(make_float2(v, v)).x : v;
    const float2 dl2 = make_float2(Delta * kLog2e, Delta * kLog2e);
    const float2 uu = make_float2(Delta * xv, Delta * xv);
    float2 acc = make_float2(0.0f, 0.0f);
    if (live) {
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int n = n0 + 4 * q;
            if (n < N) {
                const float4 A4 = quad<float, VEC>(p.A, d, N, n);
                const float4 B4 = quad<T, VEC>(p.B, b, N, n);
                const float4 C4 = quad<T, VEC>(p.C, b, N, n);
                const float2 e01 = __fmul2_rn(dl2, make_float2(A4.x, A4.y));
                const float2 e23 = __fmul2_rn(dl2, make_float2(A4.z, A4.w));
                float2 h01 = __ffma2_rn(make_float2(ex2(e01.x), ex2(e01.y)), make_float2(h[q].x, h[q].y),
                                        __fmul2_rn(uu, make_float2(B4.x, B4.y)));
                float2 h23 = __ffma2_rn(make_float2(ex2(e23.x), ex2(e23.y)), make_float2(h[q].z, h[q].w),
                                        __fmul2_rn(uu, make_float2(B4.z, B4.w)));
                acc = __ffma2_rn(make_float2(C4.x, C4.y), h01, acc);
                acc = __ffma2_rn(make_float2(C4.z, C4.w), h23, acc);
                h[q] = make_float4(h01.x, h01.y, h23.x, h23.y);
            }
        }
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
            const int n = n0 + 4 * q;
            if (n < N) {
                if (VEC) {
                    *reinterpret_cast<float4 *>(srow + n) = h[q];
                } else {
                    srow[n] = h[q].x;
                    if (n + 1 < N) srow[n + 1] = h[q].y;
                    if (n + 2 < N) srow[n + 2] = h[q].z;
                    if (n + 3 < N) srow[n + 3] = h[q].w;
                }
            }
        }
    }
    float sum = acc.x + acc.y;
    // every lane of the warp reaches the shuffles (the grid covers whole warps)
#pragma unroll
    for (int off = G / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
    if (live && gl == 0) {
        if (p.D) sum = fmaf(__ldg(p.D + d), xv, sum);
        if (p.z) sum *= silu_f(Io<T>::ld(p.z, ch));
        Io<T>::st(p.y, ch, sum);
    }
}

// The state streamed through shared memory.  A persistent CTA of kTmaThreads
// threads walks tiles of kTmaThreads / G channels (kTmaThreads * S floats,
// 8 KB for S = 16): bulk copies bring the tiles' state rows into a kStages
// ring (completion on an mbarrier per stage, bounded waits), up to kStages
// tiles ahead; every thread updates its own S states in shared memory, and
// one bulk store per tile writes them back, so global state traffic is whole
// contiguous tiles.  The per-channel x, delta, dt_bias and z are loaded into
// registers one tile ahead.  A thread's S states sit at tid * S floats; it visits
// its S/4 quads starting at quad (tid * S / 32) mod (S / 4), so the 8 lanes
// of each 128-byte shared-memory phase touch 8 different 16-byte bank groups.
constexpr int kTmaThreads = 128;
// Three stages: 14.46 us per step against 14.87 with four (the smaller ring
// lets 8 CTAs of 63 registers share an SM instead of 6), 256 x 2048 x 16 bf16.
constexpr int kStages = 3;

template <int S>
constexpr uint32_t tile_bytes_full() { return (uint32_t)kTmaThreads * S * 4; }

template <typename T, int S, int G>
__global__ void __launch_bounds__(kTmaThreads, 1) step_tma_kernel(const StepArgs p, unsigned int *status) {
    constexpr int NQ = S / 4;
    constexpr int TCH = kTmaThreads / G;                   // channels per tile
    constexpr uint32_t kTile = tile_bytes_full<S>();
    extern __shared__ __align__(128) unsigned char smem[];
    float *ring = reinterpret_cast<float *>(smem);         // [kStages][kTmaThreads * S]
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + kStages * kTile);

    const int tid = threadIdx.x;
    const int N = p.N;                                     // == S * G
    const uint32_t nchan = (uint32_t)((int64_t)p.batch * p.dim);
    const uint32_t dim = (uint32_t)p.dim;
    const uint32_t ntiles = (nchan + TCH - 1) / TCH;
    const uint32_t stride = gridDim.x;
    auto bytes_of = [&](uint32_t t) -> uint32_t {
        const uint32_t c0 = t * TCH;
        const uint32_t nc = nchan - c0 < (uint32_t)TCH ? nchan - c0 : (uint32_t)TCH;
        return nc * (uint32_t)N * 4u;
    };
    // tiles of this CTA: blockIdx.x + k * stride, k = 0, 1, ...
    const uint32_t mine_n = blockIdx.x < ntiles ? (ntiles - blockIdx.x + stride - 1) / stride : 0;
    if (tid == 0) {
        for (int s = 0; s < kStages; ++s) mbar_init(&full[s], 1);
        fence_mbar_init();
    }
    __syncthreads();
    auto issue = [&](uint32_t k) {                         // load the CTA's k-th tile into stage k % kStages
        const uint32_t t = blockIdx.x + k * stride;
        const int s = (int)(k % kStages);
        mbar_arrive_expect_tx(&full[s], bytes_of(t));
        bulk_load(ring + s * kTmaThreads * S, p.state + (int64_t)t * TCH * N, bytes_of(t), &full[s]);
    };
    uint32_t issued = 0;                                   // tiles whose load has been issued (tid 0)
    if (tid == 0)   // tiles 0 .. kStages-2; from k = 1 on, tile k + kStages - 2 is loaded at iteration k
        for (; issued < mine_n && issued < (uint32_t)kStages - 1; ++issued) issue(issued);

    const int gl = tid % G;
    const int r = (tid * NQ / 8) % NQ;                     // first quad this thread visits
    // the per-channel inputs (x, delta, dt_bias, z) of a tile, loaded one
    // tile ahead so that their DRAM latency overlaps the previous tile's
    // work: raw bits from addresses clamped into the problem, converted (and
    // dt_bias added) only when the tile is processed
    struct Inputs {
        uint32_t x, dl, z;
        float bias;
    };
    auto load_inputs = [&](uint32_t kk) -> Inputs {
        Inputs in;
        const uint32_t c = (blockIdx.x + kk * stride) * TCH + (uint32_t)(tid / G);
        const uint32_t ch = (kk < mine_n && c < nchan) ? c : 0u;
        in.x = ld_bits<T>(p.x, ch);
        in.dl = ld_bits<T>(p.delta, ch);
        in.z = p.z ? ld_bits<T>(p.z, ch) : 0u;
        in.bias = p.dt_bias ? __ldg(p.dt_bias + ch % dim) : 0.0f;
        return in;
    };
    Inputs next = load_inputs(0);
    bool aborted = false;
    uint32_t k = 0;
    for (; k < mine_n; ++k) {
        const int st = (int)(k % kStages);
        const uint32_t t = blockIdx.x + k * stride;
        // load tile k + kStages - 2 into the stage of tile k - 2 once that tile's store
        // (issued a whole tile ago) has read it; tile k - 1's store may still
        // be reading its own stage
        if (tid == 0 && k > 0 && issued < mine_n) {
            bulk_wait_read<1>();
            issue(issued);
            ++issued;
        }
        const Inputs cur = next;
        next = load_inputs(k + 1);
        const uint32_t c0 = t * TCH;
        const uint32_t ch = c0 + (uint32_t)(tid / G);
        const bool live = ch < nchan;
        const uint32_t b = live ? ch / dim : 0u;
        const uint32_t d = live ? ch - b * dim : 0u;
        // A, B and C do not depend on the state: load them before the wait
        // (b and d are clamped into the problem; dead lanes' results are unused)
        float4 A4[NQ];
        typename QuadRaw<T>::type Br[NQ], Cr[NQ];
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            const int n = gl * S + 4 * ((j + r) % NQ);
            A4[j] = Quad<float>::ld(p.A, (int64_t)d * N + n);
            Br[j] = QuadRaw<T>::ld(p.B, (int64_t)b * N + n);
            Cr[j] = QuadRaw<T>::ld(p.C, (int64_t)b * N + n);
        }
        const bool ok = wait_parity(&full[st], (uint32_t)((k / kStages) & 1), status);
        if (!__syncthreads_and(ok)) { aborted = true; break; }
        const float xv = of_bits<T>(cur.x), v = of_bits<T>(cur.dl) + cur.bias, zv = of_bits<T>(cur.z);
        float4 B4[NQ], C4[NQ];
#pragma unroll
        for (int j = 0; j < NQ; ++j) {
            B4[j] = QuadRaw<T>::cvt(Br[j]);
            C4[j] = QuadRaw<T>::cvt(Cr[j]);
        }

        const float Delta = p.softplus ? softplus2(make_float2(v, v)).x : v;
        const float2 dl2 = make_float2(Delta * kLog2e, Delta * kLog2e);
        const float2 uu = make_float2(Delta * xv, Delta * xv);
        float2 acc = make_float2(0.0f, 0.0f);
        float *mine = ring + st * kTmaThreads * S + tid * S;
        if (live) {
#pragma unroll
            for (int j = 0; j < NQ; ++j) {
                const int q = (j + r) % NQ;
                float4 *hp = reinterpret_cast<float4 *>(mine + 4 * q);
                const float4 h = *hp;
                const float2 e01 = __fmul2_rn(dl2, make_float2(A4[j].x, A4[j].y));
                const float2 e23 = __fmul2_rn(dl2, make_float2(A4[j].z, A4[j].w));
                const float2 h01 = __ffma2_rn(make_float2(ex2(e01.x), ex2(e01.y)), make_float2(h.x, h.y),
                                              __fmul2_rn(uu, make_float2(B4[j].x, B4[j].y)));
                const float2 h23 = __ffma2_rn(make_float2(ex2(e23.x), ex2(e23.y)), make_float2(h.z, h.w),
                                              __fmul2_rn(uu, make_float2(B4[j].z, B4[j].w)));
                acc = __ffma2_rn(make_float2(C4[j].x, C4[j].y), h01, acc);
                acc = __ffma2_rn(make_float2(C4[j].z, C4[j].w), h23, acc);
                *hp = make_float4(h01.x, h01.y, h23.x, h23.y);
            }
        }
        float sum = acc.x + acc.y;
#pragma unroll
        for (int off = G / 2; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
        if (live && gl == 0) {
            if (p.D) sum = fmaf(__ldg(p.D + d), xv, sum);
            if (p.z) sum *= silu_f(zv);
            Io<T>::st(p.y, ch, sum);
        }
        // hand the updated tile to the async proxy and store it
        fence_proxy_async();
        __syncthreads();
        if (tid == 0) {
            bulk_store(p.state + (int64_t)c0 * N, ring + st * kTmaThreads * S, bytes_of(t));
            bulk_commit();
        }
    }
    if (tid == 0) {
        // no CTA leaves with a copy in flight: after an abort wait (bounded)
        // for the loads still outstanding, and always for the stores
        if (aborted)
            for (uint32_t j = k; j < issued; ++j)
                wait_parity(&full[j % kStages], (uint32_t)((j / kStages) & 1), status, 1ll << 28);
        bulk_wait_all();
    }
}

struct TmaLaunch {
    int blocks_per_sm = 0;
    int sms = 0;
};

template <typename T, int S, int G>
cudaError_t launch_tma(const StepArgs &a, cudaStream_t st) {
    unsigned int *status = device_status_word();
    if (!status) return cudaErrorInvalidSymbol;
    auto kern = step_tma_kernel<T, S, G>;
    const size_t smem = (size_t)kStages * tile_bytes_full<S>() + kStages * sizeof(uint64_t);

    static std::mutex mu;
    static TmaLaunch cache[64];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    TmaLaunch lc;
    {
        std::lock_guard<std::mutex> lk(mu);
        if (cache[dev].sms == 0) {
            int nb = 0, sms = 0;
            e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kTmaThreads, smem);
            if (e != cudaSuccess) return e;
            e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
            if (e != cudaSuccess) return e;
            cache[dev].blocks_per_sm = nb > 0 ? nb : 1;
            cache[dev].sms = sms > 0 ? sms : 1;
        }
        lc = cache[dev];
    }
    const int64_t nchan = (int64_t)a.batch * a.dim;
    const int64_t ntiles = (nchan + kTmaThreads / G - 1) / (kTmaThreads / G);
    const int64_t resident = (int64_t)lc.blocks_per_sm * lc.sms;
    const unsigned grid = (unsigned)(ntiles < resident ? ntiles : resident);
    kern<<<grid, kTmaThreads, smem, st>>>(a, status);
    return cudaGetLastError();
}

template <typename T, int S, int G>
cudaError_t launch_g(const StepArgs &a, bool vec, cudaStream_t st) {
    const int64_t threads = (int64_t)a.batch * a.dim * G;
    const unsigned grid = (unsigned)((threads + kThreads - 1) / kThreads);
    if (vec) step_kernel<T, S, G, true><<<grid, kThreads, 0, st>>>(a);
    else step_kernel<T, S, G, false><<<grid, kThreads, 0, st>>>(a);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_t(const StepArgs &a, bool vec, cudaStream_t st) {
    const int N = a.N;
    if (vec) {   // whole-tile streaming when the state rows are 4, 8, 16, 32 or 64 floats
        if (N == 4) return launch_tma<T, 4, 1>(a, st);
        if (N == 8) return launch_tma<T, 8, 1>(a, st);
        if (N == 16) return launch_tma<T, 16, 1>(a, st);
        if (N == 32) return launch_tma<T, 16, 2>(a, st);
        if (N == 64) return launch_tma<T, 16, 4>(a, st);
    }
    if (N <= 4) return launch_g<T, 4, 1>(a, vec, st);
    if (N <= 8) return launch_g<T, 8, 1>(a, vec, st);
    if (N <= 16) return launch_g<T, 16, 1>(a, vec, st);
    if (N <= 32) return launch_g<T, 16, 2>(a, vec, st);
    return launch_g<T, 16, 4>(a, vec, st);
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Span {
    uintptr_t lo, hi;
};

Span span(const void *p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Span{a, a + (p ? bytes : 0)};
}

bool overlap(Span a, Span b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

}  // namespace
}  // namespace ssm

extern "C" int ssm_scan_step(float *state, const void *x, const void *delta, const float *A, const void *B,
                             const void *C, const float *D, const void *z, const float *dt_bias,
                             int delta_softplus, void *y, int batch, int dim, int dstate, int io_dtype,
                             void *stream) {
    using namespace ssm;
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (batch < 0 || dim < 0 || dstate < 1 || dstate > 64) return SSM_ERR_DIMS;
    if ((int64_t)batch * dim > ((int64_t)1 << 31)) return SSM_ERR_DIMS;
    if (batch == 0 || dim == 0) return SSM_OK;
    if (!state || !x || !delta || !A || !B || !C || !y) return SSM_ERR_NULL;
    const size_t es = io_dtype == SSM_BF16 ? 2 : 4;
    const void *iop[] = {x, delta, B, C, z, y};
    for (const void *q : iop)
        if (q && !aligned(q, es)) return SSM_ERR_ALIGN;
    const void *fp[] = {state, A, D, dt_bias};
    for (const void *q : fp)
        if (q && !aligned(q, 4)) return SSM_ERR_ALIGN;
    const size_t nc = (size_t)batch * dim;
    const Span ins[] = {span(x, nc * es), span(delta, nc * es), span(z, nc * es),
                        span(B, (size_t)batch * dstate * es), span(C, (size_t)batch * dstate * es),
                        span(A, (size_t)dim * dstate * 4), span(D, (size_t)dim * 4), span(dt_bias, (size_t)dim * 4)};
    const Span sy = span(y, nc * es), ss = span(state, nc * dstate * 4);
    for (const Span &i : ins)
        if (overlap(sy, i) || overlap(ss, i)) return SSM_ERR_ALIAS;
    if (overlap(sy, ss)) return SSM_ERR_ALIAS;
    StepArgs a{state, x, delta, A, B, C, D, z, dt_bias, delta_softplus ? 1 : 0, y, batch, dim, dstate};
    // 16-byte state and A rows, 4-element B and C loads
    const bool vec = dstate % 4 == 0 && aligned(state, 16) && aligned(A, 16) && aligned(B, 4 * es) &&
                     aligned(C, 4 * es);
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const cudaError_t e = io_dtype == SSM_BF16 ? launch_t<__nv_bfloat16>(a, vec, st) : launch_t<float>(a, vec, st);
    return e == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}
