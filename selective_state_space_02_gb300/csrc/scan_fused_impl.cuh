// Channel-parallel, time-serial forward selective scan (FUSED variant, and
// both passes of the TWOPASS variant).
//
// "Mamba hardware-aware parallel associative scan" (pwwt.cn/news/6375169):
//   sect. 2.2, third approach -- parallelism over channels; a thread owns part
//     of one channel's state in registers and walks the sequence in order;
//   sect. 2.2 / 3.3 -- two-pass chunk carry: per-chunk totals (A_k, B_k), a
//     small scan over the totals, then a fix-up pass from each chunk's start
//     state;
//   sect. 4.1 -- discretisation, scan, C contraction, D skip and gate fused
//     in one kernel; neither (a, b) nor h_t ever reaches global memory
//     ("Mamba (part 2)", scwacadex.pages.dev, sect. 4.1-4.2).
//
// Warp-specialised CTA: one producer warp and NW consumer warps.
//   producer : per tile of kTC steps, waits for the stage to be free, issues
//              2-D TMA copies of x, delta, z (DT rows) and B, C (NP rows) that
//              complete on the stage's `full` mbarrier (or, for rows that are
//              not 16-byte aligned, loads the tile element by element), then
//              re-lays B and C out as float32 [state-in-group][group][step]
//              and arrives on `ready`.
//   consumers: a consumer warp owns CPW = 32 / NS channels; each channel's NP
//              (padded) states are split over NS lanes, S states per lane.
//              Per block of kBlk steps (warp-synchronous, no CTA barrier):
//                1. each lane computes Delta = softplus(delta + dt_bias) and
//                   u = Delta * x for kBlk / NS steps of its channel and
//                   shares them through warp-private shared memory;
//                2. each lane advances its S recurrences through the block
//                   with packed f32x2 arithmetic: a = 2^(Delta * A log2 e),
//                   h = a h + u B, partial y = sum_s C h;
//                3. the NS partial sums of each (channel, step) are added by
//                   the lane that owns the step, which applies the skip D x and
//                   the gate silu(z) and stores y.
//              After a tile every consumer warp arrives on the stage's `empty`
//              mbarrier, releasing it to the producer.
// Padding is the identity step (1, 0): states n >= dstate have A = B = C = 0,
// steps t >= L and channels d >= dim have Delta = u = 0.  Every mbarrier wait
// is bounded; a wait that gives up flags the status word and the CTA stops.
#pragma once

#include "scan_internal.h"
#include "scan_device.cuh"
#include "scan_tma.cuh"

namespace ssm {
namespace fused {

constexpr int kBlk = 16;           // steps per warp-synchronous block
constexpr int kDU = 4 * kBlk + 4;  // float stride of one channel's {Delta, Delta, u, u} block (conflict free)
constexpr int kYP = kBlk + 4;      // float stride of one lane's partial sums

// Steps per tile (TMA box width): 32, or 16 for wide states so that four
// pipeline stages of B/C tiles still fit in shared memory.
__host__ __device__ constexpr int tile_steps(int np) { return np >= 32 ? 16 : 32; }
constexpr int kStagesMax = 4;

#ifndef SSM_MINB
#define SSM_MINB 1
#endif

enum Mode { kWhole = 0, kTotals = 1, kSeeded = 2 };

struct SegArgs {
    int64_t seg_len;   // steps per segment (the last one may be shorter)
    int nseg;          // number of segments in this launch
    float *ws_h;       // [nseg][batch*dim][dstate]: B_k after pass 1, h_init after the small scan
    float *ws_s;       // [nseg][batch*dim]: sum of Delta over the segment
};

struct TileMaps {
    CUtensorMap x, dl, z, B, C;
};

__host__ __device__ constexpr size_t align128(size_t n) { return (n + 127) / 128 * 128; }

template <typename T, int NP, int S, int NW, bool GATE, int MODE>
struct Layout {
    static constexpr int NS = NP / S;            // lanes per channel
    static constexpr int CPW = 32 / NS;          // channels per consumer warp
    static constexpr int DT = NW * CPW;          // channels per CTA
    static constexpr int NT = (NW + 1) * 32;     // consumer warps + producer warp
    static constexpr int E = kBlk / NS;          // steps per lane in the element phases
    static constexpr bool kY = MODE != kTotals;
    static constexpr bool kZ = GATE && kY;
    static constexpr int TC = tile_steps(NP);     // steps per tile
    static constexpr int NST = kStagesMax;        // pipeline depth
    static constexpr int YPC = NS * kYP + 4;      // float stride of one channel's partial sums (conflict free)
    static constexpr size_t row_bytes = (size_t)DT * TC * sizeof(T);
    static constexpr size_t bc_bytes = (size_t)NP * TC * sizeof(T);
    // one pipeline stage
    static constexpr size_t off_x = 0;
    static constexpr size_t off_dl = align128(row_bytes);
    static constexpr size_t off_z = off_dl + align128(row_bytes);
    static constexpr size_t off_B = off_z + (kZ ? align128(row_bytes) : 0);
    static constexpr size_t off_C = off_B + align128(bc_bytes);
    static constexpr size_t off_Bf = off_C + (kY ? align128(bc_bytes) : 0);   // [TC][NS][B(S) C(S)] float
    static constexpr size_t stage_bytes = off_Bf + align128((size_t)TC * NP * 2 * 4);
    static constexpr uint32_t tx_bytes = (uint32_t)(row_bytes * (kZ ? 3 : 2) + bc_bytes * (kY ? 2 : 1));
    // per consumer warp: {Delta, Delta, u, u} per step [CPW][kDU], partial sums [CPW*NS][kYP]
    static constexpr size_t warp_du = (size_t)CPW * kDU * 4;
    static constexpr size_t warp_yp = kY ? (size_t)CPW * YPC * 4 : 0;
    static constexpr size_t warp_bytes = align128(warp_du + warp_yp);
    static constexpr size_t off_warp = NST * stage_bytes;
    static constexpr size_t off_bar = off_warp + NW * warp_bytes;
    static constexpr size_t bytes = off_bar + 3 * NST * 8 + 16;
};

// Raw tile element access (shared memory).
template <typename T>
__device__ __forceinline__ float raw1(const unsigned char *base, int idx) {
    if constexpr (sizeof(T) == 4) {
        return reinterpret_cast<const float *>(base)[idx];
    } else {
        const unsigned short v = reinterpret_cast<const unsigned short *>(base)[idx];
        return __uint_as_float((uint32_t)v << 16);
    }
}

// E consecutive raw elements starting at idx (E in {1, 2, 4, 8}; idx * sizeof(T)
// aligned to E * sizeof(T)).
template <typename T, int E>
__device__ __forceinline__ void rawE(const unsigned char *base, int idx, float (&v)[E]) {
    if constexpr (sizeof(T) == 4) {
        const float *p = reinterpret_cast<const float *>(base) + idx;
        if constexpr (E % 4 == 0) {
#pragma unroll
            for (int k = 0; k < E; k += 4) {
                const float4 q = *reinterpret_cast<const float4 *>(p + k);
                v[k] = q.x; v[k + 1] = q.y; v[k + 2] = q.z; v[k + 3] = q.w;
            }
        } else if constexpr (E == 2) {
            const float2 q = *reinterpret_cast<const float2 *>(p);
            v[0] = q.x; v[1] = q.y;
        } else {
            v[0] = p[0];
        }
    } else {
        const unsigned char *p = base + (size_t)idx * 2;
        if constexpr (E >= 2) {
#pragma unroll
            for (int k = 0; k < E; k += 2) {
                const uint32_t w = *reinterpret_cast<const uint32_t *>(p + 2 * k);
                v[k] = __uint_as_float(w << 16);
                v[k + 1] = __uint_as_float(w & 0xffff0000u);
            }
        } else {
            v[0] = raw1<T>(base, idx);
        }
    }
}

// Store E consecutive outputs at global index idx (all in range) .
template <typename T, int E>
__device__ __forceinline__ void storeE(void *y, int64_t idx, bool vec, const float (&v)[E]) {
    if constexpr (sizeof(T) == 4) {
        float *p = static_cast<float *>(y) + idx;
        if (vec && E % 4 == 0) {
#pragma unroll
            for (int k = 0; k < E; k += 4) *reinterpret_cast<float4 *>(p + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
        } else if (vec && E == 2) {
            *reinterpret_cast<float2 *>(p) = make_float2(v[0], v[1]);
        } else {
#pragma unroll
            for (int k = 0; k < E; ++k) p[k] = v[k];
        }
    } else {
        __nv_bfloat16 *p = static_cast<__nv_bfloat16 *>(y) + idx;
        if constexpr (E >= 2) {
            uint32_t w[E / 2];
#pragma unroll
            for (int k = 0; k < E; k += 2) {
                const __nv_bfloat162 pr = __floats2bfloat162_rn(v[k], v[k + 1]);
                w[k / 2] = *reinterpret_cast<const uint32_t *>(&pr);
            }
            if (vec && E == 8) {
                *reinterpret_cast<uint4 *>(p) = make_uint4(w[0], w[1], w[2], w[3]);
            } else if (vec && E == 4) {
                *reinterpret_cast<uint2 *>(p) = make_uint2(w[0], w[1]);
            } else if (vec && E == 2) {
                *reinterpret_cast<uint32_t *>(p) = w[0];
            } else {
#pragma unroll
                for (int k = 0; k < E; k += 2) {
                    p[k] = __ushort_as_bfloat16((unsigned short)(w[k / 2] & 0xffffu));
                    p[k + 1] = __ushort_as_bfloat16((unsigned short)(w[k / 2] >> 16));
                }
            }
        } else {
            p[0] = __float2bfloat16_rn(v[0]);
        }
    }
}

// Gate: accurate form for float32 outputs, one-MUFU tanh form for bf16
// outputs (its ~2^-11 relative error is far below bf16 rounding).
template <typename T>
__device__ __forceinline__ float gate(float z) {
    if constexpr (sizeof(T) == 4) {
        return silu_f(z);
    } else {
        const float hz = 0.5f * z;
        float t;
        asm("tanh.approx.f32 %0, %1;" : "=f"(t) : "f"(hz));
        return fmaf(hz, t, hz);   // z * sigmoid(z) = z/2 * (1 + tanh(z/2))
    }
}

template <typename T, int NP, int S, int NW, bool GATE, int MODE, bool TMA>
__global__ void __launch_bounds__((NW + 1) * 32, SSM_MINB)
scan_kernel(const FwdArgs p, const SegArgs sg, const __grid_constant__ TileMaps maps, unsigned int *status) {
    using Ly = Layout<T, NP, S, NW, GATE, MODE>;
    constexpr int NS = Ly::NS, CPW = Ly::CPW, DT = Ly::DT, E = Ly::E, kStages = Ly::NST, kTC = Ly::TC;
    constexpr bool kY = Ly::kY, kZ = Ly::kZ;
    static_assert(S % 2 == 0 && NS >= 1 && NS <= 32 && 32 % NS == 0, "lane split");
    static_assert(kBlk % NS == 0 && E >= 1, "element split");

    extern __shared__ __align__(128) unsigned char smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Ly::off_bar);
    uint64_t *ready = full + kStages;
    uint64_t *empty = ready + kStages;
    int *abort_flag = reinterpret_cast<int *>(empty + kStages);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int d0 = blockIdx.x * DT;
    const int b = blockIdx.y;
    const int seg = blockIdx.z;
    const int dim = p.dim, N = p.dstate;
    const int64_t L = p.L;
    const int64_t ts = (int64_t)seg * sg.seg_len;
    const int64_t te = (ts + sg.seg_len < L) ? ts + sg.seg_len : L;
    const int ntiles = (int)((te - ts + kTC - 1) / kTC);
    const int64_t chan0 = (int64_t)b * dim;
    const int64_t nchan = (int64_t)p.batch * dim;
    const int64_t row0 = chan0 + d0;              // first x/delta/z row of this CTA
    const int64_t brow0 = (int64_t)b * N;         // first B/C row of this batch

    if (threadIdx.x == 0) {
        for (int s = 0; s < kStages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&ready[s], 1);
            mbar_init(&empty[s], NW);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------------------------------------ producer
        int issued = 0;
        for (int tile = 0; tile < ntiles; ++tile) {
            const int st = tile % kStages;
            const uint32_t ph = (uint32_t)((tile / kStages) & 1);
            unsigned char *base = smem + st * Ly::stage_bytes;
            const int64_t t0 = ts + (int64_t)tile * kTC;
            const int tvalid = (int)((te - t0) < kTC ? (te - t0) : kTC);
            bool ok = true;
            if (tile >= kStages) ok = wait_parity(&empty[st], ph ^ 1u, status);
            if (!ok) { *abort_flag = 1; break; }
            if constexpr (TMA) {
                if (lane == 0) {
                    fence_proxy_async();
                    mbar_arrive_expect_tx(&full[st], Ly::tx_bytes);
                    const int tc = (int)t0, r0 = (int)row0, rb = (int)brow0;
                    tma_load_2d(base + Ly::off_x, &maps.x, tc, r0, &full[st]);
                    tma_load_2d(base + Ly::off_dl, &maps.dl, tc, r0, &full[st]);
                    if constexpr (kZ) tma_load_2d(base + Ly::off_z, &maps.z, tc, r0, &full[st]);
                    tma_load_2d(base + Ly::off_B, &maps.B, tc, rb, &full[st]);
                    if constexpr (kY) tma_load_2d(base + Ly::off_C, &maps.C, tc, rb, &full[st]);
                }
                issued = tile + 1;
                if (!wait_parity(&full[st], ph, status)) { *abort_flag = 1; break; }
            } else {
                // element loads; zeros outside the problem
                for (int e = lane; e < DT * kTC; e += 32) {
                    const int r = e / kTC, c = e % kTC;
                    const bool in = d0 + r < dim && c < tvalid;
                    const int64_t idx = (row0 + r) * L + t0 + c;
                    T xv = T(0.0f), dv = T(0.0f), zv = T(0.0f);
                    if (in) {
                        xv = static_cast<const T *>(p.x)[idx];
                        dv = static_cast<const T *>(p.delta)[idx];
                        if constexpr (kZ) zv = static_cast<const T *>(p.z)[idx];
                    }
                    reinterpret_cast<T *>(base + Ly::off_x)[e] = xv;
                    reinterpret_cast<T *>(base + Ly::off_dl)[e] = dv;
                    if constexpr (kZ) reinterpret_cast<T *>(base + Ly::off_z)[e] = zv;
                }
                for (int e = lane; e < NP * kTC; e += 32) {
                    const int n = e / kTC, c = e % kTC;
                    const bool in = n < N && c < tvalid;
                    const int64_t idx = (brow0 + n) * L + t0 + c;
                    T bv = T(0.0f), cv = T(0.0f);
                    if (in) {
                        bv = static_cast<const T *>(p.B)[idx];
                        if constexpr (kY) cv = static_cast<const T *>(p.C)[idx];
                    }
                    reinterpret_cast<T *>(base + Ly::off_B)[e] = bv;
                    if constexpr (kY) reinterpret_cast<T *>(base + Ly::off_C)[e] = cv;
                }
                __syncwarp();
            }
            // B, C [n][t] raw -> float [t][n / S][B(S) C(S)], rows n >= dstate
            // zeroed (in the TMA path they hold the next batch's rows).  Each
            // lane converts 4 steps of one state.
            float *BC = reinterpret_cast<float *>(base + Ly::off_Bf);
            for (int e = lane; e < NP * (kTC / 4); e += 32) {
                const int n = e % NP, c4 = e / NP;
                const bool in = n < N;
                float v[4];
                rawE<T, 4>(base + Ly::off_B, n * kTC + 4 * c4, v);
                float *dst = BC + ((4 * c4) * NS + n / S) * (2 * S) + n % S;
#pragma unroll
                for (int k = 0; k < 4; ++k) dst[k * NS * 2 * S] = in ? v[k] : 0.0f;
                if constexpr (kY) {
                    rawE<T, 4>(base + Ly::off_C, n * kTC + 4 * c4, v);
#pragma unroll
                    for (int k = 0; k < 4; ++k) dst[k * NS * 2 * S + S] = in ? v[k] : 0.0f;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&ready[st]);
        }
        // drain: copies issued before an abort must land before the CTA exits
        if constexpr (TMA) {
            if (lane == 0 && *abort_flag) {
                for (int t = (issued > kStages ? issued - kStages : 0); t < issued; ++t)
                    wait_parity(&full[t % kStages], (uint32_t)((t / kStages) & 1), status, 1ll << 28);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumer
    static_assert(E % 2 == 0 || E == 1, "element phases work on pairs");
    const int cw = lane / NS;                 // channel within the warp
    const int g = lane % NS;                  // state group
    const int cl = warp * CPW + cw;           // channel within the CTA
    const int d = d0 + cl;
    const bool dok = d < dim;
    float *du = reinterpret_cast<float *>(smem + Ly::off_warp + warp * Ly::warp_bytes);   // [CPW][kDU]
    float *yp = du + CPW * kDU;                                                             // [CPW][YPC]
    float *my_du = du + cw * kDU;             // this channel's {Delta, Delta, u, u} per step

    float2 h2[S / 2], a2[S / 2];
#pragma unroll
    for (int q = 0; q < S / 2; ++q) {
        float v[2], hv[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int n = g * S + 2 * q + k;
            const bool ok = dok && n < N;
            v[k] = ok ? __ldg(p.A + (int64_t)d * N + n) * kLog2e : 0.0f;
            hv[k] = (MODE == kSeeded && ok) ? sg.ws_h[((int64_t)seg * nchan + chan0 + d) * N + n] : 0.0f;
        }
        a2[q] = make_float2(v[0], v[1]);
        h2[q] = make_float2(hv[0], hv[1]);
    }
    const float bias = (dok && p.dt_bias) ? __ldg(p.dt_bias + d) : 0.0f;
    const float Dd = (dok && p.D) ? __ldg(p.D + d) : 0.0f;
    const bool vec = p.vec16 != 0;
    const bool sp = p.softplus != 0;
    float dsum = 0.0f;

    for (int tile = 0; tile < ntiles; ++tile) {
        const int st = tile % kStages;
        const uint32_t ph = (uint32_t)((tile / kStages) & 1);
        const unsigned char *base = smem + st * Ly::stage_bytes;
        const float *BC = reinterpret_cast<const float *>(base + Ly::off_Bf);
        const int64_t t0 = ts + (int64_t)tile * kTC;
        const int tvalid = (int)((te - t0) < kTC ? (te - t0) : kTC);
        bool ok = wait_parity(&ready[st], ph, status);
        if (TMA && ok) ok = wait_parity(&full[st], ph, status);   // TMA writes visible to this thread
        if (!ok) { *abort_flag = 1; }
        if (__any_sync(0xffffffffu, *abort_flag != 0)) break;

#pragma unroll 1
        for (int blk = 0; blk < kTC / kBlk; ++blk) {
            const int cb = blk * kBlk;              // first column of the block in the tile
            const int ce = cb + g * E;              // first column this lane owns in element phases
            // ---- 1. Delta, u for this lane's E steps, in pairs ----------------
            {
                float dv[E], xv[E];
                rawE<T, E>(base + Ly::off_dl, cl * kTC + ce, dv);
                rawE<T, E>(base + Ly::off_x, cl * kTC + ce, xv);
#pragma unroll
                for (int k = 0; k < E; k += 2) {
                    float2 v = make_float2(dv[k], E > 1 ? dv[k + 1] : 0.0f);
                    v = __fadd2_rn(v, make_float2(bias, bias));
                    float2 Dl = sp ? softplus2(v) : v;
                    const bool in0 = dok && ce + k < tvalid;
                    const bool in1 = dok && ce + k + 1 < tvalid;
                    Dl = make_float2(in0 ? Dl.x : 0.0f, in1 ? Dl.y : 0.0f);
                    const float2 Ul = __fmul2_rn(Dl, make_float2(xv[k], E > 1 ? xv[k + 1] : 0.0f));
                    *reinterpret_cast<float4 *>(my_du + 4 * (g * E + k)) = make_float4(Dl.x, Dl.x, Ul.x, Ul.x);
                    if (E > 1)
                        *reinterpret_cast<float4 *>(my_du + 4 * (g * E + k + 1)) = make_float4(Dl.y, Dl.y, Ul.y, Ul.y);
                }
            }
            __syncwarp();
            // ---- 2. scan the block ------------------------------------------
            float yv[kBlk];
#pragma unroll
            for (int j = 0; j < kBlk; ++j) {
                const float4 du4 = *reinterpret_cast<const float4 *>(my_du + 4 * j);   // Delta, Delta, u, u
                const float2 dd = make_float2(du4.x, du4.y);
                const float2 uu = make_float2(du4.z, du4.w);
                // this step's B (S values) then C (S values), 16-byte loads
                const float *bc = BC + ((cb + j) * NS + g) * (2 * S);
                float bcv[2 * S];
#pragma unroll
                for (int k = 0; k < (kY ? 2 * S : S); k += 4) {
                    if (k + 4 <= 2 * S) {
                        const float4 v4 = *reinterpret_cast<const float4 *>(bc + k);
                        bcv[k] = v4.x; bcv[k + 1] = v4.y; bcv[k + 2] = v4.z; bcv[k + 3] = v4.w;
                    }
                }
                if constexpr (!kY && S == 2) {
                    const float2 v2 = *reinterpret_cast<const float2 *>(bc);
                    bcv[0] = v2.x; bcv[1] = v2.y;
                }
                float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
                for (int q = 0; q < S / 2; ++q) {
                    const float2 arg = __fmul2_rn(dd, a2[q]);
                    const float2 a = make_float2(ex2(arg.x), ex2(arg.y));
                    h2[q] = __ffma2_rn(a, h2[q], __fmul2_rn(uu, make_float2(bcv[2 * q], bcv[2 * q + 1])));
                    if constexpr (kY) acc = __ffma2_rn(make_float2(bcv[S + 2 * q], bcv[S + 2 * q + 1]), h2[q], acc);
                }
                yv[j] = acc.x + acc.y;
                if constexpr (!kY) dsum += du4.x;
            }
            if constexpr (kY) {
                float *myp = yp + cw * Ly::YPC + g * kYP;
#pragma unroll
                for (int q4 = 0; q4 < kBlk / 4; ++q4)
                    *reinterpret_cast<float4 *>(myp + 4 * q4) =
                        make_float4(yv[4 * q4], yv[4 * q4 + 1], yv[4 * q4 + 2], yv[4 * q4 + 3]);
                __syncwarp();
                // ---- 3. reduce the NS partial sums of this lane's E steps, skip, gate, store
                float ys[E];
#pragma unroll
                for (int k = 0; k < E; ++k) ys[k] = 0.0f;
#pragma unroll
                for (int q = 0; q < NS; ++q) {
                    float pv[E];
                    const float *src = yp + cw * Ly::YPC + q * kYP + g * E;
                    if constexpr (E % 4 == 0) {
#pragma unroll
                        for (int k = 0; k < E; k += 4) {
                            const float4 v4 = *reinterpret_cast<const float4 *>(src + k);
                            pv[k] = v4.x; pv[k + 1] = v4.y; pv[k + 2] = v4.z; pv[k + 3] = v4.w;
                        }
                    } else if constexpr (E == 2) {
                        const float2 v2 = *reinterpret_cast<const float2 *>(src);
                        pv[0] = v2.x; pv[1] = v2.y;
                    } else {
                        pv[0] = src[0];
                    }
                    if constexpr (E >= 2) {
#pragma unroll
                        for (int k = 0; k < E; k += 2) {
                            const float2 s2 = __fadd2_rn(make_float2(ys[k], ys[k + 1]), make_float2(pv[k], pv[k + 1]));
                            ys[k] = s2.x; ys[k + 1] = s2.y;
                        }
                    } else {
                        ys[0] += pv[0];
                    }
                }
                if (dok) {
                    float xv[E];
                    rawE<T, E>(base + Ly::off_x, cl * kTC + ce, xv);
                    float zv[E];
                    if constexpr (kZ) rawE<T, E>(base + Ly::off_z, cl * kTC + ce, zv);
                    if constexpr (E >= 2) {
#pragma unroll
                        for (int k = 0; k < E; k += 2) {
                            float2 v = __ffma2_rn(make_float2(Dd, Dd), make_float2(xv[k], xv[k + 1]),
                                                  make_float2(ys[k], ys[k + 1]));
                            if constexpr (kZ) v = __fmul2_rn(v, make_float2(gate<T>(zv[k]), gate<T>(zv[k + 1])));
                            ys[k] = v.x; ys[k + 1] = v.y;
                        }
                    } else {
                        float v = fmaf(Dd, xv[0], ys[0]);
                        if constexpr (kZ) v *= gate<T>(zv[0]);
                        ys[0] = v;
                    }
                    const int64_t gidx = (row0 + cl) * L + t0 + ce;
                    const int nv = tvalid - ce;
                    if (nv >= E) {
                        storeE<T, E>(p.y, gidx, vec, ys);
                    } else {
#pragma unroll
                        for (int k = 0; k < E; ++k)
                            if (k < nv) Io<T>::st(p.y, gidx + k, ys[k]);
                    }
                }
            }
            __syncwarp();
        }
        if (lane == 0) mbar_arrive(&empty[st]);
    }

    if (!dok) return;
    if constexpr (MODE == kTotals) {
#pragma unroll
        for (int q = 0; q < S / 2; ++q) {
            const int n = g * S + 2 * q;
            float *dst = sg.ws_h + ((int64_t)seg * nchan + chan0 + d) * N;
            if (n < N) dst[n] = h2[q].x;
            if (n + 1 < N) dst[n + 1] = h2[q].y;
        }
        if (g == 0) sg.ws_s[(int64_t)seg * nchan + chan0 + d] = dsum;
    } else {
        if (p.final_state && seg == sg.nseg - 1) {
#pragma unroll
            for (int q = 0; q < S / 2; ++q) {
                const int n = g * S + 2 * q;
                float *dst = p.final_state + (chan0 + d) * N;
                if (n < N) dst[n] = h2[q].x;
                if (n + 1 < N) dst[n + 1] = h2[q].y;
            }
        }
    }
}

// Launch one instantiation.
template <typename T, int NP, int S, int NW, bool GATE, int MODE, bool TMA>
cudaError_t launch_one(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps, unsigned int *status,
                       cudaStream_t st) {
    using Ly = Layout<T, NP, S, NW, GATE, MODE>;
    auto kern = scan_kernel<T, NP, S, NW, GATE, MODE, TMA>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Ly::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.dim + Ly::DT - 1) / Ly::DT), (unsigned)a.batch, (unsigned)sg.nseg);
    kern<<<grid, Ly::NT, Ly::bytes, st>>>(a, sg, maps, status);
    return cudaGetLastError();
}

// Instantiation dispatch for one I/O type (defined in scan_fused_<type>.cu).
template <typename T>
cudaError_t launch_typed(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps, unsigned int *status,
                         int mode, bool tma, int cfg, cudaStream_t st);

}  // namespace fused
}  // namespace ssm
