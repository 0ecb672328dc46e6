// FUSED and TWOPASS variants: channel-parallel, time-serial forward selective
// scan, optionally cut into sequence segments that are combined through a
// small scan over the segment totals.
//
// "Mamba hardware-aware parallel associative scan" (pwwt.cn/news/6375169):
//   sect. 2.2, third approach -- parallelism over channels; each thread owns
//     part of one channel's state in registers and walks the sequence in order;
//   sect. 2.2 / 3.3 -- two-pass chunk carry: per-chunk totals (A_k, B_k), a
//     scan over the K totals (O(log K) depth), then a fix-up pass;
//   sect. 4.1 -- discretisation, scan, C contraction, D skip and gate in one
//     kernel; neither (a, b) nor h_t is written to global memory
//     ("Mamba (part 2)", scwacadex.pages.dev, sect. 4.1-4.2).
//
// CTA = (channel tile of DT channels, batch b, sequence segment).  Each
// channel's NP (padded) states are split over NS = NP / S threads, S states
// per thread.  The CTA walks its segment in tiles of kTC steps.  Per tile:
//   1. stage   : x, delta, z, B, C of the tile are read from global memory
//                (coalesced along t) into shared memory; Delta = softplus(
//                delta + dt_bias) and u = Delta * x are computed once per
//                element; B and C are stored transposed as [t][group][S].
//   2. scan    : every thread runs its S recurrences through the tile:
//                a = 2^(Delta * A * log2 e), h = a * h + u * B, and writes the
//                partial contraction sum_s C * h of every step.
//   3. epilogue: the NS partial sums of each (channel, step) are added, the
//                skip D * x and the gate silu(z) are applied and y is stored.
// Padding is the identity step (1, 0): states n >= dstate have A = B = C = 0,
// steps t >= L and channels d >= dim have Delta = u = 0, so they leave h
// unchanged and contribute nothing.
//
// Modes: kWhole -- one segment, y and final state;  kTotals -- pass 1 of the
// two-pass variant: start from h = 0, skip y, write the segment's state h_end
// (= B_k) and the segment's sum of Delta (A_k[n] = exp(A[d,n] * sum Delta));
// kSeeded -- pass 2: start from the carried state h_init of the segment and
// write y (and the final state from the last segment).
#include "scan_internal.h"
#include "scan_device.cuh"

namespace ssm {
namespace {

template <int NP> struct FusedCfg;
template <> struct FusedCfg<8>  { static constexpr int S = 2, DT = 32; };
template <> struct FusedCfg<16> { static constexpr int S = 4, DT = 32; };
template <> struct FusedCfg<32> { static constexpr int S = 8, DT = 32; };
template <> struct FusedCfg<64> { static constexpr int S = 8, DT = 16; };

constexpr int kTC = 64;          // steps per tile
constexpr int kRow = kTC + 1;    // padded shared row (bank-conflict free)

enum Mode { kWhole = 0, kTotals = 1, kSeeded = 2 };

struct SegArgs {
    int64_t seg_len;   // steps per segment (the last one may be shorter)
    int nseg;          // number of segments
    float *ws_h;       // [nseg][batch*dim][dstate]: B_k after pass 1, h_init after the small scan
    float *ws_s;       // [nseg][batch*dim]: sum of Delta over the segment
};

template <int NP>
constexpr size_t fused_smem_bytes() {
    constexpr int S = FusedCfg<NP>::S, DT = FusedCfg<NP>::DT, NS = NP / S;
    // Delta, u, x, z rows + B/C tile + partial sums
    return sizeof(float) * (size_t)(4 * DT * kRow + kTC * NS * 2 * S + DT * NS * kRow);
}

template <typename T, int NP, bool GATE, int MODE>
__global__ void __launch_bounds__(FusedCfg<NP>::DT * (NP / FusedCfg<NP>::S))
fused_scan_kernel(FwdArgs p, SegArgs sg) {
    constexpr int S = FusedCfg<NP>::S;
    constexpr int DT = FusedCfg<NP>::DT;
    constexpr int NS = NP / S;
    constexpr int NT = DT * NS;
    constexpr bool kWriteY = MODE != kTotals;

    extern __shared__ float smem[];
    float *dsm = smem;                    // [DT][kRow] Delta
    float *usm = dsm + DT * kRow;         // [DT][kRow] Delta * x
    float *xsm = usm + DT * kRow;         // [DT][kRow] x
    float *zsm = xsm + DT * kRow;         // [DT][kRow] z
    float *bcs = zsm + DT * kRow;         // [kTC][NS][2S] B then C
    float *ysm = bcs + kTC * NS * 2 * S;  // [DT*NS][kRow] partial sums

    const int tid = threadIdx.x;
    const int g = tid % NS;               // state group of this thread
    const int dl = tid / NS;              // channel within the CTA
    const int b = blockIdx.y;
    const int seg = blockIdx.z;
    const int d0 = blockIdx.x * DT;
    const int d = d0 + dl;
    const int dim = p.dim, N = p.dstate;
    const int64_t L = p.L;
    const int64_t ts = (int64_t)seg * sg.seg_len;
    const int64_t te = (ts + sg.seg_len < L) ? ts + sg.seg_len : L;

    const int64_t chan0 = (int64_t)b * dim;      // first channel row of this batch
    const int64_t brow0 = (int64_t)b * N;        // first B/C row of this batch
    const int64_t nchan = (int64_t)p.batch * dim;

    float h[S], a2[S];
#pragma unroll
    for (int s = 0; s < S; ++s) {
        const int n = g * S + s;
        const bool ok = d < dim && n < N;
        a2[s] = ok ? p.A[(int64_t)d * N + n] * kLog2e : 0.0f;
        h[s] = 0.0f;
        if (MODE == kSeeded && ok) h[s] = sg.ws_h[((int64_t)seg * nchan + chan0 + d) * N + n];
    }
    float dsum = 0.0f;   // sum of Delta over the segment (pass 1)

    for (int64_t t0 = ts; t0 < te; t0 += kTC) {
        // ---- 1. stage the tile ------------------------------------------
        for (int e = tid; e < DT * kTC; e += NT) {
            const int r = e / kTC, c = e % kTC;
            const int dd = d0 + r;
            const int64_t t = t0 + c;
            float Delta = 0.0f, u = 0.0f, xv = 0.0f, zv = 0.0f;
            if (dd < dim && t < te) {
                const int64_t idx = (chan0 + dd) * L + t;
                xv = Io<T>::ld(p.x, idx);
                const float bias = p.dt_bias ? __ldg(p.dt_bias + dd) : 0.0f;
                Delta = step_delta(Io<T>::ld(p.delta, idx), bias, p.softplus);
                u = Delta * xv;
                if (GATE && kWriteY) zv = Io<T>::ld(p.z, idx);
            }
            dsm[r * kRow + c] = Delta;
            usm[r * kRow + c] = u;
            xsm[r * kRow + c] = xv;
            zsm[r * kRow + c] = zv;
        }
        for (int e = tid; e < NP * kTC; e += NT) {
            const int n = e / kTC, c = e % kTC;
            const int64_t t = t0 + c;
            float bv = 0.0f, cv = 0.0f;
            if (n < N && t < te) {
                const int64_t idx = (brow0 + n) * L + t;
                bv = Io<T>::ld(p.B, idx);
                if (kWriteY) cv = Io<T>::ld(p.C, idx);
            }
            float *dst = bcs + (c * NS + n / S) * 2 * S + n % S;
            dst[0] = bv;
            dst[S] = cv;
        }
        __syncthreads();

        // ---- 2. scan the tile -------------------------------------------
        {
            const float *dr = dsm + dl * kRow;
            const float *ur = usm + dl * kRow;
            float *yr = ysm + tid * kRow;
#pragma unroll 4
            for (int c = 0; c < kTC; ++c) {
                const float Delta = dr[c];
                const float u = ur[c];
                const float *bc = bcs + (c * NS + g) * 2 * S;
                float acc = 0.0f;
#pragma unroll
                for (int s = 0; s < S; ++s) {
                    const float a = ex2(Delta * a2[s]);
                    h[s] = fmaf(a, h[s], u * bc[s]);
                    if (kWriteY) acc = fmaf(bc[S + s], h[s], acc);
                }
                if (kWriteY) yr[c] = acc;
                else dsum += Delta;
            }
        }
        __syncthreads();

        // ---- 3. epilogue: reduce partials, skip, gate, store --------------
        if (kWriteY) {
            for (int e = tid; e < DT * kTC; e += NT) {
                const int r = e / kTC, c = e % kTC;
                const int dd = d0 + r;
                const int64_t t = t0 + c;
                if (dd < dim && t < te) {
                    float yv = 0.0f;
#pragma unroll
                    for (int q = 0; q < NS; ++q) yv += ysm[(r * NS + q) * kRow + c];
                    const float xv = xsm[r * kRow + c];
                    if (p.D) yv = fmaf(__ldg(p.D + dd), xv, yv);
                    if (GATE) yv *= silu_f(zsm[r * kRow + c]);
                    Io<T>::st(p.y, (chan0 + dd) * L + t, yv);
                }
            }
            __syncthreads();
        }
    }

    if (d >= dim) return;
    if (MODE == kTotals) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int n = g * S + s;
            if (n < N) sg.ws_h[((int64_t)seg * nchan + chan0 + d) * N + n] = h[s];
        }
        if (g == 0) sg.ws_s[(int64_t)seg * nchan + chan0 + d] = dsum;
    } else if (p.final_state && seg == sg.nseg - 1) {
#pragma unroll
        for (int s = 0; s < S; ++s) {
            const int n = g * S + s;
            if (n < N) p.final_state[(chan0 + d) * N + n] = h[s];
        }
    }
}

// Small scan over the segment totals ("Mamba hardware-aware parallel
// associative scan", sect. 3.3, second method), one warp per (channel, state):
// the segment pairs (A_k, B_k) = (exp(A * sum Delta_k), h_end_k) are composed
// with a warp-shuffle Hillis-Steele scan, 32 segments per round, the running
// state carried from round to round.  On return ws_h[k] holds the state at the
// start of segment k (h_init^(k); h_init^(0) = 0), which pass 2 starts from:
//   h_init^(k) = A_{k-1} * h_init^(k-1) + B_{k-1}.
__global__ void segment_carry_kernel(const float *__restrict__ A, float *ws_h,
                                     const float *__restrict__ ws_s, int64_t nchan,
                                     int dim, int N, int nseg) {
    const int lane = threadIdx.x & 31;
    const int64_t pair = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (pair >= nchan * N) return;                 // whole warp leaves together
    const int64_t ch = pair / N;
    const int n = (int)(pair % N);
    const float a2 = A[(int64_t)(ch % dim) * N + n] * kLog2e;
    float carry = 0.0f;                             // h_init of the first segment of the round
    for (int k0 = 0; k0 < nseg; k0 += 32) {
        const int k = k0 + lane;
        float Ak = 1.0f, Bk = 0.0f;                 // identity pads the last round
        if (k < nseg - 1) {                         // the last segment's total is never needed
            Ak = ex2(a2 * ws_s[(int64_t)k * nchan + ch]);
            Bk = ws_h[((int64_t)k * nchan + ch) * N + n];
        }
        // inclusive Hillis-Steele scan over the lanes: x_i <- x_i o x_{i-off}
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float Ap = __shfl_up_sync(0xffffffffu, Ak, off);
            const float Bp = __shfl_up_sync(0xffffffffu, Bk, off);
            if (lane >= off) {
                Bk = fmaf(Ak, Bp, Bk);
                Ak = Ak * Ap;
            }
        }
        // state after segment k, then shift by one lane for the start states
        const float hend = fmaf(Ak, carry, Bk);
        float hstart = __shfl_up_sync(0xffffffffu, hend, 1);
        if (lane == 0) hstart = carry;
        if (k < nseg) ws_h[((int64_t)k * nchan + ch) * N + n] = hstart;
        carry = __shfl_sync(0xffffffffu, hend, 31);
    }
}

template <typename T, int NP, bool GATE, int MODE>
cudaError_t launch_mode(const FwdArgs &a, const SegArgs &sg, cudaStream_t st) {
    constexpr int S = FusedCfg<NP>::S, DT = FusedCfg<NP>::DT, NS = NP / S;
    constexpr size_t smem = fused_smem_bytes<NP>();
    auto kern = fused_scan_kernel<T, NP, GATE, MODE>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.dim + DT - 1) / DT), (unsigned)a.batch, (unsigned)sg.nseg);
    kern<<<grid, DT * NS, smem, st>>>(a, sg);
    return cudaGetLastError();
}

template <int MODE, typename T, bool GATE>
cudaError_t launch_t(const FwdArgs &a, const SegArgs &sg, cudaStream_t st) {
    if (a.dstate <= 8) return launch_mode<T, 8, GATE, MODE>(a, sg, st);
    if (a.dstate <= 16) return launch_mode<T, 16, GATE, MODE>(a, sg, st);
    if (a.dstate <= 32) return launch_mode<T, 32, GATE, MODE>(a, sg, st);
    return launch_mode<T, 64, GATE, MODE>(a, sg, st);
}

template <int MODE>
cudaError_t launch_any(const FwdArgs &a, const SegArgs &sg, cudaStream_t st) {
    const bool gate = a.z != nullptr;
    if constexpr (MODE == kTotals) {   // pass 1 never reads z
        return a.bf16 ? launch_t<MODE, __nv_bfloat16, false>(a, sg, st)
                      : launch_t<MODE, float, false>(a, sg, st);
    } else {
        if (a.bf16) return gate ? launch_t<MODE, __nv_bfloat16, true>(a, sg, st)
                                : launch_t<MODE, __nv_bfloat16, false>(a, sg, st);
        return gate ? launch_t<MODE, float, true>(a, sg, st) : launch_t<MODE, float, false>(a, sg, st);
    }
}

}  // namespace

cudaError_t launch_fused(const FwdArgs &a, cudaStream_t st) {
    SegArgs sg{a.L, 1, nullptr, nullptr};
    return launch_any<kWhole>(a, sg, st);
}

int64_t twopass_chunk_len(int batch, int dim, int dstate, int64_t L) {
    // Enough segments that the CTAs of one pass fill every SM several times,
    // while each segment keeps at least 8 tiles of work.
    const int np = dstate <= 8 ? 8 : dstate <= 16 ? 16 : dstate <= 32 ? 32 : 64;
    const int dt = np == 64 ? 16 : 32;
    const int64_t ctas = (int64_t)batch * ((dim + dt - 1) / dt);
    const int64_t want_ctas = 152 * 8;
    int64_t nseg = (want_ctas + ctas - 1) / (ctas > 0 ? ctas : 1);
    const int64_t max_seg = (L + 8 * kTC - 1) / (8 * kTC);
    if (nseg > max_seg) nseg = max_seg;
    if (nseg < 1) nseg = 1;
    int64_t len = (L + nseg - 1) / nseg;
    len = (len + kTC - 1) / kTC * kTC;    // whole tiles
    return len > 0 ? len : kTC;
}

size_t twopass_workspace_bytes(int batch, int dim, int dstate, int64_t L) {
    const int64_t len = twopass_chunk_len(batch, dim, dstate, L);
    const int64_t nseg = L > 0 ? (L + len - 1) / len : 1;
    const int64_t nchan = (int64_t)batch * dim;
    size_t h = (size_t)nseg * nchan * dstate * sizeof(float);
    h = (h + 255) / 256 * 256;
    size_t s = (size_t)nseg * nchan * sizeof(float);
    s = (s + 255) / 256 * 256;
    return h + s;
}

cudaError_t launch_twopass(const FwdArgs &a, void *workspace, cudaStream_t st) {
    const int64_t len = twopass_chunk_len(a.batch, a.dim, a.dstate, a.L);
    const int nseg = (int)((a.L + len - 1) / len);
    const int64_t nchan = (int64_t)a.batch * a.dim;
    size_t hbytes = (size_t)nseg * nchan * a.dstate * sizeof(float);
    hbytes = (hbytes + 255) / 256 * 256;
    SegArgs sg{len, nseg, static_cast<float *>(workspace),
               reinterpret_cast<float *>(static_cast<char *>(workspace) + hbytes)};
    cudaError_t e = cudaSuccess;
    if (nseg > 1) {   // pass 1 over every segment but the last (its total is never used)
        SegArgs s1 = sg;
        s1.nseg = nseg - 1;
        e = launch_any<kTotals>(a, s1, st);
        if (e != cudaSuccess) return e;
    }
    const int64_t pairs = nchan * a.dstate;
    const int wpb = 8;
    segment_carry_kernel<<<(unsigned)((pairs + wpb - 1) / wpb), wpb * 32, 0, st>>>(
        a.A, sg.ws_h, sg.ws_s, nchan, a.dim, a.dstate, nseg);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_any<kSeeded>(a, sg, st);
}

}  // namespace ssm
