// Channel-parallel, time-serial forward selective scan (FUSED variant, both
// passes of the TWOPASS variant, and the backward's chunk-start states).
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
// Data flow.  A pre-pass (bc_prepare_kernel) writes B and C once per call as
// float32 rows [batch*L][NS][B(S) C(S) pad] -- per step, per state group,
// the group's S values of B then of C, zero for padded states, and for groups
// of 128 bytes 16 bytes of padding so that the groups of one step fall in
// different shared-memory banks -- so that the scan reads each lane's B and C
// for a step with 16-byte loads, conflict free and without conversion.  The scan CTA has NW consumer warps and one producer warp.
//   producer : per tile of TC steps, waits for the ring stage to be free and
//              issues 2-D TMA copies of x, delta, z (the CTA's DT channel
//              rows) and of the prepared B/C rows, completing on the stage's
//              `full` mbarrier (or, for rows that are not 16-byte aligned,
//              loads the tile element by element).
//   consumers: a consumer warp owns CPW = 32 / NS channels, each channel's NP
//              (padded) states split over NS lanes, S per lane.  Per block of
//              KB steps (32 when a lane holds at most 4 states, else 16):
//                1. the lane that owns KB / NS consecutive steps of its
//                   channel forms Delta = softplus(delta + dt_bias) and
//                   u = Delta * x for them (packed f32x2, in registers);
//                2. every lane advances its S recurrences through the block
//                   with packed f32x2 arithmetic, a = 2^(Delta * A log2 e),
//                   h = a h + u B, partial y = sum_s C h, receiving each
//                   step's Delta and u from the owner lane by a shuffle;
//                3. a shuffle reduce-scatter over the NS lanes leaves each
//                   owner lane the full contraction of its own steps, which it
//                   finishes with the skip D x and the gate silu(z) and stores.
//              After a tile each consumer warp arrives on the stage's `empty`
//              mbarrier.
// Padding is the identity step (1, 0): states n >= dstate have A = B = C = 0,
// steps t >= L and channels d >= dim have Delta = u = 0.  Every mbarrier wait
// is bounded; a wait that gives up flags the status word and the CTA stops.
#pragma once

#include "scan_internal.h"
#include "scan_device.cuh"
#include "scan_tma.cuh"

namespace ssm {
namespace fused {

constexpr int kNST = 4;            // TMA ring depth

// Steps per tile (TMA box width): 32, or 16 for wide states so that the
// ring's B/C tiles stay small.
__host__ __device__ constexpr int tile_steps(int np) { return np >= 32 ? 16 : 32; }

// Steps per block, the register working set of one round of the three
// phases: fewer block boundaries pay where a lane holds few states, while
// wider lanes keep 16 to stay within the register budget of 4 CTAs per SM.
__host__ __device__ constexpr int blk_steps(int S) { return S <= 4 ? 32 : 16; }

// Consumer warps per CTA (plus one producer warp).  Lanes with 16 states need
// about 160 registers, so 4 CTAs of 2 consumer warps no longer fit on an SM
// and 3 CTAs of 3 hold more of them at once; narrower lanes fit 4 or 5 CTAs of
// 2, the finer grain.
__host__ __device__ constexpr int consumer_warps(int S) { return S >= 16 ? 3 : 2; }

// kWhole: y (and the final state) over whole sequences; kTotals: per-segment
// totals of the two-pass variant, no y; kSeeded: y from each segment's start
// state; kStates: no y, the state at the start of every ck_len-step chunk.
enum Mode { kWhole = 0, kTotals = 1, kSeeded = 2, kStates = 3 };

struct SegArgs {
    int64_t seg_len;   // steps per segment (the last one may be shorter)
    int nseg;          // number of segments in this launch
    float *ws_h;       // [nseg][batch*dim][dstate]: B_k after pass 1, h_init after the small scan
    float *ws_s;       // [nseg][batch*dim]: sum of Delta over the segment
    const float *bc;   // prepared B/C rows [batch*L][bc_row(NP, S)]
    int64_t ck_len;    // kStates, or kWhole/kSeeded with checkpoints (FwdArgs::ckpt): steps per chunk
                       // (whole tiles); the states are then [nchunk][batch*dim][dstate] (kStates: in ws_h)
};

// Floats per prepared B/C row: NS groups of S B values and S C values.  A
// group of 128 bytes or more (S >= 16) gets 16 bytes of padding so that the
// groups of one step start in different shared-memory banks; smaller groups
// already do.
__host__ __device__ constexpr int bc_group(int S) { return 2 * S + (S >= 16 ? 4 : 0); }
__host__ __device__ constexpr int bc_row(int NP, int S) { return (NP / S) * bc_group(S); }
// The widest row over the configurations.
__host__ __device__ constexpr int bc_row_max(int NP) { return 2 * NP + 16; }

struct TileMaps {
    CUtensorMap x, dl, z, bc;
};

__host__ __device__ constexpr size_t align128(size_t n) { return (n + 127) / 128 * 128; }

// CK: taps of the causal convolution fused in front of the scan (0: none).
template <typename T, int NP, int S, int NW, bool GATE, int MODE, int CK = 0>
struct Layout {
    static constexpr int NS = NP / S;            // lanes per channel
    static constexpr int CPW = 32 / NS;          // channels per consumer warp
    static constexpr int DT = NW * CPW;          // channels per CTA
    static constexpr int NT = (NW + 1) * 32;     // consumers + producer
    static constexpr int KB = blk_steps(S);      // steps per block
    static constexpr int E = KB / NS;            // steps each lane owns per block
    static constexpr int TC = tile_steps(NP);
    static constexpr bool kY = MODE == kWhole || MODE == kSeeded;
    static constexpr bool kZ = GATE && kY;
    static constexpr size_t row_bytes = (size_t)DT * TC * sizeof(T);
    static constexpr int BCW = bc_row(NP, S);    // floats per prepared B/C row
    static constexpr size_t bc_bytes = (size_t)TC * BCW * 4;
    // tiles of 128-byte rows (float32) are copied with the 128-byte swizzle,
    // tiles of 64-byte rows (bf16) with the 64-byte swizzle (tile_byte);
    // their buffers start on 1024-byte boundaries
    static constexpr int kSWZ = TC * (int)sizeof(T) == 128 ? 128 : TC * (int)sizeof(T) == 64 ? 64 : 0;
    static constexpr bool kSW = kSWZ != 0;
    static constexpr size_t kAl = kSW ? 1024 : 128;
    static constexpr size_t al(size_t n) { return (n + kAl - 1) / kAl * kAl; }
    // one ring stage
    static constexpr size_t off_x = 0;
    static constexpr size_t off_dl = al(row_bytes);
    static constexpr size_t off_z = off_dl + al(row_bytes);
    static constexpr size_t off_bc = off_z + (kZ ? al(row_bytes) : 0);
    static constexpr size_t stage_bytes = off_bc + al(bc_bytes);
    static constexpr uint32_t tx_bytes = (uint32_t)(row_bytes * (kZ ? 3 : 2) + bc_bytes);
    // convolution history: the last CK raw inputs of every channel before the
    // current tile (float, [DT][CK])
    static constexpr size_t off_halo = kNST * stage_bytes;
    static constexpr size_t halo_bytes = CK > 0 ? align128((size_t)DT * CK * 4) : 0;
    static constexpr size_t off_bar = off_halo + halo_bytes;
    // (plus room to align the base of a swizzled layout)
    static constexpr size_t bytes = off_bar + 2 * kNST * 8 + 16 + (kSW ? 1024 : 0);
};

// Byte offset of element (row r, column c) of a staged x, delta or z tile of
// TC columns, the tile on a 1024-byte boundary.  The swizzled copies XOR the
// 16-byte chunk bits of an offset with the bits above the 128-byte line: the
// 128-byte mode bits 4-6 with bits 7-9 (a 128-byte row r stores chunk j at
// j ^ (r mod 8)), the 64-byte mode bits 4-5 with bits 7-8 (a 64-byte row r
// stores chunk j at j ^ ((r / 2) mod 4)).  The same column of consecutive
// rows then falls in different bank groups.
template <typename T, int TC, bool SW>
__device__ __forceinline__ int tile_byte(int r, int c) {
    constexpr int row = TC * (int)sizeof(T);
    const int off = (r * TC + c) * (int)sizeof(T);
    if constexpr (SW && row == 128) return off ^ (((off >> 7) & 7) << 4);
    if constexpr (SW && row == 64) return off ^ (((off >> 7) & 3) << 4);
    return off;
}

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

// E consecutive raw elements starting at element idx (idx * sizeof(T) aligned
// to min(E * sizeof(T), 16)).
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
        if constexpr (E % 8 == 0) {
#pragma unroll
            for (int k = 0; k < E; k += 8) {
                const uint4 w = *reinterpret_cast<const uint4 *>(p + 2 * k);
                const uint32_t ws[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    v[k + 2 * i] = __uint_as_float(ws[i] << 16);
                    v[k + 2 * i + 1] = __uint_as_float(ws[i] & 0xffff0000u);
                }
            }
        } else if constexpr (E == 4) {
            const uint2 w = *reinterpret_cast<const uint2 *>(p);
            v[0] = __uint_as_float(w.x << 16); v[1] = __uint_as_float(w.x & 0xffff0000u);
            v[2] = __uint_as_float(w.y << 16); v[3] = __uint_as_float(w.y & 0xffff0000u);
        } else if constexpr (E == 2) {
            const uint32_t w = *reinterpret_cast<const uint32_t *>(p);
            v[0] = __uint_as_float(w << 16); v[1] = __uint_as_float(w & 0xffff0000u);
        } else {
            v[0] = raw1<T>(base, idx);
        }
    }
}

// E consecutive elements of row r from column c (c * sizeof(T) aligned to
// min(E * sizeof(T), 16)) of a staged tile; every 16-byte chunk is contiguous
// in the swizzled layout too.
template <typename T, int E, int TC, bool SW>
__device__ __forceinline__ void rowE(const unsigned char *tile, int r, int c, float (&v)[E]) {
    if constexpr (!SW) {
        rawE<T, E>(tile, r * TC + c, v);
    } else if constexpr (sizeof(T) == 4) {
        if constexpr (E % 4 == 0) {
#pragma unroll
            for (int k = 0; k < E; k += 4) {
                const float4 q = *reinterpret_cast<const float4 *>(tile + tile_byte<T, TC, SW>(r, c + k));
                v[k] = q.x; v[k + 1] = q.y; v[k + 2] = q.z; v[k + 3] = q.w;
            }
        } else if constexpr (E == 2) {
            const float2 q = *reinterpret_cast<const float2 *>(tile + tile_byte<T, TC, SW>(r, c));
            v[0] = q.x; v[1] = q.y;
        } else {
            v[0] = *reinterpret_cast<const float *>(tile + tile_byte<T, TC, SW>(r, c));
        }
    } else {
        // bf16: 16-byte chunks of 8 elements, or a piece of one chunk
        if constexpr (E % 8 == 0) {
#pragma unroll
            for (int k = 0; k < E; k += 8) {
                float w[8];
                rawE<T, 8>(tile + tile_byte<T, TC, SW>(r, c + k), 0, w);
#pragma unroll
                for (int i = 0; i < 8; ++i) v[k + i] = w[i];
            }
        } else {
            rawE<T, E>(tile + tile_byte<T, TC, SW>(r, c), 0, v);
        }
    }
}

template <typename T, int TC, bool SW>
__device__ __forceinline__ float row1(const unsigned char *tile, int r, int c) {
    if constexpr (!SW) return raw1<T>(tile, r * TC + c);
    return raw1<T>(tile + tile_byte<T, TC, SW>(r, c), 0);
}

// Store E consecutive outputs at global index idx (all in range).
template <typename T, int E>
__device__ __forceinline__ void storeE(void *y, int64_t idx, bool vec, const float (&v)[E]) {
    if constexpr (sizeof(T) == 4) {
        float *p = static_cast<float *>(y) + idx;
        if (vec && E % 4 == 0) {
#pragma unroll
            for (int k = 0; k < E; k += 4)
                *reinterpret_cast<float4 *>(p + k) = make_float4(v[k], v[k + 1], v[k + 2], v[k + 3]);
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
            if (vec && E % 8 == 0) {
#pragma unroll
                for (int k = 0; k < E / 2; k += 4)
                    *reinterpret_cast<uint4 *>(p + 2 * k) = make_uint4(w[k], w[k + 1], w[k + 2], w[k + 3]);
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

// B and C of one batch, [NP rows][L] in the I/O type, re-laid out as float32
// rows [batch*L][NS][B(S) C(S) pad] with zeros for states n >= dstate and for
// the padding.  One CTA per (32 steps, batch): coalesced reads along t,
// shared-memory transpose, coalesced row writes.
template <typename T, int NP, int S>
__global__ void __launch_bounds__(256) bc_prepare_kernel(const void *Bm, const void *Cm, float *out, int N,
                                                         int64_t L) {
    constexpr int R = bc_row(NP, S);                  // floats per output row
    constexpr int G = bc_group(S);
    __shared__ float tile[32][R + 1];
    const int b = blockIdx.y;
    const int64_t t0 = (int64_t)blockIdx.x * 32;
    for (int e = threadIdx.x; e < 32 * (R + 1); e += blockDim.x) (&tile[0][0])[e] = 0.0f;
    __syncthreads();
    for (int e = threadIdx.x; e < 2 * NP * 32; e += blockDim.x) {
        const int c = e % 32, r = e / 32;             // r: 0..NP-1 B rows, NP..2NP-1 C rows
        const int n = r % NP;
        const bool isC = r >= NP;
        const int64_t t = t0 + c;
        float v = 0.0f;
        if (n < N && t < L) v = Io<T>::ld(isC ? Cm : Bm, ((int64_t)b * N + n) * L + t);
        // destination column inside the output row: group n / S, slot n % S (+S for C)
        tile[c][(n / S) * G + (isC ? S : 0) + n % S] = v;
    }
    __syncthreads();
    for (int e = threadIdx.x; e < 32 * R; e += blockDim.x) {
        const int c = e / R, k = e % R;
        const int64_t t = t0 + c;
        if (t < L) out[((int64_t)b * L + t) * R + k] = tile[c][k];
    }
}

// Reduce-scatter of per-step partial sums over the lanes of a channel.  In
// the round with xor distance M a lane keeps the half of its current LEN*2
// steps selected by bit M of its group index and sends the other half, so
// after log2(NS) rounds v[0..E) holds the full sums of the lane's own steps.
// Template recursion keeps every index a compile-time constant (registers).
template <int LEN, int M>
struct ReduceScatter {
    template <int NV>
    static __device__ __forceinline__ void run(float (&v)[NV], int g) {
        const bool hi = (g & M) != 0;
#pragma unroll
        for (int k = 0; k < LEN; ++k) {
            const float send = hi ? v[k] : v[LEN + k];
            const float keep = hi ? v[LEN + k] : v[k];
            v[k] = keep + __shfl_xor_sync(0xffffffffu, send, M);
        }
        ReduceScatter<LEN / 2, M / 2>::run(v, g);
    }
};
template <int LEN>
struct ReduceScatter<LEN, 0> {
    template <int NV>
    static __device__ __forceinline__ void run(float (&)[NV], int) {}
};

// CKPT: the forward also stores its checkpoints (FwdArgs::ckpt), the state at
// the start of every kCkptSteps-step chunk; separate instantiations, so that
// the plain forward carries none of it.  Those keep 16-state lanes at 3 CTAs
// per SM, as the plain kernel's registers allow.
template <typename T, int NP, int S, int NW, bool GATE, int MODE, bool TMA, int CK = 0, bool CKPT = false>
__global__ void __launch_bounds__((NW + 1) * 32, (CKPT && S >= 16) ? 3 : 1)
scan_kernel(const FwdArgs p, const SegArgs sg, const __grid_constant__ TileMaps maps, unsigned int *status) {
    using Ly = Layout<T, NP, S, NW, GATE, MODE, CK>;
    static_assert(CK == 0 || (MODE == kWhole && CK <= 4), "the convolution runs with whole sequences");
    static_assert(!CKPT || ((MODE == kWhole || MODE == kSeeded) && CK == 0), "checkpoints of the y passes");
    constexpr int NS = Ly::NS, CPW = Ly::CPW, DT = Ly::DT, E = Ly::E, TC = Ly::TC;
    constexpr bool kY = Ly::kY, kZ = Ly::kZ;
    static_assert(S % 2 == 0 && (NS == 1 || NS == 2 || NS == 4 || NS == 8), "lane split");
    constexpr int KB = Ly::KB;
    static_assert(E % 2 == 0 && TC % KB == 0, "block split");
    constexpr unsigned FULL = 0xffffffffu;

    extern __shared__ __align__(128) unsigned char smem_raw[];
    unsigned char *smem = smem_raw;
    if constexpr (Ly::kSW) smem += (1024u - (smem_u32(smem_raw) & 1023u)) & 1023u;
    constexpr bool SW = Ly::kSW;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Ly::off_bar);
    uint64_t *empty = full + kNST;
    int *abort_flag = reinterpret_cast<int *>(empty + kNST);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int dim = p.dim, N = p.dstate;
    const int b = blockIdx.y;
    const int seg = blockIdx.z;
    const int d0 = blockIdx.x * DT;
    const int64_t L = p.L;
    const int64_t ts = (int64_t)seg * sg.seg_len;
    const int64_t te = (ts + sg.seg_len < L) ? ts + sg.seg_len : L;
    const int ntiles = (int)((te - ts + TC - 1) / TC);
    const int64_t chan0 = (int64_t)b * dim;
    const int64_t nchan = (int64_t)p.batch * dim;
    const int64_t row0 = chan0 + d0;                  // first x/delta/z row of this CTA
    const int nw_live = (dim - d0 + CPW - 1) / CPW < NW ? (dim - d0 + CPW - 1) / CPW : NW;   // consumer warps with channels

    if (threadIdx.x == 0) {
        for (int s = 0; s < kNST; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], nw_live);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    if (warp == NW) {
        // ------------------------------------------------------------ producer
        int issued = 0;
        for (int tile = 0; tile < ntiles; ++tile) {
            const int st = tile % kNST;
            const uint32_t ph = (uint32_t)((tile / kNST) & 1);
            unsigned char *base = smem + st * Ly::stage_bytes;
            const int64_t t0 = ts + (int64_t)tile * TC;
            const int tvalid = (int)((te - t0) < TC ? (te - t0) : TC);
            const bool ok = tile < kNST || wait_parity(&empty[st], ph ^ 1u, status);
            if (!__all_sync(FULL, ok)) { *abort_flag = 1; break; }
            if constexpr (TMA) {
                if (lane == 0) {
                    fence_proxy_async();
                    mbar_arrive_expect_tx(&full[st], Ly::tx_bytes);
                    const int tc = (int)t0, r0 = (int)row0, rb = (int)((int64_t)b * L + t0);
                    tma_load_2d(base + Ly::off_x, &maps.x, tc, r0, &full[st]);
                    tma_load_2d(base + Ly::off_dl, &maps.dl, tc, r0, &full[st]);
                    if constexpr (kZ) tma_load_2d(base + Ly::off_z, &maps.z, tc, r0, &full[st]);
                    tma_load_2d(base + Ly::off_bc, &maps.bc, 0, rb, &full[st]);
                }
                issued = tile + 1;
            } else {
                // element loads; zeros outside the problem
                for (int e = lane; e < DT * TC; e += 32) {
                    const int r = e / TC, c = e % TC;
                    const bool in = d0 + r < dim && c < tvalid;
                    const int64_t idx = (row0 + r) * L + t0 + c;
                    T xv = T(0.0f), dv = T(0.0f), zv = T(0.0f);
                    if (in) {
                        xv = static_cast<const T *>(p.x)[idx];
                        dv = static_cast<const T *>(p.delta)[idx];
                        if constexpr (kZ) zv = static_cast<const T *>(p.z)[idx];
                    }
                    const int tb = tile_byte<T, TC, SW>(r, c);
                    *reinterpret_cast<T *>(base + Ly::off_x + tb) = xv;
                    *reinterpret_cast<T *>(base + Ly::off_dl + tb) = dv;
                    if constexpr (kZ) *reinterpret_cast<T *>(base + Ly::off_z + tb) = zv;
                }
                float *bcs = reinterpret_cast<float *>(base + Ly::off_bc);
                for (int e = lane; e < TC * Ly::BCW; e += 32) {
                    const int c = e / Ly::BCW;
                    bcs[e] = c < tvalid ? sg.bc[((int64_t)b * L + t0) * Ly::BCW + e] : 0.0f;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&full[st]);
            }
        }
        if constexpr (TMA) {
            // No CTA may exit while its bulk copies are in flight.  The
            // consumers wait on every tile's barrier; the producer also waits
            // for the copies it issued last (after an abort they may be the
            // only waits left) before it returns.
            if (lane == 0) {
                for (int t = issued > kNST ? issued - kNST : 0; t < issued; ++t)
                    wait_parity(&full[t % kNST], (uint32_t)((t / kNST) & 1), status, 1ll << 28);
            }
        }
        return;
    }

    // ---------------------------------------------------------------- consumer
    if (warp >= nw_live) return;                       // no channels for this warp
    // channel within the warp; with swizzled tiles and two lanes a channel
    // the channels are permuted (bits 1 and 2 of the index swapped) so that
    // a quarter-warp's four channels sit in rows 0, 1, 4, 5 (or 2, 3, 6, 7)
    // modulo 8 and its 16-byte tile reads fall in eight bank groups
    const int cw = (SW && NS == 2) ? (((lane / NS) & 9) | (((lane / NS) & 2) << 1) | (((lane / NS) & 4) >> 1))
                                   : lane / NS;
    const int g = lane % NS;                            // state group
    const int cl = warp * CPW + cw;                     // channel within the CTA
    const int d = d0 + cl;
    const bool dok = d < dim;
    const int own0 = g * E;                             // first step of each block this lane owns

    float2 h2[S / 2], a2[S / 2];
#pragma unroll
    for (int q = 0; q < S / 2; ++q) {
        float v[2], hv[2];
#pragma unroll
        for (int k = 0; k < 2; ++k) {
            const int n = g * S + 2 * q + k;
            const bool ok = dok && n < N;
            v[k] = ok ? __ldg(p.A + (int64_t)d * N + n) * kLog2e : 0.0f;
            hv[k] = (MODE == kSeeded && ok)               ? sg.ws_h[((int64_t)seg * nchan + chan0 + d) * N + n]
                    : (MODE != kSeeded && MODE != kTotals && ok && p.h0) ? p.h0[(chan0 + d) * N + n]
                                                         : 0.0f;
        }
        a2[q] = make_float2(v[0], v[1]);
        h2[q] = make_float2(hv[0], hv[1]);
    }
    const float bias = (dok && p.dt_bias) ? __ldg(p.dt_bias + d) : 0.0f;
    const float Dd = (dok && p.D) ? __ldg(p.D + d) : 0.0f;
    // fused convolution: the filter right-aligned in CK taps (zero taps in
    // front for narrower filters), and the history before the sequence
    float cw4[CK > 0 ? CK : 1];
    float cbias = 0.0f;
    float *halo = reinterpret_cast<float *>(smem + Ly::off_halo) + cl * (CK > 0 ? CK : 1);
    if constexpr (CK > 0) {
        const int K = p.conv_k;
#pragma unroll
        for (int j = 0; j < CK; ++j) {
            const int i = j - (CK - K);               // tap index of the filter
            cw4[j] = (dok && i >= 0) ? __ldg(p.conv_w + (int64_t)d * K + i) : 0.0f;
        }
        cbias = (dok && p.conv_b) ? __ldg(p.conv_b + d) : 0.0f;
        if (g == 0) {
            // halo[m] holds the raw input at step m - CK of the current tile
#pragma unroll
            for (int m = 0; m < CK; ++m) {
                const int i = m - (CK - (K - 1));     // index into the K-1 inputs before t = 0
                float v = 0.0f;
                if (dok && p.conv_state && i >= 0)
                    v = Io<T>::ld(p.conv_state, (chan0 + d) * (int64_t)(K - 1) + i);
                halo[m] = v;
            }
        }
        __syncwarp();
    }
    const bool vec = p.vec16 != 0;
    const bool sp = p.softplus != 0;
    float dsum = 0.0f;
    bool aborted = false;

    for (int tile = 0; tile < ntiles; ++tile) {
        const int st = tile % kNST;
        const unsigned char *base = smem + st * Ly::stage_bytes;
        const float *BC = reinterpret_cast<const float *>(base + Ly::off_bc);   // [TC][BCW]
        const int64_t t0 = ts + (int64_t)tile * TC;
        const int tvalid = (int)((te - t0) < TC ? (te - t0) : TC);
        const bool ok = wait_parity(&full[st], (uint32_t)((tile / kNST) & 1), status);
        if (!__all_sync(FULL, ok && *abort_flag == 0)) { aborted = true; break; }
        if constexpr (MODE == kStates || CKPT) {
            // the state at the start of every chunk: the state pass's output
            // (ck_len-step chunks), or the forward's checkpoints (kCkptSteps)
            float *const ck = MODE == kStates ? sg.ws_h : p.ckpt;
            const int64_t ckl = MODE == kStates ? sg.ck_len : (int64_t)kCkptSteps;
            if (dok && t0 % ckl == 0) {
                float *dst = ck + ((t0 / ckl) * nchan + chan0 + d) * N;
#pragma unroll
                for (int q = 0; q < S / 2; ++q) {
                    const int n = g * S + 2 * q;
                    if (n < N) dst[n] = h2[q].x;
                    if (n + 1 < N) dst[n + 1] = h2[q].y;
                }
            }
        }

#pragma unroll 1
        for (int blk = 0; blk < TC / KB; ++blk) {
            const int cb = blk * KB;
            const int ce = cb + own0;                     // first tile column this lane owns
            // ---- 1. Delta and u of the lane's own E steps (registers) ---------
            float Dl[E], Ul[E], xv[E];
            {
                float dv[E];
                rowE<T, E, TC, SW>(base + Ly::off_dl, cl, ce, dv);
                rowE<T, E, TC, SW>(base + Ly::off_x, cl, ce, xv);
                if constexpr (CK > 0) {
                    // x = silu(bias + sum_j w_j raw_{t-CK+1+j}): the lane's E raw
                    // inputs and the CK-1 before them (from the tile, or for
                    // the first steps of a tile from the history)
                    float win[E + CK - 1];
#pragma unroll
                    for (int k = 0; k < E; ++k) win[CK - 1 + k] = xv[k];
#pragma unroll
                    for (int i = 1; i < CK; ++i) {
                        const int c = ce - i;          // both reads stay in bounds
                        const float tv = row1<T, TC, SW>(base + Ly::off_x, cl, c >= 0 ? c : 0);
                        const float hv = halo[CK + (c < 0 ? c : -1)];
                        win[CK - 1 - i] = c >= 0 ? tv : hv;
                    }
#pragma unroll
                    for (int k = 0; k < E; ++k) {
                        float acc = cbias;
#pragma unroll
                        for (int j = 0; j < CK; ++j) acc = fmaf(cw4[j], win[k + j], acc);
                        xv[k] = dok ? gate<T>(acc) : 0.0f;
                    }
                    if (blk == TC / KB - 1) {
                        // the tile's last CK raw inputs become the next tile's history
                        __syncwarp();
                        if (g == NS - 1) {
#pragma unroll
                            for (int m = 0; m < CK; ++m) halo[m] = win[E - 1 + m];
                        }
                        __syncwarp();
                    }
                }
#pragma unroll
                for (int k = 0; k < E; k += 2) {
                    const float2 v = __fadd2_rn(make_float2(dv[k], dv[k + 1]), make_float2(bias, bias));
                    float2 Dv = sp ? softplus2(v) : v;
                    Dv = make_float2((dok && ce + k < tvalid) ? Dv.x : 0.0f,
                                     (dok && ce + k + 1 < tvalid) ? Dv.y : 0.0f);
                    const float2 Uv = __fmul2_rn(Dv, make_float2(xv[k], xv[k + 1]));
                    Dl[k] = Dv.x; Dl[k + 1] = Dv.y;
                    Ul[k] = Uv.x; Ul[k + 1] = Uv.y;
                }
            }
            // ---- 2. scan the block --------------------------------------------
            // Batches of JB steps: first everything that does not depend on the
            // state (Delta/u exchange, B/C loads, a = 2^(Delta A log2 e), u B)
            // for all JB steps, then the JB dependent updates h = a h + u B and
            // the contraction.  The independent half gives the scheduler JB
            // steps of special-function and load latency to overlap: 8 steps
            // for narrow lanes of four or more a channel (mid-size shape:
            // 106.5 -> 104.4 us against 4), 4 for 8 states, 2 for 16 (registers).
            constexpr int JB = S >= 16 ? 2 : (S <= 4 && NS >= 4) ? 8 : 4;
            float pv[KB];
#pragma unroll
            for (int j0 = 0; j0 < KB; j0 += JB) {
                float2 av[JB][S / 2], bv[JB][S / 2], cv[JB][S / 2];
#pragma unroll
                for (int jj = 0; jj < JB; ++jj) {
                    const int j = j0 + jj;
                    float Dj, Uj;
                    if constexpr (NS == 1) {
                        Dj = Dl[j];
                        Uj = Ul[j];
                    } else {
                        const int src = (lane & ~(NS - 1)) | (j / E);      // owner of step j
                        Dj = __shfl_sync(FULL, Dl[j % E], src);
                        Uj = __shfl_sync(FULL, Ul[j % E], src);
                    }
                    const float2 dd = make_float2(Dj, Dj);
                    const float2 uu = make_float2(Uj, Uj);
                    const float *bc = BC + (cb + j) * Ly::BCW + g * bc_group(S);
                    float bcv[2 * S];
#pragma unroll
                    for (int k = 0; k < (kY ? 2 * S : S); k += 4) {
                        const float4 v4 = *reinterpret_cast<const float4 *>(bc + k);
                        bcv[k] = v4.x; bcv[k + 1] = v4.y; bcv[k + 2] = v4.z; bcv[k + 3] = v4.w;
                    }
#pragma unroll
                    for (int q = 0; q < S / 2; ++q) {
                        const float2 arg = __fmul2_rn(dd, a2[q]);
                        av[jj][q] = make_float2(ex2(arg.x), ex2(arg.y));
                        bv[jj][q] = __fmul2_rn(uu, make_float2(bcv[2 * q], bcv[2 * q + 1]));
                        if constexpr (kY) cv[jj][q] = make_float2(bcv[S + 2 * q], bcv[S + 2 * q + 1]);
                    }
                    if constexpr (!kY) dsum += Dj;
                }
#pragma unroll
                for (int jj = 0; jj < JB; ++jj) {
                    // two accumulators halve the dependent chain of the contraction
                    float2 acc0 = make_float2(0.0f, 0.0f), acc1 = make_float2(0.0f, 0.0f);
#pragma unroll
                    for (int q = 0; q < S / 2; ++q) {
                        h2[q] = __ffma2_rn(av[jj][q], h2[q], bv[jj][q]);
                        if constexpr (kY) {
                            if (q % 2 == 0) acc0 = __ffma2_rn(cv[jj][q], h2[q], acc0);
                            else acc1 = __ffma2_rn(cv[jj][q], h2[q], acc1);
                        }
                    }
                    const float2 acc = __fadd2_rn(acc0, acc1);
                    pv[j0 + jj] = acc.x + acc.y;
                }
            }
            if constexpr (kY) {
                // ---- 3. reduce-scatter the partial sums over the NS lanes -------
                ReduceScatter<KB / 2, NS / 2>::run(pv, g);
                float ys[E];
#pragma unroll
                for (int k = 0; k < E; ++k) ys[k] = pv[k];
                // ---- skip, gate, store the lane's own steps ---------------------
                if (dok) {
                    float zv[E];
                    if constexpr (kZ) rowE<T, E, TC, SW>(base + Ly::off_z, cl, ce, zv);
#pragma unroll
                    for (int k = 0; k < E; k += 2) {
                        float2 v = __ffma2_rn(make_float2(Dd, Dd), make_float2(xv[k], xv[k + 1]),
                                              make_float2(ys[k], ys[k + 1]));
                        if constexpr (kZ) v = __fmul2_rn(v, make_float2(gate<T>(zv[k]), gate<T>(zv[k + 1])));
                        ys[k] = v.x; ys[k + 1] = v.y;
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
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[st]);
    }
    if (aborted) { *abort_flag = 1; return; }
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
template <typename T, int NP, int S, int NW, bool GATE, int MODE, bool TMA, int CK = 0, bool CKPT = false>
cudaError_t launch_one(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps, unsigned int *status,
                       cudaStream_t st) {
    using Ly = Layout<T, NP, S, NW, GATE, MODE, CK>;
    auto kern = scan_kernel<T, NP, S, NW, GATE, MODE, TMA, CK, CKPT>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Ly::bytes);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)((a.dim + Ly::DT - 1) / Ly::DT), (unsigned)a.batch, (unsigned)sg.nseg);
    kern<<<grid, Ly::NT, Ly::bytes, st>>>(a, sg, maps, status);
    return cudaGetLastError();
}

// Prepare the B/C rows for states-per-lane S.
template <typename T, int NP, int S>
cudaError_t launch_prepare(const FwdArgs &a, float *out, cudaStream_t st) {
    dim3 grid((unsigned)((a.L + 31) / 32), (unsigned)a.batch);
    bc_prepare_kernel<T, NP, S><<<grid, 256, 0, st>>>(a.B, a.C, out, a.dstate, a.L);
    return cudaGetLastError();
}

// Instantiation dispatch for one I/O type (defined in scan_fused_<type>.cu):
// prepares B/C when `prepare` is set, then runs the scan in `mode`.
template <typename T>
cudaError_t launch_typed(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps, unsigned int *status,
                         int mode, bool tma, int cfg, bool prepare, cudaStream_t st);
// The same for the forward that stores checkpoints (kWhole and kSeeded only;
// defined in scan_fused_ckpt_<type>.cu).
template <typename T>
cudaError_t launch_typed_ckpt(const FwdArgs &a, const SegArgs &sg, const TileMaps &maps, unsigned int *status,
                              int mode, bool tma, int cfg, bool prepare, cudaStream_t st);

}  // namespace fused
}  // namespace ssm
