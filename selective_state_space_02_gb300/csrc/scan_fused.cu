// Host side of the FUSED and TWOPASS variants: tile-configuration choice,
// TMA tensor maps, the segment plan of the two-pass variant and its small
// scan over segment totals, and the device status word of the bounded waits.
//
// "Mamba hardware-aware parallel associative scan" (pwwt.cn/news/6375169),
// sect. 2.2 and 3.3: chunked two-pass scheme and the chunk-start formula
//   h_init^(k) = A_tot^(k-1) * h_init^(k-1) + B_tot^(k-1),  h_init^(0) = 0,
// where (A_tot, B_tot) is the composition of all of a chunk's pairs; for the
// diagonal A of the selective scan, A_tot[n] = exp(A[d,n] * sum of Delta).
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "scan_fused_impl.cuh"

namespace ssm {

__device__ unsigned int g_scan_status = 0;

namespace {

constexpr int kSMs = 152;

// Device address of g_scan_status on the current device, looked up on every
// call (a cudaDeviceReset reloads the module, possibly at a new address).
unsigned int *status_ptr() {
    void *p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scan_status) != cudaSuccess) return nullptr;
    return static_cast<unsigned int *>(p);
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

int padded_states(int N) { return N <= 8 ? 8 : N <= 16 ? 16 : N <= 32 ? 32 : 64; }

// States per lane of each configuration (see scan_fused_dispatch.cuh).
int fused_states(int np, int cfg, bool tma) {
    if (np == 8) return (tma && cfg == 0) ? 8 : 4;
    if (np == 16) return !tma ? 8 : cfg == 0 ? 16 : cfg == 1 ? 8 : cfg == 2 ? 4 : 2;
    if (np == 32) return (tma && cfg == 0) ? 16 : 8;
    return 16;
}

int max_cfg(int np) { return np == 16 ? 3 : np == 64 ? 0 : 1; }

// Configuration of the two-pass variant: segments supply the parallelism, and
// four states per lane (two for N <= 8, eight for N <= 32, sixteen for N <= 64)
// measured fastest for segmented runs.
int twopass_cfg(int np) {
#ifdef SSM_TUNE
    if (const char *e = std::getenv("SSM_TWOPASS_CFG")) {
        const int c = std::atoi(e);
        return c < 0 ? 0 : c > max_cfg(np) ? max_cfg(np) : c;
    }
#endif
    return np == 64 ? 0 : 1;
}

// Consumer warps per SM that the segment plan of the two-pass variant aims
// for.  Measured on GB300 with the long-sequence workload (768 channels, 16
// states, 131072 steps, float32): 8 states a lane with 8 warps per SM (25
// segments) took 0.82 ms, against 0.95 ms for 4 states a lane and 1.28 ms for
// 16; plans of 6, 9 or 12 warps per SM were 25-40% slower (partial waves).
int resident_warps(int np, int cfg) {
    const int S = fused_states(np, cfg, true);
    return S >= 16 ? 9 : 8;
}

// Channels per warp (the TMA box height of x, delta and z).
int warp_channels(int np, int cfg, bool tma) { return 32 / (np / fused_states(np, cfg, tma)); }

// The configuration with the most states per lane that still gives at least
// one warp per SM sub-partition (4 per SM); fewer states per lane only when
// the problem has too few channels for that.
int choose_cfg(int64_t nchan, int np, int64_t nseg) {
#ifdef SSM_TUNE
    if (const char *e = std::getenv("SSM_FUSED_CFG")) {
        const int c = std::atoi(e);
        return c < 0 ? 0 : c > max_cfg(np) ? max_cfg(np) : c;
    }
#endif
    for (int cfg = 0; cfg < max_cfg(np); ++cfg) {
        const int64_t warps = nchan * nseg / warp_channels(np, cfg, true);
        if (warps >= (int64_t)kSMs * 4) return cfg;
    }
    return max_cfg(np);
}

// Tensor maps for the TMA path; false selects the element-load path (rows not
// 16-byte aligned, coordinates beyond 32 bits, or no driver entry point).
bool make_maps(const FwdArgs &a, int cfg, const float *bc, fused::TileMaps &m) {
    std::memset(&m, 0, sizeof(m));
    if (!a.vec16) return false;
    const int64_t rows = (int64_t)a.batch * a.dim;
    const int64_t brows = (int64_t)a.batch * a.L;
    if (a.L >= ((int64_t)1 << 31) || rows >= ((int64_t)1 << 31) || brows >= ((int64_t)1 << 31)) return false;
    const int np = padded_states(a.dstate);
    const uint32_t dt = (uint32_t)(warp_channels(np, cfg, true) * fused::consumer_warps(fused_states(np, cfg, true)));
    const uint64_t L = (uint64_t)a.L;
    const bool bf = a.bf16 != 0;
    const uint32_t tc = (uint32_t)fused::tile_steps(np);
    const int S = fused_states(np, cfg, true);
    const int bcw = fused::bc_row(np, S);
    // tiles of 128-byte rows take the 128-byte swizzle, of 64-byte rows the
    // 64-byte swizzle (the layouts the kernel reads through tile_byte)
    const uint32_t rowb = tc * (bf ? 2u : 4u);
    const int sw = rowb == 128 ? 128 : rowb == 64 ? 64 : 0;
    return encode_tile_map(&m.x, a.x, bf, (uint64_t)rows, L, dt, tc, sw) &&
           encode_tile_map(&m.dl, a.delta, bf, (uint64_t)rows, L, dt, tc, sw) &&
           encode_f32_map(&m.bc, bc, (uint64_t)brows, (uint64_t)bcw, tc, (uint32_t)bcw) &&
           (!a.z || encode_tile_map(&m.z, a.z, bf, (uint64_t)rows, L, dt, tc, sw));
}

// Bytes of the prepared B/C rows: [batch * L][widest row] float.
size_t bc_bytes(int batch, int dstate, int64_t L) {
    const size_t n = (size_t)batch * (size_t)L * fused::bc_row_max(padded_states(dstate)) * sizeof(float);
    return (n + 255) / 256 * 256;
}

cudaError_t launch_mode(const FwdArgs &a, const fused::SegArgs &sg, int mode, int cfg, bool prepare,
                        cudaStream_t st) {
    unsigned int *status = status_ptr();
    if (!status) return cudaErrorInvalidSymbol;
    fused::TileMaps maps;
    const bool tma = make_maps(a, cfg, sg.bc, maps);
    if (a.ckpt && (mode == fused::kWhole || mode == fused::kSeeded)) {   // the forward's y pass with checkpoints
        if (a.bf16) return fused::launch_typed_ckpt<__nv_bfloat16>(a, sg, maps, status, mode, tma, cfg, prepare, st);
        return fused::launch_typed_ckpt<float>(a, sg, maps, status, mode, tma, cfg, prepare, st);
    }
    if (a.bf16) return fused::launch_typed<__nv_bfloat16>(a, sg, maps, status, mode, tma, cfg, prepare, st);
    return fused::launch_typed<float>(a, sg, maps, status, mode, tma, cfg, prepare, st);
}

// Carry over the segment totals ("Mamba hardware-aware parallel associative
// scan", sect. 3.3): for every (channel, state) pair, in segment order,
// h_init^(k+1) = A_k h_init^(k) + B_k with the segment's pair (A_k, B_k) =
// (exp(A * sum Delta_k), its end state from the zero state).  On return
// ws_h[k] holds the state at the start of segment k, h_init^(0) being the
// start state h0 of the whole sequence (zero when h0 is null).  The last
// segment's total is never read (pass 1 does not form it).
//
// Two levels, so that every load is coalesced and a long chain of segments
// still has parallelism: a CTA takes 32 consecutive pairs (lane = pair) and
// kCarryWarps warps, warp w a contiguous group of the segments.
//   1. each warp composes its group's pairs into one (A_g, B_g), A_g from the
//      group's summed Delta (one exponential, the log-domain form);
//   2. through shared memory each warp composes the groups before its own
//      with the start state into its group's start;
//   3. each warp walks its group again from that start, writing the segment
//      start states.
constexpr int kCarryWarps = 16;

__global__ void __launch_bounds__(kCarryWarps * 32) segment_carry_kernel(const float *__restrict__ A, float *ws_h,
                                                                          const float *__restrict__ ws_s,
                                                                          const float *__restrict__ h0,
                                                                          int64_t nchan, int dim, int N, int nseg) {
    __shared__ float gA[kCarryWarps][32], gB[kCarryWarps][32];
    const int lane = threadIdx.x & 31;
    const int w = threadIdx.x >> 5;
    const int64_t npair = nchan * N;
    const int64_t pair = (int64_t)blockIdx.x * 32 + lane;
    const bool ok = pair < npair;
    const int64_t pc = ok ? pair : 0;               // a valid pair for the loads of idle lanes
    const int64_t ch = pc / N;
    const int n = (int)(pc % N);
    const float a2 = A[(ch % dim) * N + n] * kLog2e;
    const int per = (nseg + kCarryWarps - 1) / kCarryWarps;
    const int k0 = w * per;
    const int k1 = (k0 + per < nseg) ? k0 + per : nseg;
    const int kt = k1 < nseg - 1 ? k1 : nseg - 1;   // segments of the group that have totals
    // 1. the group's composition from the zero state (loads issued U segments
    // ahead of the dependent multiply-adds)
    constexpr int U = 8;
    float hg = 0.0f, sg = 0.0f;
    int k = k0;
    for (; k + U <= kt; k += U) {
        float Bv[U], sv[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            Bv[j] = ws_h[(int64_t)(k + j) * npair + pc];
            sv[j] = ws_s[(int64_t)(k + j) * nchan + ch];
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            hg = fmaf(ex2(a2 * sv[j]), hg, Bv[j]);
            sg += sv[j];
        }
    }
    for (; k < kt; ++k) {
        const float sk = ws_s[(int64_t)k * nchan + ch];
        hg = fmaf(ex2(a2 * sk), hg, ws_h[(int64_t)k * npair + pc]);
        sg += sk;
    }
    gA[w][lane] = ex2(a2 * sg);
    gB[w][lane] = hg;
    __syncthreads();
    // 2. the group's start state
    float h = (ok && h0) ? h0[pair] : 0.0f;
    for (int v = 0; v < w; ++v) h = fmaf(gA[v][lane], h, gB[v][lane]);
    // 3. the segment start states of the group
    k = k0;
    for (; k + U <= kt; k += U) {
        float Bv[U], sv[U];
#pragma unroll
        for (int j = 0; j < U; ++j) {
            Bv[j] = ws_h[(int64_t)(k + j) * npair + pc];
            sv[j] = ws_s[(int64_t)(k + j) * nchan + ch];
        }
#pragma unroll
        for (int j = 0; j < U; ++j) {
            if (ok) ws_h[(int64_t)(k + j) * npair + pc] = h;
            h = fmaf(ex2(a2 * sv[j]), h, Bv[j]);
        }
    }
    for (; k < k1; ++k) {
        const int64_t i = (int64_t)k * npair + pc;
        const bool has = k < nseg - 1;
        const float Bk = has ? ws_h[i] : 0.0f;
        const float sk = has ? ws_s[(int64_t)k * nchan + ch] : 0.0f;
        if (ok) ws_h[i] = h;
        h = fmaf(ex2(a2 * sk), h, Bk);
    }
}

}  // namespace

bool encode_tile_map(CUtensorMap *map, const void *base, bool bf16, uint64_t rows, uint64_t cols,
                     uint32_t box_rows, uint32_t box_cols, int swizzle) {
    auto fn = encode_fn();
    if (!fn) return false;
    const size_t es = bf16 ? 2 : 4;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * es};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    if (swizzle && box_cols * es != (uint32_t)swizzle) return false;
    CUresult r = fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2,
                    const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    swizzle == 128 ? CU_TENSOR_MAP_SWIZZLE_128B
                    : swizzle == 64 ? CU_TENSOR_MAP_SWIZZLE_64B
                                    : CU_TENSOR_MAP_SWIZZLE_NONE,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool encode_f32_map(CUtensorMap *map, const void *base, uint64_t rows, uint64_t cols, uint32_t box_rows,
                    uint32_t box_cols) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {cols * 4};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, const_cast<void *>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

size_t fused_workspace_bytes(int batch, int dim, int dstate, int64_t L) {
    (void)dim;
    return bc_bytes(batch, dstate, L);
}

cudaError_t launch_fused(const FwdArgs &a, void *workspace, cudaStream_t st) {
    const int64_t nchan = (int64_t)a.batch * a.dim;
    fused::SegArgs sg{a.L, 1, nullptr, nullptr, static_cast<const float *>(workspace), kCkptSteps};
    return launch_mode(a, sg, fused::kWhole, choose_cfg(nchan, padded_states(a.dstate), 1), true, st);
}

int64_t twopass_chunk_len(int batch, int dim, int dstate, int64_t L) {
    // As many segments as keep one pass within about 8 consumer warps per SM
    // (4 resident CTAs: rounding up would leave a second, nearly empty wave),
    // while each segment keeps at least 8 tiles of work.
    const int np = padded_states(dstate);
    const int cfg = twopass_cfg(np);
    const int cpw = warp_channels(np, cfg, true);
    const int64_t warps = (int64_t)batch * ((dim + cpw - 1) / cpw);
    int64_t want = (int64_t)kSMs * resident_warps(np, cfg);
#ifdef SSM_TUNE
    if (const char *e = std::getenv("SSM_TWOPASS_WANT")) want = (int64_t)kSMs * std::atoi(e);
#endif
    int64_t nseg = want / (warps > 0 ? warps : 1);
    const int64_t tcs = fused::tile_steps(np);
    const int64_t max_seg = (L + 8 * tcs - 1) / (8 * tcs);
    if (nseg > max_seg) nseg = max_seg;
    if (nseg < 1) nseg = 1;
    int64_t len = (L + nseg - 1) / nseg;
    len = (len + tcs - 1) / tcs * tcs;   // whole tiles
    return len > 0 ? len : tcs;
}

size_t twopass_workspace_bytes(int batch, int dim, int dstate, int64_t L) {
    const int64_t len = twopass_chunk_len(batch, dim, dstate, L);
    const int64_t nseg = L > 0 ? (L + len - 1) / len : 1;
    const int64_t nchan = (int64_t)batch * dim;
    size_t h = (size_t)nseg * nchan * dstate * sizeof(float);
    h = (h + 255) / 256 * 256;
    size_t s = (size_t)nseg * nchan * sizeof(float);
    s = (s + 255) / 256 * 256;
    return h + s + bc_bytes(batch, dstate, L);
}

cudaError_t launch_twopass(const FwdArgs &a, void *workspace, cudaStream_t st) {
    const int64_t len = twopass_chunk_len(a.batch, a.dim, a.dstate, a.L);
    const int nseg = (int)((a.L + len - 1) / len);
    const int64_t nchan = (int64_t)a.batch * a.dim;
    size_t hbytes = (size_t)nseg * nchan * a.dstate * sizeof(float);
    hbytes = (hbytes + 255) / 256 * 256;
    size_t sbytes = (size_t)nseg * nchan * sizeof(float);
    sbytes = (sbytes + 255) / 256 * 256;
    char *ws = static_cast<char *>(workspace);
    fused::SegArgs sg{len, nseg, reinterpret_cast<float *>(ws), reinterpret_cast<float *>(ws + hbytes),
                      reinterpret_cast<const float *>(ws + hbytes + sbytes), kCkptSteps};
    const int cfg = twopass_cfg(padded_states(a.dstate));
    cudaError_t e = cudaSuccess;
    bool prepared = false;
    if (nseg > 1) {   // pass 1 over every segment but the last (its total is never used)
        fused::SegArgs s1 = sg;
        s1.nseg = nseg - 1;
        e = launch_mode(a, s1, fused::kTotals, cfg, true, st);
        if (e != cudaSuccess) return e;
        prepared = true;
    }
    const int64_t pairs = nchan * a.dstate;
    segment_carry_kernel<<<(unsigned)((pairs + 31) / 32), kCarryWarps * 32, 0, st>>>(a.A, sg.ws_h, sg.ws_s, a.h0,
                                                                                    nchan, a.dim, a.dstate, nseg);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    return launch_mode(a, sg, fused::kSeeded, cfg, !prepared, st);
}

unsigned int *device_status_word() { return status_ptr(); }

size_t chunk_states_workspace_bytes(int batch, int dim, int dstate, int64_t L, int64_t seg_len) {
    const int64_t nseg = L > 0 ? (L + seg_len - 1) / seg_len : 0;
    const int64_t nchan = (int64_t)batch * dim;
    size_t h = (size_t)nseg * nchan * dstate * sizeof(float);
    size_t s = (size_t)nseg * nchan * sizeof(float);
    return (h + 255) / 256 * 256 + (s + 255) / 256 * 256 + bc_bytes(batch, dstate, L);
}

namespace {

// Whether chunk_start_states takes the one-pass route: channels for at least
// one consumer warp per SM sub-partition, segments of whole tiles.
bool states_in_one_pass(int batch, int dim, int dstate, int64_t seg_len) {
    const int64_t nchan = (int64_t)batch * dim;
    const int np = padded_states(dstate);
    const int cfg = choose_cfg(nchan, np, 1);
    bool one = nchan / warp_channels(np, cfg, true) >= (int64_t)kSMs * 4 && seg_len % fused::tile_steps(np) == 0;
#ifdef SSM_TUNE
    if (const char *e = std::getenv("SSM_CKPT")) one = one && std::atoi(e) != 0;
#endif
    return one;
}

}  // namespace

int chunk_start_states_kernels(int batch, int dim, int dstate, int64_t L, int64_t seg_len) {
    if (states_in_one_pass(batch, dim, dstate, seg_len)) return 2;   // B/C re-layout, the pass
    const int64_t nseg = (L + seg_len - 1) / seg_len;
    return nseg > 1 ? 3 : 1;                                        // (re-layout, totals,) carry scan
}

cudaError_t chunk_start_states(const FwdArgs &a, int64_t seg_len, void *workspace, cudaStream_t st) {
    const int nseg = (int)((a.L + seg_len - 1) / seg_len);
    const int64_t nchan = (int64_t)a.batch * a.dim;
    size_t hbytes = (size_t)nseg * nchan * a.dstate * sizeof(float);
    hbytes = (hbytes + 255) / 256 * 256;
    size_t sbytes = (size_t)nseg * nchan * sizeof(float);
    sbytes = (sbytes + 255) / 256 * 256;
    char *ws = static_cast<char *>(workspace);
    fused::SegArgs sg{seg_len, nseg, reinterpret_cast<float *>(ws), reinterpret_cast<float *>(ws + hbytes),
                      reinterpret_cast<const float *>(ws + hbytes + sbytes), seg_len};
    // With channels for at least one consumer warp per SM sub-partition, one
    // pass of the whole-sequence kernel from the start state writes the state
    // at every segment start as it goes.
    const int np = padded_states(a.dstate);
    const int wcfg = choose_cfg(nchan, np, 1);
    if (states_in_one_pass(a.batch, a.dim, a.dstate, seg_len)) {
        sg.seg_len = a.L;
        sg.nseg = 1;
        return launch_mode(a, sg, fused::kStates, wcfg, true, st);
    }
    // Otherwise the first two steps of the two-pass forward with segments of
    // seg_len steps: per-segment totals from the zero state, then the carry
    // scan over the segments seeded with the start state.
    const int cfg = twopass_cfg(np);
    cudaError_t e = cudaSuccess;
    if (nseg > 1) {
        fused::SegArgs s1 = sg;
        s1.nseg = nseg - 1;
        e = launch_mode(a, s1, fused::kTotals, cfg, true, st);
        if (e != cudaSuccess) return e;
    }
    const int64_t pairs = nchan * a.dstate;
    segment_carry_kernel<<<(unsigned)((pairs + 31) / 32), kCarryWarps * 32, 0, st>>>(a.A, sg.ws_h, sg.ws_s, a.h0,
                                                                                    nchan, a.dim, a.dstate, nseg);
    return cudaGetLastError();
}

namespace {

// One thread waits, bounded, on an mbarrier that no thread arrives on and no
// copy targets; the wait runs out, flags the status word and returns.
__global__ void wait_timeout_kernel(unsigned int *status, long long limit) {
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    mbar_init(&bar, 1);
    fence_mbar_init();
    wait_parity(&bar, 0u, status, limit);
}

}  // namespace

cudaError_t selftest_wait_timeout(long long limit, cudaStream_t st) {
    unsigned int *status = status_ptr();
    if (!status) return cudaErrorInvalidSymbol;
    wait_timeout_kernel<<<1, 32, 0, st>>>(status, limit);
    return cudaGetLastError();
}

int read_device_status(cudaStream_t st, bool clear, unsigned int *out) {
    unsigned int *p = status_ptr();
    if (!p) return -1;
    unsigned int v = 0;
    if (cudaMemcpyAsync(&v, p, sizeof(v), cudaMemcpyDeviceToHost, st) != cudaSuccess) return -1;
    if (clear && cudaMemsetAsync(p, 0, sizeof(v), st) != cudaSuccess) return -1;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    *out = v;
    return 0;
}

}  // namespace ssm
