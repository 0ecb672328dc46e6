// C ABI of libssmscan: argument validation, variant selection and the
// device- and host-buffer entry points.  Declared in include/ssm_scan.h.
#include "../../include/ssm_scan.h"
#include "../../include/ssm_conv.h"
#include "scan_internal.h"

#include <cstring>
#include <mutex>

namespace {

constexpr int kVersion = (1 << 16) | 2;
constexpr int kFusedConvTaps = 4;   // widest filter the fused kernel takes

bool valid_sizes(int batch, int dim, int dstate, int64_t seqlen) {
    return batch >= 0 && dim >= 0 && dstate >= 1 && dstate <= 64 && seqlen >= 0;
}

size_t elem_size(int io_dtype) { return io_dtype == SSM_BF16 ? 2 : 4; }

int resolve_variant(int batch, int dim, int dstate, int64_t seqlen, int io_dtype, int variant) {
    if (variant == SSM_VARIANT_AUTO) return ssm_scan_select_variant(batch, dim, dstate, seqlen, io_dtype);
    if (variant < SSM_VARIANT_FUSED || variant > SSM_VARIANT_TWOPASS) return SSM_ERR_VARIANT;
    return variant;
}

// The variant of a forward that writes checkpoints: FUSED and TWOPASS store
// them as they go; where AUTO would pick CHUNKED it takes TWOPASS.
int ckpt_variant(int batch, int dim, int dstate, int64_t seqlen, int io_dtype, int variant) {
    const int v = resolve_variant(batch, dim, dstate, seqlen, io_dtype, variant);
    if (v != SSM_VARIANT_CHUNKED) return v;
    return variant == SSM_VARIANT_AUTO ? SSM_VARIANT_TWOPASS : SSM_ERR_UNSUPPORTED;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

struct Range {
    uintptr_t lo, hi;   // [lo, hi)
};

Range range_of(const void *p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return Range{a, a + bytes};
}

bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi && a.lo != a.hi && b.lo != b.hi; }

// Shared validation of the entry points.  Returns SSM_OK or an error code.
// The start state h0 (nullable) is an input that final_state may replace in
// place: the two may be the same array, but no other overlap is allowed.
int validate(const void *x, const void *delta, const float *A, const void *B, const void *C,
             const float *D, const void *z, const float *dt_bias, void *y, float *final_state,
             int batch, int dim, int dstate, int64_t seqlen, int io_dtype, const float *h0 = nullptr) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (!valid_sizes(batch, dim, dstate, seqlen)) return SSM_ERR_DIMS;
    // sizes whose element counts would not fit the 64-bit index arithmetic
    if (seqlen > ((int64_t)1 << 40) || (int64_t)batch * dim > ((int64_t)1 << 31)) return SSM_ERR_DIMS;
    const bool empty = batch == 0 || dim == 0;
    if (!empty) {
        if (!A) return SSM_ERR_NULL;
        if (seqlen > 0 && (!x || !delta || !B || !C || !y)) return SSM_ERR_NULL;
    }
    const size_t es = elem_size(io_dtype);
    const void *iop[] = {x, delta, B, C, z, y};
    for (const void *q : iop)
        if (q && !aligned(q, es)) return SSM_ERR_ALIGN;
    const void *fp[] = {A, D, dt_bias, final_state, h0};
    for (const void *q : fp)
        if (q && !aligned(q, 4)) return SSM_ERR_ALIGN;
    const size_t ns = (size_t)batch * dim * dstate * 4;
    if (h0 && final_state && h0 != final_state && overlap(range_of(h0, ns), range_of(final_state, ns)))
        return SSM_ERR_ALIAS;
    if (empty || seqlen == 0) return SSM_OK;
    // outputs must not overlap inputs
    const size_t nx = (size_t)batch * dim * (size_t)seqlen * es;
    const size_t nb = (size_t)batch * dstate * (size_t)seqlen * es;
    const Range ins[] = {range_of(x, nx), range_of(delta, nx), range_of(z, z ? nx : 0),
                         range_of(B, nb), range_of(C, nb),
                         range_of(A, (size_t)dim * dstate * 4), range_of(D, D ? (size_t)dim * 4 : 0),
                         range_of(dt_bias, dt_bias ? (size_t)dim * 4 : 0)};
    if (h0 && overlap(range_of(y, nx), range_of(h0, ns))) return SSM_ERR_ALIAS;
    const Range outs[] = {range_of(y, nx),
                          range_of(final_state, final_state ? (size_t)batch * dim * dstate * 4 : 0)};
    for (const Range &o : outs)
        for (const Range &i : ins)
            if (overlap(o, i)) return SSM_ERR_ALIAS;
    if (overlap(outs[0], outs[1])) return SSM_ERR_ALIAS;
    return SSM_OK;
}

size_t workspace_for(int batch, int dim, int dstate, int64_t seqlen, int variant) {
    if (batch <= 0 || dim <= 0 || seqlen <= 0) return 0;
    if (variant == SSM_VARIANT_TWOPASS) return ssm::twopass_workspace_bytes(batch, dim, dstate, seqlen);
    if (variant == SSM_VARIANT_FUSED) return ssm::fused_workspace_bytes(batch, dim, dstate, seqlen);
    if (variant == SSM_VARIANT_CHUNKED) return ssm::chunked_workspace_bytes(batch, dim, dstate, seqlen);
    return 0;
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

// Time chunks of the host-buffer entry point.  The inputs are copied, scanned
// and copied back chunk after chunk on three streams, so that the copies of
// chunk j+1 overlap the scan of chunk j and the copy back of chunk j-1; each
// chunk starts from the state the previous one ended in.  Measured on GB300
// (pinned memory, about 200 GB/s each way alone and 150 GB/s each way
// together), three chunks gave the shortest calls on the 100 MB - 1.2 GB
// problems: fewer leave the scan and the copy back exposed, more let the copy
// back slow the copy in for longer and add per-chunk overhead.  Problems of
// 48 MiB or more (x, delta, z and y) run in three chunks, from 16 MiB in two,
// smaller ones in one; chunk boundaries fall on whole 64-step tiles (16-byte
// aligned rows in either dtype), so only the last chunk can be ragged.
constexpr int kMaxHostChunks = 3;

struct HostPlan {
    int64_t start[kMaxHostChunks + 1];   // chunk j covers steps [start[j], start[j + 1])
    int n;                               // number of chunks
    int64_t len(int j) const { return start[j + 1] - start[j]; }
};

// Chunk shares of the sequence, largest first: the last chunk's scan and copy
// back are the exposed tail of the pipeline.  0.40 / 0.35 / 0.25 measured
// 1-5% faster than equal thirds on the 100 MB - 1.2 GB problems.
constexpr double kShare2[2] = {0.55, 0.45};
constexpr double kShare3[3] = {0.40, 0.35, 0.25};

HostPlan host_plan(int batch, int dim, int64_t seqlen, int io_dtype, bool has_z) {
    const size_t bytes = (size_t)batch * dim * (size_t)seqlen * elem_size(io_dtype) * (has_z ? 4 : 3);
    const int k = bytes >= ((size_t)48 << 20) ? 3 : bytes >= ((size_t)16 << 20) ? 2 : 1;
    const double *share = k == 3 ? kShare3 : kShare2;
    HostPlan hp{};
    hp.start[0] = 0;
    hp.n = 0;
    double acc = 0.0;
    for (int j = 0; j < k; ++j) {
        int64_t end = seqlen;
        if (j + 1 < k) {
            acc += share[j];
            end = ((int64_t)(acc * (double)seqlen) + 63) / 64 * 64;   // whole 64-step tiles
        }
        if (end <= hp.start[hp.n]) continue;
        if (end > seqlen) end = seqlen;
        hp.start[++hp.n] = end;
        if (end == seqlen) break;
    }
    if (hp.n == 0) { hp.start[1] = seqlen; hp.n = 1; }
    return hp;
}

// Copy streams and events of one device for the host-buffer entry point,
// created by its first call on that device and kept until the process exits.
// The mutex serialises calls on the device, which share them.
struct HostStreams {
    std::mutex mu;
    cudaStream_t in = nullptr, out = nullptr;
    cudaEvent_t start = nullptr;
    cudaEvent_t ready[kMaxHostChunks] = {};
    cudaEvent_t done[kMaxHostChunks] = {};
};

HostStreams *host_streams() {
    static std::mutex mu;
    static HostStreams *cache[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(mu);
    if (cache[dev]) return cache[dev];
    HostStreams *h = new HostStreams();
    bool ok = cudaStreamCreateWithFlags(&h->in, cudaStreamNonBlocking) == cudaSuccess &&
              cudaStreamCreateWithFlags(&h->out, cudaStreamNonBlocking) == cudaSuccess &&
              cudaEventCreateWithFlags(&h->start, cudaEventDisableTiming) == cudaSuccess;
    for (int i = 0; ok && i < kMaxHostChunks; ++i)
        ok = cudaEventCreateWithFlags(&h->ready[i], cudaEventDisableTiming) == cudaSuccess &&
             cudaEventCreateWithFlags(&h->done[i], cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
        if (h->in) cudaStreamDestroy(h->in);
        if (h->out) cudaStreamDestroy(h->out);
        if (h->start) cudaEventDestroy(h->start);
        for (int i = 0; i < kMaxHostChunks; ++i) {
            if (h->ready[i]) cudaEventDestroy(h->ready[i]);
            if (h->done[i]) cudaEventDestroy(h->done[i]);
        }
        delete h;
        return nullptr;
    }
    cache[dev] = h;
    return h;
}

}  // namespace

extern "C" {

int ssm_scan_version(void) { return kVersion; }

const char *ssm_scan_status_string(int status) {
    switch (status) {
        case SSM_OK: return "ok";
        case SSM_ERR_NULL: return "a required pointer is NULL";
        case SSM_ERR_DIMS: return "a size is out of range";
        case SSM_ERR_ALIGN: return "a pointer is not aligned to its element size";
        case SSM_ERR_DTYPE: return "unknown io dtype";
        case SSM_ERR_WORKSPACE: return "workspace missing, too small or misaligned";
        case SSM_ERR_LAUNCH: return "the CUDA runtime rejected a launch or copy";
        case SSM_ERR_UNSUPPORTED: return "the variant cannot run this shape";
        case SSM_ERR_ALIAS: return "an output overlaps an input";
        case SSM_ERR_VARIANT: return "unknown variant";
        case SSM_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of the allocation-free entry point";
        default: return "unknown status";
    }
}

int ssm_scan_select_variant(int batch, int dim, int dstate, int64_t seqlen, int io_dtype) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return SSM_ERR_DTYPE;
    if (!valid_sizes(batch, dim, dstate, seqlen)) return SSM_ERR_DIMS;
    // Channel-parallel walking wins once there are enough channels to keep
    // the GPU busy.  With fewer, short sequences go to the time-parallel
    // CHUNKED variant and longer ones are cut into segments combined by the
    // two-pass chunk carry.  Boundaries timed on GB300 with 16 states, gate
    // on, over 256-6144 channels and 512-32768 steps, for each I/O type (bf16
    // rows are half the bytes, so the fused variant needs more channels
    // before it wins).
    const int64_t nchan = (int64_t)batch * dim;
    if (nchan >= 4096) return SSM_VARIANT_FUSED;
    const bool bf16 = io_dtype == SSM_BF16;
    if (nchan >= 3072) return (bf16 && seqlen > 2048) ? SSM_VARIANT_TWOPASS : SSM_VARIANT_FUSED;
    if (nchan >= 2048 && !bf16) return seqlen <= 2048 ? SSM_VARIANT_FUSED : SSM_VARIANT_TWOPASS;
    return seqlen <= 2048 ? SSM_VARIANT_CHUNKED : SSM_VARIANT_TWOPASS;
}

size_t ssm_scan_fwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                                   int variant) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return (size_t)-1;
    if (!valid_sizes(batch, dim, dstate, seqlen)) return (size_t)-1;
    const int v = resolve_variant(batch, dim, dstate, seqlen, io_dtype, variant);
    if (v < 0) return (size_t)-1;
    return workspace_for(batch, dim, dstate, seqlen, v);
}

size_t ssm_scan_fwd_ckpt_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                                        int variant) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return (size_t)-1;
    if (!valid_sizes(batch, dim, dstate, seqlen)) return (size_t)-1;
    const int v = ckpt_variant(batch, dim, dstate, seqlen, io_dtype, variant);
    if (v < 0) return (size_t)-1;
    return workspace_for(batch, dim, dstate, seqlen, v);
}

}  // extern "C"

namespace {

// Causal convolution fused in front of the scan (ssm_scan_fwd_conv, fused
// mode): filter, bias and history; conv_k = 0 means none.
struct ConvArgs {
    int conv_k = 0;
    const float *w = nullptr;
    const float *b = nullptr;
    const void *state = nullptr;
};

// The device-buffer forward behind ssm_scan_fwd_variant,
// ssm_scan_fwd_from_state and ssm_scan_fwd_conv; h0 is the nullable start
// state.
int fwd_device(const void *x, const void *delta, const float *A, const void *B, const void *C, const float *D,
               const void *z, const float *dt_bias, int delta_softplus, const float *h0, void *y,
               float *final_state, int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
               void *workspace, size_t workspace_bytes, void *stream, int variant,
               const ConvArgs &conv = ConvArgs{}, float *ckpt = nullptr) {
    int rc = validate(x, delta, A, B, C, D, z, dt_bias, y, final_state, batch, dim, dstate, seqlen,
                      io_dtype, h0);
    if (rc != SSM_OK) return rc;
    if (ckpt) {   // the checkpoints overlap nothing else
        if (!aligned(ckpt, 4)) return SSM_ERR_ALIGN;
        const size_t es = elem_size(io_dtype);
        const size_t nx = (size_t)batch * dim * (size_t)seqlen * es;
        const size_t nb = (size_t)batch * dstate * (size_t)seqlen * es;
        const size_t ns = (size_t)batch * dim * dstate * 4;
        const Range ck = range_of(ckpt, ssm_scan_ckpt_size(batch, dim, dstate, seqlen));
        const Range others[] = {range_of(x, nx), range_of(delta, nx), range_of(z, z ? nx : 0),
                                range_of(B, nb), range_of(C, nb), range_of(A, (size_t)dim * dstate * 4),
                                range_of(D, D ? (size_t)dim * 4 : 0), range_of(dt_bias, dt_bias ? (size_t)dim * 4 : 0),
                                range_of(h0, h0 ? ns : 0), range_of(y, nx), range_of(final_state, final_state ? ns : 0)};
        for (const Range &o : others)
            if (overlap(ck, o)) return SSM_ERR_ALIAS;
    }
    const int v = ckpt ? ckpt_variant(batch, dim, dstate, seqlen, io_dtype, variant)
                       : resolve_variant(batch, dim, dstate, seqlen, io_dtype, variant);
    if (v < 0) return v;
    const size_t need = workspace_for(batch, dim, dstate, seqlen, v);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256)))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (batch == 0 || dim == 0) return SSM_OK;
    if (seqlen == 0) {   // the state is unchanged: final = start (or zero)
        const size_t ns = (size_t)batch * dim * dstate * sizeof(float);
        cudaError_t e = cudaSuccess;
        if (final_state && h0 && final_state != h0)
            e = cudaMemcpyAsync(final_state, h0, ns, cudaMemcpyDeviceToDevice, st);
        else if (final_state && !h0)
            e = cudaMemsetAsync(final_state, 0, ns, st);
        return e == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
    }
    ssm::FwdArgs a;
    a.x = x; a.delta = delta; a.A = A; a.B = B; a.C = C; a.D = D; a.z = z; a.dt_bias = dt_bias;
    a.softplus = delta_softplus ? 1 : 0;
    a.y = y; a.final_state = final_state; a.h0 = h0;
    a.batch = batch; a.dim = dim; a.dstate = dstate; a.L = seqlen;
    a.bf16 = io_dtype == SSM_BF16;
    const size_t es = elem_size(io_dtype);
    bool v16 = ((size_t)seqlen * es) % 16 == 0;
    const void *iop[] = {x, delta, B, C, z, y};
    for (const void *q : iop)
        if (q && !aligned(q, 16)) v16 = false;
    a.vec16 = v16 ? 1 : 0;
    a.conv_k = conv.conv_k;
    a.conv_w = conv.w;
    a.conv_b = conv.b;
    a.conv_state = conv.state;
    a.ckpt = ckpt;
    if (conv.conv_k > 0 && v != SSM_VARIANT_FUSED) return SSM_ERR_UNSUPPORTED;
    cudaError_t e;
    switch (v) {
        case SSM_VARIANT_FUSED: e = ssm::launch_fused(a, workspace, st); break;
        case SSM_VARIANT_CHUNKED: e = ssm::launch_chunked(a, workspace, st); break;
        case SSM_VARIANT_TWOPASS: e = ssm::launch_twopass(a, workspace, st); break;
        default: return SSM_ERR_VARIANT;
    }
    return e == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

}  // namespace

extern "C" {

int ssm_scan_fwd_variant(const void *x, const void *delta, const float *A, const void *B,
                         const void *C, const float *D, const void *z, const float *dt_bias,
                         int delta_softplus, void *y, float *final_state,
                         int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                         void *workspace, size_t workspace_bytes, void *stream, int variant) {
    return fwd_device(x, delta, A, B, C, D, z, dt_bias, delta_softplus, nullptr, y, final_state, batch, dim,
                      dstate, seqlen, io_dtype, workspace, workspace_bytes, stream, variant);
}

int ssm_scan_fwd_from_state(const void *x, const void *delta, const float *A, const void *B,
                            const void *C, const float *D, const void *z, const float *dt_bias,
                            int delta_softplus, const float *initial_state, void *y, float *final_state,
                            int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                            void *workspace, size_t workspace_bytes, void *stream, int variant) {
    return fwd_device(x, delta, A, B, C, D, z, dt_bias, delta_softplus, initial_state, y, final_state, batch,
                      dim, dstate, seqlen, io_dtype, workspace, workspace_bytes, stream, variant);
}

int ssm_scan_fwd_ckpt(const void *x, const void *delta, const float *A, const void *B, const void *C,
                      const float *D, const void *z, const float *dt_bias, int delta_softplus,
                      const float *initial_state, void *y, float *final_state, float *ckpt, int batch, int dim,
                      int dstate, int64_t seqlen, int io_dtype, void *workspace, size_t workspace_bytes,
                      void *stream, int variant) {
    if (!ckpt && batch > 0 && dim > 0 && seqlen > 0) return SSM_ERR_NULL;
    return fwd_device(x, delta, A, B, C, D, z, dt_bias, delta_softplus, initial_state, y, final_state, batch,
                      dim, dstate, seqlen, io_dtype, workspace, workspace_bytes, stream, variant, ConvArgs{},
                      ckpt);
}

int ssm_scan_fwd(const void *x, const void *delta, const float *A, const void *B, const void *C,
                 const float *D, const void *z, const float *dt_bias, int delta_softplus, void *y,
                 float *final_state, int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                 void *workspace, size_t workspace_bytes, void *stream) {
    return ssm_scan_fwd_variant(x, delta, A, B, C, D, z, dt_bias, delta_softplus, y, final_state,
                                batch, dim, dstate, seqlen, io_dtype, workspace, workspace_bytes,
                                stream, SSM_VARIANT_AUTO);
}

int ssm_scan_device_status(void *stream, int clear) {
    unsigned int v = 0;
    if (ssm::read_device_status(static_cast<cudaStream_t>(stream), clear != 0, &v) != 0) return SSM_ERR_LAUNCH;
    return (int)(v & 0x7fffffffu);
}

int ssm_scan_selftest_wait_timeout(long long limit_cycles, void *stream) {
    if (limit_cycles < 1 || limit_cycles > (1ll << 31)) return SSM_ERR_DIMS;
    return ssm::selftest_wait_timeout(limit_cycles, static_cast<cudaStream_t>(stream)) == cudaSuccess
               ? SSM_OK
               : SSM_ERR_LAUNCH;
}

size_t ssm_scan_fwd_host_buffer_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                                     int has_D, int has_z, int has_dt_bias, int has_final_state,
                                     int variant) {
    (void)has_final_state;   // the chunk-to-chunk state buffer is always present
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return (size_t)-1;
    if (!valid_sizes(batch, dim, dstate, seqlen)) return (size_t)-1;
    if (resolve_variant(batch, dim, dstate, seqlen, io_dtype, variant) < 0) return (size_t)-1;
    const HostPlan hp = host_plan(batch, dim, seqlen, io_dtype, has_z != 0);
    size_t ws = 0;
    for (int j = 0; j < hp.n; ++j) {
        const int64_t len = hp.len(j);
        const int v = resolve_variant(batch, dim, dstate, len, io_dtype, variant);
        if (v < 0) return (size_t)-1;
        const size_t w = workspace_for(batch, dim, dstate, len, v);
        ws = w > ws ? w : ws;
    }
    const size_t es = elem_size(io_dtype);
    const size_t nx = (size_t)batch * dim * (size_t)seqlen * es;
    const size_t nb = (size_t)batch * dstate * (size_t)seqlen * es;
    size_t total = round256(ws);
    total += 3 * round256(nx) + (has_z ? round256(nx) : 0);      // x, delta, y (, z)
    total += 2 * round256(nb);                                      // B, C
    total += round256((size_t)dim * dstate * 4);                    // A
    total += has_D ? round256((size_t)dim * 4) : 0;
    total += has_dt_bias ? round256((size_t)dim * 4) : 0;
    total += round256((size_t)batch * dim * dstate * 4);            // state carried from chunk to chunk
    return total;
}

int ssm_scan_fwd_host(const void *x, const void *delta, const float *A, const void *B, const void *C,
                      const float *D, const void *z, const float *dt_bias, int delta_softplus,
                      void *y, float *final_state, int batch, int dim, int dstate, int64_t seqlen,
                      int io_dtype, void *device_buffer, size_t device_buffer_bytes, void *stream,
                      int variant) {
    int rc = validate(x, delta, A, B, C, D, z, dt_bias, y, final_state, batch, dim, dstate, seqlen,
                      io_dtype);
    if (rc != SSM_OK) return rc;
    if (resolve_variant(batch, dim, dstate, seqlen, io_dtype, variant) < 0) return SSM_ERR_VARIANT;
    const size_t need = ssm_scan_fwd_host_buffer_size(batch, dim, dstate, seqlen, io_dtype, D != nullptr,
                                                      z != nullptr, dt_bias != nullptr,
                                                      final_state != nullptr, variant);
    if (need == (size_t)-1) return SSM_ERR_DIMS;
    if (!device_buffer || device_buffer_bytes < need || !aligned(device_buffer, 256))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t es = elem_size(io_dtype);
    const size_t nx = (size_t)batch * dim * (size_t)seqlen * es;
    const size_t nb = (size_t)batch * dstate * (size_t)seqlen * es;
    const size_t ns = (size_t)batch * dim * dstate * 4;
    const HostPlan hp = host_plan(batch, dim, seqlen, io_dtype, z != nullptr);
    size_t wsb = 0;
    for (int j = 0; j < hp.n; ++j) {
        const int64_t len = hp.len(j);
        const size_t w = workspace_for(batch, dim, dstate, len, resolve_variant(batch, dim, dstate, len, io_dtype, variant));
        wsb = w > wsb ? w : wsb;
    }
    char *cur = static_cast<char *>(device_buffer);
    auto carve = [&](size_t bytes) { char *r = cur; cur += round256(bytes); return r; };
    char *ws = carve(wsb);
    char *dx = carve(nx), *dd = carve(nx), *dy = carve(nx);
    char *dz = z ? carve(nx) : nullptr;
    char *dB = carve(nb), *dC = carve(nb);
    float *dA = reinterpret_cast<float *>(carve((size_t)dim * dstate * 4));
    float *dD = D ? reinterpret_cast<float *>(carve((size_t)dim * 4)) : nullptr;
    float *dbias = dt_bias ? reinterpret_cast<float *>(carve((size_t)dim * 4)) : nullptr;
    float *dstate_buf = reinterpret_cast<float *>(carve(ns));

    HostStreams *hs = host_streams();
    if (!hs) return SSM_ERR_LAUNCH;
    std::lock_guard<std::mutex> lk(hs->mu);
    // Everything already queued on `stream` comes first; the copy streams
    // join it, and the call returns only after all three are idle.
    bool fail = cudaEventRecord(hs->start, st) != cudaSuccess ||
                cudaStreamWaitEvent(hs->in, hs->start, 0) != cudaSuccess ||
                cudaStreamWaitEvent(hs->out, hs->start, 0) != cudaSuccess;
    const struct { void *dst; const void *src; size_t n; } small[] = {
        {dA, A, (size_t)dim * dstate * 4}, {dD, D, D ? (size_t)dim * 4 : 0},
        {dbias, dt_bias, dt_bias ? (size_t)dim * 4 : 0}};
    for (const auto &c : small)
        if (!fail && c.n) fail = cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, hs->in) != cudaSuccess;
    const size_t rows = (size_t)batch * dim, brows = (size_t)batch * dstate, pitch = (size_t)seqlen * es;
    if (seqlen == 0 || rows == 0) {
        // nothing to copy in; the forward still sets final_state (zeros)
        if (!fail) fail = cudaEventRecord(hs->ready[0], hs->in) != cudaSuccess ||
                          cudaStreamWaitEvent(st, hs->ready[0], 0) != cudaSuccess;
        if (!fail) rc = ssm_scan_fwd_variant(dx, dd, dA, dB, dC, dD, dz, dbias, delta_softplus, dy,
                                             final_state ? dstate_buf : nullptr, batch, dim, dstate, seqlen,
                                             io_dtype, ws, wsb, stream, variant);
        if (!fail && rc == SSM_OK && final_state && ns)
            fail = cudaMemcpyAsync(final_state, dstate_buf, ns, cudaMemcpyDeviceToHost, st) != cudaSuccess;
    } else {
        for (int j = 0; j < hp.n && !fail && rc == SSM_OK; ++j) {
            // chunk j: steps [t0, t0 + len), stored chunk after chunk in the device
            // buffers, each chunk's rows contiguous
            const int64_t t0 = hp.start[j];
            const int64_t len = hp.len(j);
            const size_t wb = (size_t)len * es, off = (size_t)t0 * es;
            char *cx = dx + rows * off, *cd = dd + rows * off, *cy = dy + rows * off;
            char *cz = dz ? dz + rows * off : nullptr;
            char *cB = dB + brows * off, *cC = dC + brows * off;
            const struct { char *dst; const void *src; size_t h; } in[] = {
                {cx, x, rows}, {cd, delta, rows}, {cz, z, z ? rows : 0}, {cB, B, brows}, {cC, C, brows}};
            for (const auto &c : in)
                if (!fail && c.h)
                    fail = cudaMemcpy2DAsync(c.dst, wb, static_cast<const char *>(c.src) + off, pitch, wb, c.h,
                                             cudaMemcpyHostToDevice, hs->in) != cudaSuccess;
            if (fail) break;
            fail = cudaEventRecord(hs->ready[j], hs->in) != cudaSuccess ||
                   cudaStreamWaitEvent(st, hs->ready[j], 0) != cudaSuccess;
            if (fail) break;
            rc = fwd_device(cx, cd, dA, cB, cC, dD, cz, dbias, delta_softplus, j ? dstate_buf : nullptr, cy,
                            dstate_buf, batch, dim, dstate, len, io_dtype, ws, wsb, stream, variant);
            if (rc != SSM_OK) break;
            fail = cudaEventRecord(hs->done[j], st) != cudaSuccess ||
                   cudaStreamWaitEvent(hs->out, hs->done[j], 0) != cudaSuccess ||
                   cudaMemcpy2DAsync(static_cast<char *>(y) + off, pitch, cy, wb, wb, rows, cudaMemcpyDeviceToHost,
                                     hs->out) != cudaSuccess;
        }
        if (!fail && rc == SSM_OK && final_state)
            fail = cudaMemcpyAsync(final_state, dstate_buf, ns, cudaMemcpyDeviceToHost, hs->out) != cudaSuccess;
    }
    // Wait for every queued copy before returning, also after a failure: the
    // copies read and write the caller's host buffers.
    const bool s1 = cudaStreamSynchronize(hs->in) == cudaSuccess;
    const bool s2 = cudaStreamSynchronize(st) == cudaSuccess;
    const bool s3 = cudaStreamSynchronize(hs->out) == cudaSuccess;
    if (rc != SSM_OK) return rc;
    return (!fail && s1 && s2 && s3) ? SSM_OK : SSM_ERR_LAUNCH;
}

}  // extern "C"

// ---------------------------------------------------------------------------
// Convolution in front of the scan.
namespace {

bool conv_fusable(int batch, int dim, int dstate, int64_t seqlen, int io_dtype, int width) {
    return width <= kFusedConvTaps &&
           ssm_scan_select_variant(batch, dim, dstate, seqlen, io_dtype) == SSM_VARIANT_FUSED;
}

int resolve_conv_mode(int batch, int dim, int dstate, int64_t seqlen, int io_dtype, int width, int mode) {
    if (mode == SSM_CONV_AUTO)
        return conv_fusable(batch, dim, dstate, seqlen, io_dtype, width) ? SSM_CONV_FUSED : SSM_CONV_SEPARATE;
    if (mode == SSM_CONV_FUSED) return width <= kFusedConvTaps ? SSM_CONV_FUSED : SSM_ERR_UNSUPPORTED;
    if (mode == SSM_CONV_SEPARATE) return SSM_CONV_SEPARATE;
    return SSM_ERR_VARIANT;
}

size_t conv_out_bytes(int batch, int dim, int64_t seqlen, int io_dtype) {
    return round256((size_t)batch * dim * (size_t)seqlen * elem_size(io_dtype));
}

}  // namespace

extern "C" {

size_t ssm_scan_fwd_conv_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int conv_width,
                                        int io_dtype, int mode) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return (size_t)-1;
    if (!valid_sizes(batch, dim, dstate, seqlen) || conv_width < 1 || conv_width > 8) return (size_t)-1;
    const int m = resolve_conv_mode(batch, dim, dstate, seqlen, io_dtype, conv_width, mode);
    if (m < 0) return (size_t)-1;
    if (m == SSM_CONV_FUSED) return workspace_for(batch, dim, dstate, seqlen, SSM_VARIANT_FUSED);
    const int v = resolve_variant(batch, dim, dstate, seqlen, io_dtype, SSM_VARIANT_AUTO);
    if (batch <= 0 || dim <= 0 || seqlen <= 0) return 0;
    return conv_out_bytes(batch, dim, seqlen, io_dtype) + workspace_for(batch, dim, dstate, seqlen, v);
}

int ssm_scan_fwd_conv(const void *x, const float *conv_weight, const float *conv_bias, const void *conv_state,
                      int conv_width, const void *delta, const float *A, const void *B, const void *C,
                      const float *D, const void *z, const float *dt_bias, int delta_softplus, void *y,
                      float *final_state, int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                      void *workspace, size_t workspace_bytes, void *stream, int mode) {
    int rc = validate(x, delta, A, B, C, D, z, dt_bias, y, final_state, batch, dim, dstate, seqlen, io_dtype);
    if (rc != SSM_OK) return rc;
    if (conv_width < 1 || conv_width > 8) return SSM_ERR_DIMS;
    const int m = resolve_conv_mode(batch, dim, dstate, seqlen, io_dtype, conv_width, mode);
    if (m < 0) return m;
    const bool empty = batch == 0 || dim == 0 || seqlen == 0;
    if (!empty && !conv_weight) return SSM_ERR_NULL;
    if ((conv_weight && !aligned(conv_weight, 4)) || (conv_bias && !aligned(conv_bias, 4)) ||
        (conv_state && !aligned(conv_state, elem_size(io_dtype))))
        return SSM_ERR_ALIGN;
    if (!empty) {
        // the outputs must not overlap the convolution's inputs either
        const size_t nx = (size_t)batch * dim * (size_t)seqlen * elem_size(io_dtype);
        const Range cin[] = {range_of(conv_weight, (size_t)dim * conv_width * 4),
                             range_of(conv_bias, conv_bias ? (size_t)dim * 4 : 0),
                             range_of(conv_state, conv_state ? (size_t)batch * dim * (conv_width - 1) *
                                                                    elem_size(io_dtype)
                                                              : 0)};
        const Range outs[] = {range_of(y, nx),
                              range_of(final_state, final_state ? (size_t)batch * dim * dstate * 4 : 0)};
        for (const Range &o : outs)
            for (const Range &i : cin)
                if (overlap(o, i)) return SSM_ERR_ALIAS;
    }
    const size_t need = ssm_scan_fwd_conv_workspace_size(batch, dim, dstate, seqlen, conv_width, io_dtype, m);
    if (need > 0 && (!workspace || workspace_bytes < need || !aligned(workspace, 256))) return SSM_ERR_WORKSPACE;
    if (m == SSM_CONV_FUSED) {
        ConvArgs cv;
        cv.conv_k = empty ? 0 : conv_width;
        cv.w = conv_weight;
        cv.b = conv_bias;
        cv.state = conv_state;
        return fwd_device(x, delta, A, B, C, D, z, dt_bias, delta_softplus, nullptr, y, final_state, batch, dim,
                          dstate, seqlen, io_dtype, workspace, workspace_bytes, stream, SSM_VARIANT_FUSED, cv);
    }
    // separate: the convolution's output goes to the front of the workspace,
    // the scan reads it from there
    if (empty)
        return fwd_device(x, delta, A, B, C, D, z, dt_bias, delta_softplus, nullptr, y, final_state, batch, dim,
                          dstate, seqlen, io_dtype, workspace, workspace_bytes, stream, SSM_VARIANT_AUTO);
    const size_t xb = conv_out_bytes(batch, dim, seqlen, io_dtype);
    rc = ssm_conv1d_fwd(x, conv_weight, conv_bias, conv_state, workspace, nullptr, 1, batch, dim, seqlen,
                        conv_width, io_dtype, stream);
    if (rc != SSM_OK) return rc;
    return fwd_device(workspace, delta, A, B, C, D, z, dt_bias, delta_softplus, nullptr, y, final_state, batch,
                      dim, dstate, seqlen, io_dtype, static_cast<char *>(workspace) + xb, workspace_bytes - xb,
                      stream, SSM_VARIANT_AUTO);
}

}  // extern "C"
