// C ABI of libssmscan: argument validation, variant selection and the
// device- and host-buffer entry points.  Declared in include/ssm_scan.h.
#include "../../include/ssm_scan.h"
#include "scan_internal.h"

#include <cstring>

namespace {

constexpr int kVersion = (1 << 16) | 0;

bool valid_sizes(int batch, int dim, int dstate, int64_t seqlen) {
    return batch >= 0 && dim >= 0 && dstate >= 1 && dstate <= 64 && seqlen >= 0;
}

size_t elem_size(int io_dtype) { return io_dtype == SSM_BF16 ? 2 : 4; }

int resolve_variant(int batch, int dim, int dstate, int64_t seqlen, int io_dtype, int variant) {
    if (variant == SSM_VARIANT_AUTO) return ssm_scan_select_variant(batch, dim, dstate, seqlen, io_dtype);
    if (variant < SSM_VARIANT_FUSED || variant > SSM_VARIANT_TWOPASS) return SSM_ERR_VARIANT;
    return variant;
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
    return 0;
}

size_t round256(size_t n) { return (n + 255) / 256 * 256; }

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
    // Channel-parallel walking fills the GPU when there are enough channels
    // (or the sequence is short); otherwise the sequence is cut into
    // segments combined by the two-pass chunk carry.  The warp-shuffle
    // CHUNKED variant is available on request.
    const int64_t nchan = (int64_t)batch * dim;
    if (nchan >= 4096 || seqlen <= 2048) return SSM_VARIANT_FUSED;
    return SSM_VARIANT_TWOPASS;
}

size_t ssm_scan_fwd_workspace_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                                   int variant) {
    if (io_dtype != SSM_F32 && io_dtype != SSM_BF16) return (size_t)-1;
    if (!valid_sizes(batch, dim, dstate, seqlen)) return (size_t)-1;
    const int v = resolve_variant(batch, dim, dstate, seqlen, io_dtype, variant);
    if (v < 0) return (size_t)-1;
    return workspace_for(batch, dim, dstate, seqlen, v);
}

}  // extern "C"

namespace {

// The device-buffer forward behind ssm_scan_fwd_variant and
// ssm_scan_fwd_from_state; h0 is the nullable start state.
int fwd_device(const void *x, const void *delta, const float *A, const void *B, const void *C, const float *D,
               const void *z, const float *dt_bias, int delta_softplus, const float *h0, void *y,
               float *final_state, int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
               void *workspace, size_t workspace_bytes, void *stream, int variant) {
    int rc = validate(x, delta, A, B, C, D, z, dt_bias, y, final_state, batch, dim, dstate, seqlen,
                      io_dtype, h0);
    if (rc != SSM_OK) return rc;
    const int v = resolve_variant(batch, dim, dstate, seqlen, io_dtype, variant);
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
    cudaError_t e;
    switch (v) {
        case SSM_VARIANT_FUSED: e = ssm::launch_fused(a, workspace, st); break;
        case SSM_VARIANT_CHUNKED: e = ssm::launch_chunked(a, st); break;
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

size_t ssm_scan_fwd_host_buffer_size(int batch, int dim, int dstate, int64_t seqlen, int io_dtype,
                                     int has_D, int has_z, int has_dt_bias, int has_final_state,
                                     int variant) {
    const size_t ws = ssm_scan_fwd_workspace_size(batch, dim, dstate, seqlen, io_dtype, variant);
    if (ws == (size_t)-1) return (size_t)-1;
    const size_t es = elem_size(io_dtype);
    const size_t nx = (size_t)batch * dim * (size_t)seqlen * es;
    const size_t nb = (size_t)batch * dstate * (size_t)seqlen * es;
    size_t total = round256(ws);
    total += 3 * round256(nx) + (has_z ? round256(nx) : 0);      // x, delta, y (, z)
    total += 2 * round256(nb);                                      // B, C
    total += round256((size_t)dim * dstate * 4);                    // A
    total += has_D ? round256((size_t)dim * 4) : 0;
    total += has_dt_bias ? round256((size_t)dim * 4) : 0;
    total += has_final_state ? round256((size_t)batch * dim * dstate * 4) : 0;
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
    const int v = resolve_variant(batch, dim, dstate, seqlen, io_dtype, variant);
    if (v < 0) return v;
    const size_t need = ssm_scan_fwd_host_buffer_size(batch, dim, dstate, seqlen, io_dtype, D != nullptr,
                                                      z != nullptr, dt_bias != nullptr,
                                                      final_state != nullptr, v);
    if (!device_buffer || device_buffer_bytes < need || !aligned(device_buffer, 256))
        return SSM_ERR_WORKSPACE;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const size_t es = elem_size(io_dtype);
    const size_t nx = (size_t)batch * dim * (size_t)seqlen * es;
    const size_t nb = (size_t)batch * dstate * (size_t)seqlen * es;
    char *cur = static_cast<char *>(device_buffer);
    auto carve = [&](size_t bytes) { char *r = cur; cur += round256(bytes); return r; };
    void *ws = carve(workspace_for(batch, dim, dstate, seqlen, v));
    void *dx = carve(nx), *dd = carve(nx), *dy = carve(nx);
    void *dz = z ? carve(nx) : nullptr;
    void *dB = carve(nb), *dC = carve(nb);
    float *dA = reinterpret_cast<float *>(carve((size_t)dim * dstate * 4));
    float *dD = D ? reinterpret_cast<float *>(carve((size_t)dim * 4)) : nullptr;
    float *dbias = dt_bias ? reinterpret_cast<float *>(carve((size_t)dim * 4)) : nullptr;
    float *dfs = final_state ? reinterpret_cast<float *>(carve((size_t)batch * dim * dstate * 4)) : nullptr;
    struct Copy { void *dst; const void *src; size_t n; };
    const Copy in[] = {{dx, x, nx}, {dd, delta, nx}, {dz, z, z ? nx : 0}, {dB, B, nb}, {dC, C, nb},
                       {dA, A, (size_t)dim * dstate * 4}, {dD, D, D ? (size_t)dim * 4 : 0},
                       {dbias, dt_bias, dt_bias ? (size_t)dim * 4 : 0}};
    for (const Copy &c : in)
        if (c.n && cudaMemcpyAsync(c.dst, c.src, c.n, cudaMemcpyHostToDevice, st) != cudaSuccess)
            return SSM_ERR_LAUNCH;
    rc = ssm_scan_fwd_variant(dx, dd, dA, dB, dC, dD, dz, dbias, delta_softplus, dy, dfs, batch, dim,
                              dstate, seqlen, io_dtype, ws, round256(workspace_for(batch, dim, dstate, seqlen, v)),
                              stream, v);
    if (rc != SSM_OK) return rc;
    if (nx && cudaMemcpyAsync(y, dy, nx, cudaMemcpyDeviceToHost, st) != cudaSuccess) return SSM_ERR_LAUNCH;
    if (dfs && cudaMemcpyAsync(final_state, dfs, (size_t)batch * dim * dstate * 4, cudaMemcpyDeviceToHost,
                               st) != cudaSuccess)
        return SSM_ERR_LAUNCH;
    return cudaStreamSynchronize(st) == cudaSuccess ? SSM_OK : SSM_ERR_LAUNCH;
}

}  // extern "C"
