// gdn_api.cu -- the C ABI declared in include/gdn.h: host-side argument
// validation, workspace carving and kernel launches.  No allocation, no
// synchronisation.
#include <atomic>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>

#include "gdn.h"
#include "gdn_testing.h"
#include "gdn_internal.cuh"

namespace {

thread_local std::string g_last_error;

gdn_status fail(gdn_status s, const char* fmt, ...) __attribute__((format(printf, 2, 3)));
gdn_status fail(gdn_status s, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
    return s;
}

// First CUDA error the library has seen that leaves the context unusable (a fault of an earlier
// kernel, which every later launch and copy reports), kept for gdn_last_async_error; 0 = none yet.
std::atomic<int> g_sticky_error{0};

// the error codes CUDA documents as corrupting the context: once one is seen, every later call in
// the process returns it, so it is kept rather than reported once
bool context_fatal(cudaError_t e)
{
    switch (e) {
    case cudaErrorIllegalAddress:
    case cudaErrorLaunchFailure:
    case cudaErrorIllegalInstruction:
    case cudaErrorMisalignedAddress:
    case cudaErrorInvalidAddressSpace:
    case cudaErrorInvalidPc:
    case cudaErrorHardwareStackError:
    case cudaErrorLaunchTimeout:
    case cudaErrorAssert:
    case cudaErrorECCUncorrectable:
        return true;
    default:
        return false;
    }
}

void note_cuda_error(cudaError_t e)
{
    int none = 0;
    if (context_fatal(e)) g_sticky_error.compare_exchange_strong(none, (int)e);
}

gdn_status cuda_fail(cudaError_t e, const char* what)
{
    note_cuda_error(e);
    return fail(GDN_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

gdn_status check_dims(const gdn_dims* d)
{
    if (!d) return fail(GDN_ERR_INVALID_ARG, "dims is NULL");
    if (d->hk < 1 || d->hv < 1 || d->hv % d->hk != 0)
        return fail(GDN_ERR_INVALID_ARG, "need hk >= 1 and hv a multiple of hk (hk=%d hv=%d)", d->hk, d->hv);
    if (d->dk != gdn::kHeadDim || d->dv != gdn::kHeadDim)
        return fail(GDN_ERR_UNSUPPORTED, "only dk = dv = 128 is implemented (dk=%d dv=%d)", d->dk, d->dv);
    if (d->hv > 4096) return fail(GDN_ERR_UNSUPPORTED, "hv=%d above 4096", d->hv);
    if (!(d->eps > 0.0f) || !std::isfinite(d->eps))
        return fail(GDN_ERR_INVALID_ARG, "eps must be finite and > 0");
    return GDN_OK;
}

gdn_status check_batch(int32_t n_seq, int32_t T, const int32_t* cu)
{
    if (n_seq < 0 || T < 0) return fail(GDN_ERR_INVALID_ARG, "negative n_seq or total_tokens");
    if (n_seq == 0 && T != 0) return fail(GDN_ERR_INVALID_ARG, "tokens without sequences");
    if (n_seq > 65535) return fail(GDN_ERR_UNSUPPORTED, "n_seq=%d above 65535", n_seq);
    if (n_seq > 0 && !cu) return fail(GDN_ERR_INVALID_ARG, "cu_seqlens is NULL");
    if (cu && (reinterpret_cast<uintptr_t>(cu) & 3u)) return fail(GDN_ERR_ALIGNMENT, "cu_seqlens not 4-byte aligned");
    return GDN_OK;
}

struct Buf {
    const void* p;
    size_t bytes;
    const char* name;
};

// every non-empty buffer present and 16-byte aligned
gdn_status check_bufs(const Buf* b, int n)
{
    for (int i = 0; i < n; ++i) {
        if (b[i].bytes == 0) continue;
        if (!b[i].p) return fail(GDN_ERR_INVALID_ARG, "%s is NULL", b[i].name);
        if (!aligned16(b[i].p)) return fail(GDN_ERR_ALIGNMENT, "%s is not 16-byte aligned", b[i].name);
    }
    return GDN_OK;
}

bool overlap(const Buf& a, const Buf& b)
{
    if (a.bytes == 0 || b.bytes == 0) return false;
    auto pa = reinterpret_cast<uintptr_t>(a.p), pb = reinterpret_cast<uintptr_t>(b.p);
    return pa < pb + b.bytes && pb < pa + a.bytes;
}

// no output may overlap another output or any input
gdn_status check_disjoint(const Buf* outs, int n_out, const Buf* ins, int n_in)
{
    for (int i = 0; i < n_out; ++i) {
        for (int j = i + 1; j < n_out; ++j)
            if (overlap(outs[i], outs[j]))
                return fail(GDN_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, outs[j].name);
        for (int j = 0; j < n_in; ++j)
            if (overlap(outs[i], ins[j]))
                return fail(GDN_ERR_INVALID_ARG, "%s overlaps %s", outs[i].name, ins[j].name);
    }
    return GDN_OK;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int channels(const gdn_dims* d) { return 2 * d->hk * d->dk + d->hv * d->dv; }

}  // namespace

namespace gdn {
void set_last_error(const char* msg) { g_last_error = msg; }
}  // namespace gdn

extern "C" {

const char* gdn_status_string(gdn_status s)
{
    switch (s) {
    case GDN_OK: return "GDN_OK";
    case GDN_ERR_INVALID_ARG: return "GDN_ERR_INVALID_ARG";
    case GDN_ERR_UNSUPPORTED: return "GDN_ERR_UNSUPPORTED";
    case GDN_ERR_ALIGNMENT: return "GDN_ERR_ALIGNMENT";
    case GDN_ERR_WORKSPACE: return "GDN_ERR_WORKSPACE";
    case GDN_ERR_CUDA: return "GDN_ERR_CUDA";
    case GDN_ERR_TIMEOUT: return "GDN_ERR_TIMEOUT";
    }
    return "GDN_ERR_UNKNOWN";
}

const char* gdn_last_error_string(void) { return g_last_error.c_str(); }

gdn_status gdn_last_async_error(void)
{
    // what the runtime has already observed (peek: no synchronisation, nothing cleared)
    note_cuda_error(cudaPeekAtLastError());
    const int e = g_sticky_error.load();
    if (e == 0) return GDN_OK;
    return fail(GDN_ERR_CUDA, "an earlier kernel faulted and the CUDA context is unusable: %s",
                cudaGetErrorString((cudaError_t)e));
}

}  // extern "C"

namespace {

gdn_status prep_pre(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                    const uint16_t* qkv, const float* conv_w, const uint16_t* hist_in, uint16_t* hist_out,
                    const uint16_t* a, const uint16_t* b, const float* A_log, const float* dt_bias, float* qn,
                    float* kn, float* vc, float* glog, float* beta, gdn::PreParams& p, bool kq_images = false)
{
    gdn_status st;
    if ((st = check_dims(dims)) != GDN_OK) return st;
    if ((st = check_batch(n_seq, T, cu_seqlens)) != GDN_OK) return st;
    const size_t C = (size_t)channels(dims), hk = dims->hk, hv = dims->hv, d = dims->dk, tt = (size_t)T;
    const Buf bufs[] = {
        {qkv, tt * C * 2, "qkv"},        {conv_w, C * 16, "conv_w"},
        {hist_in, n_seq * C * 6, "hist_in"}, {hist_out, n_seq * C * 6, "hist_out"},
        {a, tt * hv * 2, "a"},           {b, tt * hv * 2, "b"},
        {A_log, hv * 4, "A_log"},        {dt_bias, hv * 4, "dt_bias"},
        // inside gdn_layer q and k go to the scan's images instead (no qn / kn buffers)
        {qn, kq_images ? 0 : tt * hk * d * 4, "qn"}, {kn, kq_images ? 0 : tt * hk * d * 4, "kn"},
        {vc, tt * hv * d * 4, "vc"},     {glog, tt * hv * 4, "glog"},
        {beta, tt * hv * 4, "beta"},
    };
    if ((st = check_bufs(bufs, sizeof bufs / sizeof bufs[0])) != GDN_OK) return st;
    // hist_out may be hist_in itself (the history is then written by a trailing launch, after every
    // read of the old history); any other overlap is rejected
    const bool hist_in_place = hist_out == hist_in && bufs[3].bytes > 0;
    const Buf ins[] = {bufs[0], bufs[1], bufs[2], bufs[4], bufs[5], bufs[6], bufs[7]};
    const Buf outs[] = {bufs[3], bufs[8], bufs[9], bufs[10], bufs[11], bufs[12]};
    if (hist_in_place) {
        const Buf ins_x[] = {bufs[0], bufs[1], bufs[4], bufs[5], bufs[6], bufs[7]};
        if ((st = check_disjoint(outs, 6, ins_x, 6)) != GDN_OK) return st;
        for (int i = 1; i < 6; ++i)
            if (overlap(outs[i], bufs[2])) return fail(GDN_ERR_INVALID_ARG, "%s overlaps hist_in", outs[i].name);
    } else if ((st = check_disjoint(outs, 6, ins, 7)) != GDN_OK) {
        return st;
    }
    p = gdn::PreParams{};
    p.hist_in_place = hist_in_place ? 1 : 0;
    p.hk = dims->hk; p.hv = dims->hv; p.C = (int)C; p.T = T; p.n_seq = n_seq; p.eps = dims->eps;
    p.cu_seqlens = cu_seqlens;
    p.qkv = reinterpret_cast<const __half*>(qkv);
    p.conv_w = conv_w;
    p.hist_in = reinterpret_cast<const __half*>(hist_in);
    p.hist_out = reinterpret_cast<__half*>(hist_out);
    p.a = reinterpret_cast<const __half*>(a);
    p.b = reinterpret_cast<const __half*>(b);
    p.A_log = A_log; p.dt_bias = dt_bias;
    p.qn = qn; p.kn = kn; p.vc = vc; p.glog = glog; p.beta = beta;
    return GDN_OK;
}

gdn_status run_pre(const gdn::PreParams& p, struct CUstream_st* stream)
{
    if (p.n_seq == 0) return GDN_OK;
    cudaError_t e = gdn::launch_pre(p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_pre launch");
}

gdn_status prep_scan(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                     const float* qn, const float* kn, const float* vc, const float* glog, const float* beta,
                     const float* S_in, float* S_out, float* o, void* workspace, size_t workspace_bytes,
                     gdn::ScanParams& p, bool kq_images = false)
{
    gdn_status st;
    if ((st = check_dims(dims)) != GDN_OK) return st;
    if ((st = check_batch(n_seq, T, cu_seqlens)) != GDN_OK) return st;
    const size_t hk = dims->hk, hv = dims->hv, d = dims->dk, tt = (size_t)T;
    const Buf bufs[] = {
        {qn, kq_images ? 0 : tt * hk * d * 4, "qn"}, {kn, kq_images ? 0 : tt * hk * d * 4, "kn"},
        {vc, tt * hv * d * 4, "vc"},
        {glog, tt * hv * 4, "glog"},   {beta, tt * hv * 4, "beta"},
        {S_in, n_seq * hv * d * d * 4, "S_in"}, {S_out, n_seq * hv * d * d * 4, "S_out"},
        {o, tt * hv * d * 4, "o"},
    };
    if ((st = check_bufs(bufs, sizeof bufs / sizeof bufs[0])) != GDN_OK) return st;
    if (bufs[5].p != bufs[6].p && overlap(bufs[5], bufs[6]))
        return fail(GDN_ERR_INVALID_ARG, "S_out partially overlaps S_in (identical buffers are allowed)");
    const Buf ins[] = {bufs[0], bufs[1], bufs[2], bufs[3], bufs[4]};
    const Buf outs[] = {bufs[6], bufs[7]};
    if ((st = check_disjoint(outs, 2, ins, 5)) != GDN_OK) return st;
    if (overlap(bufs[7], bufs[5])) return fail(GDN_ERR_INVALID_ARG, "o overlaps S_in");
    const size_t need = gdn::scan_workspace_bytes(dims->hk, dims->hv, n_seq, T);
    if (workspace_bytes < need || (need && !workspace))
        return fail(GDN_ERR_WORKSPACE, "scan workspace %zu bytes, need %zu", workspace_bytes, need);
    if (need && !aligned16(workspace)) return fail(GDN_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
    p = gdn::ScanParams{};
    p.hk = dims->hk; p.hv = dims->hv; p.T = T; p.n_seq = n_seq; p.cu_seqlens = cu_seqlens;
    p.qn = qn; p.kn = kn; p.vc = vc; p.glog = glog; p.beta = beta; p.S_in = S_in; p.S_out = S_out; p.o = o;
    p.workspace = workspace; p.workspace_bytes = workspace_bytes;
    return GDN_OK;
}

gdn_status run_scan(const gdn::ScanParams& p, struct CUstream_st* stream)
{
    if (p.n_seq == 0) {  // nothing to compute; the failure record still starts clean
        cudaError_t e = p.workspace ? cudaMemsetAsync(p.workspace, 0, 4, reinterpret_cast<cudaStream_t>(stream))
                                    : cudaSuccess;
        return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_scan workspace clear");
    }
    cudaError_t e = gdn::launch_scan(p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_scan launch");
}

// the scan's failure record: the first 4 bytes of its workspace
gdn_status read_failure_word(const void* word, struct CUstream_st* stream)
{
    if (!word) return fail(GDN_ERR_INVALID_ARG, "workspace is NULL");
    uint32_t h = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    cudaError_t e = cudaMemcpyAsync(&h, word, sizeof h, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "reading the scan's failure record");
    if (h) return fail(GDN_ERR_TIMEOUT, "a bounded wait in the scan kernels expired (record 0x%x); outputs are invalid", h);
    return GDN_OK;
}

// offset of the scan workspace inside a gdn_layer workspace (the stage tensors vc, o, glog and beta
// come first; q and k live only in the scan workspace's images)
size_t layer_scan_offset(const gdn_dims* dims, int32_t T)
{
    const size_t hv = dims->hv, d = dims->dk, tt = (size_t)T;
    return align256(tt * hv * d * 4) * 2 + align256(tt * hv * 4) * 2;
}

gdn_status prep_post(const gdn_dims* dims, int32_t T, const float* o, const uint16_t* z, const float* gamma,
                     int32_t out_f32, void* y, gdn::PostParams& p)
{
    gdn_status st;
    if ((st = check_dims(dims)) != GDN_OK) return st;
    if (T < 0) return fail(GDN_ERR_INVALID_ARG, "negative total_tokens");
    if (out_f32 != 0 && out_f32 != 1) return fail(GDN_ERR_INVALID_ARG, "out_f32 must be 0 or 1");
    const size_t hv = dims->hv, d = dims->dv, tt = (size_t)T;
    const Buf bufs[] = {
        {o, tt * hv * d * 4, "o"}, {z, tt * hv * d * 2, "z"}, {gamma, d * 4, "gamma"},
        {y, tt * hv * d * (out_f32 ? 4 : 2), "y"},
    };
    if ((st = check_bufs(bufs, 4)) != GDN_OK) return st;
    if (overlap(bufs[3], bufs[0]) || overlap(bufs[3], bufs[1]))
        return fail(GDN_ERR_INVALID_ARG, "y overlaps an input");
    p = gdn::PostParams{};
    p.hv = dims->hv; p.T = T; p.eps = dims->eps; p.o = o; p.z = reinterpret_cast<const __half*>(z);
    p.gamma = gamma; p.out_f32 = out_f32; p.y = y;
    return GDN_OK;
}

gdn_status run_post(const gdn::PostParams& p, struct CUstream_st* stream)
{
    cudaError_t e = gdn::launch_post(p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_post launch");
}

}  // namespace

extern "C" {

gdn_status gdn_pre(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                   const uint16_t* qkv, const float* conv_w, const uint16_t* hist_in, uint16_t* hist_out,
                   const uint16_t* a, const uint16_t* b, const float* A_log, const float* dt_bias, float* qn,
                   float* kn, float* vc, float* glog, float* beta, struct CUstream_st* stream)
{
    gdn::PreParams p;
    gdn_status st = prep_pre(dims, n_seq, T, cu_seqlens, qkv, conv_w, hist_in, hist_out, a, b, A_log, dt_bias,
                             qn, kn, vc, glog, beta, p);
    return st != GDN_OK ? st : run_pre(p, stream);
}

size_t gdn_scan_workspace_bytes(const gdn_dims* dims, int32_t n_seq, int32_t T)
{
    if (!dims || n_seq < 0 || T < 0) return 0;
    return gdn::scan_workspace_bytes(dims->hk, dims->hv, n_seq, T);
}

gdn_status gdn_scan(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                    const float* qn, const float* kn, const float* vc, const float* glog, const float* beta,
                    const float* S_in, float* S_out, float* o, void* workspace, size_t workspace_bytes,
                    struct CUstream_st* stream)
{
    gdn::ScanParams p;
    gdn_status st = prep_scan(dims, n_seq, T, cu_seqlens, qn, kn, vc, glog, beta, S_in, S_out, o, workspace,
                              workspace_bytes, p);
    return st != GDN_OK ? st : run_scan(p, stream);
}

gdn_status gdn_scan_fast(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                         const float* qn, const float* kn, const float* vc, const float* glog, const float* beta,
                         const float* S_in, float* S_out, float* o, void* workspace, size_t workspace_bytes,
                         struct CUstream_st* stream)
{
    gdn::ScanParams p;
    gdn_status st = prep_scan(dims, n_seq, T, cu_seqlens, qn, kn, vc, glog, beta, S_in, S_out, o, workspace,
                              workspace_bytes, p);
    if (st != GDN_OK) return st;
    p.fast = 1;
    return run_scan(p, stream);
}

gdn_status gdn_post(const gdn_dims* dims, int32_t T, const float* o, const uint16_t* z, const float* gamma,
                    int32_t out_f32, void* y, struct CUstream_st* stream)
{
    gdn::PostParams p;
    gdn_status st = prep_post(dims, T, o, z, gamma, out_f32, y, p);
    return st != GDN_OK ? st : run_post(p, stream);
}

size_t gdn_layer_workspace_bytes(const gdn_dims* dims, int32_t n_seq, int32_t T)
{
    if (!dims || n_seq < 0 || T < 0) return 0;
    const size_t hv = dims->hv, d = dims->dk, tt = (size_t)T;
    size_t total = 0;                         // no qn, kn: q and k go straight into the scan's images
    total += align256(tt * hv * d * 4) * 2;  // vc, o
    total += align256(tt * hv * 4) * 2;      // glog, beta
    total += align256(gdn::scan_workspace_bytes(dims->hk, dims->hv, n_seq, T));
    return total;
}

static gdn_status layer_impl(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                             const uint16_t* qkv, const float* conv_w, const uint16_t* hist_in, uint16_t* hist_out,
                             const uint16_t* a, const uint16_t* b, const uint16_t* z, const float* A_log,
                             const float* dt_bias, const float* gamma, const float* S_in, float* S_out,
                             int32_t out_f32, void* y, void* workspace, size_t workspace_bytes,
                             struct CUstream_st* stream, int fast, int stages)
{
    gdn_status st;
    if (stages < 0 || stages > 7) return fail(GDN_ERR_INVALID_ARG, "stage mask %d outside 0..7", stages);
    if ((st = check_dims(dims)) != GDN_OK) return st;
    if ((st = check_batch(n_seq, T, cu_seqlens)) != GDN_OK) return st;
    const size_t need = gdn_layer_workspace_bytes(dims, n_seq, T);
    if (workspace_bytes < need || (need && !workspace))
        return fail(GDN_ERR_WORKSPACE, "layer workspace %zu bytes, need %zu", workspace_bytes, need);
    if (need && !aligned16(workspace)) return fail(GDN_ERR_ALIGNMENT, "workspace is not 16-byte aligned");
    const size_t hv = dims->hv, d = dims->dk, tt = (size_t)T;
    char* w = static_cast<char*>(workspace);
    auto carve = [&](size_t bytes) { char* r = w; w += align256(bytes); return r; };
    // (no qn / kn: q and k go from the pre kernel straight into the scan's [K; Q] operand images,
    // bf16 hi / lo split exactly as the scan splits fp32 inputs, and the scan's gram kernel only
    // copies them in)
    float* vc = reinterpret_cast<float*>(carve(tt * hv * d * 4));
    float* o = reinterpret_cast<float*>(carve(tt * hv * d * 4));
    float* glog = reinterpret_cast<float*>(carve(tt * hv * 4));
    float* beta = reinterpret_cast<float*>(carve(tt * hv * 4));
    const size_t scan_ws = gdn::scan_workspace_bytes(dims->hk, dims->hv, n_seq, T);
    void* sws = scan_ws ? carve(scan_ws) : nullptr;
    // the y buffer must not alias the stage inputs the later stages still read
    const Buf ybuf{y, tt * hv * d * (out_f32 ? 4 : 2), "y"};
    const Buf ins[] = {{qkv, tt * (size_t)channels(dims) * 2, "qkv"}, {z, tt * hv * d * 2, "z"},
                       {workspace, need, "workspace"}};
    for (const Buf& in : ins)
        if (overlap(ybuf, in)) return fail(GDN_ERR_INVALID_ARG, "y overlaps %s", in.name);
    // validate all three stages before anything is enqueued
    gdn::PreParams pp;
    gdn::ScanParams sp;
    gdn::PostParams op;
    if ((st = prep_pre(dims, n_seq, T, cu_seqlens, qkv, conv_w, hist_in, hist_out, a, b, A_log, dt_bias, nullptr,
                       nullptr, vc, glog, beta, pp, true)) != GDN_OK)
        return st;
    if ((st = prep_scan(dims, n_seq, T, cu_seqlens, nullptr, nullptr, vc, glog, beta, S_in, S_out, o, sws, scan_ws,
                        sp, true)) != GDN_OK)
        return st;
    if ((st = prep_post(dims, T, o, z, gamma, out_f32, y, op)) != GDN_OK) return st;
    sp.fast = fast;
    if (T > 0) {
        pp.kq_images = static_cast<unsigned char*>(sws) + gdn::scan_kq_images_offset(dims->hk, dims->hv, n_seq, T);
        sp.kq_written = 1;
    }
    if ((stages & 1) && (st = run_pre(pp, stream)) != GDN_OK) return st;
    if ((stages & 2) && (st = run_scan(sp, stream)) != GDN_OK) return st;
    return (stages & 4) ? run_post(op, stream) : GDN_OK;
}

gdn_status gdn_layer(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                     const uint16_t* qkv, const float* conv_w, const uint16_t* hist_in, uint16_t* hist_out,
                     const uint16_t* a, const uint16_t* b, const uint16_t* z, const float* A_log,
                     const float* dt_bias, const float* gamma, const float* S_in, float* S_out,
                     int32_t out_f32, void* y, void* workspace, size_t workspace_bytes,
                     struct CUstream_st* stream)
{
    return layer_impl(dims, n_seq, T, cu_seqlens, qkv, conv_w, hist_in, hist_out, a, b, z, A_log, dt_bias, gamma,
                      S_in, S_out, out_f32, y, workspace, workspace_bytes, stream, 0, 7);
}

gdn_status gdn_layer_fast(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                          const uint16_t* qkv, const float* conv_w, const uint16_t* hist_in, uint16_t* hist_out,
                          const uint16_t* a, const uint16_t* b, const uint16_t* z, const float* A_log,
                          const float* dt_bias, const float* gamma, const float* S_in, float* S_out,
                          int32_t out_f32, void* y, void* workspace, size_t workspace_bytes,
                          struct CUstream_st* stream)
{
    return layer_impl(dims, n_seq, T, cu_seqlens, qkv, conv_w, hist_in, hist_out, a, b, z, A_log, dt_bias, gamma,
                      S_in, S_out, out_f32, y, workspace, workspace_bytes, stream, 1, 7);
}

gdn_status gdn_layer_selftest_stages(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                                     const uint16_t* qkv, const float* conv_w, const uint16_t* hist_in,
                                     uint16_t* hist_out, const uint16_t* a, const uint16_t* b, const uint16_t* z,
                                     const float* A_log, const float* dt_bias, const float* gamma, const float* S_in,
                                     float* S_out, int32_t out_f32, void* y, void* workspace, size_t workspace_bytes,
                                     int32_t fast, int32_t stages, struct CUstream_st* stream)
{
    return layer_impl(dims, n_seq, T, cu_seqlens, qkv, conv_w, hist_in, hist_out, a, b, z, A_log, dt_bias, gamma,
                      S_in, S_out, out_f32, y, workspace, workspace_bytes, stream, fast ? 1 : 0, stages);
}

}  // extern "C"

extern "C" {

gdn_status gdn_step(const gdn_dims* dims, int32_t n_seq, const uint16_t* qkv, const float* conv_w,
                    const uint16_t* hist_in, uint16_t* hist_out, const uint16_t* a, const uint16_t* b,
                    const uint16_t* z, const float* A_log, const float* dt_bias, const float* gamma,
                    const float* S_in, float* S_out, int32_t out_f32, void* y, struct CUstream_st* stream)
{
    gdn_status st;
    if ((st = check_dims(dims)) != GDN_OK) return st;
    if (n_seq < 0) return fail(GDN_ERR_INVALID_ARG, "negative n_seq");
    if (n_seq > 65535) return fail(GDN_ERR_UNSUPPORTED, "n_seq=%d above 65535", n_seq);
    if (out_f32 != 0 && out_f32 != 1) return fail(GDN_ERR_INVALID_ARG, "out_f32 must be 0 or 1");
    const size_t C = (size_t)channels(dims), hv = dims->hv, d = dims->dk, ns = (size_t)n_seq;
    const Buf bufs[] = {
        {qkv, ns * C * 2, "qkv"},          {conv_w, C * 16, "conv_w"},
        {hist_in, ns * C * 6, "hist_in"},  {a, ns * hv * 2, "a"},
        {b, ns * hv * 2, "b"},             {z, ns * hv * d * 2, "z"},
        {A_log, hv * 4, "A_log"},          {dt_bias, hv * 4, "dt_bias"},
        {gamma, d * 4, "gamma"},           {S_in, ns * hv * d * d * 4, "S_in"},
        {hist_out, ns * C * 6, "hist_out"}, {S_out, ns * hv * d * d * 4, "S_out"},
        {y, ns * hv * d * (out_f32 ? 4 : 2), "y"},
    };
    if ((st = check_bufs(bufs, sizeof bufs / sizeof bufs[0])) != GDN_OK) return st;
    if (bufs[9].p != bufs[11].p && overlap(bufs[9], bufs[11]))
        return fail(GDN_ERR_INVALID_ARG, "S_out partially overlaps S_in (identical buffers are allowed)");
    const Buf ins[] = {bufs[0], bufs[1], bufs[2], bufs[3], bufs[4], bufs[5], bufs[6], bufs[7], bufs[8]};
    const Buf outs[] = {bufs[10], bufs[11], bufs[12]};
    if ((st = check_disjoint(outs, 3, ins, 9)) != GDN_OK) return st;
    if (overlap(bufs[10], bufs[9]) || overlap(bufs[12], bufs[9]))
        return fail(GDN_ERR_INVALID_ARG, "hist_out or y overlaps S_in");
    if (n_seq == 0) return GDN_OK;
    gdn::StepParams p{};
    p.hk = dims->hk; p.hv = dims->hv; p.C = (int)C; p.n_seq = n_seq; p.eps = dims->eps;
    p.qkv = reinterpret_cast<const __half*>(qkv);
    p.conv_w = conv_w;
    p.hist_in = reinterpret_cast<const __half*>(hist_in);
    p.hist_out = reinterpret_cast<__half*>(hist_out);
    p.a = reinterpret_cast<const __half*>(a);
    p.b = reinterpret_cast<const __half*>(b);
    p.z = reinterpret_cast<const __half*>(z);
    p.A_log = A_log; p.dt_bias = dt_bias; p.gamma = gamma;
    p.S_in = S_in; p.S_out = S_out; p.out_f32 = out_f32; p.y = y;
    cudaError_t e = gdn::launch_step(p, reinterpret_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? GDN_OK : cuda_fail(e, "gdn_step launch");
}

}  // extern "C"

extern "C" {

gdn_status gdn_scan_check(const void* workspace, struct CUstream_st* stream)
{
    return read_failure_word(workspace, stream);
}

gdn_status gdn_layer_check(const gdn_dims* dims, int32_t n_seq, int32_t T, const void* workspace,
                           struct CUstream_st* stream)
{
    gdn_status st;
    if ((st = check_dims(dims)) != GDN_OK) return st;
    if (n_seq < 0 || T < 0) return fail(GDN_ERR_INVALID_ARG, "negative n_seq or total_tokens");
    if (!workspace) return fail(GDN_ERR_INVALID_ARG, "workspace is NULL");
    return read_failure_word(static_cast<const char*>(workspace) + layer_scan_offset(dims, T), stream);
}

gdn_status gdn_scan_selftest_timeout(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                                     const float* qn, const float* kn, const float* vc, const float* glog,
                                     const float* beta, const float* S_in, float* S_out, float* o, void* workspace,
                                     size_t workspace_bytes, struct CUstream_st* stream)
{
    gdn::ScanParams p;
    gdn_status st = prep_scan(dims, n_seq, T, cu_seqlens, qn, kn, vc, glog, beta, S_in, S_out, o, workspace,
                              workspace_bytes, p);
    if (st != GDN_OK) return st;
    p.withhold_first_copy = 1;
    return run_scan(p, stream);
}

gdn_status gdn_scan_selftest_withhold_flag(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                                           const float* qn, const float* kn, const float* vc, const float* glog,
                                           const float* beta, const float* S_in, float* S_out, float* o,
                                           void* workspace, size_t workspace_bytes, struct CUstream_st* stream)
{
    gdn::ScanParams p;
    gdn_status st = prep_scan(dims, n_seq, T, cu_seqlens, qn, kn, vc, glog, beta, S_in, S_out, o, workspace,
                              workspace_bytes, p);
    if (st != GDN_OK) return st;
    p.withhold_flag = 1;
    return run_scan(p, stream);
}

gdn_status gdn_scan_selftest_one_taker(const gdn_dims* dims, int32_t n_seq, int32_t T, const int32_t* cu_seqlens,
                                       const float* qn, const float* kn, const float* vc, const float* glog,
                                       const float* beta, const float* S_in, float* S_out, float* o,
                                       void* workspace, size_t workspace_bytes, struct CUstream_st* stream)
{
    gdn::ScanParams p;
    gdn_status st = prep_scan(dims, n_seq, T, cu_seqlens, qn, kn, vc, glog, beta, S_in, S_out, o, workspace,
                              workspace_bytes, p);
    if (st != GDN_OK) return st;
    p.prep_no_keepers = 1;
    return run_scan(p, stream);
}

}  // extern "C"
