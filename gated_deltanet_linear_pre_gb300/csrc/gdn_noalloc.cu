// gdn_noalloc.cu -- gdn_scan_noalloc: the scan for callers that cannot
// allocate device memory (see include/gdn.h).  Its scratch is one file-scope
// device array of GDN_SCAN_NOALLOC_MAX_BYTES; the scan itself is the same
// gdn_scan path, handed that array as its workspace.
#include <cstdio>
#include <mutex>

#include "gdn.h"
#include "gdn_internal.cuh"

namespace {

// Scratch of the allocation-free scan.  Every device that loads the library
// holds it until the process exits.
static __device__ __align__(256) unsigned char g_scan_scratch[GDN_SCAN_NOALLOC_MAX_BYTES];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

int current_device(gdn_status* st)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        gdn::set_last_error(cudaGetErrorString(e));
        *st = GDN_ERR_CUDA;
        return -1;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        gdn::set_last_error("gdn_scan_noalloc: device ordinal beyond the supported 64");
        *st = GDN_ERR_UNSUPPORTED;
        return -1;
    }
    *st = GDN_OK;
    return dev;
}

// Device address of this device's scratch array, with that device current.  In host code the
// array's name is only a host-side handle; kernels must be given this address.  Looked up on
// every call outside stream capture (after a device reset the module, and with it the array, is
// loaded afresh); under capture the address of the last call outside capture is used, so the
// first call on a device must come before any capture.
gdn_status scratch_for_current_device(cudaStream_t stream, void** out)
{
    gdn_status st;
    const int dev = current_device(&st);
    if (st != GDN_OK) return st;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) {
        gdn::set_last_error(cudaGetErrorString(e));
        return GDN_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (cs == cudaStreamCaptureStatusNone) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_scan_scratch);
        if (e != cudaSuccess || !ptr) {
            gdn::set_last_error(e != cudaSuccess ? cudaGetErrorString(e)
                                                 : "gdn_scan_noalloc: scratch symbol has no device address");
            return GDN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
    } else if (!g_scratch_ptr[dev]) {
        gdn::set_last_error("gdn_scan_noalloc: the first call on a device must come before any stream capture");
        return GDN_ERR_INVALID_ARG;
    }
    *out = g_scratch_ptr[dev];
    return GDN_OK;
}

}  // namespace

extern "C" gdn_status gdn_scan_noalloc(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                                       const int32_t* cu_seqlens, const float* qn, const float* kn,
                                       const float* vc, const float* glog, const float* beta,
                                       const float* S_in, float* S_out, float* o, struct CUstream_st* stream)
{
    if (!dims || n_seq < 0 || total_tokens < 0) {
        gdn::set_last_error("gdn_scan_noalloc: dims is NULL or a size is negative");
        return GDN_ERR_INVALID_ARG;
    }
    const size_t need = gdn_scan_workspace_bytes(dims, n_seq, total_tokens);
    if (need > GDN_SCAN_NOALLOC_MAX_BYTES) {
        char msg[256];
        snprintf(msg, sizeof msg,
                 "gdn_scan_noalloc: this batch needs %zu bytes of scan scratch, above the fixed %zu-byte "
                 "maximum (GDN_SCAN_NOALLOC_MAX_BYTES); use gdn_scan with a workspace",
                 need, (size_t)GDN_SCAN_NOALLOC_MAX_BYTES);
        gdn::set_last_error(msg);
        return GDN_ERR_UNSUPPORTED;
    }
    void* scratch = nullptr;
    gdn_status st = scratch_for_current_device(reinterpret_cast<cudaStream_t>(stream), &scratch);
    if (st != GDN_OK) return st;
    // the same validation and launches as gdn_scan; the scan clears the part of
    // its scratch that must start at zero on every call
    return gdn_scan(dims, n_seq, total_tokens, cu_seqlens, qn, kn, vc, glog, beta, S_in, S_out, o, scratch,
                    GDN_SCAN_NOALLOC_MAX_BYTES, stream);
}

extern "C" gdn_status gdn_scan_noalloc_check(struct CUstream_st* stream)
{
    gdn_status st;
    const int dev = current_device(&st);
    if (st != GDN_OK) return st;
    void* scratch = nullptr;
    {
        std::lock_guard<std::mutex> lock(g_setup_mutex);
        scratch = g_scratch_ptr[dev];
    }
    if (!scratch) {
        gdn::set_last_error("gdn_scan_noalloc_check: gdn_scan_noalloc has not run on this device");
        return GDN_ERR_INVALID_ARG;
    }
    return gdn_scan_check(scratch, stream);
}
