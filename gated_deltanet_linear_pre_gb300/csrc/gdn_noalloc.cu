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

// Device address of this device's scratch array, looked up once per device
// with that device current.  In host code the array's name is only a
// host-side handle; kernels must be given this address.
gdn_status scratch_for_current_device(void** out)
{
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        gdn::set_last_error(cudaGetErrorString(e));
        return GDN_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        gdn::set_last_error("gdn_scan_noalloc: device ordinal beyond the supported 64");
        return GDN_ERR_UNSUPPORTED;
    }
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    if (!g_scratch_ptr[dev]) {
        void* ptr = nullptr;
        e = cudaGetSymbolAddress(&ptr, g_scan_scratch);
        if (e != cudaSuccess || !ptr) {
            gdn::set_last_error(e != cudaSuccess ? cudaGetErrorString(e)
                                                 : "gdn_scan_noalloc: scratch symbol has no device address");
            return GDN_ERR_CUDA;
        }
        g_scratch_ptr[dev] = ptr;
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
    gdn_status st = scratch_for_current_device(&scratch);
    if (st != GDN_OK) return st;
    // the same validation and launches as gdn_scan; the scan clears the part of
    // its scratch that must start at zero on every call
    return gdn_scan(dims, n_seq, total_tokens, cu_seqlens, qn, kn, vc, glog, beta, S_in, S_out, o, scratch,
                    GDN_SCAN_NOALLOC_MAX_BYTES, stream);
}
