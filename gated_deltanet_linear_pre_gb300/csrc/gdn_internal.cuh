// gdn_internal.cuh -- declarations shared by the library's translation units.
// Nothing here is part of the public ABI (include/gdn.h is).
#pragma once

#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace gdn {

constexpr int kHeadDim = 128;  // dk == dv == 128: one head is 32 lanes x 4 channels
constexpr int kChunk = 64;     // tokens per scan chunk

// The scan's [K; Q] operand image of one (chunk slot, key head): 128 rows (the chunk's 64 k rows and
// 64 q rows, k first for chunks at an even index within their sequence, q first for odd ones) x 128
// columns, bf16 split into hi and lo planes, in 16 groups of 8 rows, each group its hi plane (2 KB,
// 16 no-swizzle core matrices along the columns) then its lo plane.  Byte offset of (row r, column k)
// in the hi plane; the lo plane is 2048 bytes behind.  Chunk slots: sequence s owns slots from
// cu[s] / 64 + s on.
constexpr size_t kKqImageBytes = 128 * 128 * 2 * 2;
__host__ __device__ __forceinline__ int kq_off(int r, int k)
{
    return (r >> 3) * 4096 + (k >> 3) * 128 + (r & 7) * 16 + (k & 7) * 2;
}

struct PreParams {
    int hk, hv, C, T, n_seq;
    float eps;
    const int32_t* cu_seqlens;
    const __half* qkv;
    const float* conv_w;
    const __half* hist_in;
    __half* hist_out;
    const __half* a;
    const __half* b;
    const float* A_log;
    const float* dt_bias;
    float* qn;
    float* kn;
    float* vc;
    float* glog;
    float* beta;
    // inside gdn_layer: q and k go straight into the scan's [K; Q] images (qn and kn unused); the
    // images of slot `slot`, key head j start at kq_images + (slot * hk + j) * kKqImageBytes
    unsigned char* kq_images;
    int hist_in_place;  // hist_out == hist_in: the history is written by a second launch after the conv
};

struct ScanParams {
    int hk, hv, T, n_seq;
    const int32_t* cu_seqlens;
    const float* qn;
    const float* kn;
    const float* vc;
    const float* glog;
    const float* beta;
    const float* S_in;
    float* S_out;
    float* o;
    void* workspace;
    size_t workspace_bytes;
    int withhold_first_copy;  // failure-report self-test only (gdn_scan_selftest_timeout)
    int prep_no_keepers;      // prep fallback self-test only (gdn_scan_selftest_one_taker)
    int withhold_flag;        // cross-kernel wait self-test only (gdn_scan_selftest_withhold_flag)
    int fast;                 // one-pass bf16 products (gdn_scan_fast / gdn_layer_fast)
    int prep_sms, prep_keep;  // SMs of the device; SMs whose prep CTAs stay after round one (set by launch_scan)
    int kq_written;           // the pre kernel wrote the [K; Q] images (qn and kn unused; gdn_layer)
};

struct PostParams {
    int hv, T;
    float eps;
    const float* o;
    const __half* z;
    const float* gamma;
    int out_f32;
    void* y;
};

// one decode step: one token per sequence, the three stages fused
struct StepParams {
    int hk, hv, C, n_seq;
    float eps;
    const __half* qkv;      // [n_seq][C]
    const float* conv_w;    // [C][4]
    const __half* hist_in;  // [n_seq][C][3]
    __half* hist_out;
    const __half* a;        // [n_seq][hv]
    const __half* b;
    const __half* z;        // [n_seq][hv][dv]
    const float* A_log;
    const float* dt_bias;
    const float* gamma;
    const float* S_in;      // [n_seq][hv][dk][dv]
    float* S_out;
    int out_f32;
    void* y;                // [n_seq][hv][dv]
};

cudaError_t launch_pre(const PreParams& p, cudaStream_t stream);
cudaError_t launch_step(const StepParams& p, cudaStream_t stream);
size_t scan_workspace_bytes(int hk, int hv, int n_seq, int T);
size_t scan_kq_images_offset(int hk, int hv, int n_seq, int T);  // byte offset of the [K; Q] images in the workspace
cudaError_t launch_scan(const ScanParams& p, cudaStream_t stream);
cudaError_t launch_post(const PostParams& p, cudaStream_t stream);

// record the detail string returned by gdn_last_error_string on this thread
void set_last_error(const char* msg);

// ---- programmatic dependent launch ---------------------------------------------
// Kernels launched with launch_k(..., pdl = true) may start while the previous
// kernel on the stream is still draining.  Every kernel calls pdl_wait() before
// its first read of global memory (a no-op when launched without the
// attribute) and pdl_launch_dependents() early, which lets the next kernel's
// CTAs be scheduled once every CTA of this one has started.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream, bool pdl,
                     Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = pdl ? attr : nullptr;
    cfg.numAttrs = pdl ? 1 : 0;
    return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- small device helpers ---------------------------------------------------
__device__ __forceinline__ float warp_sum(float v)
{
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    return v;
}

// cu_seqlens[s] clamped into [0, T]: a malformed offsets array gives wrong
// results, never an out-of-bounds access
__device__ __forceinline__ int cu_at(const int32_t* cu, int s, int T)
{
    return min(max(__ldg(cu + s), 0), T);
}

__device__ __forceinline__ float sigmoidf_(float x) { return 1.0f / (1.0f + expf(-x)); }

__device__ __forceinline__ float siluf_(float x) { return x / (1.0f + expf(-x)); }

// SiLU with the fast exponential and reciprocal intrinsics (a few ulp; for
// x -> -inf the reciprocal of inf is 0, so the result goes to -0 cleanly)
__device__ __forceinline__ float silu_fast(float x) { return x * __fdividef(1.0f, 1.0f + __expf(-x)); }

}  // namespace gdn
