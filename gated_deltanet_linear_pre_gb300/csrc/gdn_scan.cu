// gdn_scan.cu -- stage 2 of the GDN prefill path: the gated delta rule.
//
// Per value head h (key head h / (hv/hk)), fp32 state S in R^{128x128}:
//     S <- g S;  u = beta (v - S^T k);  S <- S + k u^T;  o = S^T q / sqrt(dk)
// ("Round 30 Track C Audit: gdn_pre, gdn_post, and gdn_scanr_4", section 1:
// gdn_scan_r keeps the fp32 state in registers, decays and updates it every
// token and forms the k and q products against it.)
//
// Token-sequential CUDA-core form.  One block owns 32 value columns of one
// (sequence, value head): 128 threads, each holding 32 state entries (one
// column, one quarter of the keys) in registers.  A token costs three 32-long
// dot products per thread (S^T k, S^T q, k.q), two xor-shuffles to finish
// them across the key quarters, and one fused update of the 32 entries,
// using o = g (S_old^T q) + (k.q) u.  Chunks of 64 tokens of k, q, v, g and
// beta are staged in shared memory.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kSlice = 32;              // value columns per block
constexpr int kThreads = 128;
constexpr int kGroupPad = 36;           // key quarter stride in shared memory (bank spread)
constexpr int kRowPad = 4 * kGroupPad;  // 144 floats per staged k/q row

struct ScanSmem {
    float k[kChunk * kRowPad];
    float q[kChunk * kRowPad];
    float v[kChunk * kSlice];
    float g[kChunk];
    float b[kChunk];
};

__global__ void __launch_bounds__(kThreads) scan_seq_kernel(ScanParams p)
{
    extern __shared__ __align__(16) unsigned char smem_raw[];
    ScanSmem& sm = *reinterpret_cast<ScanSmem*>(smem_raw);

    const int slices = kHeadDim / kSlice;
    const int h = blockIdx.x / slices, slice = blockIdx.x % slices;
    const int s = blockIdx.y;
    const int j = h / (p.hv / p.hk);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int col = warp * 8 + (lane >> 2);  // 0..31 within the slice
    const int kg = lane & 3;                 // key quarter
    const int vcol = slice * kSlice + col;

    const int t0 = cu_at(p.cu_seqlens, s, p.T), t1 = max(cu_at(p.cu_seqlens, s + 1, p.T), t0);
    const size_t sbase = ((size_t)s * p.hv + h) * kHeadDim * kHeadDim;

    float S[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) S[i] = p.S_in[sbase + (size_t)(kg * 32 + i) * kHeadDim + vcol];

    const float qscale = rsqrtf((float)kHeadDim);
    for (int c0 = t0; c0 < t1; c0 += kChunk) {
        const int n = min(kChunk, t1 - c0);
        __syncthreads();  // previous chunk fully consumed
        for (int idx = threadIdx.x; idx < n * 32; idx += kThreads) {
            const int row = idx >> 5, part = idx & 31;
            const size_t src = ((size_t)(c0 + row) * p.hk + j) * kHeadDim + part * 4;
            const int dst = row * kRowPad + (part >> 3) * kGroupPad + (part & 7) * 4;
            *reinterpret_cast<float4*>(&sm.k[dst]) = __ldg(reinterpret_cast<const float4*>(p.kn + src));
            *reinterpret_cast<float4*>(&sm.q[dst]) = __ldg(reinterpret_cast<const float4*>(p.qn + src));
        }
        for (int idx = threadIdx.x; idx < n * (kSlice / 4); idx += kThreads) {
            const int row = idx / (kSlice / 4), part = idx % (kSlice / 4);
            const size_t src = ((size_t)(c0 + row) * p.hv + h) * kHeadDim + slice * kSlice + part * 4;
            *reinterpret_cast<float4*>(&sm.v[row * kSlice + part * 4]) =
                __ldg(reinterpret_cast<const float4*>(p.vc + src));
        }
        for (int idx = threadIdx.x; idx < n; idx += kThreads) {
            sm.g[idx] = expf(__ldg(p.glog + (size_t)(c0 + idx) * p.hv + h));
            sm.b[idx] = __ldg(p.beta + (size_t)(c0 + idx) * p.hv + h);
        }
        __syncthreads();

        for (int i = 0; i < n; ++i) {
            const float* kr = &sm.k[i * kRowPad + kg * kGroupPad];
            const float* qr = &sm.q[i * kRowPad + kg * kGroupPad];
            float sk = 0.f, sq = 0.f, kq = 0.f;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 kk = *reinterpret_cast<const float4*>(kr + e);
                const float4 qq = *reinterpret_cast<const float4*>(qr + e);
                sk = fmaf(S[e], kk.x, sk); sk = fmaf(S[e + 1], kk.y, sk);
                sk = fmaf(S[e + 2], kk.z, sk); sk = fmaf(S[e + 3], kk.w, sk);
                sq = fmaf(S[e], qq.x, sq); sq = fmaf(S[e + 1], qq.y, sq);
                sq = fmaf(S[e + 2], qq.z, sq); sq = fmaf(S[e + 3], qq.w, sq);
                kq = fmaf(kk.x, qq.x, kq); kq = fmaf(kk.y, qq.y, kq);
                kq = fmaf(kk.z, qq.z, kq); kq = fmaf(kk.w, qq.w, kq);
            }
#pragma unroll
            for (int off = 1; off <= 2; off <<= 1) {
                sk += __shfl_xor_sync(0xffffffffu, sk, off);
                sq += __shfl_xor_sync(0xffffffffu, sq, off);
                kq += __shfl_xor_sync(0xffffffffu, kq, off);
            }
            const float g = sm.g[i], b = sm.b[i];
            const float u = b * (sm.v[i * kSlice + col] - g * sk);
            const float o = (g * sq + kq * u) * qscale;
#pragma unroll
            for (int e = 0; e < 32; e += 4) {
                const float4 kk = *reinterpret_cast<const float4*>(kr + e);
                S[e] = fmaf(kk.x, u, g * S[e]);
                S[e + 1] = fmaf(kk.y, u, g * S[e + 1]);
                S[e + 2] = fmaf(kk.z, u, g * S[e + 2]);
                S[e + 3] = fmaf(kk.w, u, g * S[e + 3]);
            }
            if (kg == 0) p.o[((size_t)(c0 + i) * p.hv + h) * kHeadDim + vcol] = o;
        }
    }

#pragma unroll
    for (int i = 0; i < 32; ++i) p.S_out[sbase + (size_t)(kg * 32 + i) * kHeadDim + vcol] = S[i];
}

}  // namespace

size_t scan_workspace_bytes(int, int, int, int) { return 0; }

cudaError_t launch_scan(const ScanParams& p, cudaStream_t stream)
{
    if (p.n_seq == 0) return cudaSuccess;
    const size_t smem = sizeof(ScanSmem);
    cudaError_t e = cudaFuncSetAttribute(scan_seq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.hv * (kHeadDim / kSlice)), (unsigned)p.n_seq);
    scan_seq_kernel<<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
