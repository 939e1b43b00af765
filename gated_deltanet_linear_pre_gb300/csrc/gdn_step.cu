// gdn_step.cu -- one decode step of the GDN layer: one new token for each of
// n_seq sequences, pre + scan + post fused into one kernel.
//
// Per sequence s and value head h (key head j = h / (hv/hk)), for the token x:
//   conv + SiLU of its q (head j), k (head j) and v (head h) channels against
//   the carried 3-token history, q and k L2-normalised (eps);
//   lam = -exp(A_log) softplus(a + dt_bias), g = e^lam, beta = sigmoid(b);
//   S <- g S;  u = beta (v - S^T k);  S <- S + k u^T;  o = S^T q / sqrt(dk);
//   y = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z);
//   history <- the last 3 inputs (old slots 1, 2 and x).
// This is the token-sequential recurrence that the pages' scan kernel runs per
// token ("Round 30 Track C Audit: gdn_pre, gdn_post, and gdn_scanr_4", section
// 1: gdn_scan_r decays and updates the fp32 state per token and forms the k
// and q products against it), with the pre and post arithmetic of the same
// section for a single token.
//
// HBM-bound on the state: each CTA reads its 64 KB fp32 state slice once
// (issued before the conv so its latency hides behind it) and writes it once.
// One CTA per (sequence, value head), 256 threads; in the state phase thread
// (rg, cg) = (tid / 32, tid % 32) owns rows [16 rg, 16 rg + 16) x columns
// [4 cg, 4 cg + 4), so every warp-wide access is one contiguous 512-byte row.
#include "gdn_internal.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 256;
constexpr int kRows = 16;  // state rows per thread

__device__ __forceinline__ float conv4(float w0, float w1, float w2, float w3, float x0, float x1, float x2,
                                       float x3)
{
    float acc = w0 * x0;  // taps oldest first, the current token last
    acc = fmaf(w1, x1, acc);
    acc = fmaf(w2, x2, acc);
    acc = fmaf(w3, x3, acc);
    return acc;
}

// SiLU(conv) of channel ch of sequence s; writes its shifted history when asked
__device__ __forceinline__ float conv_channel(const StepParams& p, int s, int ch, bool write_hist)
{
    const __half* hi = p.hist_in + ((size_t)s * p.C + ch) * 3;
    const __half h0 = hi[0], h1 = hi[1], h2 = hi[2];
    const __half x = p.qkv[(size_t)s * p.C + ch];
    const float4 w = __ldg(reinterpret_cast<const float4*>(p.conv_w) + ch);
    if (write_hist) {
        __half* ho = p.hist_out + ((size_t)s * p.C + ch) * 3;
        ho[0] = h1;
        ho[1] = h2;
        ho[2] = x;
    }
    return silu_fast(conv4(w.x, w.y, w.z, w.w, __half2float(h0), __half2float(h1), __half2float(h2),
                           __half2float(x)));
}

__global__ void __launch_bounds__(kThreads, 3) step_kernel(StepParams p)
{
    __shared__ float sq[kHeadDim], sk[kHeadDim], sv[kHeadDim];
    __shared__ float red[8][kHeadDim];  // per-row-group partial column sums
    __shared__ float wsum[8];
    __shared__ float s_g, s_beta;

    pdl_launch_dependents();
    pdl_wait();
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x, s = blockIdx.y;
    const int group = p.hv / p.hk, j = h / group;
    const int rg = tid >> 5, cg = tid & 31;
    const size_t sbase = ((size_t)s * p.hv + h) * kHeadDim * kHeadDim;

    // ---- state slice loads first --------------------------------------------------------
    float4 S[kRows];
#pragma unroll
    for (int r = 0; r < kRows; ++r)
        S[r] = __ldg(reinterpret_cast<const float4*>(p.S_in + sbase + (size_t)(kRows * rg + r) * kHeadDim) + cg);

    // ---- conv + SiLU: threads 0-127 q channel tid and v channel tid, 128-255 k channel -------
    const int c = tid & 127;
    const bool own_qk = (h % group) == 0;  // one value head per key head writes the q/k history
    float yqk;
    if (tid < 128) {
        yqk = conv_channel(p, s, j * kHeadDim + c, own_qk);
        sv[c] = conv_channel(p, s, 2 * p.hk * kHeadDim + h * kHeadDim + c, true);
    } else {
        yqk = conv_channel(p, s, p.hk * kHeadDim + j * kHeadDim + c, own_qk);
    }
    // L2 norms of q (warps 0-3) and k (warps 4-7)
    float ss = warp_sum(yqk * yqk);
    if (lane == 0) wsum[warp] = ss;
    if (tid == 0) {
        const float av = __half2float(p.a[(size_t)s * p.hv + h]) + __ldg(p.dt_bias + h);
        const float bv = __half2float(p.b[(size_t)s * p.hv + h]);
        const float sp = fmaxf(av, 0.0f) + log1pf(expf(-fabsf(av)));  // softplus
        s_g = expf(-expf(__ldg(p.A_log + h)) * sp);
        s_beta = sigmoidf_(bv);
    }
    __syncthreads();
    {
        const int w0 = tid < 128 ? 0 : 4;
        const float tot = wsum[w0] + wsum[w0 + 1] + wsum[w0 + 2] + wsum[w0 + 3];
        const float v = yqk * rsqrtf(tot + p.eps);
        if (tid < 128) sq[c] = v; else sk[c] = v;
    }
    __syncthreads();

    // ---- S^T k over this thread's rows, combined across the 8 row groups ---------------------
    const float g = s_g, beta = s_beta;
    {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const float kr = sk[kRows * rg + r];
            acc.x = fmaf(S[r].x, kr, acc.x); acc.y = fmaf(S[r].y, kr, acc.y);
            acc.z = fmaf(S[r].z, kr, acc.z); acc.w = fmaf(S[r].w, kr, acc.w);
        }
        *reinterpret_cast<float4*>(&red[rg][4 * cg]) = acc;
    }
    __syncthreads();
    float4 u;
    {
        float4 t = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 x = *reinterpret_cast<const float4*>(&red[q][4 * cg]);
            t.x += x.x; t.y += x.y; t.z += x.z; t.w += x.w;
        }
        const float4 vv = *reinterpret_cast<const float4*>(&sv[4 * cg]);
        // (g S)^T k = g (S^T k)
        u = make_float4(beta * (vv.x - g * t.x), beta * (vv.y - g * t.y), beta * (vv.z - g * t.z),
                        beta * (vv.w - g * t.w));
    }
    __syncthreads();  // red is reused below

    // ---- S <- g S + k u^T (written out), then S^T q -----------------------------------------
    {
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int r = 0; r < kRows; ++r) {
            const int row = kRows * rg + r;
            const float kr = sk[row], qr = sq[row];
            float4 x = S[r];
            x.x = fmaf(g, x.x, kr * u.x); x.y = fmaf(g, x.y, kr * u.y);
            x.z = fmaf(g, x.z, kr * u.z); x.w = fmaf(g, x.w, kr * u.w);
            reinterpret_cast<float4*>(p.S_out + sbase + (size_t)row * kHeadDim)[cg] = x;
            acc.x = fmaf(x.x, qr, acc.x); acc.y = fmaf(x.y, qr, acc.y);
            acc.z = fmaf(x.z, qr, acc.z); acc.w = fmaf(x.w, qr, acc.w);
        }
        *reinterpret_cast<float4*>(&red[rg][4 * cg]) = acc;
    }
    __syncthreads();

    // ---- o and the gated RMSNorm: warp 0, 4 columns per lane ----------------------------------
    if (warp == 0) {
        float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 x = *reinterpret_cast<const float4*>(&red[q][4 * lane]);
            o.x += x.x; o.y += x.y; o.z += x.z; o.w += x.w;
        }
        const float qs = rsqrtf((float)kHeadDim);
        o.x *= qs; o.y *= qs; o.z *= qs; o.w *= qs;
        const float sso = warp_sum(o.x * o.x + o.y * o.y + o.z * o.z + o.w * o.w);
        const float inv = rsqrtf(sso * (1.0f / kHeadDim) + p.eps);
        const size_t row = ((size_t)s * p.hv + h) * kHeadDim + 4 * lane;
        const uint2 zr = __ldg(reinterpret_cast<const uint2*>(p.z + row));
        const float2 z01 = __half22float2(*reinterpret_cast<const __half2*>(&zr.x));
        const float2 z23 = __half22float2(*reinterpret_cast<const __half2*>(&zr.y));
        const float4 gm = __ldg(reinterpret_cast<const float4*>(p.gamma) + lane);
        const float y0 = o.x * inv * (gm.x * silu_fast(z01.x)), y1 = o.y * inv * (gm.y * silu_fast(z01.y));
        const float y2 = o.z * inv * (gm.z * silu_fast(z23.x)), y3 = o.w * inv * (gm.w * silu_fast(z23.y));
        if (p.out_f32) {
            *reinterpret_cast<float4*>(static_cast<float*>(p.y) + row) = make_float4(y0, y1, y2, y3);
        } else {
            __half2 a01 = __floats2half2_rn(y0, y1), a23 = __floats2half2_rn(y2, y3);
            uint2 out;
            out.x = *reinterpret_cast<uint32_t*>(&a01);
            out.y = *reinterpret_cast<uint32_t*>(&a23);
            *reinterpret_cast<uint2*>(static_cast<__half*>(p.y) + row) = out;
        }
    }
}

}  // namespace

cudaError_t launch_step(const StepParams& p, cudaStream_t stream)
{
    if (p.n_seq == 0) return cudaSuccess;
    return launch_k(step_kernel, dim3((unsigned)p.hv, (unsigned)p.n_seq), dim3(kThreads), 0, stream, true, p);
}

}  // namespace gdn
