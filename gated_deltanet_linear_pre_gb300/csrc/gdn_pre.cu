// gdn_pre.cu -- stage 1 of the GDN prefill path.
//
// Width-4 causal depthwise conv over the packed q|k|v channels with a carried
// 3-token history, SiLU, L2 normalisation of each q/k head, and the gates
// lam = -exp(A_log) * softplus(a + dt_bias), beta = sigmoid(b).
// ("Round 30 Track C Audit: gdn_pre, gdn_post, and gdn_scanr_4", section 1:
// gdn_pre's 4-tap conv loop, its history write at the last token and its
// per-key-head sum-of-squares reductions; "round 10 track b: gdn
// vectorization and scan", variants: four multiply-adds per output in tap
// order, vectorised tap loads, history kept channel by channel.)
//
// HBM-bound.  One warp owns one 128-channel head for a block of 16 consecutive
// tokens.  It first copies the block's rows of its head (and the 3 rows before
// them) into shared memory with 16-byte asynchronous copies, one
// commit group per 8 tokens, so that many rows are in flight per SM without
// holding registers; then each lane, holding 4 channels' taps in registers,
// reads its 8 bytes of each row from shared memory, slides the 3-token window
// in registers and writes 16-byte fp32 stores.  The q/k norms are warp
// reductions.  A separate row of blocks writes the carried history of every
// sequence.
#include <cuda_bf16.h>

#include "gdn_internal.cuh"

namespace gdn {
namespace {

// tokens per warp task (a multiple of 8, at most 32)
template <bool kImg>
constexpr int kTokBlkFor = 16;
constexpr int kWarps = 4;     // warps (heads) per block (128-thread blocks schedule finer than 256)
constexpr int kThreads = kWarps * 32;
constexpr int kHistThreads = kThreads;  // one history channel per thread

struct F4 {
    float x, y, z, w;
};

__device__ __forceinline__ F4 unpack_half4(uint2 raw)
{
    __half2 lo = *reinterpret_cast<__half2*>(&raw.x);
    __half2 hi = *reinterpret_cast<__half2*>(&raw.y);
    float2 a = __half22float2(lo), b = __half22float2(hi);
    return {a.x, a.y, b.x, b.y};
}

__device__ __forceinline__ F4 load_half4(const __half* p)
{
    return unpack_half4(__ldg(reinterpret_cast<const uint2*>(p)));
}

// The 4 channels [c, c+4) of the input at position `pos` of sequence `seq`
// (pos < 0 reads the carried history, slot 3 + pos).
__device__ __forceinline__ F4 tap4(const PreParams& p, int seq, int seq_start, int pos, int c)
{
    if (pos >= 0) return load_half4(p.qkv + (size_t)min(seq_start + pos, p.T - 1) * p.C + c);
    const __half* h = p.hist_in + ((size_t)seq * p.C + c) * 3 + (3 + max(pos, -3));
    return {__half2float(h[0]), __half2float(h[3]), __half2float(h[6]), __half2float(h[9])};
}

__device__ __forceinline__ int find_seq(const int32_t* cu, int n_seq, int t)
{
    // last s with cu[s] <= t (skips empty sequences)
    int lo = 0, hi = n_seq - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (__ldg(cu + mid) <= t) lo = mid; else hi = mid - 1;
    }
    return lo;  // in [0, n_seq - 1] whatever cu holds
}

__device__ __forceinline__ float conv4(float w0, float w1, float w2, float w3, float x0, float x1,
                                       float x2, float x3)
{
    // taps in order: oldest first, current token last
    float acc = w0 * x0;
    acc = fmaf(w1, x1, acc);
    acc = fmaf(w2, x2, acc);
    acc = fmaf(w3, x3, acc);
    return acc;
}

// One token's normalised q or k head (4 channels per lane) into the scan's [K; Q] image:
// bf16 hi / lo split (hi = bf16(x), lo = bf16(x - hi), as the scan splits its fp32
// inputs), then lanes 2m and 2m+1, which hold columns 8m..8m+7, trade halves so
// that the even lane stores the 16-byte hi piece and the odd lane the lo piece.
// pos: the token's position in its sequence; slot0: the sequence's first slot.
__device__ __forceinline__ void store_kq(unsigned char* img_j, size_t slot_stride, int slot0, int pos, bool is_k,
                                         int lane, float y0, float y1, float y2, float y3)
{
    const int ci = pos >> 6, r = pos & 63;
    const bool odd = (ci & 1) != 0;
    const int row = ((is_k == odd) ? 64 : 0) + r;  // k first in even chunks, q first in odd ones
    const __nv_bfloat162 h01 = __floats2bfloat162_rn(y0, y1), h23 = __floats2bfloat162_rn(y2, y3);
    const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
    const __nv_bfloat162 l01 = __floats2bfloat162_rn(y0 - f01.x, y1 - f01.y);
    const __nv_bfloat162 l23 = __floats2bfloat162_rn(y2 - f23.x, y3 - f23.y);
    const uint32_t uh01 = *reinterpret_cast<const uint32_t*>(&h01), uh23 = *reinterpret_cast<const uint32_t*>(&h23);
    const uint32_t ul01 = *reinterpret_cast<const uint32_t*>(&l01), ul23 = *reinterpret_cast<const uint32_t*>(&l23);
    const bool ev = (lane & 1) == 0;
    const uint32_t g0 = __shfl_xor_sync(0xffffffffu, ev ? ul01 : uh01, 1);
    const uint32_t g1 = __shfl_xor_sync(0xffffffffu, ev ? ul23 : uh23, 1);
    const uint4 out = ev ? make_uint4(uh01, uh23, g0, g1) : make_uint4(g0, g1, ul01, ul23);
    unsigned char* dst = img_j + (size_t)(slot0 + ci) * slot_stride + kq_off(row, 8 * (lane >> 1)) + (ev ? 0 : 2048);
    *reinterpret_cast<uint4*>(dst) = out;
}

// The token rows of one warp task, one head of each: the 3 rows before the block (when they lie
// inside the sequence) and the block's rows, 256 bytes each, copied in by 16-byte asynchronous
// copies so that many rows are in flight per SM without holding registers.
static_assert(kTokBlkFor<false> % 8 == 0 && kTokBlkFor<false> <= 32 && kTokBlkFor<true> % 8 == 0 && kTokBlkFor<true> <= 32,
              "one commit group per 8 tokens, at most 4 in flight; one gate lane per token");
constexpr int kRowBytes = kHeadDim * 2;

// copy rows [r_lo, r_hi) of the stage (row r = token t_begin - 3 + r, channels of head `slot`) as
// one commit group: 16 bytes per lane and copy, a warp moving two rows per instruction
__device__ __forceinline__ void stage_rows(unsigned char* stage, const __half* qkv, int C, int slot, int t_begin,
                                           int r_lo, int r_hi, int lane)
{
    const int pieces = (r_hi - r_lo) * (kRowBytes / 16);
    for (int i = lane; i < pieces; i += 32) {
        const int r = r_lo + i / (kRowBytes / 16), k = i % (kRowBytes / 16);
        const __half* src = qkv + (size_t)(t_begin - 3 + r) * C + slot * kHeadDim + 8 * k;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"((uint32_t)__cvta_generic_to_shared(
                         stage + r * kRowBytes + 16 * k)),
                     "l"(src)
                     : "memory");
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
}

// wait until at most n of this thread's commit groups are still in flight (n < 4)
__device__ __forceinline__ void cp_async_wait_groups(int n)
{
    switch (n) {
        case 0: asm volatile("cp.async.wait_group 0;" ::: "memory"); break;
        case 1: asm volatile("cp.async.wait_group 1;" ::: "memory"); break;
        case 2: asm volatile("cp.async.wait_group 2;" ::: "memory"); break;
        default: asm volatile("cp.async.wait_group 3;" ::: "memory"); break;
    }
}

__device__ __forceinline__ F4 stage_row(const unsigned char* stage, int r, int lane)
{
    return unpack_half4(*reinterpret_cast<const uint2*>(stage + r * kRowBytes + lane * 8));
}

// kImg: q and k go to the scan's [K; Q] images (inside gdn_layer) instead of qn / kn
template <bool kImg>
__global__ void __launch_bounds__(kThreads, 8)
pre_kernel(PreParams p, int n_slots, int head_groups, int n_conv_blocks)
{
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    pdl_launch_dependents();
    pdl_wait();

    if ((int)blockIdx.x >= n_conv_blocks) {
        // ---- carried history: the last 3 inputs of sequence s, channel c --
        const long long idx = (long long)(blockIdx.x - n_conv_blocks) * kHistThreads + threadIdx.x;
        const int s = (int)(idx / p.C), c = (int)(idx % p.C);
        if (s >= p.n_seq) return;
        const int start = cu_at(p.cu_seqlens, s, p.T);
        const int len = max(cu_at(p.cu_seqlens, s + 1, p.T) - start, 0);
        __half v[3];
#pragma unroll
        for (int i = 0; i < 3; ++i) {  // all loads first, then the stores
            const int pos = len - 3 + i;
            v[i] = pos >= 0 ? p.qkv[(size_t)(start + pos) * p.C + c]
                            : p.hist_in[((size_t)s * p.C + c) * 3 + (3 + pos)];
        }
#pragma unroll
        for (int i = 0; i < 3; ++i) p.hist_out[((size_t)s * p.C + c) * 3 + i] = v[i];
        return;
    }

    // head slot (q heads | k heads | v heads) and token block of this warp
    const int slot = (blockIdx.x % head_groups) * kWarps + warp;
    const int tb = blockIdx.x / head_groups;
    if (slot >= n_slots) return;
    const int c = slot * kHeadDim + lane * 4;
    constexpr int kTokBlk = kTokBlkFor<kImg>;
    constexpr int kStageRows = kTokBlk + 3;
    // the image variant stages each 8-row output group in the same array: its hi plane over input rows
    // 0-7 (token i writes row i, whose input token i - 3 has been read), its lo plane in 8 rows behind
    // the inputs
    constexpr int kAllRows = kStageRows + (kImg ? 8 : 0);
    const int t_begin = tb * kTokBlk;
    const int t_end = min(p.T, t_begin + kTokBlk);

    const int hk = p.hk;
    const bool is_q = slot < hk, is_k = !is_q && slot < 2 * hk;
    const int vh = slot - 2 * hk;  // value head (valid when >= 0)

    int seq = find_seq(p.cu_seqlens, p.n_seq, t_begin);
    int seq_start = min(cu_at(p.cu_seqlens, seq, p.T), t_begin);
    int seq_end = cu_at(p.cu_seqlens, seq + 1, p.T);
    const bool whole = t_end - t_begin == kTokBlk && t_end <= seq_end;  // the common case
    const int pos0 = t_begin - seq_start;
    __shared__ __align__(16) unsigned char in_stage[kWarps][kAllRows * kRowBytes];
    unsigned char* stage = in_stage[warp];
    if (whole) {
        // the block's rows in one commit group per 8 tokens (the first with the 3 rows before the block,
        // when those lie in the sequence; otherwise the window comes from the carried history below)
        const int r0 = pos0 >= 3 ? 0 : 3;
#pragma unroll
        for (int g = 0; g < kTokBlk / 8; ++g)
            stage_rows(stage, p.qkv, p.C, slot, t_begin, g == 0 ? r0 : 3 + 8 * g, 3 + 8 * (g + 1), lane);
    }

    // taps of my 4 channels
    const float4 w0 = __ldg(reinterpret_cast<const float4*>(p.conv_w) + c + 0);
    const float4 w1 = __ldg(reinterpret_cast<const float4*>(p.conv_w) + c + 1);
    const float4 w2 = __ldg(reinterpret_cast<const float4*>(p.conv_w) + c + 2);
    const float4 w3 = __ldg(reinterpret_cast<const float4*>(p.conv_w) + c + 3);

    F4 win0, win1, win2;  // inputs at positions pos-3, pos-2, pos-1
    if (!whole || pos0 < 3) {
        win0 = tap4(p, seq, seq_start, pos0 - 3, c);
        win1 = tap4(p, seq, seq_start, pos0 - 2, c);
        win2 = tap4(p, seq, seq_start, pos0 - 1, c);
    }

    // inside gdn_layer, q and k go to the scan's images
    const size_t slot_stride = (size_t)hk * kKqImageBytes;
    unsigned char* img_j = kImg ? p.kq_images + (size_t)(is_q ? slot : slot - hk) * kKqImageBytes : nullptr;

    if (whole) {
        cp_async_wait_groups(kTokBlk / 8 - 1);  // the first 8 rows (and the rows before them)
        __syncwarp();
        if (pos0 >= 3) {
            win0 = stage_row(stage, 0, lane);
            win1 = stage_row(stage, 1, lane);
            win2 = stage_row(stage, 2, lane);
        }
        // output of one token: a normalised q/k row or a v row
        float* dst = nullptr;
        size_t dstride = 0;
        if (vh >= 0) {
            dst = p.vc + ((size_t)t_begin * p.hv + vh) * kHeadDim + lane * 4;
            dstride = (size_t)p.hv * kHeadDim;
        } else if (!kImg) {
            dst = (is_k ? p.kn : p.qn) + ((size_t)t_begin * hk + (is_q ? slot : slot - hk)) * kHeadDim + lane * 4;
            dstride = (size_t)hk * kHeadDim;
        }
        // image output: when the sequence starts at a multiple of 8, each 8 tokens of the block are one
        // 8-row group of one chunk's image, 4 contiguous KB (hi plane, lo plane): staged in shared memory
        // (row-major 256-byte rows whose 16-byte pieces are permuted by the row index, piece m of row
        // r at m ^ r, so that neither side's accesses conflict) and written with 512 contiguous bytes
        // per warp store.  Otherwise each token goes out on its own.
        constexpr int kRow = 256, kPlane = kStageRows * kRow;  // the lo plane's offset from the hi plane
        const bool grouped = (pos0 & 7) == 0;
        const int slot0 = seq_start / kChunk + seq;
#pragma unroll(kImg ? 1 : kTokBlk / 8)
        for (int h8 = 0; h8 < kTokBlk / 8; ++h8) {
            if (h8 > 0) {
                cp_async_wait_groups(kTokBlk / 8 - 1 - h8);
                __syncwarp();
            }
#pragma unroll
            for (int i8 = 0; i8 < 8; ++i8) {
                const int i = 8 * h8 + i8;
                const F4 x = stage_row(stage, 3 + i, lane);
                float y0 = silu_fast(conv4(w0.x, w0.y, w0.z, w0.w, win0.x, win1.x, win2.x, x.x));
                float y1 = silu_fast(conv4(w1.x, w1.y, w1.z, w1.w, win0.y, win1.y, win2.y, x.y));
                float y2 = silu_fast(conv4(w2.x, w2.y, w2.z, w2.w, win0.z, win1.z, win2.z, x.z));
                float y3 = silu_fast(conv4(w3.x, w3.y, w3.z, w3.w, win0.w, win1.w, win2.w, x.w));
                win0 = win1;
                win1 = win2;
                win2 = x;
                if (vh < 0) {
                    const float inv = rsqrtf(warp_sum(y0 * y0 + y1 * y1 + y2 * y2 + y3 * y3) + p.eps);
                    y0 *= inv; y1 *= inv; y2 *= inv; y3 *= inv;
                }
                if (kImg && vh < 0) {
                    if (grouped) {
                        unsigned char* stg = stage;
                        const __nv_bfloat162 h01 = __floats2bfloat162_rn(y0, y1), h23 = __floats2bfloat162_rn(y2, y3);
                        const float2 f01 = __bfloat1622float2(h01), f23 = __bfloat1622float2(h23);
                        const __nv_bfloat162 l01 = __floats2bfloat162_rn(y0 - f01.x, y1 - f01.y);
                        const __nv_bfloat162 l23 = __floats2bfloat162_rn(y2 - f23.x, y3 - f23.y);
                        const int so = i8 * kRow + (((lane >> 1) ^ i8) << 4) + (lane & 1) * 8;
                        *reinterpret_cast<uint2*>(stg + so) =
                            make_uint2(*reinterpret_cast<const uint32_t*>(&h01), *reinterpret_cast<const uint32_t*>(&h23));
                        *reinterpret_cast<uint2*>(stg + kPlane + so) =
                            make_uint2(*reinterpret_cast<const uint32_t*>(&l01), *reinterpret_cast<const uint32_t*>(&l23));
                    } else {
                        store_kq(img_j, slot_stride, slot0, pos0 + i, is_k, lane, y0, y1, y2, y3);
                    }
                } else {
                    *reinterpret_cast<float4*>(dst) = make_float4(y0, y1, y2, y3);
                    dst += dstride;
                }
            }
            if (kImg && vh < 0 && grouped) {
                __syncwarp();
                const unsigned char* stg = stage;
                const int pg = pos0 + 8 * h8, ci = pg >> 6;
                const int row0 = ((is_k == ((ci & 1) != 0)) ? 64 : 0) + (pg & 63);
                unsigned char* gdst = img_j + (size_t)(slot0 + ci) * slot_stride + (row0 >> 3) * 4096;
                // 16-byte piece `lane` of each 512-byte run: plane k / 4, core matrix 4 (k % 4) + lane / 8
                // (columns 8 m .. 8 m + 7), row lane % 8
#pragma unroll
                for (int k = 0; k < 8; ++k) {
                    const int m = (k & 3) * 4 + (lane >> 3), r = lane & 7;
                    *reinterpret_cast<uint4*>(gdst + k * 512 + lane * 16) =
                        *reinterpret_cast<const uint4*>(stg + (k >> 2) * kPlane + r * kRow + ((m ^ r) << 4));
                }
                __syncwarp();  // the stage is refilled by the next 8 tokens
            }
        }
    } else {
    // a block that crosses a sequence end or is cut by T: token by token
    for (int i = 0; i < kTokBlk; ++i) {
        const int t = t_begin + i;
        if (t >= t_end) break;
        if (t >= seq_end) {
            // first token of a new sequence: window comes from that sequence's history
            while (t >= seq_end && seq + 1 < p.n_seq) {
                ++seq;
                seq_start = seq_end;
                seq_end = cu_at(p.cu_seqlens, seq + 1, p.T);
            }
            seq_start = min(seq_start, t);
            win0 = tap4(p, seq, seq_start, -3, c);
            win1 = tap4(p, seq, seq_start, -2, c);
            win2 = tap4(p, seq, seq_start, -1, c);
        }
        const F4 x = load_half4(p.qkv + (size_t)t * p.C + c);
        float y0 = silu_fast(conv4(w0.x, w0.y, w0.z, w0.w, win0.x, win1.x, win2.x, x.x));
        float y1 = silu_fast(conv4(w1.x, w1.y, w1.z, w1.w, win0.y, win1.y, win2.y, x.y));
        float y2 = silu_fast(conv4(w2.x, w2.y, w2.z, w2.w, win0.z, win1.z, win2.z, x.z));
        float y3 = silu_fast(conv4(w3.x, w3.y, w3.z, w3.w, win0.w, win1.w, win2.w, x.w));
        win0 = win1;
        win1 = win2;
        win2 = x;
        float* dst;
        if (vh >= 0) {
            dst = p.vc + ((size_t)t * p.hv + vh) * kHeadDim + lane * 4;
        } else {
            float ss = y0 * y0 + y1 * y1 + y2 * y2 + y3 * y3;
            ss = warp_sum(ss);
            const float inv = rsqrtf(ss + p.eps);
            y0 *= inv; y1 *= inv; y2 *= inv; y3 *= inv;
            if constexpr (kImg) {
                store_kq(img_j, slot_stride, seq_start / kChunk + seq, t - seq_start, is_k, lane, y0, y1, y2, y3);
                continue;
            }
            const int j = is_q ? slot : slot - hk;
            dst = (is_k ? p.kn : p.qn) + ((size_t)t * hk + j) * kHeadDim + lane * 4;
        }
        *reinterpret_cast<float4*>(dst) = make_float4(y0, y1, y2, y3);
    }
    }

    // gates of value head vh for the block's tokens: one lane per token
    if (vh >= 0 && lane < t_end - t_begin) {
        const int t = t_begin + lane;
        const float av = __half2float(p.a[(size_t)t * p.hv + vh]) + __ldg(p.dt_bias + vh);
        const float bv = __half2float(p.b[(size_t)t * p.hv + vh]);
        // softplus as max(x, 0) + log1p(e^-|x|): for strongly negative x the sum 1 + e^-|x| would round
        // most of e^-|x| away, and log1p keeps it (relative error of lam stays at the fp32 level)
        const float sp = fmaxf(av, 0.0f) + log1pf(__expf(-fabsf(av)));
        p.glog[(size_t)t * p.hv + vh] = -__expf(__ldg(p.A_log + vh)) * sp;
        p.beta[(size_t)t * p.hv + vh] = __fdividef(1.0f, 1.0f + __expf(-bv));
    }
}

}  // namespace

cudaError_t launch_pre(const PreParams& p, cudaStream_t stream)
{
    const int n_slots = 2 * p.hk + p.hv;
    const int tok_blk = p.kq_images ? kTokBlkFor<true> : kTokBlkFor<false>;
    const long long n_tblocks = (p.T + tok_blk - 1) / tok_blk;
    const int head_groups = (n_slots + kWarps - 1) / kWarps;
    const long long n_conv_blocks = n_tblocks * head_groups;
    const long long n_hist_blocks = ((long long)p.n_seq * p.C + kHistThreads - 1) / kHistThreads;
    if (n_conv_blocks + n_hist_blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    auto launch = [&](long long blocks, int conv_blocks) {
        if (blocks == 0) return cudaSuccess;
        return p.kq_images ? launch_k(pre_kernel<true>, dim3((unsigned)blocks), dim3(kThreads), 0, stream, true, p,
                                      n_slots, head_groups, conv_blocks)
                           : launch_k(pre_kernel<false>, dim3((unsigned)blocks), dim3(kThreads), 0, stream, true, p,
                                      n_slots, head_groups, conv_blocks);
    };
    if (!p.hist_in_place) return launch(n_conv_blocks + n_hist_blocks, (int)n_conv_blocks);
    // history in place: the conv blocks (the readers of the old history) first; the history blocks in a
    // second launch, whose grid-dependency wait returns only once the first grid has completed
    cudaError_t e = launch(n_conv_blocks, (int)n_conv_blocks);
    return e != cudaSuccess ? e : launch(n_hist_blocks, 0);
}

}  // namespace gdn
