// gdn_scan.cu -- stage 2 of the GDN prefill path: the gated delta rule,
// chunk-wise on the tcgen05 tensor cores.
//
// Per value head h (key head j = h / (hv/hk)), fp32 state S in R^{128x128}:
//     S <- g S;  u = beta (v - S^T k);  S <- S + k u^T;  o = S^T q / sqrt(dk)
// ("Round 30 Track C Audit: gdn_pre, gdn_post, and gdn_scanr_4", section 1:
// gdn_scan_r keeps the fp32 state on chip, decays and updates it per token
// and forms the k and q products against it.)
//
// Chunk algebra (exact in exact arithmetic; 64-token chunks, S0 = state at
// the chunk start, G_i = running sum of lam = log g inside the chunk, L the
// last row):
//   A_ij = beta_i e^{G_i-G_j} (k_i.k_j) (j < i),   T = (I + A)^-1
//   P_ij = e^{G_i-G_j} (q_i.k_j) / sqrt(dk) (j <= i)
//   X    = beta (V - e^G (K S0))                   U = T X
//   O    = e^G (Q S0) / sqrt(dk) + P U             S = e^{G_L} S0 + K^T (e^{G_L-G} U)
// Every dense product runs on the tensor core with bf16 operands split as
// x = hi + lo (hi = bf16(x), lo = bf16(x - hi)) and three MMAs hi*hi + hi*lo
// + lo*hi accumulated in fp32 in TMEM (about 16 significant bits per operand).
// Products are stacked to fill the 128 rows of one MMA:
//   [K; Q] K^T -> (K K^T ; Q K^T)          P T (rows 0-63 of an M=128 MMA)
//   [K; Q] S0  -> (K S0 ; Q S0)            [T; P T] X -> (U ; P U)
// so (Q S0) and (P U) land in the same TMEM lanes and O needs no exchange.
//
// Three kernels:
//  * scan_gram_kernel, one CTA per (chunk, key head), fully parallel: splits
//    [K; Q] into the tensor-core layout (the chain's [K; Q] image) and forms
//    (K K^T ; Q K^T) in fp32.
//  * scan_prep_kernel, one CTA per (chunk, key head), fully parallel: for each
//    value head reading that key head, A and P, the inverse of I + A
//    (recursive halving with 16x16 diagonal blocks by forward substitution,
//    on CUDA cores) and P T on the tensor core; writes the [T; P T] image per
//    (chunk, value head).
//  * scan_chain_kernel, one CTA per (sequence, value head, 64-column slice):
//    the state-dependent part, chunk after chunk, with the fp32 state slice
//    in registers.  The images stream in with bulk asynchronous copies one
//    chunk ahead ([K; Q] double-buffered), V and the gates through registers
//    one chunk ahead, so each chunk costs three MMA groups and three short
//    CUDA-core phases.  K^T for the state update is
//    the K half of the [K; Q] image read through an MN-major descriptor.
//
// Every MMA is issued by one thread and completes on an mbarrier; every wait
// is bounded and, on expiry, the CTA records an error code in the workspace,
// drains its own copies in flight (bounded), frees its TMEM and stops.
#include "gdn_internal.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr float kLamFloor = -110.0f;  // e^-110 is below the smallest fp32 denormal: g = 0 exactly
constexpr uint32_t kErrTimeout = 1u;
constexpr size_t kAmBytes = 128 * 64 * 2 * 2;     // [T; P T] image, bf16 hi + lo
constexpr size_t kKqBytes = 128 * 128 * 2 * 2;    // [K; Q] image, bf16 hi + lo
constexpr size_t kGramBytes = 128 * 64 * 4;       // (K K^T ; Q K^T), fp32 rows
constexpr size_t kWsHeader = 4096;                // error words
constexpr int kDVS = 64;                          // value columns per chain CTA

// element offsets inside no-swizzle core-matrix tiles (bf16, 64 elements per core matrix)
__device__ __forceinline__ int kmaj(int r, int k, int Kd) { return ((r >> 3) * (Kd >> 3) + (k >> 3)) * 64 + (r & 7) * 8 + (k & 7); }
__device__ __forceinline__ int mnmaj(int mn, int k, int Kd) { return ((mn >> 3) * (Kd >> 3) + (k >> 3)) * 64 + (k & 7) * 8 + (mn & 7); }

__device__ __forceinline__ uint32_t bf2_bits(__nv_bfloat162 v) { return *reinterpret_cast<uint32_t*>(&v); }

// split 8 fp32 values into bf16 hi / lo vectors (packed conversions)
__device__ __forceinline__ void split8(const float* x, uint4& hi, uint4& lo)
{
    uint32_t h[4], l[4];
#pragma unroll
    for (int e = 0; e < 4; ++e) {
        const __nv_bfloat162 hh = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
        const float2 hf = __bfloat1622float2(hh);
        h[e] = bf2_bits(hh);
        l[e] = bf2_bits(__floats2bfloat162_rn(x[2 * e] - hf.x, x[2 * e + 1] - hf.y));
    }
    hi = make_uint4(h[0], h[1], h[2], h[3]);
    lo = make_uint4(l[0], l[1], l[2], l[3]);
}

__device__ __forceinline__ void store_split8(uint16_t* hi, uint16_t* lo, const float* x)
{
    uint4 vh, vl;
    split8(x, vh, vl);
    *reinterpret_cast<uint4*>(hi) = vh;
    *reinterpret_cast<uint4*>(lo) = vl;
}

// Three-pass split product D = A * B over `ksteps` 16-wide K steps; a_kstep /
// b_kstep are the byte advances of one K step in each tile.  Descriptors are
// built once per operand and advanced by adding to their start-address field.
__device__ __forceinline__ void mma_split(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t a_lbo, uint32_t a_sbo,
                                          uint32_t a_kstep, uint32_t b_hi, uint32_t b_lo, uint32_t b_sbo,
                                          uint32_t b_kstep, int ksteps, uint32_t idesc)
{
    const uint64_t dah = umma::desc(a_hi, a_lbo, a_sbo), dal = umma::desc(a_lo, a_lbo, a_sbo);
    const uint64_t dbh = umma::desc(b_hi, 128, b_sbo), dbl = umma::desc(b_lo, 128, b_sbo);
    const uint64_t sa = a_kstep >> 4, sb = b_kstep >> 4;
    for (int ks = 0; ks < ksteps; ++ks) umma::mma_bf16(d, dah + ks * sa, dbh + ks * sb, idesc, ks != 0);
    for (int ks = 0; ks < ksteps; ++ks) umma::mma_bf16(d, dah + ks * sa, dbl + ks * sb, idesc, 1u);
    for (int ks = 0; ks < ksteps; ++ks) umma::mma_bf16(d, dal + ks * sa, dbh + ks * sb, idesc, 1u);
}

// Split product in two instruction groups: D[:, 0:2N] = A_hi [B_hi | B_lo], then
// D[:, 0:N] += A_lo B_hi, so D[:, 0:N] + D[:, N:2N] = A B to ~16 bits.  Needs B_lo
// to follow B_hi directly along N in shared memory (b_hilo is the start of
// both).  Two thirds of the instructions of mma_split for the same tensor work.
__device__ __forceinline__ void mma_split2(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t a_lbo, uint32_t a_sbo,
                                           uint32_t a_kstep, uint32_t b_hilo, uint32_t b_sbo, uint32_t b_kstep,
                                           int ksteps, int N, bool a_mn, bool b_mn)
{
    const uint64_t dah = umma::desc(a_hi, a_lbo, a_sbo), dal = umma::desc(a_lo, a_lbo, a_sbo);
    const uint64_t db = umma::desc(b_hilo, 128, b_sbo);
    const uint64_t sa = a_kstep >> 4, sb = b_kstep >> 4;
    const uint32_t wide = umma::idesc_bf16(128, 2 * N, a_mn, b_mn), narrow = umma::idesc_bf16(128, N, a_mn, b_mn);
    for (int ks = 0; ks < ksteps; ++ks) umma::mma_bf16(d, dah + ks * sa, db + ks * sb, wide, ks != 0);
    for (int ks = 0; ks < ksteps; ++ks) umma::mma_bf16(d, dal + ks * sa, db + ks * sb, narrow, 1u);
}

// Chunk slots: sequence s owns slots [base(s), base(s) + ceil(len_s / 64)) with
// base(s) = floor(cu[s] / 64) + s, which never overlap and need no prefix sum;
// floor(T / 64) + n_seq slots cover every batch.
__device__ __forceinline__ int slot_base(const ScanParams& p, int s) { return cu_at(p.cu_seqlens, s, p.T) / kChunk + s; }

__host__ __device__ inline size_t n_slots(int T, int n_seq) { return (size_t)(T / kChunk) + (size_t)n_seq; }

__device__ __forceinline__ unsigned char* am_image(const ScanParams& p, size_t slot, int h)
{
    return static_cast<unsigned char*>(p.workspace) + kWsHeader + (slot * p.hv + h) * kAmBytes;
}

__device__ __forceinline__ unsigned char* kq_image(const ScanParams& p, size_t slot, int j)
{
    return static_cast<unsigned char*>(p.workspace) + kWsHeader + n_slots(p.T, p.n_seq) * p.hv * kAmBytes +
           (slot * p.hk + j) * kKqBytes;
}

__device__ __forceinline__ float* gram_rows(const ScanParams& p, size_t slot, int j)
{
    return reinterpret_cast<float*>(static_cast<unsigned char*>(p.workspace) + kWsHeader +
                                    n_slots(p.T, p.n_seq) * ((size_t)p.hv * kAmBytes + (size_t)p.hk * kKqBytes) +
                                    (slot * p.hk + j) * kGramBytes);
}

// slot -> (sequence, first token, token count); false for a slot no sequence uses
__device__ __forceinline__ bool slot_chunk(const ScanParams& p, int slot, int& c0, int& n)
{
    int lo = 0, hi = p.n_seq - 1;
    while (lo < hi) {  // last s with base(s) <= slot
        const int mid = (lo + hi + 1) >> 1;
        if (slot_base(p, mid) <= slot) lo = mid; else hi = mid - 1;
    }
    const int start = cu_at(p.cu_seqlens, lo, p.T), end = max(cu_at(p.cu_seqlens, lo + 1, p.T), start);
    c0 = start + (slot - slot_base(p, lo)) * kChunk;
    n = min(kChunk, end - c0);
    return slot >= slot_base(p, lo) && c0 < end;
}

// running log-decay of one chunk from warp 0: lam[q] for tokens lane + 32 q in,
// inclusive sums out; returns the chunk total
__device__ __forceinline__ float warp_chunk_cumsum(float (&lam)[2], int lane)
{
#pragma unroll
    for (int q = 0; q < 2; ++q)
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const float y = __shfl_up_sync(0xffffffffu, lam[q], off);
            if (lane >= off) lam[q] += y;
        }
    lam[1] += __shfl_sync(0xffffffffu, lam[0], 31);
    return __shfl_sync(0xffffffffu, lam[1], 31);
}

// =======================================================================================
// gram: one CTA per (chunk slot, key head): split [K; Q] (the chain's operand
// image) and (K K^T ; Q K^T) in fp32 for the prep kernel
// =======================================================================================
constexpr int kGramThreads = 256;

struct __align__(1024) GramSmem {
    uint16_t akq[2][128 * 128];  // split [K; Q] (K-major)
    uint32_t tmem_base;
    int abort_flag;
    uint64_t mbar;
};

__global__ void __launch_bounds__(kGramThreads) scan_gram_kernel(ScanParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    GramSmem& sm = *reinterpret_cast<GramSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int L = tid & 127, wg = tid >> 7;
    const int slot = blockIdx.x, j = blockIdx.y;
    uint32_t* err = reinterpret_cast<uint32_t*>(p.workspace);
    int c0, n;
    if (!slot_chunk(p, slot, c0, n)) return;  // unused slot (whole CTA)

    if (warp == 0) umma::tmem_alloc(&sm.tmem_base, 64);
    if (tid == 0) {
        umma::mbar_init(&sm.mbar, 1);
        sm.abort_flag = 0;
    }
    // Unit u = (matrix, token group, column group, row in group), row fastest so
    // that 8 consecutive lanes fill one 128-byte core matrix; all loads in flight together.
    {
        constexpr int kU = 2 * 64 * 16 / kGramThreads;
        float4 ld[2 * kU];
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int u = tid + kGramThreads * q;
            const int mat = u >> 10, tg = (u >> 7) & 7, g = (u >> 3) & 15, t = tg * 8 + (u & 7);
            if (t < n) {
                const float4* src = reinterpret_cast<const float4*>(
                    (mat ? p.qn : p.kn) + ((size_t)(c0 + t) * p.hk + j) * kHeadDim + g * 8);
                ld[2 * q] = __ldg(src);
                ld[2 * q + 1] = __ldg(src + 1);
            } else {
                ld[2 * q] = ld[2 * q + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        unsigned char* img = kq_image(p, slot, j);
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            const int u = tid + kGramThreads * q;
            const int mat = u >> 10, tg = (u >> 7) & 7, g = (u >> 3) & 15, t = tg * 8 + (u & 7);
            const float x[8] = {ld[2 * q].x, ld[2 * q].y, ld[2 * q].z, ld[2 * q].w,
                                ld[2 * q + 1].x, ld[2 * q + 1].y, ld[2 * q + 1].z, ld[2 * q + 1].w};
            uint4 vh, vl;
            split8(x, vh, vl);
            const int off = kmaj(mat * 64 + t, g * 8, 128);
            *reinterpret_cast<uint4*>(&sm.akq[0][off]) = vh;
            *reinterpret_cast<uint4*>(&sm.akq[1][off]) = vl;
            *reinterpret_cast<uint4*>(img + off * 2) = vh;
            *reinterpret_cast<uint4*>(img + kKqBytes / 2 + off * 2) = vl;
        }
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    // (K K^T ; Q K^T) = [K; Q] K^T  (B = the K rows of the same tile)
    if (tid == 0) {
        const uint32_t a_hi = umma::smem_u32(sm.akq[0]), a_lo = umma::smem_u32(sm.akq[1]);
        mma_split(tmem, a_hi, a_lo, 128, 2048, 256, a_hi, a_lo, 2048, 256, 8, umma::idesc_bf16(128, 64, false, false));
        umma::commit(&sm.mbar);
    }
    if (!umma::mbar_wait(&sm.mbar, 0)) { sm.abort_flag = 1; atomicOr(err, kErrTimeout); }
    __syncthreads();
    if (!sm.abort_flag) {
        umma::fence_after_sync();
        float d[32];
        umma::tmem_ld32(tmem + ((uint32_t)((warp & 3) * 32) << 16) + 32 * wg, d);
        umma::tmem_wait_ld();
        float4* dst = reinterpret_cast<float4*>(gram_rows(p, slot, j) + L * 64 + 32 * wg);
#pragma unroll
        for (int q = 0; q < 8; ++q) dst[q] = make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(sm.tmem_base, 64);
}

// =======================================================================================
// prep: one CTA per (chunk slot, key head); its value heads one after another
// =======================================================================================
constexpr int kPrepThreads = 256;  // two warpgroups: each covers all 128 TMEM lanes, half the columns

struct __align__(1024) PrepSmem {
    uint16_t ap[2][64 * 64];   // P (K-major, 64 rows); an M = 128 descriptor reads its rows 64-127 from
    uint16_t bt[2][64 * 64];   //   the next 16 KB (here), whose products are never read
    float A[64 * 68];          // fp32 A and T (rows padded to 68 floats)
    float T[64 * 68];
    float W[32 * 32];          // off-diagonal block products of the solve
    float G[64], beta[64];
    uint32_t tmem_base;
    int abort_flag;
    uint64_t mbar;
};

__global__ void __launch_bounds__(kPrepThreads, 3) scan_prep_kernel(ScanParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    PrepSmem& sm = *reinterpret_cast<PrepSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = tid & 127, wg = tid >> 7;  // TMEM lane, column half
    const int slot = blockIdx.x, j = blockIdx.y;
    const int group = p.hv / p.hk;
    uint32_t* err = reinterpret_cast<uint32_t*>(p.workspace);
    constexpr int ST = 68;  // fp32 row stride of A and T
    int c0, n;
    if (!slot_chunk(p, slot, c0, n)) return;  // unused slot (whole CTA)
    const float qscale = rsqrtf((float)kHeadDim);

    if (warp == 0) umma::tmem_alloc(&sm.tmem_base, 64);
    if (tid == 0) {
        umma::mbar_init(&sm.mbar, 1);
        sm.abort_flag = 0;
    }
    // raw gates of a value head, loaded by warp 0 one head ahead
    float raw_lam[2] = {0.f, 0.f}, raw_beta[2] = {0.f, 0.f};
    auto load_gates = [&](int h) {
        if (warp == 0) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int t = lane + 32 * q;
                raw_lam[q] = t < n ? __ldg(p.glog + (size_t)(c0 + t) * p.hv + h) : 0.0f;
                raw_beta[q] = t < n ? __ldg(p.beta + (size_t)(c0 + t) * p.hv + h) : 0.0f;
            }
        }
    };
    load_gates(j * group);
    // this thread's 32 entries of the gram rows: row L (K K^T for L < 64, Q K^T
    // for L >= 64), columns [32 wg, 32 wg + 32); shared by all value heads
    float d[32];
    {
        const float4* src = reinterpret_cast<const float4*>(gram_rows(p, slot, j) + L * 64 + 32 * wg);
#pragma unroll
        for (int q = 0; q < 8; ++q) {
            const float4 x = __ldg(src + q);
            d[4 * q] = x.x; d[4 * q + 1] = x.y; d[4 * q + 2] = x.z; d[4 * q + 3] = x.w;
        }
    }
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t a_p[2] = {umma::smem_u32(sm.ap[0]), umma::smem_u32(sm.ap[1])};
    const uint32_t b_t[2] = {umma::smem_u32(sm.bt[0]), umma::smem_u32(sm.bt[1])};
    uint32_t phase = 0;
    float* A = sm.A;
    float* Tm = sm.T;

    for (int hh = 0; hh < group; ++hh) {
        const int h = j * group + hh;
        // gates of value head h: running log-decay G and beta
        if (warp == 0) {
            float lam[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) lam[q] = (lane + 32 * q) < n ? fmaxf(raw_lam[q], kLamFloor) : 0.0f;
            const float b0 = raw_beta[0], b1 = raw_beta[1];
            if (hh + 1 < group) load_gates(h + 1);
            warp_chunk_cumsum(lam, lane);
            sm.G[lane] = lam[0];
            sm.G[lane + 32] = lam[1];
            sm.beta[lane] = b0;
            sm.beta[lane + 32] = b1;
        }
        __syncthreads();

        // A (fp32, rows L < 64) and P (split, rows L - 64 for L >= 64), columns of wg
        {
            const int i = L & 63, cb = 32 * wg;
            const float Gi = sm.G[i];
            const float4* G4 = reinterpret_cast<const float4*>(sm.G + cb);
            if (L < 64) {
                const float bi = sm.beta[i];
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 g = G4[q];
                    const float gg[4] = {g.x, g.y, g.z, g.w};
                    float a[4];
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const int jj = cb + 4 * q + e;
                        a[e] = jj < i ? bi * __expf(Gi - gg[e]) * d[4 * q + e] : 0.0f;
                    }
                    *reinterpret_cast<float4*>(&A[i * ST + cb + 4 * q]) = make_float4(a[0], a[1], a[2], a[3]);
                }
            } else {
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const float4 ga = G4[2 * q], gb = G4[2 * q + 1];
                    const float gg[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                    float pr[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) {
                        const int jj = cb + 8 * q + e;
                        pr[e] = jj <= i ? __expf(Gi - gg[e]) * d[8 * q + e] * qscale : 0.0f;
                    }
                    store_split8(&sm.ap[0][kmaj(i, cb + 8 * q, 64)], &sm.ap[1][kmaj(i, cb + 8 * q, 64)], pr);
                }
            }
        }
        __syncthreads();

        // T = (I + A)^-1 (A strictly lower), recursively by halves: T = [[T1, 0], [-T2 A21 T1, T2]].
        // (1) the four 16x16 diagonal blocks by forward substitution (thread (b, c): column c;
        //     col[r] = [r == c] - sum_{m<r} A[r][m] col[m], the entries above c come out zero);
        // (2) the two 32x32 halves: T_(b,b-1) = -T_(b,b) A_(b,b-1) T_(b-1,b-1) for b = 1, 3;
        // (3) the 32x32 off-diagonal block: T21 = -T2 (A21 T1).
        // Only the block lower triangle of T is written; readers treat the rest as zero.
        {
            if (tid < 64) {
                const int b = tid >> 4, c = tid & 15, o = 16 * b;
                float col[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float acc = (r == c) ? 1.0f : 0.0f;
#pragma unroll
                    for (int m4 = 0; m4 < r; m4 += 4) {
                        const float4 a4 = *reinterpret_cast<const float4*>(&A[(o + r) * ST + o + m4]);
                        if (m4 + 0 < r) acc = fmaf(-a4.x, col[m4 + 0], acc);
                        if (m4 + 1 < r) acc = fmaf(-a4.y, col[m4 + 1], acc);
                        if (m4 + 2 < r) acc = fmaf(-a4.z, col[m4 + 2], acc);
                        if (m4 + 3 < r) acc = fmaf(-a4.w, col[m4 + 3], acc);
                    }
                    col[r] = acc;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tm[(o + r) * ST + o + c] = col[r];
            }
            __syncthreads();
            {   // (2) pairs b = 1 (rows 16-31 x cols 0-15) and b = 3 (rows 48-63 x cols 32-47)
                const int pr = tid >> 7, r = (tid >> 3) & 15, c2 = 2 * (tid & 7);
                const int ro = 32 * pr + 16, co = 32 * pr;  // block (b, b-1) origin
                float w0 = 0.f, w1 = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float a = A[(ro + r) * ST + co + m];
                    const float2 t2 = *reinterpret_cast<const float2*>(&Tm[(co + m) * ST + co + c2]);
                    w0 = fmaf(a, t2.x, w0);
                    w1 = fmaf(a, t2.y, w1);
                }
                *reinterpret_cast<float2*>(&sm.W[pr * 256 + r * 16 + c2]) = make_float2(w0, w1);
                __syncthreads();
                float t0 = 0.f, t1 = 0.f;
#pragma unroll
                for (int m = 0; m < 16; ++m) {
                    const float a = Tm[(ro + r) * ST + ro + m];
                    const float2 w2 = *reinterpret_cast<const float2*>(&sm.W[pr * 256 + m * 16 + c2]);
                    t0 = fmaf(a, w2.x, t0);
                    t1 = fmaf(a, w2.y, t1);
                }
                *reinterpret_cast<float2*>(&Tm[(ro + r) * ST + co + c2]) = make_float2(-t0, -t1);
            }
            __syncthreads();
            {   // (3) rows 32-63 x cols 0-31; T1 and T2 are block lower triangular
                const int r = tid >> 3, c4 = 4 * (tid & 7);
                float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                for (int m = 0; m < 32; ++m) {
                    if ((m >> 4) < (c4 >> 4)) continue;  // T1[m][c] = 0 above the block diagonal
                    const float a = A[(32 + r) * ST + m];
                    const float4 t4 = *reinterpret_cast<const float4*>(&Tm[m * ST + c4]);
                    acc[0] = fmaf(a, t4.x, acc[0]); acc[1] = fmaf(a, t4.y, acc[1]);
                    acc[2] = fmaf(a, t4.z, acc[2]); acc[3] = fmaf(a, t4.w, acc[3]);
                }
                *reinterpret_cast<float4*>(&sm.W[r * 32 + c4]) = make_float4(acc[0], acc[1], acc[2], acc[3]);
                __syncthreads();
                float t[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll 8
                for (int m = 0; m < 32; ++m) {
                    if ((m >> 4) > (r >> 4)) continue;  // T2[r][m] = 0 above the block diagonal
                    const float a = Tm[(32 + r) * ST + 32 + m];
                    const float4 w4 = *reinterpret_cast<const float4*>(&sm.W[m * 32 + c4]);
                    t[0] = fmaf(a, w4.x, t[0]); t[1] = fmaf(a, w4.y, t[1]);
                    t[2] = fmaf(a, w4.z, t[2]); t[3] = fmaf(a, w4.w, t[3]);
                }
                *reinterpret_cast<float4*>(&Tm[(32 + r) * ST + c4]) = make_float4(-t[0], -t[1], -t[2], -t[3]);
            }
            __syncthreads();
            // T -> MN-major B tile (element (n = column, k = row)); row fastest across
            // lanes; column groups right of the row's diagonal block are zero
            for (int u = tid; u < 64 * 8; u += kPrepThreads) {
                const int m = u & 63, g = u >> 6;
                float tr[8];
                if ((g >> 1) <= (m >> 4)) {
                    const float4 x0 = *reinterpret_cast<const float4*>(&Tm[m * ST + g * 8]);
                    const float4 x1 = *reinterpret_cast<const float4*>(&Tm[m * ST + g * 8 + 4]);
                    tr[0] = x0.x; tr[1] = x0.y; tr[2] = x0.z; tr[3] = x0.w;
                    tr[4] = x1.x; tr[5] = x1.y; tr[6] = x1.z; tr[7] = x1.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 8; ++e) tr[e] = 0.0f;
                }
                store_split8(&sm.bt[0][mnmaj(g * 8, m, 64)], &sm.bt[1][mnmaj(g * 8, m, 64)], tr);
            }
        }
        umma::fence_proxy_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();

        // P T  (M = 128 descriptor over the 64-row P tile; rows 64-127 of the product unused)
        if (tid == 0) {
            mma_split(tmem, a_p[0], a_p[1], 128, 1024, 256, b_t[0], b_t[1], 1024, 256, 4,
                      umma::idesc_bf16(128, 64, false, true));
            umma::commit(&sm.mbar);
        }
        if (!umma::mbar_wait(&sm.mbar, phase)) { sm.abort_flag = 1; atomicOr(err, kErrTimeout); }
        phase ^= 1u;
        __syncthreads();
        if (sm.abort_flag) goto done;
        umma::fence_after_sync();

        // [T; P T] image (K-major, split): threads L >= 64 write row L - 64 (T, from shared
        // memory), threads L < 64 write row 64 + L (P T, from TMEM lane L); columns of wg
        {
            unsigned char* img = am_image(p, slot, h);
            const int cb = 32 * wg;
            float x[32];
            int row;
            if (L < 64) {
                umma::tmem_ld32(tmem + lane_off + cb, x);
                umma::tmem_wait_ld();
                row = 64 + L;
            } else {
                const int m = L - 64;
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int g = (cb + 4 * q) >> 3;
                    float4 t4 = make_float4(0.f, 0.f, 0.f, 0.f);
                    if ((g >> 1) <= (m >> 4)) t4 = *reinterpret_cast<const float4*>(&Tm[m * ST + cb + 4 * q]);
                    x[4 * q] = t4.x; x[4 * q + 1] = t4.y; x[4 * q + 2] = t4.z; x[4 * q + 3] = t4.w;
                }
                row = m;
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 vh, vl;
                split8(x + 8 * q, vh, vl);
                const int off = kmaj(row, cb + 8 * q, 64);
                *reinterpret_cast<uint4*>(img + off * 2) = vh;
                *reinterpret_cast<uint4*>(img + kAmBytes / 2 + off * 2) = vl;
            }
        }
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
    }

done:
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(sm.tmem_base, 64);
}

// =======================================================================================
// chain: one CTA per (sequence, value head, kDVS-column slice)
// =======================================================================================
constexpr int kChainWG = 4;                   // warpgroups; each covers all 128 TMEM lanes
constexpr int kChainThreads = 128 * kChainWG;  // and kDVS / kChainWG of the columns

template <int DVS>
struct __align__(1024) ChainSmem {
    uint16_t akq[2][2][128 * 128];  // [K; Q] image, double-buffered: [buffer][hi/lo]
    uint16_t am[2][128 * 64];       // [T; P T] image
    uint16_t bs[2][128 * DVS];      // S slice (MN-major B, dk x DVS)
    uint16_t bx[2][64 * DVS];       // X, then e^{G_L-G} U (MN-major B, 64 x DVS)
    float v[64 * (DVS + 4)];        // V tile of the slice (rows padded by 16 bytes), later the O tile
    float eG[64], beta[64], kdec[64];
    float gL;
    uint32_t tmem_base;
    int abort_flag;
    uint64_t mbar_mma, mbar_kq[2], mbar_am;
};

template <int COLS>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&d)[COLS])
{
    static_assert(COLS == 16 || COLS == 32, "column count");
    if constexpr (COLS == 16) umma::tmem_ld16(taddr, d);
    else umma::tmem_ld32(taddr, d);
}

template <int DVS>
__global__ void __launch_bounds__(kChainThreads, 1) scan_chain_kernel(ScanParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    ChainSmem<DVS>& sm = *reinterpret_cast<ChainSmem<DVS>*>(smem_raw);
    constexpr int SLICES = kHeadDim / DVS;
    constexpr int COLS = DVS / kChainWG;  // columns per thread
    constexpr uint32_t kTmemCols = 512;
    // each product takes 2*DVS columns: [hi*hi + lo*hi | hi*lo]
    constexpr uint32_t cD2 = 0, cD3 = 2 * DVS, cD4 = 4 * DVS;
    static_assert(6 * DVS <= (int)kTmemCols, "TMEM columns");
    constexpr int kGateWarp = 3;   // computes the gates while thread 0 issues MMAs
    constexpr int kCopyThread = 64;  // issues the bulk copies

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = tid & 127;            // TMEM lane of this thread
    const int wg = tid >> 7;            // column group
    const int cb = wg * COLS;           // first column of this thread within the slice
    const int h = blockIdx.x / SLICES, slice = blockIdx.x % SLICES, s = blockIdx.y;
    const int j = h / (p.hv / p.hk);
    const int v0 = slice * DVS;
    const int t0 = cu_at(p.cu_seqlens, s, p.T), t1 = max(cu_at(p.cu_seqlens, s + 1, p.T), t0);
    const int n_chunks = (t1 - t0 + kChunk - 1) / kChunk;
    const size_t base = (size_t)slot_base(p, s);
    const size_t sbase = ((size_t)s * p.hv + h) * kHeadDim * kHeadDim;
    const float qscale = rsqrtf((float)kHeadDim);
    uint32_t* err = reinterpret_cast<uint32_t*>(p.workspace);

    if (warp == 0) umma::tmem_alloc(&sm.tmem_base, kTmemCols);
    if (tid == 0) {
        umma::mbar_init(&sm.mbar_mma, 1);
        umma::mbar_init(&sm.mbar_kq[0], 1);
        umma::mbar_init(&sm.mbar_kq[1], 1);
        umma::mbar_init(&sm.mbar_am, 1);
        sm.abort_flag = 0;
    }

    // state slice: thread (L, wg) holds row L (key index), columns v0 + cb + [0, COLS)
    float S[COLS];
    {
        const float* src = p.S_in + sbase + (size_t)L * kHeadDim + v0 + cb;
#pragma unroll
        for (int c = 0; c < COLS; c += 4) {
            const float4 x = *reinterpret_cast<const float4*>(src + c);
            S[c] = x.x; S[c + 1] = x.y; S[c + 2] = x.z; S[c + 3] = x.w;
        }
#pragma unroll
        for (int c = 0; c < COLS; c += 8)
            store_split8(&sm.bs[0][mnmaj(cb + c, L, 128)], &sm.bs[1][mnmaj(cb + c, L, 128)], S + c);
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();

    const uint32_t tmem = sm.tmem_base;
    const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t b_s = umma::smem_u32(sm.bs[0]);
    const uint32_t b_x = umma::smem_u32(sm.bx[0]);
    const uint32_t a_m[2] = {umma::smem_u32(sm.am[0]), umma::smem_u32(sm.am[1])};
    uint32_t ph_mma = 0;
    // outstanding bulk copies (uniform across threads): issued but not yet waited
    bool pend_kq[2] = {false, false}, pend_am = false;

    // ---- bulk-copy issue helpers -----------------------------------------------------------
    auto issue_kq = [&](int c) {  // [K; Q] image of chunk c into buffer c & 1
        if (tid == kCopyThread) {
            uint64_t* mb = &sm.mbar_kq[c & 1];
            umma::mbar_arrive_expect_tx(mb, (uint32_t)kKqBytes);
            umma::bulk_g2s(sm.akq[c & 1], kq_image(p, base + c, j), (uint32_t)kKqBytes, mb);
        }
        pend_kq[c & 1] = true;
    };
    auto issue_am = [&](int c) {
        if (tid == kCopyThread) {
            umma::mbar_arrive_expect_tx(&sm.mbar_am, (uint32_t)kAmBytes);
            umma::bulk_g2s(sm.am, am_image(p, base + c, h), (uint32_t)kAmBytes, &sm.mbar_am);
        }
        pend_am = true;
    };
    // V tile of a chunk: every thread loads its float4s into registers one chunk ahead
    constexpr int kVq = 64 * DVS / 4 / kChainThreads;
    float4 vpre[kVq];
    auto load_v = [&](int c) {
        const int cc0 = t0 + c * kChunk, nn = min(kChunk, t1 - cc0);
#pragma unroll
        for (int q = 0; q < kVq; ++q) {
            const int u = tid + kChainThreads * q, t = u / (DVS / 4), c4 = (u % (DVS / 4)) * 4;
            vpre[q] = t < nn ? __ldg(reinterpret_cast<const float4*>(p.vc + ((size_t)(cc0 + t) * p.hv + h) * kHeadDim + v0 + c4))
                             : make_float4(0.f, 0.f, 0.f, 0.f);
        }
    };
    auto store_v = [&]() {
#pragma unroll
        for (int q = 0; q < kVq; ++q) {
            const int u = tid + kChainThreads * q, t = u / (DVS / 4), c4 = (u % (DVS / 4)) * 4;
            *reinterpret_cast<float4*>(&sm.v[t * (DVS + 4) + c4]) = vpre[q];
        }
    };
    // gates of one chunk, raw values prefetched into the gate warp's registers one chunk ahead
    float lam_nx[2] = {0.f, 0.f}, bet_nx[2] = {0.f, 0.f};
    int n_nx = 0;
    auto load_gates = [&](int c) {
        const int cc0 = t0 + c * kChunk, nn = min(kChunk, t1 - cc0);
        n_nx = nn;
        if (warp == kGateWarp) {
#pragma unroll
            for (int q = 0; q < 2; ++q) {
                const int t = lane + 32 * q;
                lam_nx[q] = t < nn ? __ldg(p.glog + (size_t)(cc0 + t) * p.hv + h) : 0.0f;
                bet_nx[q] = t < nn ? __ldg(p.beta + (size_t)(cc0 + t) * p.hv + h) : 0.0f;
            }
        }
    };

#define GDN_WAIT(mbar, parity)                                                 \
    do {                                                                       \
        if (!umma::mbar_wait((mbar), (parity))) {                              \
            sm.abort_flag = 1;                                                 \
            atomicOr(err, kErrTimeout);                                        \
        }                                                                      \
    } while (0)
#define GDN_SYNC_OR_ABORT()                                                    \
    do {                                                                       \
        __syncthreads();                                                       \
        if (sm.abort_flag) goto done;                                          \
        umma::fence_after_sync();                                              \
    } while (0)
#define GDN_PUBLISH()                                                          \
    do {                                                                       \
        umma::fence_proxy_async();                                             \
        umma::fence_before_sync();                                             \
        __syncthreads();                                                       \
        umma::fence_after_sync();                                              \
    } while (0)

    if (n_chunks > 0) {
        issue_kq(0);
        issue_am(0);
        load_gates(0);
        load_v(0);
        store_v();
    }

    for (int c = 0; c < n_chunks; ++c) {
        const int c0 = t0 + c * kChunk, n = min(kChunk, t1 - c0);
        const bool more = c + 1 < n_chunks;
        if (more) issue_kq(c + 1);  // its buffer was last read by chunk c-1's state update

        // ---- (K S0 ; Q S0) = [K; Q] S0 ------------------------------------------------------------
        GDN_WAIT(&sm.mbar_kq[c & 1], (c >> 1) & 1);
        pend_kq[c & 1] = false;
        GDN_SYNC_OR_ABORT();
        const uint32_t a_kq_hi = umma::smem_u32(sm.akq[c & 1][0]), a_kq_lo = umma::smem_u32(sm.akq[c & 1][1]);
        if (tid == 0) {
            mma_split2(tmem + cD2, a_kq_hi, a_kq_lo, 128, 2048, 256, b_s, 2048, 256, 8, DVS, false, true);
            umma::commit(&sm.mbar_mma);
        }
        // ---- meanwhile: gates e^G, beta, e^{G_L - G}, e^{G_L}; next chunk's gates and V ---------
        if (warp == kGateWarp) {
            float lam[2];
#pragma unroll
            for (int q = 0; q < 2; ++q) lam[q] = (lane + 32 * q) < n_nx ? fmaxf(lam_nx[q], kLamFloor) : 0.0f;
            const float b0 = bet_nx[0], b1 = bet_nx[1];
            if (more) load_gates(c + 1);
            const float GL = warp_chunk_cumsum(lam, lane);
            sm.eG[lane] = __expf(lam[0]);
            sm.eG[lane + 32] = __expf(lam[1]);
            sm.kdec[lane] = __expf(GL - lam[0]);
            sm.kdec[lane + 32] = __expf(GL - lam[1]);
            sm.beta[lane] = b0;
            sm.beta[lane + 32] = b1;
            if (lane == 0) sm.gL = __expf(GL);
        } else if (more) {
            n_nx = min(kChunk, t1 - (c0 + kChunk));
        }
        if (more) load_v(c + 1);
        GDN_WAIT(&sm.mbar_mma, ph_mma);
        ph_mma ^= 1u;
        GDN_SYNC_OR_ABORT();

        // ---- X = beta (V - e^G K S0) -> bx;  keep e^G Q S0 / sqrt(dk) --------------------------------
        float qs[COLS];
        {
            const int t = L & 63;
            float d[COLS], d2[COLS];
            tmem_ld_cols<COLS>(tmem + lane_off + cD2 + cb, d);
            tmem_ld_cols<COLS>(tmem + lane_off + cD2 + DVS + cb, d2);
            umma::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < COLS; ++e) d[e] += d2[e];
            if (L < 64) {
                const float bt = sm.beta[t], eg = sm.eG[t];
                const float4* vr = reinterpret_cast<const float4*>(&sm.v[t * (DVS + 4) + cb]);
#pragma unroll
                for (int cc = 0; cc < COLS; cc += 8) {
                    const float4 va = vr[cc / 4], vb = vr[cc / 4 + 1];
                    const float vv[8] = {va.x, va.y, va.z, va.w, vb.x, vb.y, vb.z, vb.w};
                    float x[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) x[e] = bt * (vv[e] - eg * d[cc + e]);
                    store_split8(&sm.bx[0][mnmaj(cb + cc, t, 64)], &sm.bx[1][mnmaj(cb + cc, t, 64)], x);
                }
            } else {
                const float f = sm.eG[t] * qscale;
#pragma unroll
                for (int e = 0; e < COLS; ++e) qs[e] = f * d[e];
            }
        }
        GDN_PUBLISH();

        // ---- (U ; P U) = [T; P T] X --------------------------------------------------------------------
        GDN_WAIT(&sm.mbar_am, c & 1);
        pend_am = false;
        GDN_SYNC_OR_ABORT();
        if (tid == 0) {
            mma_split2(tmem + cD3, a_m[0], a_m[1], 128, 1024, 256, b_x, 1024, 256, 4, DVS, false, true);
            umma::commit(&sm.mbar_mma);
        }
        GDN_WAIT(&sm.mbar_mma, ph_mma);
        ph_mma ^= 1u;
        GDN_SYNC_OR_ABORT();
        if (more) issue_am(c + 1);  // [T; P T] image consumed

        // ---- e^{G_L-G} U -> bx;  O = e^G Q S0 / sqrt(dk) + P U -> the V tile ----------------------------
        {
            const int t = L & 63;
            float d[COLS], d2[COLS];
            tmem_ld_cols<COLS>(tmem + lane_off + cD3 + cb, d);
            tmem_ld_cols<COLS>(tmem + lane_off + cD3 + DVS + cb, d2);
            umma::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < COLS; ++e) d[e] += d2[e];
            if (L < 64) {
                const float kd = sm.kdec[t];
#pragma unroll
                for (int e = 0; e < COLS; ++e) d[e] *= kd;
#pragma unroll
                for (int cc = 0; cc < COLS; cc += 8)
                    store_split8(&sm.bx[0][mnmaj(cb + cc, t, 64)], &sm.bx[1][mnmaj(cb + cc, t, 64)], d + cc);
            } else {  // O row t -> the (consumed) V tile, written out coalesced below
                float* dst = &sm.v[t * (DVS + 4) + cb];
#pragma unroll
                for (int e = 0; e < COLS; e += 4)
                    *reinterpret_cast<float4*>(dst + e) =
                        make_float4(qs[e] + d[e], qs[e + 1] + d[e + 1], qs[e + 2] + d[e + 2], qs[e + 3] + d[e + 3]);
            }
        }
        GDN_PUBLISH();

        // ---- dS = K^T (e^{G_L-G} U): K^T is the K half of the [K; Q] image, MN-major ------------------
        if (tid == 0) {
            mma_split2(tmem + cD4, a_kq_hi, a_kq_lo, 2048, 128, 4096, b_x, 1024, 256, 4, DVS, true, true);
            umma::commit(&sm.mbar_mma);
        }
        // O tile -> global while the state update runs: DVS/4 threads per row
#pragma unroll
        for (int q = 0; q < kVq; ++q) {
            const int u = tid + kChainThreads * q, t = u / (DVS / 4), c4 = (u % (DVS / 4)) * 4;
            if (t < n)
                __stcs(reinterpret_cast<float4*>(p.o + ((size_t)(c0 + t) * p.hv + h) * kHeadDim + v0 + c4),
                       *reinterpret_cast<const float4*>(&sm.v[t * (DVS + 4) + c4]));
        }
        GDN_WAIT(&sm.mbar_mma, ph_mma);
        ph_mma ^= 1u;
        GDN_SYNC_OR_ABORT();
        if (more) store_v();  // O tile written out: the next chunk's V goes in

        // ---- S = e^{G_L} S + dS -> registers and bs ----------------------------------------------------
        {
            const float gl = sm.gL;
            float d[COLS], d2[COLS];
            tmem_ld_cols<COLS>(tmem + lane_off + cD4 + cb, d);
            tmem_ld_cols<COLS>(tmem + lane_off + cD4 + DVS + cb, d2);
            umma::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < COLS; ++e) S[e] = fmaf(gl, S[e], d[e] + d2[e]);
#pragma unroll
            for (int cc = 0; cc < COLS; cc += 8)
                store_split8(&sm.bs[0][mnmaj(cb + cc, L, 128)], &sm.bs[1][mnmaj(cb + cc, L, 128)], S + cc);
        }
        GDN_PUBLISH();
    }

    {
        float* dst = p.S_out + sbase + (size_t)L * kHeadDim + v0 + cb;
#pragma unroll
        for (int c = 0; c < COLS; c += 4)
            *reinterpret_cast<float4*>(dst + c) = make_float4(S[c], S[c + 1], S[c + 2], S[c + 3]);
    }

done:
    // drain any copy still in flight into this CTA's shared memory (bounded), free TMEM
    if (tid == kCopyThread) {
        for (int b = 0; b < 2; ++b)
            if (pend_kq[b]) umma::mbar_wait(&sm.mbar_kq[b], 0, 1u << 16), umma::mbar_wait(&sm.mbar_kq[b], 1, 1u << 16);
        if (pend_am) umma::mbar_wait(&sm.mbar_am, 0, 1u << 16), umma::mbar_wait(&sm.mbar_am, 1, 1u << 16);
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(sm.tmem_base, kTmemCols);
#undef GDN_WAIT
#undef GDN_SYNC_OR_ABORT
#undef GDN_PUBLISH
}

}  // namespace

size_t scan_workspace_bytes(int hk, int hv, int n_seq, int T)
{
    return kWsHeader + n_slots(T, n_seq) * ((size_t)hv * kAmBytes + (size_t)hk * (kKqBytes + kGramBytes));
}

cudaError_t launch_scan(const ScanParams& p, cudaStream_t stream)
{
    if (p.n_seq == 0) return cudaSuccess;
    const size_t gram_smem = sizeof(GramSmem), prep_smem = sizeof(PrepSmem), chain_smem = sizeof(ChainSmem<kDVS>);
    cudaError_t e = cudaFuncSetAttribute(scan_gram_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gram_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(scan_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(scan_chain_kernel<kDVS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chain_smem);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p.workspace, 0, 4, stream);
    if (e != cudaSuccess) return e;
    const size_t slots = n_slots(p.T, p.n_seq);
    if (p.T > 0) {
        scan_gram_kernel<<<dim3((unsigned)slots, (unsigned)p.hk), kGramThreads, gram_smem, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
        scan_prep_kernel<<<dim3((unsigned)slots, (unsigned)p.hk), kPrepThreads, prep_smem, stream>>>(p);
        e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    scan_chain_kernel<kDVS><<<dim3((unsigned)(p.hv * (kHeadDim / kDVS)), (unsigned)p.n_seq), kChainThreads,
                              chain_smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
