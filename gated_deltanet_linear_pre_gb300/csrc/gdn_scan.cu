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
// the chunk start, G_i = running sum of lam = log g inside the chunk):
//   A_ij = beta_i e^{G_i-G_j} (k_i.k_j) (j < i),   T = (I + A)^-1
//   P_ij = e^{G_i-G_j} (q_i.k_j) / sqrt(dk) (j <= i)
//   X    = beta (V - e^G (K S0))                   U = T X
//   O    = e^G (Q S0) / sqrt(dk) + P U             S = e^{G_L} S0 + Kd^T U
// with Kd = diag(e^{G_L - G_j}) K.  Every dense product runs on the tensor
// core with bf16 operands split as x = hi + lo (hi = bf16(x), lo = bf16(x -
// hi)) and three MMAs hi*hi + hi*lo + lo*hi accumulated in fp32 in TMEM,
// which keeps ~16 significant bits per operand.  Two products are stacked to
// fill the M = 128 rows of one MMA:
//   [K; Q] K^T -> (K K^T ; Q K^T)          [I; P] T -> (T ; P T)
//   [K; Q] S0  -> (K S0 ; Q S0)            [T; P T] X -> (U ; P U)
//   Kd^T U     -> the state update
// so (Q S0) and (P U) land in the same TMEM lanes and O needs no exchange.
// The 64x64 unit lower-triangular inverse is a blocked forward substitution
// (16x16 diagonal blocks, then off-diagonal blocks by distance) on CUDA cores.
//
// One CTA (128 threads, thread i <-> TMEM lane i) owns DVS value columns of
// one (sequence, value head) and carries its fp32 state slice in registers
// through every chunk of the sequence.  Each MMA is issued by thread 0 and
// completes on an mbarrier; every wait is bounded and, on expiry, the CTA
// records an error code in the workspace and stops.
#include "gdn_internal.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr int kThreads = 128;
constexpr float kLamFloor = -110.0f;  // e^-110 is below the smallest fp32 denormal: g = 0 exactly
constexpr uint32_t kErrTimeout = 1u;

// element offsets inside no-swizzle core-matrix tiles (bf16, 64 elements per core matrix)
__device__ __forceinline__ int kmaj(int r, int k, int Kd) { return ((r >> 3) * (Kd >> 3) + (k >> 3)) * 64 + (r & 7) * 8 + (k & 7); }
__device__ __forceinline__ int mnmaj(int mn, int k, int Kd) { return ((mn >> 3) * (Kd >> 3) + (k >> 3)) * 64 + (k & 7) * 8 + (mn & 7); }

// split 8 fp32 values into bf16 hi and lo and store them as two 16-byte vectors
__device__ __forceinline__ void store_split8(uint16_t* hi, uint16_t* lo, const float* x)
{
    uint16_t h[8], l[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) umma::split_bf16(x[e], h[e], l[e]);
    uint4 vh, vl;
    vh.x = h[0] | ((uint32_t)h[1] << 16); vh.y = h[2] | ((uint32_t)h[3] << 16);
    vh.z = h[4] | ((uint32_t)h[5] << 16); vh.w = h[6] | ((uint32_t)h[7] << 16);
    vl.x = l[0] | ((uint32_t)l[1] << 16); vl.y = l[2] | ((uint32_t)l[3] << 16);
    vl.z = l[4] | ((uint32_t)l[5] << 16); vl.w = l[6] | ((uint32_t)l[7] << 16);
    *reinterpret_cast<uint4*>(hi) = vh;
    *reinterpret_cast<uint4*>(lo) = vl;
}

template <int DVS>
struct __align__(1024) ScanSmem {
    uint16_t akq[2][128 * 128];  // [K; Q] (K-major, 128 rows x dk): A of KK^T/QK^T and of KS/QS; rows 0-63 are B of KK^T
    uint16_t akt[2][128 * 64];   // Kd^T (MN-major, dk x 64 tokens): A of the state update
    struct { float A[64 * 64]; float T[64 * 64]; } f;  // fp32 A and T while solving
    uint16_t am[2][128 * 64];    // [I; P] (A of P T), then [T; P T] (A of U / P U); K-major
    union {
        uint16_t bt[2][64 * 64];  // T (MN-major B, 64 x 64)
        float W[3 * 256];         // off-diagonal block sums of the solve
    } u2;
    uint16_t bs[2][128 * DVS];   // S slice (MN-major B, dk x DVS)
    uint16_t bx[2][64 * DVS];    // X, then U (MN-major B, 64 x DVS)
    float v[64 * DVS];           // V tile of the slice
    float G[64], eG[64], beta[64], kdec[64];
    float gL;
    uint32_t tmem_base;
    int abort_flag;
    uint64_t mbar;
};

// Three-pass split product D = A * B over `ksteps` 16-wide K steps.
__device__ __forceinline__ void mma_split(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t a_sbo, uint32_t b_hi,
                                          uint32_t b_lo, uint32_t b_sbo, int ksteps, uint32_t idesc)
{
    const uint32_t as[3] = {a_hi, a_hi, a_lo};
    const uint32_t bs[3] = {b_hi, b_lo, b_hi};
#pragma unroll
    for (int pass = 0; pass < 3; ++pass)
        for (int ks = 0; ks < ksteps; ++ks) {
            const uint64_t da = umma::desc(as[pass] + ks * 256, 128, a_sbo);
            const uint64_t db = umma::desc(bs[pass] + ks * 256, 128, b_sbo);
            umma::mma_bf16(d, da, db, idesc, (pass | ks) != 0);
        }
}

template <int DVS>
__global__ void __launch_bounds__(kThreads, 1) scan_tc_kernel(ScanParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    ScanSmem<DVS>& sm = *reinterpret_cast<ScanSmem<DVS>*>(smem_raw);
    constexpr int SLICES = kHeadDim / DVS;
    constexpr uint32_t kTmemCols = 256;
    // TMEM columns: [0,64) K K^T|Q K^T, then (K S0 ; Q S0); [64,128) T|P T, then (U ; P U); [128, 128+DVS) dS
    constexpr uint32_t cKQ = 0, cPT = 64, cD2 = 0, cD3 = 64, cD4 = 128;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x / SLICES, slice = blockIdx.x % SLICES, s = blockIdx.y;
    const int j = h / (p.hv / p.hk);
    const int v0 = slice * DVS;
    const int t0 = cu_at(p.cu_seqlens, s, p.T), t1 = max(cu_at(p.cu_seqlens, s + 1, p.T), t0);
    const size_t sbase = ((size_t)s * p.hv + h) * kHeadDim * kHeadDim;
    const float qscale = rsqrtf((float)kHeadDim);
    uint32_t* err = reinterpret_cast<uint32_t*>(p.workspace);

    if (warp == 0) umma::tmem_alloc(&sm.tmem_base, kTmemCols);
    if (tid == 0) {
        umma::mbar_init(&sm.mbar, 1);
        sm.abort_flag = 0;
    }

    // state slice: thread i holds row i (key index) of S[:, v0:v0+DVS]
    float S[DVS];
#pragma unroll
    for (int c = 0; c < DVS; c += 4) {
        const float4 x = *reinterpret_cast<const float4*>(p.S_in + sbase + (size_t)tid * kHeadDim + v0 + c);
        S[c] = x.x; S[c + 1] = x.y; S[c + 2] = x.z; S[c + 3] = x.w;
    }
#pragma unroll
    for (int c = 0; c < DVS; c += 8) store_split8(&sm.bs[0][mnmaj(c, tid, 128)], &sm.bs[1][mnmaj(c, tid, 128)], S + c);

    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;
    uint32_t phase = 0;

    const uint32_t a_kq[2] = {umma::smem_u32(sm.akq[0]), umma::smem_u32(sm.akq[1])};
    const uint32_t a_kt[2] = {umma::smem_u32(sm.akt[0]), umma::smem_u32(sm.akt[1])};
    const uint32_t a_m[2] = {umma::smem_u32(sm.am[0]), umma::smem_u32(sm.am[1])};
    const uint32_t b_t[2] = {umma::smem_u32(sm.u2.bt[0]), umma::smem_u32(sm.u2.bt[1])};
    const uint32_t b_s[2] = {umma::smem_u32(sm.bs[0]), umma::smem_u32(sm.bs[1])};
    const uint32_t b_x[2] = {umma::smem_u32(sm.bx[0]), umma::smem_u32(sm.bx[1])};

#define GDN_MMA_WAIT()                                                         \
    do {                                                                       \
        if (!umma::mbar_wait(&sm.mbar, phase)) {                               \
            sm.abort_flag = 1;                                                 \
            atomicOr(err, kErrTimeout);                                        \
        }                                                                      \
        phase ^= 1u;                                                           \
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

    for (int c0 = t0; c0 < t1; c0 += kChunk) {
        const int n = min(kChunk, t1 - c0);

        // ---- 1-2. gates (warp 0), [K; Q] -> akq, Kd^T -> akt, V tile --------------------------
        // Each thread owns 16 (matrix, token, 8-column group) units; their global loads are
        // issued in two batches of 8 so that only two load latencies sit on this path.
        {
            float4 ld[16];
            float4 vv[DVS / 8];
            auto unit_src = [&](int u) -> const float* {
                const int mat = u >> 10, t = (u >> 4) & 63, g = u & 15;
                return (mat ? p.qn : p.kn) + ((size_t)(c0 + t) * p.hk + j) * kHeadDim + g * 8;
            };
            auto issue = [&](int batch) {
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int u = tid + kThreads * (8 * batch + q);
                    const int t = (u >> 4) & 63;
                    if (t < n) {
                        ld[2 * q] = __ldg(reinterpret_cast<const float4*>(unit_src(u)));
                        ld[2 * q + 1] = __ldg(reinterpret_cast<const float4*>(unit_src(u)) + 1);
                    } else {
                        ld[2 * q] = ld[2 * q + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            };
            issue(0);
#pragma unroll
            for (int q = 0; q < DVS / 8; ++q) {
                const int u = tid + kThreads * q;
                const int t = u / (DVS / 4), c = (u % (DVS / 4)) * 4;
                vv[q] = t < n ? __ldg(reinterpret_cast<const float4*>(p.vc + ((size_t)(c0 + t) * p.hv + h) * kHeadDim + v0 + c))
                              : make_float4(0.f, 0.f, 0.f, 0.f);
            }
            if (warp == 0) {
                float lam[2], bb[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int t = lane + 32 * q;
                    lam[q] = t < n ? fmaxf(__ldg(p.glog + (size_t)(c0 + t) * p.hv + h), kLamFloor) : 0.0f;
                    bb[q] = t < n ? __ldg(p.beta + (size_t)(c0 + t) * p.hv + h) : 0.0f;
                }
#pragma unroll
                for (int q = 0; q < 2; ++q)
#pragma unroll
                    for (int off = 1; off < 32; off <<= 1) {
                        const float y = __shfl_up_sync(0xffffffffu, lam[q], off);
                        if (lane >= off) lam[q] += y;
                    }
                lam[1] += __shfl_sync(0xffffffffu, lam[0], 31);
                const float GL = __shfl_sync(0xffffffffu, lam[1], 31);
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int t = lane + 32 * q;
                    sm.G[t] = lam[q];
                    sm.eG[t] = expf(lam[q]);
                    sm.beta[t] = bb[q];
                    sm.kdec[t] = expf(GL - lam[q]);
                }
                if (lane == 0) sm.gL = expf(GL);
            }
#pragma unroll
            for (int q = 0; q < DVS / 8; ++q) {
                const int u = tid + kThreads * q;
                const int t = u / (DVS / 4), c = (u % (DVS / 4)) * 4;
                *reinterpret_cast<float4*>(&sm.v[t * DVS + c]) = vv[q];
            }
            __syncthreads();  // G, kdec visible
#pragma unroll
            for (int batch = 0; batch < 2; ++batch) {
                if (batch == 1) issue(1);
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const int u = tid + kThreads * (8 * batch + q);
                    const int mat = u >> 10, t = (u >> 4) & 63, g = u & 15;
                    float x[8] = {ld[2 * q].x, ld[2 * q].y, ld[2 * q].z, ld[2 * q].w,
                                  ld[2 * q + 1].x, ld[2 * q + 1].y, ld[2 * q + 1].z, ld[2 * q + 1].w};
                    const int r = mat * 64 + t;
                    store_split8(&sm.akq[0][kmaj(r, g * 8, 128)], &sm.akq[1][kmaj(r, g * 8, 128)], x);
                    if (mat == 0) {
                        const float kd = sm.kdec[t];
#pragma unroll
                        for (int e = 0; e < 8; ++e) x[e] *= kd;
                        // element (m = key index, k = token) of the MN-major A tile
                        store_split8(&sm.akt[0][mnmaj(g * 8, t, 64)], &sm.akt[1][mnmaj(g * 8, t, 64)], x);
                    }
                }
            }
        }
        GDN_PUBLISH();

        // ---- 3. (K K^T ; Q K^T) = [K; Q] K^T ------------------------------------------------
        if (tid == 0) {
            mma_split(tmem + cKQ, a_kq[0], a_kq[1], 2048, a_kq[0], a_kq[1], 2048, 8,
                      umma::idesc_bf16(128, 64, false, false));
            umma::commit(&sm.mbar);
        }
        GDN_MMA_WAIT();

        // ---- 4. A (fp32, rows 0-63) and [I; P] (split, rows 64-127 P, rows 0-63 I) ----------
        {
            const int i = tid & 63;
            const float Gi = sm.G[i];
#pragma unroll 1
            for (int c = 0; c < 64; c += 16) {
                float d[16];
                umma::tmem_ld16(tmem + lane_off + cKQ + c, d);
                umma::tmem_wait_ld();
                if (tid < 64) {
                    const float bi = sm.beta[i];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int jj = c + e;
                        sm.f.A[i * 64 + jj] = jj < i ? bi * expf(Gi - sm.G[jj]) * d[e] : 0.0f;
                    }
                } else {
                    float pr[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) {
                        const int jj = c + e;
                        pr[e] = jj <= i ? expf(Gi - sm.G[jj]) * d[e] * qscale : 0.0f;
                    }
                    store_split8(&sm.am[0][kmaj(64 + i, c, 64)], &sm.am[1][kmaj(64 + i, c, 64)], pr);
                    store_split8(&sm.am[0][kmaj(64 + i, c + 8, 64)], &sm.am[1][kmaj(64 + i, c + 8, 64)], pr + 8);
                }
            }
            if (tid < 64) {
#pragma unroll
                for (int c = 0; c < 64; c += 8) {
                    float idr[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) idr[e] = (c + e == i) ? 1.0f : 0.0f;
                    store_split8(&sm.am[0][kmaj(i, c, 64)], &sm.am[1][kmaj(i, c, 64)], idr);
                }
            }
        }
        __syncthreads();

        // ---- 5. T = (I + A)^-1 -----------------------------------------------------------------
        {
            float* A = sm.f.A;
            float* Tm = sm.f.T;
            for (int e = tid; e < 64 * 64; e += kThreads) Tm[e] = 0.0f;
            __syncthreads();
            if (tid < 64) {  // diagonal 16x16 blocks: column c of block b by forward substitution
                const int b = tid >> 4, c = tid & 15, o = 16 * b;
                float col[16];
#pragma unroll
                for (int r = 0; r < 16; ++r) {
                    float acc = (r == c) ? 1.0f : 0.0f;
                    if (r > c) {
#pragma unroll
                        for (int m = 0; m < 16; ++m)
                            if (m >= c && m < r) acc -= A[(o + r) * 64 + o + m] * col[m];
                    }
                    col[r] = r >= c ? acc : 0.0f;
                }
#pragma unroll
                for (int r = 0; r < 16; ++r) Tm[(o + r) * 64 + o + c] = col[r];
            }
            __syncthreads();
            float* W = sm.u2.W;
            for (int dist = 1; dist < 4; ++dist) {
                const int pairs = 4 - dist;
                // W_(bi,bj) = sum_{m=bj}^{bi-1} A_(bi,m) T_(m,bj)
                for (int e = tid; e < pairs * 256; e += kThreads) {
                    const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
                    const int bj = pr, bi = pr + dist;
                    float acc = 0.0f;
                    for (int m = 16 * bj; m < 16 * bi; ++m) acc += A[(16 * bi + r) * 64 + m] * Tm[m * 64 + 16 * bj + c];
                    W[e] = acc;
                }
                __syncthreads();
                // T_(bi,bj) = -T_(bi,bi) W
                for (int e = tid; e < pairs * 256; e += kThreads) {
                    const int pr = e >> 8, r = (e >> 4) & 15, c = e & 15;
                    const int bj = pr, bi = pr + dist;
                    float acc = 0.0f;
#pragma unroll
                    for (int m = 0; m < 16; ++m) acc += Tm[(16 * bi + r) * 64 + 16 * bi + m] * W[(pr << 8) + m * 16 + c];
                    Tm[(16 * bi + r) * 64 + 16 * bj + c] = -acc;
                }
                __syncthreads();
            }
            // T -> bt (MN-major B: element (n = column, k = row))
            for (int u = tid; u < 64 * 8; u += kThreads) {
                const int m = u >> 3, g = u & 7;
                store_split8(&sm.u2.bt[0][mnmaj(g * 8, m, 64)], &sm.u2.bt[1][mnmaj(g * 8, m, 64)], &Tm[m * 64 + g * 8]);
            }
        }
        GDN_PUBLISH();

        // ---- 6. (T ; P T) = [I; P] T ---------------------------------------------------------
        if (tid == 0) {
            mma_split(tmem + cPT, a_m[0], a_m[1], 1024, b_t[0], b_t[1], 1024, 4,
                      umma::idesc_bf16(128, 64, false, true));
            umma::commit(&sm.mbar);
        }
        GDN_MMA_WAIT();

        // ---- 7. [T; P T] -> am (split) -----------------------------------------------------------
#pragma unroll 1
        for (int c = 0; c < 64; c += 16) {
            float d[16];
            umma::tmem_ld16(tmem + lane_off + cPT + c, d);
            umma::tmem_wait_ld();
            store_split8(&sm.am[0][kmaj(tid, c, 64)], &sm.am[1][kmaj(tid, c, 64)], d);
            store_split8(&sm.am[0][kmaj(tid, c + 8, 64)], &sm.am[1][kmaj(tid, c + 8, 64)], d + 8);
        }
        GDN_PUBLISH();

        // ---- 8. (K S0 ; Q S0) = [K; Q] S0 ------------------------------------------------------
        if (tid == 0) {
            mma_split(tmem + cD2, a_kq[0], a_kq[1], 2048, b_s[0], b_s[1], 2048, 8,
                      umma::idesc_bf16(128, DVS, false, true));
            umma::commit(&sm.mbar);
        }
        GDN_MMA_WAIT();

        // ---- 9. X = beta (V - e^G K S0) -> bx;  keep e^G Q S0 / sqrt(dk) ----------------------
        float qs[DVS];
        {
            const int t = tid & 63;
#pragma unroll
            for (int c = 0; c < DVS; c += 16) {
                float d[16];
                umma::tmem_ld16(tmem + lane_off + cD2 + c, d);
                umma::tmem_wait_ld();
                if (tid < 64) {
                    const float bt = sm.beta[t], eg = sm.eG[t];
                    float x[16];
#pragma unroll
                    for (int e = 0; e < 16; ++e) x[e] = bt * (sm.v[t * DVS + c + e] - eg * d[e]);
                    store_split8(&sm.bx[0][mnmaj(c, t, 64)], &sm.bx[1][mnmaj(c, t, 64)], x);
                    store_split8(&sm.bx[0][mnmaj(c + 8, t, 64)], &sm.bx[1][mnmaj(c + 8, t, 64)], x + 8);
                } else {
                    const float f = sm.eG[t] * qscale;
#pragma unroll
                    for (int e = 0; e < 16; ++e) qs[c + e] = f * d[e];
                }
            }
        }
        GDN_PUBLISH();

        // ---- 10. (U ; P U) = [T; P T] X ------------------------------------------------------------
        if (tid == 0) {
            mma_split(tmem + cD3, a_m[0], a_m[1], 1024, b_x[0], b_x[1], 1024, 4,
                      umma::idesc_bf16(128, DVS, false, true));
            umma::commit(&sm.mbar);
        }
        GDN_MMA_WAIT();

        // ---- 11. U -> bx;  O = e^G Q S0 / sqrt(dk) + P U -> o ----------------------------------------
        {
            const int t = tid & 63;
#pragma unroll
            for (int c = 0; c < DVS; c += 16) {
                float d[16];
                umma::tmem_ld16(tmem + lane_off + cD3 + c, d);
                umma::tmem_wait_ld();
                if (tid < 64) {
                    store_split8(&sm.bx[0][mnmaj(c, t, 64)], &sm.bx[1][mnmaj(c, t, 64)], d);
                    store_split8(&sm.bx[0][mnmaj(c + 8, t, 64)], &sm.bx[1][mnmaj(c + 8, t, 64)], d + 8);
                } else if (t < n) {
                    float* dst = p.o + ((size_t)(c0 + t) * p.hv + h) * kHeadDim + v0 + c;
#pragma unroll
                    for (int e = 0; e < 16; e += 4)
                        *reinterpret_cast<float4*>(dst + e) =
                            make_float4(qs[c + e] + d[e], qs[c + e + 1] + d[e + 1], qs[c + e + 2] + d[e + 2],
                                        qs[c + e + 3] + d[e + 3]);
                }
            }
        }
        GDN_PUBLISH();

        // ---- 12. dS = Kd^T U ---------------------------------------------------------------------------
        if (tid == 0) {
            mma_split(tmem + cD4, a_kt[0], a_kt[1], 1024, b_x[0], b_x[1], 1024, 4,
                      umma::idesc_bf16(128, DVS, true, true));
            umma::commit(&sm.mbar);
        }
        GDN_MMA_WAIT();

        // ---- 13. S = e^{G_L} S + dS -> registers and bs -------------------------------------------------
        {
            const float gl = sm.gL;
#pragma unroll
            for (int c = 0; c < DVS; c += 16) {
                float d[16];
                umma::tmem_ld16(tmem + lane_off + cD4 + c, d);
                umma::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 16; ++e) S[c + e] = fmaf(gl, S[c + e], d[e]);
            }
#pragma unroll
            for (int c = 0; c < DVS; c += 8)
                store_split8(&sm.bs[0][mnmaj(c, tid, 128)], &sm.bs[1][mnmaj(c, tid, 128)], S + c);
        }
        GDN_PUBLISH();
    }

#pragma unroll
    for (int c = 0; c < DVS; c += 4)
        *reinterpret_cast<float4*>(p.S_out + sbase + (size_t)tid * kHeadDim + v0 + c) =
            make_float4(S[c], S[c + 1], S[c + 2], S[c + 3]);

done:
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(tmem, kTmemCols);
#undef GDN_MMA_WAIT
#undef GDN_PUBLISH
}

constexpr int kDVS = 32;

}  // namespace

size_t scan_workspace_bytes(int, int, int, int) { return 256; }  // error word

cudaError_t launch_scan(const ScanParams& p, cudaStream_t stream)
{
    if (p.n_seq == 0) return cudaSuccess;
    const size_t smem = sizeof(ScanSmem<kDVS>);
    cudaError_t e = cudaFuncSetAttribute(scan_tc_kernel<kDVS>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    e = cudaMemsetAsync(p.workspace, 0, 4, stream);
    if (e != cudaSuccess) return e;
    dim3 grid((unsigned)(p.hv * (kHeadDim / kDVS)), (unsigned)p.n_seq);
    scan_tc_kernel<kDVS><<<grid, kThreads, smem, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace gdn
