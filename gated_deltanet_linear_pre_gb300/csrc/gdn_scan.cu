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
//   [K; Q] K^T -> (K K^T ; Q K^T)          [A; P] diag(T1, T2) -> (A diag(T1, T2) ; P diag(T1, T2))
//   [K; Q] S0  -> (K S0 ; Q S0)            [T; P T] X -> (U ; P U)
// so (Q S0) and (P U) land in the same TMEM lanes and O needs no exchange.
//
// Three kernels:
//  * scan_gram_kernel, one CTA per (two chunks, key head), fully parallel: splits
//    [K; Q] into the tensor-core layout (the chain's [K; Q] image), forms
//    (K K^T ; Q K^T) in fp32, and M = [K; Q] K_prev^T against the previous
//    chunk's keys (the chain's look-ahead operand).  Inside gdn_layer the pre
//    kernel writes the images itself and scan_gram_img_kernel (one CTA per
//    (chunk, key head)) copies them in and forms the same products.
//  * scan_prep_kernel, persistent CTAs taking (chunk, value head) tasks in
//    order, beside the chain once it runs: A and P from the key head's gram
//    rows and the head's gates; the inverse T of I + A by halves (16x16
//    diagonal blocks by forward substitution and their 16x16 couplings on CUDA
//    cores, the 32x32 coupling and P T as two products on the tensor core);
//    writes the [T; P T] image and the chain's gate row.
//  * scan_chain_kernel, one CTA per (sequence, value head, 64-column slice):
//    the state-dependent part, chunk after chunk, with the fp32 state slice
//    in registers.  The next chunk's [K; Q] S is split into a part issued a
//    chunk early and a K = 64 correction through M, so the chunk-to-chunk path
//    is two MMA groups and two short CUDA-core phases; one warp issues the
//    MMAs, one the operand copies, sixteen do the CUDA-core work.
//
// Every MMA is issued by one thread and completes on an mbarrier; every wait
// is bounded and, on expiry, the CTA records an error code in the workspace,
// drains its own copies in flight (bounded), frees its TMEM and stops.

#include <cstddef>

#include "gdn_internal.cuh"
#include "umma.cuh"

namespace gdn {
namespace {

constexpr float kLamFloor = -110.0f;  // e^-110 is below the smallest fp32 denormal: g = 0 exactly
constexpr uint32_t kErrTimeout = 1u;
constexpr size_t kAmBytes = 128 * 64 * 2 * 2;     // [T; P T] image, bf16 hi + lo
constexpr size_t kKqBytes = 128 * 128 * 2 * 2;    // [K; Q] image, bf16 hi + lo
constexpr size_t kGramBytes = 128 * 64 * 4;       // (K K^T ; Q K^T), fp32 rows
constexpr size_t kMBytes = 128 * 64 * 2 * 2;      // [K; Q] of a chunk times K^T of the previous one, bf16 hi + lo
constexpr size_t kGateBytes = 1024;               // per-chunk gate row of a value head (784 bytes used)
constexpr size_t kAmBlock = kAmBytes + kGateBytes; // [T; P T] image followed by the gate row
constexpr size_t kWsHeader = 4096;                // error words
constexpr int kDVS = 64;                          // value columns per chain CTA

// [K; Q] image of a chunk: kq_off (the shared header); any run of row groups, e.g. one 64-row
// half, is one contiguous block
static_assert(kKqBytes == kKqImageBytes, "[K; Q] image size");

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

// 8 fp32 values -> bf16 (round to nearest even), the hi plane only (fast mode)
__device__ __forceinline__ void store_hi8(uint16_t* hi, const float* x)
{
    uint32_t h[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) h[q] = bf2_bits(__floats2bfloat162_rn(x[2 * q], x[2 * q + 1]));
    *reinterpret_cast<uint4*>(hi) = make_uint4(h[0], h[1], h[2], h[3]);
}

template <bool FAST>
__device__ __forceinline__ void store_op8(uint16_t* hi, uint16_t* lo, const float* x)
{
    if constexpr (FAST) store_hi8(hi, x);
    else store_split8(hi, lo, x);
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

// One-pass product D = A_hi * B_hi (fast mode: bf16 operands, fp32 accumulation)
__device__ __forceinline__ void mma_one(uint32_t d, uint32_t a_hi, uint32_t a_lbo, uint32_t a_sbo, uint32_t a_kstep,
                                        uint32_t b_hi, uint32_t b_sbo, uint32_t b_kstep, int ksteps, uint32_t idesc)
{
    const uint64_t dah = umma::desc(a_hi, a_lbo, a_sbo), dbh = umma::desc(b_hi, 128, b_sbo);
    const uint64_t sa = a_kstep >> 4, sb = b_kstep >> 4;
    for (int ks = 0; ks < ksteps; ++ks) umma::mma_bf16(d, dah + ks * sa, dbh + ks * sb, idesc, ks != 0);
}

// Split product in two instruction groups: D[:, 0:2N] = A_hi [B_hi | B_lo], then
// D[:, 0:N] += A_lo B_hi, so D[:, 0:N] + D[:, N:2N] = A B to ~16 bits.  Needs B_lo
// to follow B_hi directly along N in shared memory (b_hilo is the start of
// both).  Two thirds of the instructions of mma_split for the same tensor work.
// The K-step count and every stride are compile-time constants so that the
// issuing thread spends as few instructions as possible per MMA.
template <int KSTEPS, int N, uint32_t A_LBO, uint32_t A_SBO, uint32_t A_KSTEP, uint32_t B_SBO, uint32_t B_KSTEP,
          bool A_MN, bool B_MN, bool ACC = false, bool FAST = false>
__device__ __forceinline__ void mma_split2(uint32_t d, uint32_t a_hi, uint32_t a_lo, uint32_t b_hilo)
{
    const uint64_t dah = umma::desc(a_hi, A_LBO, A_SBO), dal = umma::desc(a_lo, A_LBO, A_SBO);
    const uint64_t db = umma::desc(b_hilo, 128, B_SBO);
    constexpr uint32_t wide = umma::idesc_bf16(128, 2 * N, A_MN, B_MN), narrow = umma::idesc_bf16(128, N, A_MN, B_MN);
    if constexpr (FAST) {  // one pass, A_hi * B_hi into D[:, 0:N]
#pragma unroll
        for (int ks = 0; ks < KSTEPS; ++ks)
            umma::mma_bf16(d, dah + ks * (A_KSTEP >> 4), db + ks * (B_KSTEP >> 4), narrow, (ACC || ks != 0) ? 1u : 0u);
        return;
    }
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks)
        umma::mma_bf16(d, dah + ks * (A_KSTEP >> 4), db + ks * (B_KSTEP >> 4), wide, (ACC || ks != 0) ? 1u : 0u);
#pragma unroll
    for (int ks = 0; ks < KSTEPS; ++ks)
        umma::mma_bf16(d, dal + ks * (A_KSTEP >> 4), db + ks * (B_KSTEP >> 4), narrow, 1u);
}

// Chunk slots: sequence s owns slots [base(s), base(s) + ceil(len_s / 64)) with
// base(s) = floor(cu[s] / 64) + s, which never overlap and need no prefix sum;
// floor(T / 64) + n_seq slots cover every batch.
__device__ __forceinline__ int slot_base(const ScanParams& p, int s) { return cu_at(p.cu_seqlens, s, p.T) / kChunk + s; }

__host__ __device__ inline size_t n_slots(int T, int n_seq) { return (size_t)(T / kChunk) + (size_t)n_seq; }

__device__ __forceinline__ unsigned char* am_image(const ScanParams& p, size_t slot, int h)
{
    return static_cast<unsigned char*>(p.workspace) + kWsHeader + (slot * p.hv + h) * kAmBlock;
}

__device__ __forceinline__ unsigned char* kq_image(const ScanParams& p, size_t slot, int j)
{
    return static_cast<unsigned char*>(p.workspace) + kWsHeader + n_slots(p.T, p.n_seq) * p.hv * kAmBlock +
           (slot * p.hk + j) * kKqBytes;
}

// (K K^T ; Q K^T) of a (chunk slot, key head): 128 rows x 64 fp32, stored by 4-column groups,
// the float4 of (row r, columns [4 g, 4 g + 4)) at index g * 128 + r, so that the gram kernels,
// which write a row per thread, and prep, which reads one the same way, both move 512 contiguous
// bytes per warp access
__device__ __forceinline__ int gram_f4(int r, int g) { return g * 128 + r; }

__device__ __forceinline__ float* gram_rows(const ScanParams& p, size_t slot, int j)
{
    return reinterpret_cast<float*>(static_cast<unsigned char*>(p.workspace) + kWsHeader +
                                    n_slots(p.T, p.n_seq) * ((size_t)p.hv * kAmBlock + (size_t)p.hk * kKqBytes) +
                                    (slot * p.hk + j) * kGramBytes);
}

__device__ __forceinline__ unsigned char* m_image(const ScanParams& p, size_t slot, int j)
{
    return static_cast<unsigned char*>(p.workspace) + kWsHeader +
           n_slots(p.T, p.n_seq) * ((size_t)p.hv * kAmBlock + (size_t)p.hk * (kKqBytes + kGramBytes)) +
           (slot * p.hk + j) * kMBytes;
}

// gates of one chunk of one value head as the chain consumes them: e^{G_t},
// beta_t, e^{G_L - G_t} and e^{G_L} (rows past the chunk's end: lam = beta = 0)
struct ChainGates {
    float eG[64], beta[64], kdec[64];
    float gL, pad[3];
};
static_assert(sizeof(ChainGates) % 16 == 0 && sizeof(ChainGates) <= kGateBytes, "gate row");

// per (chunk slot, value head): zeroed by gram, 1 once prep has written that chunk's [T; P T]
// image and gate row (and, through its wait on gram, everything before it is complete)
__device__ __forceinline__ unsigned long long* ready_flag(const ScanParams& p, size_t slot, int h)
{
    return reinterpret_cast<unsigned long long*>(
               static_cast<unsigned char*>(p.workspace) + kWsHeader +
               n_slots(p.T, p.n_seq) * ((size_t)p.hv * kAmBlock + (size_t)p.hk * (kKqBytes + kGramBytes + kMBytes))) +
           slot * p.hv + h;
}

// the ready flag that the failure-report self-test of the cross-kernel wait leaves unset: chunk slot 1,
// value head 0 (the chain's copy warp for that head then waits for it until its bound runs out)
__device__ __forceinline__ bool withheld(const ScanParams& p, int slot, int h)
{
    return p.withhold_flag && slot == 1 && h == 0;
}

__device__ __forceinline__ void flag_publish(unsigned long long* f, unsigned long long v)
{
    asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(f), "l"(v) : "memory");
}

__device__ __forceinline__ unsigned long long flag_read(const unsigned long long* f)
{
    unsigned long long v;
    asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(f) : "memory");
    return v;
}

// bounded wait (about two seconds of SM clock) for a ready flag; false on expiry
__device__ __forceinline__ bool flag_wait(const unsigned long long* f, unsigned long long v)
{
    const long long start = clock64();
    while (flag_read(f) != v) {
        if (clock64() - start > (4ll << 30)) return false;
        __nanosleep(128);
    }
    return true;
}

// prep's task counter, count of CTAs done with round one and count of CTAs that stay (header
// words 16, 17 and 18), cleared by gram
__device__ __forceinline__ unsigned int* prep_counter(const ScanParams& p)
{
    return reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(p.workspace) + 64);
}

// per SM id (header bytes 1024..2047): prep CTAs that have arrived on that SM, cleared by gram
constexpr int kSmSlots = 256;
__device__ __forceinline__ unsigned int* prep_sm_arrivals(const ScanParams& p)
{
    return reinterpret_cast<unsigned int*>(static_cast<unsigned char*>(p.workspace) + 1024);
}

// whether this CTA's SM keeps taking prep tasks after round one: the SMs in the first
// prep_keep / prep_sms of the SM-id range (ids may leave gaps up to %nsmid)
__device__ __forceinline__ bool prep_sm_stays(const ScanParams& p)
{
    uint32_t smid, nsmid;
    asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
    asm volatile("mov.u32 %0, %%nsmid;" : "=r"(nsmid));
    return (unsigned long long)smid * (unsigned)p.prep_sms < (unsigned long long)p.prep_keep * nsmid;
}

__device__ __forceinline__ ChainGates* gate_row(const ScanParams& p, size_t slot, int h)
{
    return reinterpret_cast<ChainGates*>(am_image(p, slot, h) + kAmBytes);
}

// slot -> (sequence, first token, token count); false for a slot no sequence uses
// (has_prev: the chunk has a predecessor in its sequence; odd: its index within the
// sequence is odd, which fixes the row order of its M and [T; P T] images)
__device__ __forceinline__ bool slot_chunk(const ScanParams& p, int slot, int& c0, int& n, bool* has_prev = nullptr,
                                           bool* odd = nullptr)
{
    int lo = 0, hi = p.n_seq - 1;
    while (lo < hi) {  // last s with base(s) <= slot
        const int mid = (lo + hi + 1) >> 1;
        if (slot_base(p, mid) <= slot) lo = mid; else hi = mid - 1;
    }
    const int start = cu_at(p.cu_seqlens, lo, p.T), end = max(cu_at(p.cu_seqlens, lo + 1, p.T), start);
    c0 = start + (slot - slot_base(p, lo)) * kChunk;
    n = min(kChunk, end - c0);
    if (has_prev) *has_prev = slot > slot_base(p, lo);
    if (odd) *odd = ((slot - slot_base(p, lo)) & 1) != 0;
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
// gram: one CTA per (pair of consecutive chunk slots, key head); per chunk: split
// [K; Q] (the chain's operand image), (K K^T ; Q K^T) in fp32 for the prep kernel,
// and, for every chunk but a sequence's first, M = [K; Q] K_prev^T against the
// previous chunk's keys (the chain's look-ahead operand).  The second chunk's
// loads overlap the first one's products, and its K_prev is the first one's K,
// still in shared memory.
// =======================================================================================
constexpr int kGramThreads = 256;
static_assert(kGramThreads == kSmSlots, "gram's first CTA clears one SM slot per thread");

struct __align__(1024) GramSmem {
    uint16_t akq[2][128 * 128];  // split [K; Q] (K-major); the image-input kernel: the [K; Q] image
    uint16_t bkp[2][64 * 128];   // split K of the previous chunk (K-major B, 64 rows); image input: its image half
    uint32_t tmem_base;
    int abort_flag;
    uint64_t mbar;
    uint64_t mb_load;  // image input: the bulk copies
};
// bulk-copy destinations and operand tiles on 16-byte boundaries
static_assert(offsetof(GramSmem, akq) % 16 == 0 && offsetof(GramSmem, bkp) % 16 == 0 &&
                  offsetof(GramSmem, mbar) % 8 == 0 && offsetof(GramSmem, mb_load) % 8 == 0,
              "gram shared-memory alignment");

// 64 token rows x 128 fp32 of one key head, 32 values per thread: unit u = tid + kThreads q
// covers row t (8 rows per group of 8 core-matrix rows) and columns [8 g, 8 g + 8)
template <int kThreads>
struct RowTile {
    static constexpr int kU = 64 * 16 / kThreads;
    float4 v[2 * kU];
    __device__ __forceinline__ static void unit(int u, int& t, int& g)
    {
        const int tg = (u >> 7) & 7;
        g = (u >> 3) & 15;
        t = tg * 8 + (u & 7);
    }
    // issue the loads (rows t >= n read as zero)
    __device__ __forceinline__ void fetch(const float* src_base, size_t row_stride, int n, int tid)
    {
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            int t, g;
            unit(tid + kThreads * q, t, g);
            if (t < n) {
                const float4* src = reinterpret_cast<const float4*>(src_base + (size_t)t * row_stride + g * 8);
                v[2 * q] = __ldg(src);
                v[2 * q + 1] = __ldg(src + 1);
            } else {
                v[2 * q] = v[2 * q + 1] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
    }
    // split into a K-major bf16 tile (rows row0 + t), optionally mirrored to rows img_row0 + t of a
    // [K; Q] image
    __device__ __forceinline__ void store(uint16_t* hi, uint16_t* lo, int row0, int tile_k, unsigned char* img,
                                          int img_row0, int tid) const
    {
#pragma unroll
        for (int q = 0; q < kU; ++q) {
            int t, g;
            unit(tid + kThreads * q, t, g);
            const float x[8] = {v[2 * q].x, v[2 * q].y, v[2 * q].z, v[2 * q].w,
                                v[2 * q + 1].x, v[2 * q + 1].y, v[2 * q + 1].z, v[2 * q + 1].w};
            uint4 vh, vl;
            split8(x, vh, vl);
            const int off = kmaj(row0 + t, g * 8, tile_k);
            *reinterpret_cast<uint4*>(hi + off) = vh;
            *reinterpret_cast<uint4*>(lo + off) = vl;
            if (img) {
                const int io = kq_off(img_row0 + t, g * 8);
                *reinterpret_cast<uint4*>(img + io) = vh;
                *reinterpret_cast<uint4*>(img + io + 2048) = vl;
            }
        }
    }
};

__global__ void __launch_bounds__(kGramThreads, 2) scan_gram_kernel(ScanParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    GramSmem& sm = *reinterpret_cast<GramSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int L = tid & 127, wg = tid >> 7;
    // two consecutive chunk slots of key head j; key head fastest, so the slots complete in order
    const int j = blockIdx.x, slot0 = 2 * (int)blockIdx.y;
    uint32_t* err = reinterpret_cast<uint32_t*>(p.workspace);
    // no early trigger: prep (and through it the chain) launches once gram has completed, so both
    // see the state this kernel leaves in the workspace header and the ready flags
    pdl_wait();
    // the failure record, prep's counters and its per-SM arrival counts start clean: the first CTA
    // clears them before anything could use them (the later kernels of the scan start only after
    // this one ends)
    if (slot0 == 0 && j == 0 && tid == 0) {
        *err = 0u;
        prep_counter(p)[0] = 0u;
        prep_counter(p)[1] = 0u;
        prep_counter(p)[2] = 0u;
    }
    if (slot0 == 0 && j == 0) prep_sm_arrivals(p)[tid] = 0u;  // kGramThreads == kSmSlots
    // this CTA's two slots' ready flags, for the value heads of key head j, start at zero.  Clearing
    // them here, rather than tagging flags with a per-call value, keeps whatever the workspace held
    // irrelevant and needs nothing from the host per call, so a scan replayed from a captured CUDA
    // graph is correct too
    {
        const int per = p.hv / p.hk;
        for (int i = tid; i < 2 * per; i += kGramThreads) {
            const int s = slot0 + i / per, h = j * per + i % per;
            if ((size_t)s < n_slots(p.T, p.n_seq)) *ready_flag(p, (size_t)s, h) = 0ull;
        }
    }
    int c0[2], n[2];
    bool has_prev[2], odd[2], used[2];
    used[0] = slot_chunk(p, slot0, c0[0], n[0], &has_prev[0], &odd[0]);
    used[1] = (size_t)(slot0 + 1) < n_slots(p.T, p.n_seq) &&
              slot_chunk(p, slot0 + 1, c0[1], n[1], &has_prev[1], &odd[1]);
    if (!used[0] && !used[1]) return;  // unused slots (whole CTA)

    if (warp == 0) umma::tmem_alloc(&sm.tmem_base, 128);
    if (tid == 0) {
        umma::mbar_init(&sm.mbar, 1);
        sm.abort_flag = 0;
    }
    const size_t rs = (size_t)p.hk * kHeadDim;
    const float* kbase = p.kn + (size_t)j * kHeadDim;
    const float* qbase = p.qn + (size_t)j * kHeadDim;
    RowTile<kGramThreads> tk, tq;
    {   // K and Q loads of the first used slot in flight together
        const int f = used[0] ? 0 : 1;
        tk.fetch(kbase + (size_t)(f ? c0[1] : c0[0]) * rs, rs, f ? n[1] : n[0], tid);
        tq.fetch(qbase + (size_t)(f ? c0[1] : c0[0]) * rs, rs, f ? n[1] : n[0], tid);
    }
    uint32_t phase = 0;
#pragma unroll
    for (int t = 0; t < 2; ++t) {
        if (!used[t]) continue;
        const int slot = slot0 + t;
        unsigned char* img = kq_image(p, slot, j);
        // the second chunk's predecessor is the first one, whose split K is still in the tile
        const bool prev_here = t == 1 && used[0] && has_prev[1];
        if (prev_here) {
            const uint4* src0 = reinterpret_cast<const uint4*>(sm.akq[0]);
            const uint4* src1 = reinterpret_cast<const uint4*>(sm.akq[1]);
            uint4* dst0 = reinterpret_cast<uint4*>(sm.bkp[0]);
            uint4* dst1 = reinterpret_cast<uint4*>(sm.bkp[1]);
#pragma unroll
            for (int q = 0; q < (64 * 128 * 2) / (16 * kGramThreads); ++q) {
                dst0[tid + kGramThreads * q] = src0[tid + kGramThreads * q];
                dst1[tid + kGramThreads * q] = src1[tid + kGramThreads * q];
            }
            __syncthreads();
        }
        // image rows in the chunk's stacking order: [K; Q] for even chunks, [Q; K] for odd ones
        tk.store(sm.akq[0], sm.akq[1], 0, 128, img, odd[t] ? 64 : 0, tid);
        if (has_prev[t] && !prev_here) tk.fetch(kbase + (size_t)(c0[t] - kChunk) * rs, rs, kChunk, tid);
        tq.store(sm.akq[0], sm.akq[1], 64, 128, img, odd[t] ? 0 : 64, tid);
        if (has_prev[t] && !prev_here) tk.store(sm.bkp[0], sm.bkp[1], 0, 128, nullptr, 0, tid);
        umma::fence_proxy_async();
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
        const uint32_t tmem = sm.tmem_base;
        // (K K^T ; Q K^T) = [K; Q] K^T  (B = the K rows of the same tile);  M = [K; Q] K_prev^T
        if (tid == 0) {
            const uint32_t a_hi = umma::smem_u32(sm.akq[0]), a_lo = umma::smem_u32(sm.akq[1]);
            constexpr uint32_t id = umma::idesc_bf16(128, 64, false, false);
            if (p.fast) {
                mma_one(tmem, a_hi, 128, 2048, 256, a_hi, 2048, 256, 8, id);
                if (has_prev[t]) mma_one(tmem + 64, a_hi, 128, 2048, 256, umma::smem_u32(sm.bkp[0]), 2048, 256, 8, id);
            } else {
                mma_split(tmem, a_hi, a_lo, 128, 2048, 256, a_hi, a_lo, 2048, 256, 8, id);
                if (has_prev[t])
                    mma_split(tmem + 64, a_hi, a_lo, 128, 2048, 256, umma::smem_u32(sm.bkp[0]), umma::smem_u32(sm.bkp[1]),
                              2048, 256, 8, id);
            }
            umma::commit(&sm.mbar);
        }
        // the second chunk's K and Q loads fly while this chunk's products and epilogue run
        if (t == 0 && used[1]) {
            tk.fetch(kbase + (size_t)c0[1] * rs, rs, n[1], tid);
            tq.fetch(qbase + (size_t)c0[1] * rs, rs, n[1], tid);
        }
        if (!umma::mbar_wait(&sm.mbar, phase)) { sm.abort_flag = 1; atomicOr(err, kErrTimeout); }
        phase ^= 1u;
        __syncthreads();
        if (sm.abort_flag) break;
        umma::fence_after_sync();
        {
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            float d[32];
            umma::tmem_ld32(tmem + lane_off + 32 * wg, d);
            umma::tmem_wait_ld();
            float4* dst = reinterpret_cast<float4*>(gram_rows(p, slot, j));
            // only the groups prep reads: A and P are lower triangular, so row i's columns up to i
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (4 * (8 * wg + q) <= (L & 63))
                    dst[gram_f4(L, 8 * wg + q)] = make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
            if (has_prev[t]) {  // M rows -> split K-major image (K = 64 tokens of the previous chunk), Q rows first for odd chunks
                const int mrow = odd[t] ? (L ^ 64) : L;
                umma::tmem_ld32(tmem + lane_off + 64 + 32 * wg, d);
                umma::tmem_wait_ld();
                unsigned char* mimg = m_image(p, slot, j);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 vh, vl;
                    split8(d + 8 * q, vh, vl);
                    const int off = kmaj(mrow, 32 * wg + 8 * q, 64);
                    *reinterpret_cast<uint4*>(mimg + off * 2) = vh;
                    *reinterpret_cast<uint4*>(mimg + kMBytes / 2 + off * 2) = vl;
                }
            }
        }
        // TMEM read out and the tiles consumed before the next chunk overwrites them
        umma::fence_before_sync();
        __syncthreads();
        umma::fence_after_sync();
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(sm.tmem_base, 128);
}

// gram with the [K; Q] images already written (by the pre kernel, inside gdn_layer): one CTA
// per (chunk slot, key head) bulk-copies the slot's image and the previous chunk's k half,
// zeroes the rows past a ragged last chunk (in shared memory for its products and in the
// image for the chain) and forms the same products as scan_gram_kernel.  The image rows are in
// the chunk's stacking order, so the products' rows are too: (K K^T ; Q K^T) rows are swapped
// back for odd chunks, the M image keeps them.
constexpr uint32_t kHalfBytes = 64 * 128 * 2 * 2;  // one 64-row half of an image, hi + lo

__global__ void __launch_bounds__(kGramThreads, 2) scan_gram_img_kernel(ScanParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    GramSmem& sm = *reinterpret_cast<GramSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5;
    const int L = tid & 127, wg = tid >> 7;
    const int j = blockIdx.x, slot = (int)blockIdx.y;
    uint32_t* err = reinterpret_cast<uint32_t*>(p.workspace);
    // no early trigger (as scan_gram_kernel): prep and the chain start after this kernel completes
    pdl_wait();
    if (slot == 0 && j == 0 && tid == 0) {
        *err = 0u;
        prep_counter(p)[0] = 0u;
        prep_counter(p)[1] = 0u;
        prep_counter(p)[2] = 0u;
    }
    if (slot == 0 && j == 0) prep_sm_arrivals(p)[tid] = 0u;  // kGramThreads == kSmSlots
    {   // this slot's ready flags, for the value heads of key head j, start at zero
        const int per = p.hv / p.hk;
        for (int i = tid; i < per; i += kGramThreads) *ready_flag(p, (size_t)slot, j * per + i) = 0ull;
    }
    int c0, n;
    bool has_prev, odd;
    if (!slot_chunk(p, slot, c0, n, &has_prev, &odd)) return;  // a slot no sequence uses

    unsigned char* img_s = reinterpret_cast<unsigned char*>(sm.akq);
    unsigned char* kp_s = reinterpret_cast<unsigned char*>(sm.bkp);
    unsigned char* img = kq_image(p, (size_t)slot, j);
    if (warp == 0) umma::tmem_alloc(&sm.tmem_base, 128);
    if (tid == 0) {
        umma::mbar_init(&sm.mbar, 1);
        umma::mbar_init(&sm.mb_load, 1);
        sm.abort_flag = 0;
        // the previous chunk's k half: its first half if that chunk is even (k first), else its second
        umma::mbar_arrive_expect_tx(&sm.mb_load, (uint32_t)kKqBytes + (has_prev ? kHalfBytes : 0u));
        umma::bulk_g2s(img_s, img, (uint32_t)kKqBytes, &sm.mb_load);
        if (has_prev) umma::bulk_g2s(kp_s, kq_image(p, (size_t)slot - 1, j) + (odd ? 0u : kHalfBytes), kHalfBytes, &sm.mb_load);
    }
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (!umma::mbar_wait(&sm.mb_load, 0)) { sm.abort_flag = 1; atomicOr(err, kErrTimeout); }
    if (n < kChunk) {  // rows past the chunk's end (both halves): zero here and in the image
        for (int i = tid; i < 128 * 32; i += kGramThreads) {
            const int row = i >> 5, pc = i & 31;
            if ((row & 63) < n) continue;
            const int off = (row >> 3) * 4096 + (pc & 15) * 128 + (row & 7) * 16 + (pc >> 4) * 2048;
            *reinterpret_cast<uint4*>(img_s + off) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(img + off) = make_uint4(0u, 0u, 0u, 0u);
        }
    }
    umma::fence_proxy_async();
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    if (!sm.abort_flag) {
        const uint32_t tmem = sm.tmem_base;
        if (tid == 0) {
            const uint32_t a_hi = umma::smem_u32(img_s), b_hi = a_hi + (odd ? kHalfBytes : 0u), kp = umma::smem_u32(kp_s);
            constexpr uint32_t id = umma::idesc_bf16(128, 64, false, false);
            if (p.fast) {
                mma_one(tmem, a_hi, 128, 4096, 256, b_hi, 4096, 256, 8, id);
                if (has_prev) mma_one(tmem + 64, a_hi, 128, 4096, 256, kp, 4096, 256, 8, id);
            } else {
                mma_split(tmem, a_hi, a_hi + 2048, 128, 4096, 256, b_hi, b_hi + 2048, 4096, 256, 8, id);
                if (has_prev) mma_split(tmem + 64, a_hi, a_hi + 2048, 128, 4096, 256, kp, kp + 2048, 4096, 256, 8, id);
            }
            umma::commit(&sm.mbar);
        }
        if (!umma::mbar_wait(&sm.mbar, 0)) { sm.abort_flag = 1; atomicOr(err, kErrTimeout); }
        __syncthreads();
        umma::fence_after_sync();
        if (!sm.abort_flag) {
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            float d[32];
            umma::tmem_ld32(tmem + lane_off + 32 * wg, d);
            umma::tmem_wait_ld();
            // gram rows in (K K^T ; Q K^T) order: image row L of an odd chunk is row L ^ 64 there
            float4* dst = reinterpret_cast<float4*>(gram_rows(p, (size_t)slot, j));
            const int grow = odd ? (L ^ 64) : L;
            // only the groups prep reads: A and P are lower triangular, so row i's columns up to i
#pragma unroll
            for (int q = 0; q < 8; ++q)
                if (4 * (8 * wg + q) <= (L & 63))
                    dst[gram_f4(grow, 8 * wg + q)] = make_float4(d[4 * q], d[4 * q + 1], d[4 * q + 2], d[4 * q + 3]);
            if (has_prev) {  // M rows, already in stacking order -> split K-major image (K = 64 previous tokens)
                umma::tmem_ld32(tmem + lane_off + 64 + 32 * wg, d);
                umma::tmem_wait_ld();
                unsigned char* mimg = m_image(p, (size_t)slot, j);
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    uint4 vh, vl;
                    split8(d + 8 * q, vh, vl);
                    const int off = kmaj(L, 32 * wg + 8 * q, 64);
                    *reinterpret_cast<uint4*>(mimg + off * 2) = vh;
                    *reinterpret_cast<uint4*>(mimg + kMBytes / 2 + off * 2) = vl;
                }
            }
        }
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(sm.tmem_base, 128);
}

// =======================================================================================
// prep: persistent CTAs, one (chunk slot, value head) task at a time
// =======================================================================================
constexpr int kPrepThreads = 256;  // two warpgroups: each covers all 128 TMEM lanes, half the columns
// round-one CTAs per SM the chain takes (of the four resident): the fewer, the sooner those SMs
// are free, but the smaller the lead the staying CTAs start with over a chain that consumes
// tasks faster than they produce them (T=2048, split products: scan 134.4 us with none, 130.7
// with 1, 134.2 with 2, and 141.7 with 4 before the solve's coupling went to the tensor core, and
// 130.3 us with 1 against 133.2 with 2 since; one-pass products, whose chain consumes faster,
// layer 162.0 us with 2, 159.9 with 3, 162.4 with 4)
constexpr int kRound1PerSm = 1;
// chunk slots above which prep defers each task's ready flag into its next task (T=32768: layer
// 2459-2489 -> 2400-2454 us, the 8-sequence varlen batch 1213 -> 1200 us; one T=2048 prompt, 33
// slots, would lose 1.4 us)
constexpr int kDeferFlagsAbove = 64;
constexpr int kRound1PerSmFast = 3;

constexpr int kTS = 36;  // fp32 row stride of the 32x32 blocks of A and T (16-byte rows, no bank conflicts)

struct __align__(1024) PrepSmem {
    uint16_t ap[2][128 * 64];  // [A; P] split (K-major, 128 rows x 64; hi plane, lo plane); once its
                               // product is done, the operands of the correction product
    union {
        float A[2][32 * kTS];        // fp32 diagonal 32x32 blocks of A, for the substitution steps
        uint16_t tb[2][2][32 * 32];  // then T1 and T2 split, MN-major B tiles: [block][hi / lo]
    } u;
    float T[2][32 * kTS];      // fp32 T1, T2 (the inverses of A's diagonal 32x32 blocks plus I)
    float W[2 * 16 * 16];      // 16x16 block products of the substitution
    float G[64], beta[64];
    uint32_t tmem_base;
    int abort_flag;
    uint32_t next[2];  // the next task, broadcast from thread 0 (alternating slots)
    uint64_t mbar;
};
// operand tiles (tensor-core descriptors, 16-byte vector accesses) on 16-byte boundaries; four
// CTAs fit an SM
static_assert(offsetof(PrepSmem, ap) % 16 == 0 && offsetof(PrepSmem, u) % 16 == 0 && offsetof(PrepSmem, T) % 16 == 0 &&
                  offsetof(PrepSmem, W) % 16 == 0 && offsetof(PrepSmem, mbar) % 8 == 0,
              "prep shared-memory alignment");
static_assert(4 * (sizeof(PrepSmem) + 1024) <= 232448, "four prep CTAs per SM");

__global__ void __launch_bounds__(kPrepThreads, 4) scan_prep_kernel(ScanParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    PrepSmem& sm = *reinterpret_cast<PrepSmem*>(smem_raw);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int L = tid & 127, wg = tid >> 7;  // TMEM lane, column half
    uint32_t* err = reinterpret_cast<uint32_t*>(p.workspace);
    pdl_launch_dependents();
    pdl_wait();
    const float qscale = rsqrtf((float)kHeadDim);

    if (warp == 0) umma::tmem_alloc(&sm.tmem_base, 128);  // [A; P] Tb in columns 0-63, the correction in 64-95
    if (tid == 0) {
        umma::mbar_init(&sm.mbar, 1);
        sm.abort_flag = 0;
    }
    uint32_t phase = 0;
    // Tasks (chunk slot, value head) in slot order, the value head fastest, so the chunk slots
    // complete in order across all heads; every task index comes, in order, from the counter that
    // gram cleared.  The CTAs on the SMs chosen to stay take tasks until none is left.  On the
    // other SMs, which the chain's CTAs take as soon as they are free, only the first
    // kRound1PerSm CTAs (kRound1PerSmFast with one-pass products) to arrive take one task (round
    // one) and the rest leave at once, so that those SMs free up sooner while round one still puts
    // the stayers ahead of the chain.
    const unsigned n_tasks = (unsigned)(n_slots(p.T, p.n_seq) * (size_t)p.hv);
    bool stays = prep_sm_stays(p);
    unsigned int* counter = prep_counter(p);
    // no CTA stays: the last CTA to finish round one (or to skip it) stays whatever its SM, so the
    // remaining tasks always have a taker
    auto round_one_done = [&]() {
        if (atomicAdd(counter + 1, 1u) + 1u == gridDim.x) {
            __threadfence();
            if (atomicAdd(counter + 2, 0u) == 0u) stays = true;
        }
    };
    bool first = false;  // thread 0: this CTA's round-one task is yet to be counted
    // With many chunk slots prep is the scan's bottleneck: a task's ready flag is then published early in
    // the CTA's next task, where the fence before it (waiting for the image writes) runs under that
    // task's loads.  With few (one T=2048 prompt: 33) the chain is the bottleneck and consumes each
    // flag soon after it is set, so it is published at once.
    const bool defer_flags = n_slots(p.T, p.n_seq) > (size_t)kDeferFlagsAbove;
    int pend_slot = -1, pend_h = 0;  // the ready flag waiting to be published (deferred mode)
    if (tid == 0) {
        unsigned t = n_tasks;
        if (stays) {  // CTAs that stay register before their round one
            atomicAdd(counter + 2, 1u);
            __threadfence();
            t = atomicAdd(counter, 1u);
            first = true;
        } else {
            uint32_t smid;
            asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
            if (atomicAdd(prep_sm_arrivals(p) + (smid % kSmSlots), 1u) < (unsigned)(p.fast ? kRound1PerSmFast : kRound1PerSm)) {
                t = atomicAdd(counter, 1u);
                first = true;
            } else {  // skips round one, counted now
                round_one_done();
                if (stays) t = atomicAdd(counter, 1u);
            }
        }
        sm.next[1] = t;
    }
    __syncthreads();
    int nx = 0;
    for (unsigned task = sm.next[1]; task < n_tasks;) {
        const int h = (int)(task % (unsigned)p.hv), slot = (int)(task / (unsigned)p.hv), j = h / (p.hv / p.hk);
        int c0, n;
        bool odd;
        if (slot_chunk(p, slot, c0, n, nullptr, &odd)) {
            // gates of value head h (warp 0): running log-decay G and beta, for this CTA and the chain's
            // copy; computed while the other warps' gram-row loads are in flight, so one barrier serves both
            if (warp == 0) {
                float lam[2], bt[2];
#pragma unroll
                for (int q = 0; q < 2; ++q) {
                    const int t = lane + 32 * q;
                    lam[q] = t < n ? fmaxf(__ldg(p.glog + (size_t)(c0 + t) * p.hv + h), kLamFloor) : 0.0f;
                    bt[q] = t < n ? __ldg(p.beta + (size_t)(c0 + t) * p.hv + h) : 0.0f;
                }
                const float GL = warp_chunk_cumsum(lam, lane);
                sm.G[lane] = lam[0];
                sm.G[lane + 32] = lam[1];
                sm.beta[lane] = bt[0];
                sm.beta[lane + 32] = bt[1];
                ChainGates* gr = gate_row(p, slot, h);
                gr->eG[lane] = __expf(lam[0]);
                gr->eG[lane + 32] = __expf(lam[1]);
                gr->kdec[lane] = __expf(GL - lam[0]);
                gr->kdec[lane + 32] = __expf(GL - lam[1]);
                gr->beta[lane] = bt[0];
                gr->beta[lane + 32] = bt[1];
                if (lane == 0) gr->gL = __expf(GL);
            }
            // this thread's 32 entries of the gram rows of the key head: row L (K K^T for
            // L < 64, Q K^T for L >= 64), columns [32 wg, 32 wg + 32); gram writes only the groups
            // that reach the diagonal or below (the rest enter A and P as zeros)
            float d[32];
            {
                const float4* src = reinterpret_cast<const float4*>(gram_rows(p, slot, j));
#pragma unroll
                for (int q = 0; q < 8; ++q) {
                    const float4 x = 4 * (8 * wg + q) <= (L & 63) ? __ldg(src + gram_f4(L, 8 * wg + q))
                                                                   : make_float4(0.f, 0.f, 0.f, 0.f);
                    d[4 * q] = x.x; d[4 * q + 1] = x.y; d[4 * q + 2] = x.z; d[4 * q + 3] = x.w;
                }
            }
            // the previous task's flag: its fence (which waits for that task's image writes) runs under
            // this task's loads, in a warp that only loads here
            if (tid == kPrepThreads - 32 && pend_slot >= 0) {
                __threadfence();
                if (!withheld(p, pend_slot, pend_h)) flag_publish(ready_flag(p, (size_t)pend_slot, pend_h), 1ull);
            }
            pend_slot = -1;
            __syncthreads();
            umma::fence_after_sync();
            const uint32_t tmem = sm.tmem_base;
            const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
            constexpr uint32_t kIdN32 = umma::idesc_bf16(128, 32, false, true);  // M = 128, N = 32, B MN-major

            {
                // A (rows i = L < 64) and P (rows i = L - 64), columns [cb, cb + 32): A's diagonal 32x32
                // blocks in fp32 for the substitution steps, its lower-left block A21 and P split into the
                // [A; P] tile (the tensor core's A operand; of its rows 0-63 only A21 reaches a product
                // that is read, so the other blocks are not written).  P is zero above its diagonal.
                {
                    const int i = L & 63, cb = 32 * wg;
                    const bool is_a = L < 64;
                    const bool diag_blk = is_a && (i >> 5) == wg;
                    const bool to_tile = is_a ? (wg == 0 && i >= 32) : true;
                    const float Gi = sm.G[i];
                    const float4* G4 = reinterpret_cast<const float4*>(sm.G + cb);
                    const int row = is_a ? i : 64 + i;
                    if (!is_a && cb > i) {
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            *reinterpret_cast<uint4*>(&sm.ap[0][kmaj(row, cb + 8 * q, 64)]) = make_uint4(0u, 0u, 0u, 0u);
                            *reinterpret_cast<uint4*>(&sm.ap[1][kmaj(row, cb + 8 * q, 64)]) = make_uint4(0u, 0u, 0u, 0u);
                        }
                    } else if (diag_blk || to_tile) {
                        // A: beta_i e^{G_i - G_j} (k_i . k_j) for j < i;  P: e^{G_i - G_j} (q_i . k_j) / sqrt(dk) for j <= i
                        const float f = is_a ? sm.beta[i] : qscale;
                        float* a32 = sm.u.A[wg] + (i & 31) * kTS;
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            const float4 ga = G4[2 * q], gb = G4[2 * q + 1];
                            const float gg[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
                            float x[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) {
                                const int jj = cb + 8 * q + e;
                                x[e] = (is_a ? jj < i : jj <= i) ? f * __expf(Gi - gg[e]) * d[8 * q + e] : 0.0f;
                            }
                            if (to_tile)
                                store_split8(&sm.ap[0][kmaj(row, cb + 8 * q, 64)], &sm.ap[1][kmaj(row, cb + 8 * q, 64)], x);
                            else {
                                *reinterpret_cast<float4*>(a32 + 8 * q) = make_float4(x[0], x[1], x[2], x[3]);
                                *reinterpret_cast<float4*>(a32 + 8 * q + 4) = make_float4(x[4], x[5], x[6], x[7]);
                            }
                        }
                    }
                }
                // the writers of A's diagonal blocks (warps 0 and 5) meet the substitution warps (0, 1)
                if (L < 64) asm volatile("bar.sync 1, 128;" ::: "memory");

                // T = (I + A)^-1 (A strictly lower), by halves: with T1, T2 the inverses of the diagonal
                // 32-blocks, T = [[T1, 0], [T21, T2]], T21 = -T2 A21 T1.
                // (1) the four 16x16 diagonal blocks by forward substitution (thread (b, c): column c;
                //     col[r] = [r == c] - sum_{m<r} A[r][m] col[m], the entries above c come out zero);
                // (2) T1 and T2: their lower-left 16x16 blocks, -T_(b,b) A_(b,b-1) T_(b-1,b-1) (CUDA cores);
                // (3) on the tensor core, with Tb = diag(T1, T2) and [T; P T] = [Tb; P Tb] [[I, 0], [-W, I]],
                //     W = A21 T1: one product [A; P] Tb gives W (rows 32-63, columns 0-31 of A Tb) and
                //     P Tb, a second C = [Tb; P Tb][:, 32:64] W gives the correction of columns 0-31:
                //     T21 = -C (rows 32-63), (P T)[:, 0:32] = (P Tb)[:, 0:32] - C (rows 64-127).
                // Only the block lower triangle of T1 and T2 is written; readers treat the rest as zero.
                {
                    if (tid < 64) {
                        const int b = tid >> 4, c = tid & 15, blk = b >> 1, o = 16 * (b & 1);
                        const float* Ab = sm.u.A[blk];
                        float col[16];
#pragma unroll
                        for (int r = 0; r < 16; ++r) {
                            float acc = (r == c) ? 1.0f : 0.0f;
#pragma unroll
                            for (int m4 = 0; m4 < r; m4 += 4) {
                                const float4 a4 = *reinterpret_cast<const float4*>(&Ab[(o + r) * kTS + o + m4]);
                                if (m4 + 0 < r) acc = fmaf(-a4.x, col[m4 + 0], acc);
                                if (m4 + 1 < r) acc = fmaf(-a4.y, col[m4 + 1], acc);
                                if (m4 + 2 < r) acc = fmaf(-a4.z, col[m4 + 2], acc);
                                if (m4 + 3 < r) acc = fmaf(-a4.w, col[m4 + 3], acc);
                            }
                            col[r] = acc;
                        }
#pragma unroll
                        for (int r = 0; r < 16; ++r) sm.T[blk][(o + r) * kTS + o + c] = col[r];
                    }
                    __syncthreads();
                    {   // (2) the lower-left 16x16 block of T1 (pr = 0) and of T2 (pr = 1)
                        const int pr = tid >> 7, r = (tid >> 3) & 15, c2 = 2 * (tid & 7);
                        const float* Ab = sm.u.A[pr];
                        float* Tb = sm.T[pr];
                        float w0 = 0.f, w1 = 0.f;
#pragma unroll
                        for (int m = 0; m < 16; ++m) {
                            const float a = Ab[(16 + r) * kTS + m];
                            const float2 t2 = *reinterpret_cast<const float2*>(&Tb[m * kTS + c2]);
                            w0 = fmaf(a, t2.x, w0);
                            w1 = fmaf(a, t2.y, w1);
                        }
                        *reinterpret_cast<float2*>(&sm.W[pr * 256 + r * 16 + c2]) = make_float2(w0, w1);
                        __syncthreads();
                        float t0 = 0.f, t1 = 0.f;
#pragma unroll
                        for (int m = 0; m < 16; ++m) {
                            const float a = Tb[(16 + r) * kTS + 16 + m];
                            const float2 w2 = *reinterpret_cast<const float2*>(&sm.W[pr * 256 + m * 16 + c2]);
                            t0 = fmaf(a, w2.x, t0);
                            t1 = fmaf(a, w2.y, t1);
                        }
                        *reinterpret_cast<float2*>(&Tb[(16 + r) * kTS + c2]) = make_float2(-t0, -t1);
                    }
                    __syncthreads();
                    {   // T1, T2 -> split MN-major B tiles (element (n = column, k = row)), over A's fp32 blocks;
                        // the upper-right 16x16 block of each is zero
                        const int blk = tid >> 7, m = (tid >> 2) & 31, g = tid & 3;
                        float tr[8];
                        if (m < 16 && g >= 2) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) tr[e] = 0.0f;
                        } else {
                            const float4 x0 = *reinterpret_cast<const float4*>(&sm.T[blk][m * kTS + 8 * g]);
                            const float4 x1 = *reinterpret_cast<const float4*>(&sm.T[blk][m * kTS + 8 * g + 4]);
                            tr[0] = x0.x; tr[1] = x0.y; tr[2] = x0.z; tr[3] = x0.w;
                            tr[4] = x1.x; tr[5] = x1.y; tr[6] = x1.z; tr[7] = x1.w;
                        }
                        store_split8(&sm.u.tb[blk][0][mnmaj(8 * g, m, 32)], &sm.u.tb[blk][1][mnmaj(8 * g, m, 32)], tr);
                    }
                }
                umma::fence_proxy_async();
                umma::fence_before_sync();
                __syncthreads();
                umma::fence_after_sync();

                // [A; P] Tb: columns 0-31 (K = 32: [A; P][:, 0:32] T1) into TMEM columns 0-31, columns 32-63
                // ([A; P][:, 32:64] T2) into 32-63.  [A; P] is K-major (K = 64: core matrices 128 B apart
                // along K, 1 KB along M); the T tiles MN-major (K = 32: 128 B along K, 512 B along N).
                if (tid == 0) {
                    const uint32_t a0 = umma::smem_u32(sm.ap[0]), a1 = umma::smem_u32(sm.ap[1]);
                    const uint32_t t1h = umma::smem_u32(sm.u.tb[0][0]), t1l = umma::smem_u32(sm.u.tb[0][1]);
                    const uint32_t t2h = umma::smem_u32(sm.u.tb[1][0]), t2l = umma::smem_u32(sm.u.tb[1][1]);
                    if (p.fast) {
                        mma_one(tmem, a0, 128, 1024, 256, t1h, 512, 256, 2, kIdN32);
                        mma_one(tmem + 32, a0 + 512, 128, 1024, 256, t2h, 512, 256, 2, kIdN32);
                    } else {
                        mma_split(tmem, a0, a1, 128, 1024, 256, t1h, t1l, 512, 256, 2, kIdN32);
                        mma_split(tmem + 32, a0 + 512, a1 + 512, 128, 1024, 256, t2h, t2l, 512, 256, 2, kIdN32);
                    }
                    umma::commit(&sm.mbar);
                }
                if (!umma::mbar_wait(&sm.mbar, phase)) { sm.abort_flag = 1; atomicOr(err, kErrTimeout); }
                phase ^= 1u;
                __syncthreads();
                if (sm.abort_flag) break;
                umma::fence_after_sync();

                // operands of the correction, over the consumed [A; P] tile: [Tb; P Tb][:, 32:64] (K-major,
                // 128 rows x K = 32: rows 0-31 zero, 32-63 T2, 64-127 P Tb from TMEM columns 32-63) and W
                // (MN-major B, 32 x 32, from TMEM lanes 32-63, columns 0-31)
                uint16_t* c_hi = sm.ap[0];
                uint16_t* c_lo = sm.ap[0] + 128 * 32;
                uint16_t* w_hi = sm.ap[1];
                uint16_t* w_lo = sm.ap[1] + 32 * 32;
                if (wg == 0) {
                    if (L >= 32) {
                        float x[32];
                        umma::tmem_ld32(tmem + lane_off + (L >= 64 ? 32u : 0u), x);
                        umma::tmem_wait_ld();
#pragma unroll
                        for (int q = 0; q < 4; ++q) {
                            if (L >= 64)
                                store_split8(&c_hi[kmaj(L, 8 * q, 32)], &c_lo[kmaj(L, 8 * q, 32)], x + 8 * q);
                            else
                                store_split8(&w_hi[mnmaj(8 * q, L - 32, 32)], &w_lo[mnmaj(8 * q, L - 32, 32)], x + 8 * q);
                        }
                    }
                } else if (L < 64) {
                    const int m = L - 32;  // row of T2
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        float x[8];
                        if (L < 32 || (m < 16 && q >= 2)) {
#pragma unroll
                            for (int e = 0; e < 8; ++e) x[e] = 0.0f;
                        } else {
                            const float4 x0 = *reinterpret_cast<const float4*>(&sm.T[1][m * kTS + 8 * q]);
                            const float4 x1 = *reinterpret_cast<const float4*>(&sm.T[1][m * kTS + 8 * q + 4]);
                            x[0] = x0.x; x[1] = x0.y; x[2] = x0.z; x[3] = x0.w;
                            x[4] = x1.x; x[5] = x1.y; x[6] = x1.z; x[7] = x1.w;
                        }
                        store_split8(&c_hi[kmaj(L, 8 * q, 32)], &c_lo[kmaj(L, 8 * q, 32)], x);
                    }
                }
                umma::fence_proxy_async();
                umma::fence_before_sync();
                __syncthreads();
                umma::fence_after_sync();

                // C = [Tb; P Tb][:, 32:64] W into TMEM columns 64-95 (K = 32: 128 B along K, 512 B along M/N)
                if (tid == 0) {
                    const uint32_t ch = umma::smem_u32(c_hi), cl = umma::smem_u32(c_lo);
                    const uint32_t wh = umma::smem_u32(w_hi), wl = umma::smem_u32(w_lo);
                    if (p.fast) mma_one(tmem + 64, ch, 128, 512, 256, wh, 512, 256, 2, kIdN32);
                    else mma_split(tmem + 64, ch, cl, 128, 512, 256, wh, wl, 512, 256, 2, kIdN32);
                    umma::commit(&sm.mbar);
                }
                if (!umma::mbar_wait(&sm.mbar, phase)) { sm.abort_flag = 1; atomicOr(err, kErrTimeout); }
                phase ^= 1u;
                __syncthreads();
                if (sm.abort_flag) break;
                umma::fence_after_sync();

                // [T; P T] image (K-major, split; [P T; T] for odd chunks), columns [cb, cb + 32) of row L:
                // T rows L < 64 (T1 / T21 = -C for wg 0, zero / T2 for wg 1), P T rows L - 64 ((P Tb - C) for
                // wg 0, P Tb for wg 1)
                {
                    unsigned char* img = am_image(p, slot, h);
                    const int irow = L < 64 ? (odd ? 64 + L : L) : (odd ? L - 64 : L);
                    const bool from_tmem = L >= 32 && (wg == 0 || L >= 64);  // warp-uniform
                    const bool zero = wg == 1 && L < 32;
                    const float* src = sm.T[wg] + (L & 31) * kTS;  // T1 row (wg 0), T2 row (wg 1)
#pragma unroll
                    for (int hq = 0; hq < 2; ++hq) {  // 16 columns at a time
                        const int cl = 16 * hq;
                        float x[16];
                        if (from_tmem) {
                            if (wg == 0) {
                                umma::tmem_ld16(tmem + lane_off + 64 + cl, x);  // C
                                if (L >= 64) {
                                    float y[16];
                                    umma::tmem_ld16(tmem + lane_off + cl, y);  // P Tb, columns 0-31
                                    umma::tmem_wait_ld();
#pragma unroll
                                    for (int e = 0; e < 16; ++e) x[e] = y[e] - x[e];
                                } else {
                                    umma::tmem_wait_ld();
#pragma unroll
                                    for (int e = 0; e < 16; ++e) x[e] = -x[e];
                                }
                            } else {
                                umma::tmem_ld16(tmem + lane_off + 32 + cl, x);  // P Tb, columns 32-63
                                umma::tmem_wait_ld();
                            }
                        } else {
                            // rows 0-15 of a 32-block have their columns 16-31 in the zero block
                            const bool z = zero || (hq == 1 && (L & 31) < 16);
#pragma unroll
                            for (int e = 0; e < 16; e += 4) {
                                const float4 v = z ? make_float4(0.f, 0.f, 0.f, 0.f)
                                                   : *reinterpret_cast<const float4*>(src + cl + e);
                                x[e] = v.x; x[e + 1] = v.y; x[e + 2] = v.z; x[e + 3] = v.w;
                            }
                        }
#pragma unroll
                        for (int q = 0; q < 2; ++q) {
                            uint4 vh, vl;
                            split8(x + 8 * q, vh, vl);
                            const int off = kmaj(irow, 32 * wg + cl + 8 * q, 64);
                            *reinterpret_cast<uint4*>(img + off * 2) = vh;
                            *reinterpret_cast<uint4*>(img + kAmBytes / 2 + off * 2) = vl;
                        }
                    }
                }
                umma::fence_before_sync();
                __syncthreads();
                umma::fence_after_sync();
            }

            // everything this chunk's chain needs is written: publish it (release, GPU scope)
            if (defer_flags) {
                pend_slot = slot;
                pend_h = h;
            } else if (tid == 0) {
                __threadfence();
                if (!withheld(p, slot, h)) flag_publish(ready_flag(p, slot, h), 1ull);
            }
        }  // used slot
        // thread 0 fetches the next task (after round one, counted for the fallback above)
        if (tid == 0) {
            if (first) round_one_done();
            sm.next[nx] = stays ? atomicAdd(counter, 1u) : n_tasks;
        }
        first = false;
        __syncthreads();
        task = sm.next[nx];
        nx ^= 1;
    }

    if (tid == kPrepThreads - 32 && pend_slot >= 0) {  // the last task's flag
        __threadfence();
        if (!withheld(p, pend_slot, pend_h)) flag_publish(ready_flag(p, (size_t)pend_slot, pend_h), 1ull);
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(sm.tmem_base, 128);
}

// =======================================================================================
// chain: one CTA per (sequence, value head, kDVS-column slice)
//
// Look-ahead form of the next chunk's (K S ; Q S): with S_{c+1} = g_c S_c + K_c^T U'_c
// (U' = e^{G_L-G} U, g_c = e^{G_L} of chunk c),
//     [K; Q]_{c+1} S_{c+1} = [K; Q]_{c+1} (g_c S_c) + M_{c+1} U'_c,   M_{c+1} = [K; Q]_{c+1} K_c^T,
// so the first product is issued while chunk c is still being worked on and
// only M U' (K = 64) waits for U'_c; the state update K_c^T U'_c and the fp32
// state stay off the chunk-to-chunk path.
//
// Roles: warps 0-15 (compute; warpgroup w owns columns [16w, 16w+16) of the
// slice for all 128 TMEM lanes) run three short phases per chunk (X, state,
// U/O) and publish their operands on mbarriers; warp 16 issues every MMA;
// warp 17 issues every bulk copy (operand images and gate rows) as soon as its
// destination buffer is released, so a busy copy engine never delays an MMA.
//
// [K; Q] lives in three 64-row half slots R0 R1 R2: Q of every chunk in R1,
// K of even chunks in R0 and of odd chunks in R2, so K_c stays resident for
// its state update while both halves of chunk c+1 land.  Odd chunks thus
// stack [Q; K]; the gram and prep kernels write the [K; Q], M and [T; P T]
// images of every chunk with its two 64-row halves in that order, so each
// lands with one bulk copy (an SM's bulk copies retire at roughly one per
// 600 cycles whatever their size up to 64 KB, so a chunk takes three: [K; Q],
// M, and [T; P T] with the gate row behind it).  In chunk c the thread in TMEM
// lane L owns the K-side row L & 63 when (L >> 6) == (c & 1), else the Q-side row.
// =======================================================================================
constexpr int kChainWG = 4;                        // compute warpgroups
constexpr int kChainCompute = 128 * kChainWG;
constexpr int kMmaWarp = kChainCompute / 32;       // issues every MMA
constexpr int kCopyWarp = kMmaWarp + 1;             // issues every bulk copy
constexpr int kChainThreads = kChainCompute + 64;
constexpr uint32_t kSlotBytes = 64 * 128 * 2 * 2;  // one 64-row half of a [K; Q] image, hi + lo

template <int DVS>
struct __align__(1024) ChainSmem {
    unsigned char kh[3 * kSlotBytes];  // half slots R0 R1 R2 of the [K; Q] tiles, image layout
    uint16_t mm[2][128 * 64];      // M image of the chunk, rows in its stacking order
    uint16_t am[2][128 * 64];      // [T; P T] image, same order; the gate row lands right behind it
    ChainGates gb;
    uint16_t bs[2][128 * DVS];     // g_c S_c slice (MN-major B, dk x DVS), hi then lo
    uint16_t bx[2][64 * DVS];      // X (MN-major B, 64 x DVS); between uses the fp32 V / O staging tile
    uint16_t bu[2][64 * DVS];      // U' = e^{G_L-G} U
    uint32_t tmem_base;
    int abort_flag;
    uint64_t mb_kq, mb_m, mb_am;          // bulk copies
    uint64_t mb_f, mb_d3, mb_d4, mb_fin;  // MMA completions
    uint64_t mb_x, mb_s, mb_u;            // compute -> producer (all compute threads arrive)
    uint64_t mb_grp[2];                   // row groups of the compute threads (lanes 0-63 / 64-127)
};
// bulk-copy destinations, operand tiles and the fp32 staging tile (read as float4) on 16-byte
// boundaries; the struct fits the 227 KB a CTA may have
static_assert(offsetof(ChainSmem<64>, kh) % 16 == 0 && offsetof(ChainSmem<64>, mm) % 16 == 0 &&
                  offsetof(ChainSmem<64>, am) % 16 == 0 && offsetof(ChainSmem<64>, gb) % 16 == 0 &&
                  offsetof(ChainSmem<64>, bs) % 16 == 0 && offsetof(ChainSmem<64>, bx) % 16 == 0 &&
                  offsetof(ChainSmem<64>, bu) % 16 == 0 && offsetof(ChainSmem<64>, mb_kq) % 8 == 0,
              "chain shared-memory alignment");
static_assert(sizeof(ChainSmem<64>) <= 232448, "chain shared memory");

// fp32 64 x 64 staging tile over bx: row r, 16-byte column chunk k at chunk
// (k ^ (r & 15)) of the row, so that a warp's 32 rows hit distinct banks
__device__ __forceinline__ int stage_off(int r, int k) { return r * 64 + ((k ^ (r & 15)) << 2); }

template <int COLS>
__device__ __forceinline__ void tmem_ld_cols(uint32_t taddr, float (&d)[COLS])
{
    static_assert(COLS == 16 || COLS == 32, "column count");
    if constexpr (COLS == 16) umma::tmem_ld16(taddr, d);
    else umma::tmem_ld32(taddr, d);
}

// Wait for an mbarrier phase with the thread suspended between checks (no
// polling traffic), bounded by about two seconds of SM clock and abandoned
// once another thread of the CTA has aborted; the warp agrees on the outcome
// so that it stays converged.
__device__ __forceinline__ bool chain_wait(uint64_t* mbar, uint32_t parity, const volatile int* abort_flag)
{
    bool ok = umma::mbar_try_wait(mbar, parity);
    if (!ok) {
        const long long start = clock64();
        while (!(ok = umma::mbar_try_wait_suspend(mbar, parity, 20000u))) {
            if (*abort_flag || clock64() - start > (4ll << 30)) break;
        }
    }
    return __all_sync(0xffffffffu, ok);
}

template <int COLS>
__device__ __forceinline__ void zero_cols(float (&d)[COLS])
{
#pragma unroll
    for (int e = 0; e < COLS; ++e) d[e] = 0.0f;
}

template <int DVS, bool FAST>
__global__ void __launch_bounds__(kChainThreads, 1) scan_chain_kernel(ScanParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    ChainSmem<DVS>& sm = *reinterpret_cast<ChainSmem<DVS>*>(smem_raw);
    // no grid-wide wait on the prep kernel: the CTA waits for the ready flag of its first chunk
    // (which implies every earlier kernel of the call has completed) and the copy warp for each
    // later chunk's flag, so the recurrence starts while prep's last CTAs still run
    pdl_launch_dependents();
    constexpr int SLICES = kHeadDim / DVS;
    constexpr int COLS = DVS / kChainWG;  // columns per compute thread
    constexpr uint32_t kTmemCols = 512;
    // each product takes 2*DVS columns: [hi*hi + lo*hi | hi*lo]
    constexpr uint32_t cD2 = 0, cD3 = 2 * DVS, cD4 = 4 * DVS;
    static_assert(6 * DVS <= (int)kTmemCols, "TMEM columns");

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int h = blockIdx.x / SLICES, slice = blockIdx.x % SLICES, s = blockIdx.y;
    const int j = h / (p.hv / p.hk);
    const int v0 = slice * DVS;
    const int t0 = cu_at(p.cu_seqlens, s, p.T), t1 = max(cu_at(p.cu_seqlens, s + 1, p.T), t0);
    const int n_chunks = (t1 - t0 + kChunk - 1) / kChunk;
    const size_t base = (size_t)slot_base(p, s);
    const size_t sbase = ((size_t)s * p.hv + h) * kHeadDim * kHeadDim;
    uint32_t* err = reinterpret_cast<uint32_t*>(p.workspace);
    const volatile int* abort_flag = &sm.abort_flag;
    // copy warp's bulk copies per destination (bit 0: [K; Q], 1: M, 2: [T; P T] + gates):
    // `used` = issued at least once, `np` = parity bit the next issue will complete (drained on exit)
    uint32_t used = 0, np = 0;
    constexpr uint32_t kBitKq = 1u, kBitM = 2u, kBitAm = 4u;

    if (warp == 0) umma::tmem_alloc(&sm.tmem_base, kTmemCols);
    if (tid == 0) {
        umma::mbar_init(&sm.mb_kq, 1);
        umma::mbar_init(&sm.mb_m, 32);  // one completion arrival per copy-warp lane
        umma::mbar_init(&sm.mb_am, 1);
        umma::mbar_init(&sm.mb_f, 1);
        umma::mbar_init(&sm.mb_d3, 1);
        umma::mbar_init(&sm.mb_d4, 1);
        umma::mbar_init(&sm.mb_fin, 1);
        umma::mbar_init(&sm.mb_x, kChainCompute);
        umma::mbar_init(&sm.mb_s, kChainCompute);
        umma::mbar_init(&sm.mb_u, kChainCompute);
        umma::mbar_init(&sm.mb_grp[0], kChainCompute / 2);
        umma::mbar_init(&sm.mb_grp[1], kChainCompute / 2);
        sm.abort_flag = 0;
        if (n_chunks > 0 && !flag_wait(ready_flag(p, base, h), 1ull)) {
            sm.abort_flag = 1;
            atomicOr(err, kErrTimeout);
        }
    }
    if (n_chunks == 0) pdl_wait();  // no chunk, no flag: wait for the whole prep grid
    umma::fence_before_sync();
    __syncthreads();
    umma::fence_after_sync();
    const uint32_t tmem = sm.tmem_base;
    if (sm.abort_flag) goto done;

#define GDN_WAIT(mbar, parity)                                                 \
    do {                                                                       \
        if (!chain_wait((mbar), (parity), abort_flag)) {                       \
            if (lane == 0) {                                                   \
                sm.abort_flag = 1;                                             \
                atomicOr(err, kErrTimeout);                                    \
            }                                                                  \
            goto done;                                                         \
        }                                                                      \
    } while (0)

    if (warp == kCopyWarp) {
        // ================================ bulk copies ================================
        const bool leader = lane == 0;
        auto issue = [&](uint64_t* mb, void* dst, const void* src, uint32_t bytes, uint32_t bit) {
            if (leader) {
                umma::mbar_arrive_expect_tx(mb, bytes);
                umma::bulk_g2s(dst, src, bytes, mb);
            }
            used |= bit;
            np ^= bit;
        };
        // [K; Q] of chunk c into slots (R0, R1) (even c) or (R1, R2) (odd c)
        auto load_kq = [&](int c) {
            issue(&sm.mb_kq, sm.kh + (c & 1) * kSlotBytes, kq_image(p, base + c, j), (uint32_t)kKqBytes, kBitKq);
        };
        auto load_am = [&](int c) {  // [T; P T] and the gate row
            issue(&sm.mb_am, sm.am, am_image(p, base + c, h), (uint32_t)(kAmBytes + sizeof(ChainGates)), kBitAm);
        };

        // Each wait below precedes the copy that lets its barrier advance twice, so a
        // parity wait never sees a phase two ahead.
        if (n_chunks > 0) {
            if (!p.withhold_first_copy) load_kq(0);  // withheld only by the failure-report self-test
            load_am(0);
        }
        // [K; Q] and [T; P T] images of chunk c -> L2 two chunks ahead: their copies are issued only
        // as buffers free up, often too late to ride out DRAM latency
        auto prefetch_l2 = [&](int c) {
            if (leader && c < n_chunks) {
                umma::bulk_prefetch_l2(kq_image(p, base + c, j), (uint32_t)kKqBytes);
                umma::bulk_prefetch_l2(am_image(p, base + c, h), (uint32_t)(kAmBytes + sizeof(ChainGates)));
            }
        };
        prefetch_l2(1);
        for (int c = 0; c + 1 < n_chunks; ++c) {
            prefetch_l2(c + 2);
            {   // chunk c+1's operands are written (bounded wait for its ready flag)
                bool ok = true;
                if (leader) ok = flag_wait(ready_flag(p, base + c + 1, h), 1ull);
                if (!__shfl_sync(0xffffffffu, ok ? 1 : 0, 0)) {
                    if (leader) {
                        sm.abort_flag = 1;
                        atomicOr(err, kErrTimeout);
                    }
                    goto done;
                }
            }
            // R1 (Q_c) and M free once (K S ; Q S) of chunk c is complete; the slot of K_{c-1}
            // once that chunk's state update is done
            GDN_WAIT(&sm.mb_f, c & 1);
            if (c >= 1) GDN_WAIT(&sm.mb_d4, (c - 1) & 1);
            load_kq(c + 1);
            {   // M through the load/store path (16-byte asynchronous copies, the whole warp), which
                // keeps the bulk-copy engine free for the other two images
                const unsigned char* src = m_image(p, base + c + 1, j);
                const uint32_t dst = umma::smem_u32(sm.mm);
#pragma unroll 8
                for (int q = 0; q < (int)(kMBytes / 512); ++q)
                    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst + q * 512 + lane * 16),
                                 "l"(src + q * 512 + lane * 16)
                                 : "memory");
                asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(umma::smem_u32(&sm.mb_m))
                             : "memory");
                used |= kBitM;
                np ^= kBitM;
            }
            // [T; P T] of chunk c consumed (every compute thread read its gates at chunk start)
            GDN_WAIT(&sm.mb_d3, c & 1);
            load_am(c + 1);
        }
    } else if (warp == kMmaWarp) {
        // ================================ MMA issue ================================
        const bool leader = lane == 0;
        // [K; Q] tiles: K-major, row groups 4 KB apart with the lo plane 2 KB behind the hi one
        const uint32_t kh0 = umma::smem_u32(sm.kh);
        const uint32_t b_s = umma::smem_u32(sm.bs[0]), b_x = umma::smem_u32(sm.bx[0]), b_u = umma::smem_u32(sm.bu[0]);
        const uint32_t a_m_hi = umma::smem_u32(sm.mm[0]), a_m_lo = umma::smem_u32(sm.mm[1]);
        const uint32_t a_t_hi = umma::smem_u32(sm.am[0]), a_t_lo = umma::smem_u32(sm.am[1]);
        auto kslot = [](int c) { return (c & 1) ? 2u : 0u; };

        if (n_chunks > 0) {  // (K S0 ; Q S0) of chunk 0
            GDN_WAIT(&sm.mb_s, 0);
            GDN_WAIT(&sm.mb_kq, 0);
            umma::fence_after_sync();
            if (leader) {
                mma_split2<8, DVS, 128, 4096, 256, 2048, 256, false, true, false, FAST>(tmem + cD2, kh0, kh0 + 2048, b_s);
                umma::commit(&sm.mb_f);
            }
            __syncwarp();
        }
        for (int c = 0; c < n_chunks; ++c) {
            const bool more = c + 1 < n_chunks;
            // (U ; P U) = [T; P T] X
            GDN_WAIT(&sm.mb_x, c & 1);
            GDN_WAIT(&sm.mb_am, c & 1);
            umma::fence_after_sync();
            if (leader) {
                mma_split2<4, DVS, 128, 1024, 256, 1024, 256, false, true, false, FAST>(tmem + cD3, a_t_hi, a_t_lo, b_x);
                umma::commit(&sm.mb_d3);
            }
            __syncwarp();
            // [K; Q]_{c+1} (g_c S_c) once the compute threads have published g_c S_c
            if (more) {
                GDN_WAIT(&sm.mb_s, (c + 1) & 1);
                GDN_WAIT(&sm.mb_kq, (c + 1) & 1);
                umma::fence_after_sync();
                const uint32_t a = kh0 + ((c + 1) & 1) * kSlotBytes;  // stacked from R1 (odd) or R0 (even)
                if (leader)
                    mma_split2<8, DVS, 128, 4096, 256, 2048, 256, false, true, false, FAST>(tmem + cD2, a, a + 2048, b_s);
                __syncwarp();
            }
            // U'_c published: M_{c+1} U'_c on top (the chunk-to-chunk path), then K_c^T U'_c
            GDN_WAIT(&sm.mb_u, c & 1);
            if (more) GDN_WAIT(&sm.mb_m, c & 1);
            umma::fence_after_sync();
            if (leader) {
                if (more) {
                    mma_split2<4, DVS, 128, 1024, 256, 1024, 256, false, true, true, FAST>(tmem + cD2, a_m_hi, a_m_lo, b_u);
                    umma::commit(&sm.mb_f);
                }
                // K_c^T: MN-major view of the K half (token groups 4 KB apart, key groups 128 B)
                const uint32_t kb = kh0 + kslot(c) * kSlotBytes;
                mma_split2<4, DVS, 4096, 128, 8192, 1024, 256, true, true, false, FAST>(tmem + cD4, kb, kb + 2048, b_u);
                umma::commit(&sm.mb_d4);
            }
            __syncwarp();
        }
    } else {
        // ================================ compute ================================
        const int L = tid & 127;   // TMEM lane of this thread
        const int wg = tid >> 7;   // column group
        const int cb = wg * COLS;  // first column of this thread within the slice
        const int t = L & 63;      // chunk row this thread owns
        const int grp = L >> 6;    // row group: K side of even chunks (0) or of odd chunks (1)
        const int tig = t + 64 * wg;  // index within the row group, 0..255
        const uint32_t lane_off = (uint32_t)((warp & 3) * 32) << 16;
        const float qscale = rsqrtf((float)kHeadDim);
        float* stage = reinterpret_cast<float*>(sm.bx[0]);
        uint32_t gph = 0;  // parity of this row group's next mbarrier phase
        // all 256 threads of the row group have arrived (generic shared-memory writes published)
#define GDN_GROUP_SYNC()                                                       \
    do {                                                                       \
        umma::mbar_arrive(&sm.mb_grp[grp]);                                    \
        GDN_WAIT(&sm.mb_grp[grp], gph);                                        \
        gph ^= 1u;                                                             \
    } while (0)
        // 16-byte piece (row r, chunk k) of a chunk's V tile -> the same place of the staging
        // tile, asynchronously (rows past the chunk's end read as zero)
        auto fetch_v_piece = [&](int cc0, int nn, int r, int k) {
            const float* src = p.vc + ((size_t)(cc0 + min(r, nn - 1)) * p.hv + h) * kHeadDim + v0 + 4 * k;
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(umma::smem_u32(stage + stage_off(r, k))),
                         "l"(src), "r"(r < nn ? 16 : 0)
                         : "memory");
        };
        // completion of this thread's V pieces arrives on its row group's mbarrier
        auto v_arrive = [&]() {
            asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(umma::smem_u32(&sm.mb_grp[grp]))
                         : "memory");
        };

        // state slice: row L (key index), columns v0 + cb + [0, COLS)
        float S[COLS];
        {
            const float* src = p.S_in + sbase + (size_t)L * kHeadDim + v0 + cb;
#pragma unroll
            for (int e = 0; e < COLS; e += 4) {
                const float4 x = *reinterpret_cast<const float4*>(src + e);
                S[e] = x.x; S[e + 1] = x.y; S[e + 2] = x.z; S[e + 3] = x.w;
            }
        }
        if (n_chunks > 0) {
#pragma unroll
            for (int e = 0; e < COLS; e += 8)
                store_op8<FAST>(&sm.bs[0][mnmaj(cb + e, L, 128)], &sm.bs[1][mnmaj(cb + e, L, 128)], S + e);
            umma::fence_proxy_async();
            umma::mbar_arrive(&sm.mb_s);
            if (grp == 0) {  // V of chunk 0, by the row group that owns its K side
                const int nn = min(kChunk, t1 - t0);
#pragma unroll
                for (int q = 0; q < 4; ++q) fetch_v_piece(t0, nn, (tig + 256 * q) >> 4, (tig + 256 * q) & 15);
                v_arrive();
            }
        }
        float gl_prev = 1.0f;

        for (int c = 0; c < n_chunks; ++c) {
            const int c0 = t0 + c * kChunk, n = min(kChunk, t1 - c0);
            const bool kside = grp == (c & 1);

            // ---- X = beta (V - e^G K S) -> bx;  keep e^G Q S / sqrt(dk) ------------------------------
            GDN_WAIT(&sm.mb_am, c & 1);  // gate row of chunk c (with its [T; P T] image)
            // this thread's gates; the buffer is reloaded once every thread is past this phase
            const float g_eG = sm.gb.eG[t], g_beta = sm.gb.beta[t], g_kdec = sm.gb.kdec[t], gl = sm.gb.gL;
            GDN_WAIT(&sm.mb_f, c & 1);
            umma::fence_after_sync();
            float qs[COLS];
            {
                float d[COLS], d2[COLS];
                tmem_ld_cols<COLS>(tmem + lane_off + cD2 + cb, d);
                if constexpr (!FAST) tmem_ld_cols<COLS>(tmem + lane_off + cD2 + DVS + cb, d2); else zero_cols(d2);
                umma::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < COLS; ++e) d[e] += d2[e];
                if (kside) {
                    GDN_WAIT(&sm.mb_grp[grp], gph);  // V tile landed
                    gph ^= 1u;
                    const float bt = g_beta, eg = g_eG;
#pragma unroll
                    for (int e = 0; e < COLS; e += 4) {  // X in place of K S
                        const float4 v = *reinterpret_cast<const float4*>(stage + stage_off(t, (cb + e) >> 2));
                        d[e] = bt * (v.x - eg * d[e]);
                        d[e + 1] = bt * (v.y - eg * d[e + 1]);
                        d[e + 2] = bt * (v.z - eg * d[e + 2]);
                        d[e + 3] = bt * (v.w - eg * d[e + 3]);
                    }
                    GDN_GROUP_SYNC();  // every V read done before X overwrites the tile
#pragma unroll
                    for (int e = 0; e < COLS; e += 8)
                        store_op8<FAST>(&sm.bx[0][mnmaj(cb + e, t, 64)], &sm.bx[1][mnmaj(cb + e, t, 64)], d + e);
                    umma::fence_proxy_async();
                } else {
                    const float f = g_eG * qscale;
#pragma unroll
                    for (int e = 0; e < COLS; ++e) qs[e] = f * d[e];
                }
            }
            umma::fence_before_sync();
            umma::mbar_arrive(&sm.mb_x);
            // the next chunk's V rows -> L2 (one line per thread of half this row group), so that
            // its later fetch into the staging tile hits there
            if (!kside && c + 1 < n_chunks && tig < 128) {
                const int r = tig >> 1, cc0 = t0 + (c + 1) * kChunk;
                if (cc0 + r < t1)
                    asm volatile("prefetch.global.L2 [%0];" ::"l"(p.vc + ((size_t)(cc0 + r) * p.hv + h) * kHeadDim + v0 +
                                                                   32 * (tig & 1)));
            }

            // ---- S_c = g_{c-1} S_{c-1} + K_{c-1}^T U'_{c-1};  g_c S_c -> bs ----------------------------
            if (c > 0) {
                GDN_WAIT(&sm.mb_d4, (c - 1) & 1);
                umma::fence_after_sync();
                float d[COLS], d2[COLS];
                tmem_ld_cols<COLS>(tmem + lane_off + cD4 + cb, d);
                if constexpr (!FAST) tmem_ld_cols<COLS>(tmem + lane_off + cD4 + DVS + cb, d2); else zero_cols(d2);
                umma::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < COLS; ++e) S[e] = fmaf(gl_prev, S[e], d[e] + d2[e]);
            }
            if (c + 1 < n_chunks) {
#pragma unroll
                for (int e = 0; e < COLS; e += 8) {
                    float x[8];
#pragma unroll
                    for (int q = 0; q < 8; ++q) x[q] = gl * S[e + q];
                    store_op8<FAST>(&sm.bs[0][mnmaj(cb + e, L, 128)], &sm.bs[1][mnmaj(cb + e, L, 128)], x);
                }
                umma::fence_proxy_async();
                umma::fence_before_sync();
                umma::mbar_arrive(&sm.mb_s);
            }
            gl_prev = gl;

            // ---- U' = e^{G_L-G} U -> bu;  O = e^G Q S / sqrt(dk) + P U -> staging -> global -------------
            GDN_WAIT(&sm.mb_d3, c & 1);  // X consumed: the staging tile is free
            umma::fence_after_sync();
            {
                float d[COLS], d2[COLS];
                tmem_ld_cols<COLS>(tmem + lane_off + cD3 + cb, d);
                if constexpr (!FAST) tmem_ld_cols<COLS>(tmem + lane_off + cD3 + DVS + cb, d2); else zero_cols(d2);
                umma::tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < COLS; ++e) d[e] += d2[e];
                if (kside) {
                    const float kd = g_kdec;
#pragma unroll
                    for (int e = 0; e < COLS; e += 8) {
                        float x[8];
#pragma unroll
                        for (int q = 0; q < 8; ++q) x[q] = kd * d[e + q];
                        store_op8<FAST>(&sm.bu[0][mnmaj(cb + e, t, 64)], &sm.bu[1][mnmaj(cb + e, t, 64)], x);
                    }
                    umma::fence_proxy_async();
                } else {
#pragma unroll
                    for (int e = 0; e < COLS; e += 4)
                        *reinterpret_cast<float4*>(stage + stage_off(t, (cb + e) >> 2)) =
                            make_float4(qs[e] + d[e], qs[e + 1] + d[e + 1], qs[e + 2] + d[e + 2], qs[e + 3] + d[e + 3]);
                }
            }
            umma::fence_before_sync();
            umma::mbar_arrive(&sm.mb_u);
            if (!kside) {
                GDN_GROUP_SYNC();  // O tile staged
                // coalesced copy-out (16 threads per 256-byte row); each piece read out is at once
                // refilled with the next chunk's V piece for the same place, which this group (the
                // next chunk's K side) reads after its mbarrier completes
                const bool more = c + 1 < n_chunks;
                const int cn0 = c0 + kChunk, nn = more ? min(kChunk, t1 - cn0) : 0;
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    const int u = tig + 256 * q, r = u >> 4, k = u & 15;
                    const float4 ov = *reinterpret_cast<const float4*>(stage + stage_off(r, k));
                    // a chunk followed by another is full, so every piece is stored, and the refill
                    // is issued after that store has consumed the piece
                    if (r < n)
                        __stcs(reinterpret_cast<float4*>(p.o + ((size_t)(c0 + r) * p.hv + h) * kHeadDim + v0) + k, ov);
                    if (more) fetch_v_piece(cn0, nn, r, k);
                }
                if (more) v_arrive();
            }
        }
        if (n_chunks > 0) {  // the last chunk's state update
            GDN_WAIT(&sm.mb_d4, (n_chunks - 1) & 1);
            umma::fence_after_sync();
            float d[COLS], d2[COLS];
            tmem_ld_cols<COLS>(tmem + lane_off + cD4 + cb, d);
            if constexpr (!FAST) tmem_ld_cols<COLS>(tmem + lane_off + cD4 + DVS + cb, d2); else zero_cols(d2);
            umma::tmem_wait_ld();
#pragma unroll
            for (int e = 0; e < COLS; ++e) S[e] = fmaf(gl_prev, S[e], d[e] + d2[e]);
        }
        {
            float* dst = p.S_out + sbase + (size_t)L * kHeadDim + v0 + cb;
#pragma unroll
            for (int e = 0; e < COLS; e += 4)
                *reinterpret_cast<float4*>(dst + e) = make_float4(S[e], S[e + 1], S[e + 2], S[e + 3]);
        }
#undef GDN_GROUP_SYNC
    }

done:
    if (warp == kCopyWarp) {  // drain the copies into this CTA's shared memory (bounded)
        asm volatile("cp.async.wait_all;" ::: "memory");
        if (lane == 0) {
            auto drain = [&](uint64_t* mb, int r) {
                if ((used >> r) & 1u) umma::mbar_wait(mb, ((np >> r) & 1u) ^ 1u, 1u << 16);
            };
            drain(&sm.mb_kq, 0);
            drain(&sm.mb_m, 1);
            drain(&sm.mb_am, 2);
        }
        __syncwarp();
    } else if (warp == kMmaWarp) {  // every MMA issued has completed (bounded)
        if (lane == 0) {
            umma::commit(&sm.mb_fin);
            umma::mbar_wait(&sm.mb_fin, 0, 1u << 16);
        }
        __syncwarp();
    } else {
        asm volatile("cp.async.wait_all;" ::: "memory");  // no copy into this CTA's shared memory outlives it
    }
    umma::fence_before_sync();
    __syncthreads();
    if (warp == 0) umma::tmem_dealloc(sm.tmem_base, kTmemCols);
    // This grid completes only after prep's has: the next call's kernels wait on this grid alone,
    // and a prep CTA may still be taking its last (empty) ticket from the task counter that the next
    // call's gram clears.  By now prep has published every flag this CTA consumed, so the wait is
    // short (no measurable cost).
    pdl_wait();
#undef GDN_WAIT
}

}  // namespace

size_t scan_kq_images_offset(int hk, int hv, int n_seq, int T)
{
    (void)hk;
    return kWsHeader + n_slots(T, n_seq) * (size_t)hv * kAmBlock;
}

size_t scan_workspace_bytes(int hk, int hv, int n_seq, int T)
{
    return kWsHeader + n_slots(T, n_seq) * ((size_t)hv * (kAmBlock + 8) + (size_t)hk * (kKqBytes + kGramBytes + kMBytes));
}

int sm_count()
{
    static int cached[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cached[dev] == 0) {
        int v = 0;
        if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = v;
    }
    return cached[dev];
}

// prep grid: four CTAs per SM (its occupancy), at most one per task; sets which SMs stay after
// round one: those the chain's CTAs leave free (at least a quarter of the GPU); with more chain
// CTAs than SMs the chain runs in waves anyway and every SM stays
unsigned prep_grid(ScanParams& p, size_t slots)
{
    const long long sms = sm_count() > 0 ? sm_count() : 1;
    const long long tasks = (long long)slots * p.hv;
    const long long chain_ctas = (long long)p.hv * (kHeadDim / kDVS) * p.n_seq;
    long long keep = chain_ctas < sms ? sms - chain_ctas : sms;
    if (keep < (sms + 3) / 4) keep = (sms + 3) / 4;
    p.prep_sms = (int)sms;
    p.prep_keep = (int)keep;
    return (unsigned)(tasks < 4 * sms ? tasks : 4 * sms);
}

cudaError_t launch_scan(const ScanParams& p_in, cudaStream_t stream)
{
    ScanParams p = p_in;
    p.prep_sms = p.prep_keep = 0;
    if (p.n_seq == 0) return cudaSuccess;
    const size_t gram_smem = sizeof(GramSmem), prep_smem = sizeof(PrepSmem), chain_smem = sizeof(ChainSmem<kDVS>);
    cudaError_t e = cudaFuncSetAttribute(p.kq_written ? scan_gram_img_kernel : scan_gram_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)gram_smem);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(scan_prep_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)prep_smem);
    if (e != cudaSuccess) return e;
    auto chain = p.fast ? scan_chain_kernel<kDVS, true> : scan_chain_kernel<kDVS, false>;
    e = cudaFuncSetAttribute(chain, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)chain_smem);
    if (e != cudaSuccess) return e;
    const size_t slots = n_slots(p.T, p.n_seq);
    if (p.T == 0) {  // no gram launch to clear the failure record (rare: every sequence empty)
        e = cudaMemsetAsync(p.workspace, 0, 4, stream);
        if (e != cudaSuccess) return e;
    } else {
        // each kernel may start while its predecessor drains and waits for it before reading
        const unsigned prep_ctas = prep_grid(p, slots);
        if (p.prep_no_keepers) p.prep_keep = 0;  // self-test: the round-one fallback takes every later task
        e = p.kq_written ? launch_k(scan_gram_img_kernel, dim3((unsigned)p.hk, (unsigned)slots), dim3(kGramThreads),
                                    gram_smem, stream, true, p)
                         : launch_k(scan_gram_kernel, dim3((unsigned)p.hk, (unsigned)((slots + 1) / 2)),
                                    dim3(kGramThreads), gram_smem, stream, true, p);
        if (e != cudaSuccess) return e;
        e = launch_k(scan_prep_kernel, dim3(prep_ctas), dim3(kPrepThreads), prep_smem, stream, true, p);
        if (e != cudaSuccess) return e;
    }
    return launch_k(chain, dim3((unsigned)(p.hv * (kHeadDim / kDVS)), (unsigned)p.n_seq),
                    dim3(kChainThreads), chain_smem, stream, p.T > 0, p);
}

}  // namespace gdn
