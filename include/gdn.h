/*
 * gdn.h -- C ABI of the Gated DeltaNet (GDN) prompt-prefill library for one
 * NVIDIA GB300 GPU (sm_103a).
 *
 * The path has three stages, after the three kernels the pages benchmark
 * ("Round 30 Track C Audit: gdn_pre, gdn_post, and gdn_scanr_4", sections 1
 * and 2: gdn_pre, the gdn_scan_r recurrence and gdn_post, timed separately
 * and as one pre+scan+post total over 36 layers):
 *
 *   gdn_pre   width-4 causal depthwise conv over the packed q|k|v channels
 *             with a carried 3-token history, SiLU, L2 normalisation of every
 *             q and k head (eps), and the per-(token, value head) gates
 *             lam = log g = -exp(A_log) * softplus(a + dt_bias),
 *             beta = sigmoid(b).
 *   gdn_scan  the gated delta rule, per value head h with key head
 *             h / (hv/hk) and fp32 state S in R^{dk x dv}:
 *               S <- g S;  u = beta (v - S^T k);  S <- S + k u^T;
 *               o = S^T q / sqrt(dk).
 *   gdn_post  y = o / sqrt(mean(o^2) + eps) * gamma * SiLU(z), fp16 or fp32.
 *   gdn_layer the three stages back to back on one stream.
 *   gdn_step  one decode step (a single token per sequence) through all three.
 *
 * Conventions shared by every entry point
 * ----------------------------------------
 *  - Every array pointer is a DEVICE pointer (memory of the current CUDA
 *    device), owned by the caller, dense and row-major in the layout stated.
 *    The library allocates no device memory and keeps no pointer after the
 *    call returns; the work runs asynchronously on `stream` (NULL = legacy
 *    default stream), so buffers must stay valid until the stream reaches it.
 *  - fp16 arrays are IEEE binary16 bit patterns (uint16_t).
 *  - Shapes: hk key heads, hv value heads (hv a multiple of hk), dk = dv =
 *    128, C = 2*hk*dk + hv*dv packed channels ordered q (hk heads) | k (hk
 *    heads) | v (hv heads).  T = total tokens of a packed variable-length
 *    batch of n_seq sequences; sequence s owns tokens
 *    [cu_seqlens[s], cu_seqlens[s+1]).  cu_seqlens is a DEVICE int32 array of
 *    n_seq+1 entries, non-decreasing, cu_seqlens[0] = 0,
 *    cu_seqlens[n_seq] = T (not read on the host; a violation is undefined).
 *    Zero-length sequences are allowed: their history and state pass
 *    through unchanged.
 *  - Every pointer must be 16-byte aligned.
 *  - Errors: argument problems are detected on the host before anything is
 *    launched and return a status with nothing enqueued.  A failed launch
 *    returns GDN_ERR_CUDA (the CUDA error string is kept for
 *    gdn_last_error_string).  Asynchronous faults surface at the caller's
 *    next synchronisation, as with any CUDA library, and, without one, through
 *    gdn_last_async_error once any CUDA call of the process has observed them.
 *  - Thread safety: calls may be made from several host threads on
 *    different streams; they share no mutable state except the last-error
 *    string, which is per host thread.
 */
#ifndef GDN_H
#define GDN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st; /* cudaStream_t is `struct CUstream_st *` */

#if defined(__GNUC__)
#define GDN_API __attribute__((visibility("default")))
#else
#define GDN_API
#endif

typedef enum gdn_status {
    GDN_OK = 0,
    GDN_ERR_INVALID_ARG = 1, /* null pointer, negative size, overlap, bad value */
    GDN_ERR_UNSUPPORTED = 2, /* shape outside what the kernels implement       */
    GDN_ERR_ALIGNMENT = 3,   /* a pointer is not 16-byte aligned               */
    GDN_ERR_WORKSPACE = 4,   /* workspace missing or smaller than required     */
    GDN_ERR_CUDA = 5,        /* a CUDA runtime call or launch failed            */
    GDN_ERR_TIMEOUT = 6      /* a bounded wait inside a kernel expired: that
                                call's outputs are invalid (gdn_*_check)        */
} gdn_status;

/* Model shape.  Implemented: dk == dv == 128, 1 <= hk, hv % hk == 0,
 * hv <= 4096, eps > 0 (the pages' layer: hk=16, hv=48, eps=1e-6 -- "round 10
 * track b: gdn vectorization and scan", source and execution). */
typedef struct gdn_dims {
    int32_t hk;  /* key (and query) heads                              */
    int32_t hv;  /* value heads                                        */
    int32_t dk;  /* key head dimension (128)                           */
    int32_t dv;  /* value head dimension (128)                         */
    float eps;   /* epsilon of the L2 norms and of the RMSNorm         */
} gdn_dims;

/* Human-readable name of a status code (static storage). */
GDN_API const char* gdn_status_string(gdn_status s);

/* Detail of the last non-OK status returned on this host thread. */
GDN_API const char* gdn_last_error_string(void);

/*
 * gdn_last_async_error -- the sticky CUDA error: GDN_ERR_CUDA once the library
 * has seen an error that leaves the CUDA context unusable (a kernel that
 * faulted: illegal address or instruction, misaligned address, launch
 * failure or timeout, device assert, uncorrectable ECC), else GDN_OK.  The
 * error is seen either by one of the library's own calls (every later launch
 * or copy in a faulted context returns it) or, at this call, through the
 * CUDA runtime's last-error state.  Does not synchronise, enqueues nothing and
 * clears nothing: once set it stays set for the life of the process, as the
 * context's fault does.  The detail goes to gdn_last_error_string.
 */
GDN_API gdn_status gdn_last_async_error(void);

/*
 * gdn_pre -- stage 1 ("Round 30 Track C Audit", section 1, gdn_pre: the
 * 4-tap conv loop, the history write at the last token, the per-key-head
 * q/k sum-of-squares reductions; "round 10 track b", variants: each conv
 * output is four multiply-adds in tap order, history kept channel by
 * channel).
 *
 * In:  qkv      fp16 [T][C]             raw projections, q | k | v
 *      conv_w   fp32 [C][4]             taps; tap 3 multiplies the current
 *                                       token, tap 0 the token 3 back
 *      hist_in  fp16 [n_seq][C][3]      the 3 inputs before each sequence,
 *                                       oldest first
 *      a, b     fp16 [T][hv]            gate pre-activations
 *      A_log, dt_bias fp32 [hv]
 * Out: hist_out fp16 [n_seq][C][3]      last 3 inputs of each sequence
 *                                       (old history shifted in when the
 *                                       sequence is shorter than 3); bit
 *                                       copies, never rounded.  May be the
 *                                       same buffer as hist_in: the new
 *                                       history is then written by a second
 *                                       launch, after every read of the old
 *                                       one.  Any other overlap is rejected.
 *      qn, kn   fp32 [T][hk][dk]        SiLU(conv) / sqrt(|.|^2 + eps)
 *      vc       fp32 [T][hv][dv]        SiLU(conv) of the v channels
 *      glog     fp32 [T][hv]            lam = log g (<= 0)
 *      beta     fp32 [T][hv]            sigmoid(b)
 */
GDN_API gdn_status gdn_pre(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                   const int32_t* cu_seqlens, const uint16_t* qkv, const float* conv_w,
                   const uint16_t* hist_in, uint16_t* hist_out, const uint16_t* a,
                   const uint16_t* b, const float* A_log, const float* dt_bias, float* qn,
                   float* kn, float* vc, float* glog, float* beta, struct CUstream_st* stream);

/* Workspace bytes gdn_scan needs for this batch shape (0 is a valid answer). */
GDN_API size_t gdn_scan_workspace_bytes(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens);

/*
 * gdn_scan -- stage 2, the gated delta-rule recurrence ("Round 30 Track C
 * Audit", section 1: gdn_scan_r keeps the fp32 state on chip, decays and
 * updates it per token and forms the k and q products against it).
 * Computed chunk-wise (64 tokens), exact in exact arithmetic.
 *
 * In:  qn, kn   fp32 [T][hk][dk]        unit-norm q and k (as gdn_pre writes)
 *      vc       fp32 [T][hv][dv]
 *      glog     fp32 [T][hv]            log-decay, <= 0 (-inf allowed: g = 0)
 *      beta     fp32 [T][hv]
 *      S_in     fp32 [n_seq][hv][dk][dv]  state before each sequence
 * Out: S_out    fp32 [n_seq][hv][dk][dv]  state after each sequence; may be
 *                                       the same buffer as S_in
 *      o        fp32 [T][hv][dv]        S^T q / sqrt(dk) after each token
 * workspace: device scratch of at least gdn_scan_workspace_bytes() bytes
 *            (may be NULL when that is 0); contents on entry are ignored.
 * Stream capture: a call may be captured into a CUDA graph.  Nothing it
 * enqueues depends on host state that changes from call to call, so each
 * replay of the graph is a complete scan of what the captured buffers then
 * hold.  Calls sharing one workspace must not overlap on the GPU.
 */
GDN_API gdn_status gdn_scan(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                    const int32_t* cu_seqlens, const float* qn, const float* kn,
                    const float* vc, const float* glog, const float* beta, const float* S_in,
                    float* S_out, float* o, void* workspace, size_t workspace_bytes,
                    struct CUstream_st* stream);

/*
 * gdn_post -- stage 3, gated RMSNorm ("Round 30 Track C Audit", section 1,
 * gdn_post: per-head sum-of-squares reduction and the f32 output switch;
 * "opus_r25_gdn -- round 25 track A", shipped: the sigmoid gate and gamma).
 *
 * In:  o        fp32 [T][hv][dv]
 *      z        fp16 [T][hv][dv]
 *      gamma    fp32 [dv]               shared by all heads
 * Out: y        fp16 [T][hv][dv] when out_f32 == 0, else fp32 [T][hv][dv]
 */
GDN_API gdn_status gdn_post(const gdn_dims* dims, int32_t total_tokens, const float* o,
                    const uint16_t* z, const float* gamma, int32_t out_f32, void* y,
                    struct CUstream_st* stream);

/*
 * gdn_scan_noalloc -- gdn_scan for callers that cannot allocate device
 * memory.  The paper has no counterpart to this entry point.
 *
 * Some callers have no device allocator to hand to the library: a host
 * program that links this C ABI directly and has no workspace buffer to
 * give, or a service that forbids device allocations after start-up.  For
 * them this entry point runs the same scan with its scratch in a
 * fixed-size array that the library owns (GDN_SCAN_NOALLOC_MAX_BYTES, held
 * on every device that loads the library until the process exits).  The
 * caller still passes every input and output, exactly as for gdn_scan.
 *
 * - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 * - The first call on each device looks up that device's copy of the array
 *   (with the device current) and caches it; make that first call before
 *   any stream capture.
 * - Batches whose scan scratch (gdn_scan_workspace_bytes) exceeds
 *   GDN_SCAN_NOALLOC_MAX_BYTES are rejected with GDN_ERR_UNSUPPORTED and a
 *   message naming the limit; nothing is enqueued.
 * - All calls on a device share the one array and it keeps the last call's
 *   contents (the part that must start at zero is cleared by every call):
 *   calls whose work overlaps on the GPU -- different streams, or several
 *   host threads -- race on it.  Serialise them, e.g. on one stream.
 * - The array's device address is looked up again on every call made outside
 *   stream capture (so a device reset, after which the library's module is
 *   loaded afresh, is picked up); under capture the address from the last
 *   call outside capture is used.
 */
#define GDN_SCAN_NOALLOC_MAX_BYTES ((size_t)64 << 20)
GDN_API gdn_status gdn_scan_noalloc(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                                    const int32_t* cu_seqlens, const float* qn, const float* kn,
                                    const float* vc, const float* glog, const float* beta,
                                    const float* S_in, float* S_out, float* o,
                                    struct CUstream_st* stream);

/*
 * gdn_scan_noalloc_check -- the failure report of the last gdn_scan_noalloc on
 * the current device (as gdn_scan_check for an ordinary workspace: its
 * record is the first word of the library's own scratch array, whose address
 * the caller never holds).  Enqueues a 4-byte device-to-host copy on `stream`,
 * SYNCHRONISES it and returns GDN_OK or GDN_ERR_TIMEOUT; GDN_ERR_INVALID_ARG
 * if gdn_scan_noalloc has not run on this device yet.
 */
GDN_API gdn_status gdn_scan_noalloc_check(struct CUstream_st* stream);

/* Workspace bytes gdn_layer needs: the stage tensors vc, glog, beta, o plus
 * the scan's own workspace, each 256-byte aligned (q and k go from the pre
 * stage straight into the scan's operand images there: no qn / kn). */
GDN_API size_t gdn_layer_workspace_bytes(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens);

/*
 * gdn_layer -- the whole prefill layer: gdn_pre, gdn_scan and gdn_post on
 * `stream`, the stage tensors kept in `workspace` (the pages time the three
 * stages back to back as one pre+scan+post total, "Round 30 Track C Audit",
 * section 2).  Arguments as in the three stage calls.  S_out may equal S_in
 * and hist_out may equal hist_in (partial overlaps are rejected).  May be
 * captured into a CUDA graph, as gdn_scan.
 */
GDN_API gdn_status gdn_layer(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                     const int32_t* cu_seqlens, const uint16_t* qkv, const float* conv_w,
                     const uint16_t* hist_in, uint16_t* hist_out, const uint16_t* a,
                     const uint16_t* b, const uint16_t* z, const float* A_log,
                     const float* dt_bias, const float* gamma, const float* S_in, float* S_out,
                     int32_t out_f32, void* y, void* workspace, size_t workspace_bytes,
                     struct CUstream_st* stream);

/*
 * gdn_scan_fast / gdn_layer_fast -- the same computations with every
 * tensor-core product of the scan taken in one pass on bf16 operands (fp32
 * accumulation, fp32 state) instead of the split hi/lo passes: a third of
 * the MMA instructions, traded for accuracy.  Arguments, workspaces, layouts
 * and errors exactly as gdn_scan / gdn_layer.  The error against the fp64
 * reference is bounded by bf16 rounding of K, Q, the state and the chunk
 * intermediates rather than by the 1e-4 of the split path; the tests state the
 * bound they check.
 */
GDN_API gdn_status gdn_scan_fast(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                                 const int32_t* cu_seqlens, const float* qn, const float* kn,
                                 const float* vc, const float* glog, const float* beta,
                                 const float* S_in, float* S_out, float* o, void* workspace,
                                 size_t workspace_bytes, struct CUstream_st* stream);
GDN_API gdn_status gdn_layer_fast(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                                  const int32_t* cu_seqlens, const uint16_t* qkv, const float* conv_w,
                                  const uint16_t* hist_in, uint16_t* hist_out, const uint16_t* a,
                                  const uint16_t* b, const uint16_t* z, const float* A_log,
                                  const float* dt_bias, const float* gamma, const float* S_in,
                                  float* S_out, int32_t out_f32, void* y, void* workspace,
                                  size_t workspace_bytes, struct CUstream_st* stream);

/*
 * Failure reports of the scan.  Every wait inside the scan kernels is
 * bounded (about two seconds); one that expires makes its CTA record an
 * error in the scan workspace, release what it holds and stop, so the CUDA
 * context stays usable but the call's outputs are invalid.  These functions
 * read that record for the last gdn_scan (or gdn_layer) that used the
 * workspace: they enqueue a 4-byte device-to-host copy on `stream`,
 * SYNCHRONISE the stream and return GDN_OK or GDN_ERR_TIMEOUT (GDN_ERR_CUDA if
 * the copy fails).  gdn_layer_check takes the layer's shape to find the scan
 * part of the layer workspace.
 */
GDN_API gdn_status gdn_scan_check(const void* workspace, struct CUstream_st* stream);
GDN_API gdn_status gdn_layer_check(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                                   const void* workspace, struct CUstream_st* stream);

/*
 * gdn_step -- one decode step: a single new token for each of n_seq
 * sequences through the whole layer (pre, the recurrence for that token, and
 * post), fused into one launch.  Per token it computes exactly what gdn_layer
 * computes for a batch in which every sequence holds one token: the
 * token-sequential recurrence of "Round 30 Track C Audit: gdn_pre, gdn_post,
 * and gdn_scanr_4", section 1 (gdn_scan_r's per-token decay, delta update and
 * k/q products against the fp32 state), with that section's pre and post
 * arithmetic for the token.
 *
 * In:  qkv      fp16 [n_seq][C]         the token's raw projections, q | k | v
 *      conv_w   fp32 [C][4]             as for gdn_pre
 *      hist_in  fp16 [n_seq][C][3]      the 3 inputs before the token, oldest first
 *      a, b     fp16 [n_seq][hv]        gate pre-activations
 *      z        fp16 [n_seq][hv][dv]    output gate
 *      A_log, dt_bias fp32 [hv];  gamma fp32 [dv]
 *      S_in     fp32 [n_seq][hv][dk][dv]  state before the token
 * Out: hist_out fp16 [n_seq][C][3]      history after the token (slots 1, 2 of
 *                                       hist_in, then the token); bit copies.
 *                                       Must not overlap any input.
 *      S_out    fp32 [n_seq][hv][dk][dv]  state after the token; may be the same
 *                                       buffer as S_in (not a partial overlap)
 *      y        fp16 [n_seq][hv][dv] when out_f32 == 0, else fp32
 * No workspace.  n_seq == 0 is a no-op.  Errors as for the other entry points.
 */
GDN_API gdn_status gdn_step(const gdn_dims* dims, int32_t n_seq, const uint16_t* qkv, const float* conv_w,
                            const uint16_t* hist_in, uint16_t* hist_out, const uint16_t* a,
                            const uint16_t* b, const uint16_t* z, const float* A_log,
                            const float* dt_bias, const float* gamma, const float* S_in, float* S_out,
                            int32_t out_f32, void* y, struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_H */
