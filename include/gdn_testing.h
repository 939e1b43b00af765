/*
 * gdn_testing.h -- test hooks of the GDN prefill library (libgdn.so), kept out
 * of the product interface in gdn.h.  They compute nothing a caller wants:
 * each runs gdn_scan with one part of its machinery deliberately held back, so
 * that a test can check, without faulting or hanging a GPU, that the library
 * detects and reports what happens then (bounded waits that expire and report
 * GDN_ERR_TIMEOUT through gdn_scan_check; the prep kernel's progress guarantee).
 * Arguments, layouts and errors are those of gdn_scan in gdn.h (of gdn_layer
 * for gdn_layer_selftest_stages).
 */
#ifndef GDN_TESTING_H
#define GDN_TESTING_H

#include "gdn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * gdn_scan_selftest_timeout -- test hook of the failure report, not a
 * computation: runs gdn_scan with the recurrence kernel's first operand copy
 * withheld, so that a bounded wait in every CTA of that kernel expires (no
 * fault, no trap, no unbounded wait).  Arguments as for gdn_scan; the
 * outputs are invalid and gdn_scan_check on the workspace returns
 * GDN_ERR_TIMEOUT.  Takes about two seconds.
 */
GDN_API gdn_status gdn_scan_selftest_timeout(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                                             const int32_t* cu_seqlens, const float* qn, const float* kn,
                                             const float* vc, const float* glog, const float* beta,
                                             const float* S_in, float* S_out, float* o, void* workspace,
                                             size_t workspace_bytes, struct CUstream_st* stream);

/*
 * gdn_scan_selftest_one_taker -- test hook of the prep kernel's progress
 * guarantee: runs gdn_scan with no SM chosen to keep taking prep tasks after
 * the first round, so the one CTA that the fallback keeps (the last to finish
 * round one) takes every remaining task alone.  Arguments and results as for
 * gdn_scan (bit for bit: each task computes the same values wherever it runs);
 * only slower.
 */
GDN_API gdn_status gdn_scan_selftest_one_taker(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                                               const int32_t* cu_seqlens, const float* qn, const float* kn,
                                               const float* vc, const float* glog, const float* beta,
                                               const float* S_in, float* S_out, float* o, void* workspace,
                                               size_t workspace_bytes, struct CUstream_st* stream);

/*
 * gdn_scan_selftest_withhold_flag -- test hook of the wait across kernels:
 * runs gdn_scan with the prep kernel leaving one ready flag unset (chunk slot
 * 1, value head 0), so that the recurrence kernel's bounded wait for that flag
 * expires in the CTAs of value head 0 (no fault, no unbounded wait).  Needs a
 * batch whose first sequence spans at least two chunks.  The outputs are
 * invalid and gdn_scan_check on the workspace returns GDN_ERR_TIMEOUT.  Takes
 * about two seconds.
 */
GDN_API gdn_status gdn_scan_selftest_withhold_flag(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                                                   const int32_t* cu_seqlens, const float* qn, const float* kn,
                                                   const float* vc, const float* glog, const float* beta,
                                                   const float* S_in, float* S_out, float* o, void* workspace,
                                                   size_t workspace_bytes, struct CUstream_st* stream);

/*
 * gdn_layer_selftest_stages -- test and timing hook of gdn_layer: runs only the
 * stages of gdn_layer (or of gdn_layer_fast, fast != 0) named by the mask
 * `stages` (bit 0: the pre kernel that writes the scan's operand images, bit
 * 1: the scan, bit 2: post), on a gdn_layer workspace, so that a harness can
 * time or check the stages of the fused call one at a time.  Every argument is
 * validated as for gdn_layer whatever the mask.  A stage that is skipped leaves
 * its outputs and its part of the workspace as they were, so a later stage
 * reads what an earlier call left there: running the masks 1, 2 and 4 in turn
 * on one workspace gives gdn_layer's results bit for bit.  A mask outside 0..7
 * returns GDN_ERR_INVALID_ARG.
 */
GDN_API gdn_status gdn_layer_selftest_stages(const gdn_dims* dims, int32_t n_seq, int32_t total_tokens,
                                             const int32_t* cu_seqlens, const uint16_t* qkv, const float* conv_w,
                                             const uint16_t* hist_in, uint16_t* hist_out, const uint16_t* a,
                                             const uint16_t* b, const uint16_t* z, const float* A_log,
                                             const float* dt_bias, const float* gamma, const float* S_in,
                                             float* S_out, int32_t out_f32, void* y, void* workspace,
                                             size_t workspace_bytes, int32_t fast, int32_t stages,
                                             struct CUstream_st* stream);

#ifdef __cplusplus
}
#endif

#endif /* GDN_TESTING_H */
