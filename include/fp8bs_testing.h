/*
 * fp8bs_testing.h -- test-only export of libfp8bs.so (not for production
 * callers).  The pages have no counterpart; it exists so the failure-detection
 * test can make a device-side wait run out without faulting the GPU.
 */
#ifndef FP8BS_TESTING_H
#define FP8BS_TESTING_H

#include "fp8bs.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * fp8_blockscaled_gemm with one deliberate gap: in every CTA the producer
 * never fills the pipeline stage of that CTA's unit number `skip_unit`
 * (0-based, counted within the CTA's range), so the MMA warp's bounded wait
 * on it runs out after `timeout_ns` (1 ns .. 10 s).  The kernel then records
 * a code in the workspace status word, drains its in-flight copies, frees its
 * tensor memory and returns; the CUDA context stays usable.  Y is left
 * incomplete and the workspace counters may be non-zero afterwards: zero the
 * workspace before reusing it.  Arguments otherwise as fp8_blockscaled_gemm.
 */
FP8BS_API fp8bs_status fp8bs_testhook_gemm_stall(const uint8_t *aq, const float *as, const uint8_t *wq, const float *ws,
                                       void *y, int M, int N, int K, void *workspace, size_t workspace_bytes,
                                       int skip_unit, unsigned long long timeout_ns, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_TESTING_H */
