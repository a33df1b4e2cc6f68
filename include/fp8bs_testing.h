/*
 * fp8bs_testing.h -- test-only exports of libfp8bs.so (not for production
 * callers).  The pages have no counterpart to any of them.  They exist so
 * the tests can (1) make a device-side wait run out without faulting the
 * GPU, (2) run a GEMM under a schedule planned for another SM count, and
 * (3) see which kernels actually ran inside the process.
 *
 * (3) follows the lesson of "The profiler said the kernel ran zero times",
 * "Why it never ran": a kernel that loads is not a kernel that runs, so the
 * tests look inside the running process before they trust a result.  Every
 * kernel of the library adds one to a per-device 64-bit counter when it
 * starts (one atomic add by the first thread of the first CTA); the slot is
 * fixed per kernel instantiation, below.
 */
#ifndef FP8BS_TESTING_H
#define FP8BS_TESTING_H

#include "fp8bs.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Launch-counter slots. */
#define FP8BS_RUNS_QUANT_ACT 0      /* activation quantisation kernel */
#define FP8BS_RUNS_QUANT_WEIGHT 1   /* weight block quantisation kernel (both layouts) */
#define FP8BS_RUNS_PACK_BF16 2      /* bf16 weight tiling kernel */
#define FP8BS_RUNS_MX_QUANT_WEIGHT 3 /* MX weight quantisation kernel */
#define FP8BS_RUNS_MX_QUANT_ACT 4   /* MX activation quantisation kernel */
/* GEMM kernel instantiations: mode 0 = FP8 on pre-quantised activations,
 * 1 = FP8 with the activation cast in the kernel prologue, 2 = bf16, 3 = MX;
 * npad = the token-tile width (16, 32, 48, 64, 128 or 256); greedy = 1 for
 * the instantiation with the greedy-choice epilogue. */
#define FP8BS_RUNS_NPAD_INDEX(npad) ((npad) <= 64 ? (npad) / 16 - 1 : (npad) == 128 ? 4 : 5)
#define FP8BS_RUNS_GEMM(mode, npad, greedy) (8 + (mode) * 16 + FP8BS_RUNS_NPAD_INDEX(npad) * 2 + (greedy))
#define FP8BS_RUNS_SLOTS 128

/*
 * Synchronises the current device, then copies `count` launch counters
 * starting at slot `first` into out[0 .. count-1].  The counters count
 * kernel launches that started on this device since the library was loaded
 * into this process (they only grow).  FP8BS_ERR_INVALID_ARG when the range
 * leaves [0, FP8BS_RUNS_SLOTS) or out is NULL.
 */
FP8BS_API fp8bs_status fp8bs_testhook_kernel_runs(int first, int count, unsigned long long *out);

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

/*
 * fp8_blockscaled_gemm_fused with the schedule planned for `num_sms` SMs
 * (1 .. 4096) instead of the device's: the CTA count, the K ranges of the
 * CTAs and hence the order of the K-split reduction change with it.  Used to
 * check that the result stays within the tolerance, and bitwise
 * reproducible, under other split counts.  CTAs beyond the device's
 * capacity simply run in later waves (no CTA ever waits for another).
 * The workspace must hold fp8bs_testhook_workspace_size_sms() bytes for the
 * same num_sms.  Arguments otherwise as fp8_blockscaled_gemm_fused.
 */
FP8BS_API fp8bs_status fp8bs_testhook_gemm_fused_sms(const void *x, int ldx, const uint8_t *wq, const float *ws,
                                           void *y, int M, int N, int K, void *workspace,
                                           size_t workspace_bytes, unsigned flags, int num_sms, void *stream);

/* Workspace bytes of fp8bs_testhook_gemm_fused_sms for this shape and SM count. */
FP8BS_API fp8bs_status fp8bs_testhook_workspace_size_sms(int M, int N, int K, int num_sms, size_t *bytes);

/*
 * 1 when this copy of the library was built with FP8BS_DEBUG, 0 otherwise.
 * The FP8BS_DEBUG build (lib/libfp8bs_debug.so) adds device-side checks of
 * every tensor-load coordinate, ring stage, activation-cache slot, scale
 * index, split-K slot and arrival-counter index of the GEMM kernel: a failed
 * check records bit 5 (0x20) in the workspace status word, skips the access
 * and lets the CTA wind down through the bounded waits.  Nothing traps.  It
 * stands in for a device memory checker.
 */
FP8BS_API int fp8bs_testhook_debug_build(void);

/*
 * FP8BS_DEBUG build only (FP8BS_ERR_INVALID_ARG otherwise): the pre-quantised
 * GEMM with unit `bad_unit` of every CTA addressed one 128-row weight tile
 * past the end of Wq.  The checks must catch it: the status word then holds
 * bit 5, and the unfilled stage's bounded wait (timeout_ns, 1 ns .. 10 s)
 * adds its own time-out bit.  Zero the workspace before reusing it.
 * Arguments otherwise as fp8_blockscaled_gemm.
 */
FP8BS_API fp8bs_status fp8bs_testhook_debug_bad_tile(const uint8_t *aq, const float *as, const uint8_t *wq,
                                           const float *ws, void *y, int M, int N, int K, void *workspace,
                                           size_t workspace_bytes, int bad_unit, unsigned long long timeout_ns,
                                           void *stream);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_TESTING_H */
