/*
 * fp8bs.h -- C ABI of libfp8bs.so: the small-M FP8 block-scaled linear layer
 *
 *     Y[M,N] = dequant(Aq[M,K]) . dequant(Wq[N,K])^T
 *
 * on one GB300 (sm_103a).  M is 1..64 rows (decode / speculative-verify
 * batches; up to 512 for chunked prefill), W is E4M3 with one fp32 scale per 128x128 block, the activations
 * are cast on the fly to E4M3 with one fp32 scale per token per 128 K.
 *
 * Sources (page title, section):
 *   [P1] "A 23% faster GPU kernel, and a model that did not move",
 *        "Why this shape is hard": about 8 rows, the long dimension split
 *        across all SMs, 128x128 block scales, deterministic reduction.
 *   [P2] "The profiler said the kernel ran zero times",
 *        "What the trace showed" (casting inputs to FP8 at run time) and
 *        "The output layer, which did run" (248,320 x 5,120 output layer,
 *        one scale per 128x128 block; the same layer in 16-bit as baseline).
 *   [P3] "Kernel-Level Optimisations for LLM Inference and Training",
 *        "Quantisation kernels" (E4M3 for weights and activations).
 *
 * Numeric contract (the pages are silent; plainest reading):
 *   E4M3 is the "fn" encoding (bias 7, max finite 448, NaN 0x7F/0xFF).
 *   scale = fl32(amax / 448) by IEEE fp32 division (1.0 when amax == 0);
 *   code  = round-to-nearest-even, saturating, of fl32(x / scale); the sign of
 *   a value that rounds to zero is kept (0x80).
 *   Y is accumulated in fp32: each 128-wide K block's exact-product partial
 *   is multiplied by s_a[m,kb] * s_w[n/128,kb] and summed in K order within a
 *   CTA; K-split partials are summed in a fixed order, then rounded once to
 *   bf16 (nearest even).  Results are bitwise reproducible on one device.
 *
 * Conventions for every entry point:
 *   - All tensor pointers are DEVICE pointers owned by the caller; the
 *     library allocates no device memory and keeps no pointer after return.
 *   - Row-major layouts: X bf16 [M][ldx]; Aq u8 [M][K]; W fp32|bf16 [N][K];
 *     Wq u8 [N][K]; s_w fp32 [ceil(N/128)][K/128]; Y bf16 [M][N].
 *   - Activation scales s_a (fp32, M*(K/128) words): token-major [M][K/128]
 *     (element m*(K/128) + g) when M <= 16, K-block-major [K/128][M]
 *     (element g*M + m) when M > 16; the two coincide at M = 1.  Each is the
 *     faster one for the GEMM at that size: above 16 tokens the epilogue
 *     loads one K block's scales for a warp's tokens with one request.
 *   - `stream` is a cudaStream_t (NULL = the legacy default stream).  Work is
 *     enqueued asynchronously; no call synchronises the host except
 *     fp8bs_workspace_status().
 *   - Arguments are checked on the host before anything is enqueued; on any
 *     error nothing is launched and the status says why.  No C++ exception
 *     crosses the ABI.  Thread-safe.
 *   - Only compute capability 10.3 is accepted (FP8BS_ERR_UNSUPPORTED_DEVICE
 *     otherwise).  There is no fallback path.
 */
#ifndef FP8BS_H
#define FP8BS_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define FP8BS_API __attribute__((visibility("default")))
#else
#define FP8BS_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum fp8bs_status {
    FP8BS_OK = 0,
    FP8BS_ERR_INVALID_ARG = 1,         /* null pointer, size < 1, ldx < K, bad enum */
    FP8BS_ERR_UNSUPPORTED_SHAPE = 2,   /* M above the entry point's limit (512 for the GEMMs, 64 with the
                                          greedy choice or without a workspace), K not a multiple of 128
                                          (64 for the bf16 GEMM), sizes beyond 2^30 */
    FP8BS_ERR_MISALIGNED = 3,          /* a pointer or row stride breaks the alignment stated below */
    FP8BS_ERR_WORKSPACE_TOO_SMALL = 4, /* workspace_bytes below the *_workspace_size() answer */
    FP8BS_ERR_UNSUPPORTED_DEVICE = 5,  /* current device is not sm_103 */
    FP8BS_ERR_CUDA = 6,                /* a CUDA runtime/driver call failed (launch, attribute, ...) */
    FP8BS_ERR_DEVICE_TIMEOUT = 7       /* a kernel gave up waiting (see fp8bs_workspace_status) */
} fp8bs_status;

typedef enum fp8bs_dtype {
    FP8BS_F32 = 0,
    FP8BS_BF16 = 1
} fp8bs_dtype;

/* Flag for the GEMM entry points.  With it the kernel is launched with
 * programmatic dependent launch: it may start while the previous kernel on
 * `stream` is still finishing and begin streaming Wq/s_w (or W for the bf16
 * GEMM) before that kernel completes; it reads everything else only after
 * the previous kernel has completed.  The caller promises that no work still
 * in flight on `stream` writes the weights or their scales. */
#define FP8BS_FLAG_OVERLAP_PREV 1u

/* Flag for the GEMM entry points: the weights are in the tiled layout that
 * fp8_quant_weight_blocks_tiled (FP8) or bf16_pack_weights_tiled (bf16)
 * writes.  Every 128-row x 128-byte weight tile is then one contiguous 16 KB
 * run of memory, so each tile the GEMM streams is a single sequential HBM
 * read instead of 128 separate 128-byte pieces of 128 different rows. */
#define FP8BS_FLAG_WEIGHTS_TILED 2u

/* Flag for the fused entry points (fp8_blockscaled_gemm_fused, its greedy and
 * no-allocation variants): cast the activations in the GEMM kernel's
 * prologue, every CTA its own K blocks' token rows straight into a
 * shared-memory cache (one kernel), wherever that cache fits (at most 16
 * (K block, token) rows a CTA and 96 KB); elsewhere, and without the flag,
 * the cast runs as its own kernel before the pre-quantised GEMM.  Measured on
 * GB300, the two-kernel route is the faster one for every shape tried, 3-10 %
 * for 1 to 16 tokens, chained with or without programmatic dependent launch:
 * the prologue kernel holds one CTA per SM and repeats each K block's cast in
 * every CTA that uses it.  fp8bs_fused_route reports the route for a flag
 * set. */
#define FP8BS_FLAG_PROLOGUE_CAST 4u

/* Human-readable text of a status code (static storage, never NULL). */
FP8BS_API const char *fp8bs_status_string(fp8bs_status status);

/*
 * Activation quantisation [P2 "What the trace showed"; P3 "Quantisation
 * kernels"].  For every token m and every group g of 128 consecutive K:
 *   amax = max |x[m, 128g .. 128g+127]|
 *   s(m, g)     = amax == 0 ? 1.0f : fl32(amax / 448)
 *   xq[m*K + k] = e4m3_rn_satfinite(fl32(x[m,k] / s(m, k/128)))
 * with s(m, g) stored at xs[m*(K/128) + g] when M <= 16 and at xs[g*M + m]
 * when M > 16 (the activation-scale layouts above).
 * x : bf16, M rows, row stride ldx elements; 16-byte aligned, ldx % 8 == 0.
 * xq: u8 [M][K], 4-byte aligned.  xs: fp32, M*(K/128) words, 4-byte aligned.
 * M >= 1, K >= 128, K % 128 == 0, ldx >= K.
 * Any `flags` value other than 0 and FP8BS_FLAG_OVERLAP_PREV is rejected;
 * with the flag the kernel is launched with programmatic dependent launch and
 * waits for the previous kernel before it reads x.
 */
FP8BS_API fp8bs_status fp8_quant_act(const void *x, int M, int K, int ldx,
                           uint8_t *xq, float *xs,
                           unsigned flags, void *stream);

/*
 * Weight quantisation, one fp32 scale per 128x128 block [P1 "Why this shape
 * is hard"; P2 "The output layer, which did run"].  Run once per weight.
 * For block (nb, kb) over the rows nb*128 .. min(N, nb*128+128)-1 that exist:
 *   amax = max |w| over the block
 *   ws[nb*(K/128) + kb] = amax == 0 ? 1.0f : fl32(amax / 448)
 *   wq[n*K + k] = e4m3_rn_satfinite(fl32(w[n,k] / ws[n/128, k/128]))
 * w : fp32 or bf16 (wtype) [N][K] row-major, 16-byte aligned.
 * wq: u8 [N][K], 16-byte aligned.  ws: fp32 [ceil(N/128)][K/128].
 * N >= 1 (a ragged last block is allowed), K >= 128, K % 128 == 0.
 */
FP8BS_API fp8bs_status fp8_quant_weight_blocks(const void *w, fp8bs_dtype wtype, int N, int K,
                                     uint8_t *wq, float *ws, void *stream);

/*
 * The same quantisation (bit-identical codes and scales) written in the tiled
 * layout: the codes of block (nb, kb) occupy bytes
 *   [(nb*(K/128) + kb) * 16384, +16384)
 * with row r of the block (weight row nb*128 + r) at offset r*128, its 128
 * bytes in K order.  Rows past N in the last block are written as zeros.
 * wq must hold ceil(N/128) * 128 * K bytes, 16-byte aligned.  ws as above.
 */
FP8BS_API fp8bs_status fp8_quant_weight_blocks_tiled(const void *w, fp8bs_dtype wtype, int N, int K,
                                           uint8_t *wq, float *ws, void *stream);

/*
 * Bytes of device workspace the GEMM entry points need for this shape on the
 * current device (it depends on the SM count).  Writes *bytes; on error
 * writes 0.  The same answer serves fp8_blockscaled_gemm and
 * fp8_blockscaled_gemm_fused; bf16_gemm_ref has its own query.
 *
 * Workspace contract: zero-fill it once (e.g. cudaMemsetAsync) before its
 * first use.  Every call that completes leaves its counter words zero again,
 * so one workspace serves any number of later calls and CUDA-graph replays.
 * Calls that share a workspace must not run concurrently (same stream, or
 * ordered by events).  After FP8BS_ERR_DEVICE_TIMEOUT, zero-fill it again.
 */
FP8BS_API fp8bs_status fp8_blockscaled_gemm_workspace_size(int M, int N, int K, size_t *bytes);

/*
 * Block-scaled FP8 GEMM on pre-quantised operands [P1 "Why this shape is
 * hard"]:
 *   y[m*N + n] = bf16_rn( sum_kb s_a[m,kb] * s_w[n/128,kb]
 *                          * sum_{k in kb} dec(aq[m,k]) * dec(wq[n,k]) )
 * Swap-AB tcgen05 kernel (weights in the MMA M dimension, tokens in N),
 * 128x128 weight tiles streamed by TMA, K split across every SM with a
 * fixed-order reduction.
 * aq: u8 [M][K], 16-byte aligned.   as: fp32, laid out as fp8_quant_act writes
 * it for this M ([M][K/128] up to 16 tokens, [K/128][M] above).
 * wq: u8 [N][K], 16-byte aligned.   ws: fp32 [ceil(N/128)][K/128].
 * y : bf16 [M][N], 2-byte aligned.  With y 16-byte aligned and N % 8 == 0
 *     finished Y tiles leave through shared memory and one TMA store each
 *     (faster); otherwise the kernel stores them row by row.  Same bits.
 * 1 <= M <= 512, N >= 1, K >= 128, K % 128 == 0.  Up to 64 tokens the
 * token tile is 16, 32, 48 or 64 wide and K is split across every SM; above
 * 64 tokens (the larger-M, chunked-prefill regime, where the pages note that
 * the work turns from memory- to compute-bound: "Kernel-Level Optimisations
 * for LLM Inference and Training", "Start with the bound") the work is cut
 * into (token tile, 128-row weight tile) pairs: with at least as many
 * 128-token pairs as SMs, or with too few pairs to keep the SMs busy, K is
 * split over all the pairs' units (stream-K); otherwise each CTA computes
 * one pair over the whole K, with the widest token tile (128, 64 or 32)
 * whose pairs fit on the SMs (fp8bs_gemm_schedule reports the choice).
 * workspace: device, 256-byte aligned, >= fp8_blockscaled_gemm_workspace_size.
 * flags: any of FP8BS_FLAG_OVERLAP_PREV, FP8BS_FLAG_WEIGHTS_TILED (then wq is
 * in the tiled layout of fp8_quant_weight_blocks_tiled).
 */
FP8BS_API fp8bs_status fp8_blockscaled_gemm(const uint8_t *aq, const float *as,
                                  const uint8_t *wq, const float *ws,
                                  void *y, int M, int N, int K,
                                  void *workspace, size_t workspace_bytes,
                                  unsigned flags, void *stream);

/*
 * The whole layer from bf16 activations: activation quantisation (as
 * fp8_quant_act) fused with the GEMM (as fp8_blockscaled_gemm).  By default
 * the quantisation runs once as its own kernel into the workspace, followed
 * by the pre-quantised GEMM on the same stream.  With
 * FP8BS_FLAG_PROLOGUE_CAST, where each CTA has at most 16 (K block, token)
 * rows to cast and its cache fits 96 KB, it runs in the GEMM kernel's
 * prologue instead: every CTA quantises the token rows of the K blocks it
 * will use straight into a shared-memory cache in the tensor-core operand
 * layout (one kernel, replicated work; slower on GB300 in every
 * configuration measured, see the flag).  Either way
 * the result is bitwise identical to fp8_quant_act followed by
 * fp8_blockscaled_gemm.
 * x: bf16, M rows, row stride ldx elements, 16-byte aligned, ldx % 8 == 0.
 * flags: as fp8_blockscaled_gemm, plus FP8BS_FLAG_PROLOGUE_CAST.
 * Other arguments as fp8_blockscaled_gemm.
 */
FP8BS_API fp8bs_status fp8_blockscaled_gemm_fused(const void *x, int ldx,
                                        const uint8_t *wq, const float *ws,
                                        void *y, int M, int N, int K,
                                        void *workspace, size_t workspace_bytes,
                                        unsigned flags, void *stream);

/*
 * The output layer with the greedy next-token choice fused into its epilogue
 * [P2 "The output layer, which did run": the 248,320-wide output layer feeds
 * the choice of the next token].  Computes Y exactly as
 * fp8_blockscaled_gemm_fused (bitwise the same values) and, per token m:
 *   token[m] = the column n < N of the largest bf16 value y[m][n], compared
 *              as numbers (+0 equals -0); among equal values the lowest n;
 *   logit[m] = that value as fp32 (a zero is reported as +0).
 * Each CTA reduces the tiles it finishes while they are still in registers;
 * the logits are never read back from memory.  The choice is deterministic:
 * it depends only on Y, whose values are bitwise reproducible.
 * y: bf16 [M][N] as fp8_blockscaled_gemm_fused, or NULL to skip storing the
 *    logits.  token: int32 [M], 4-byte aligned (required).  logit: fp32 [M],
 *    4-byte aligned, or NULL.  NaN logits (NaN inputs) are outside the
 *    contract.  Workspace as fp8_blockscaled_gemm_fused (the same size query);
 *    the library leaves its greedy keys and counter at zero after every call.
 * 1 <= M <= 64 (FP8BS_ERR_UNSUPPORTED_SHAPE above).
 * Other arguments as fp8_blockscaled_gemm_fused.
 */
FP8BS_API fp8bs_status fp8_blockscaled_gemm_fused_greedy(const void *x, int ldx,
                                               const uint8_t *wq, const float *ws,
                                               void *y, int M, int N, int K,
                                               int32_t *token, float *logit,
                                               void *workspace, size_t workspace_bytes,
                                               unsigned flags, void *stream);

/*
 * fp8_blockscaled_gemm_fused without a caller-provided workspace, for callers
 * that cannot allocate device memory (code running under a graph capture
 * that must not allocate, allocator-less embedded runtimes, hooks that run
 * while a framework holds its memory pool).  The pages have no counterpart:
 * this is an interface convenience, not part of the method.
 * The split-K scratch lives in a 12 MiB array inside the library (every GPU
 * that loads the library holds it until the process exits); shapes whose
 * workspace (fp8_blockscaled_gemm_workspace_size) exceeds 12 MiB are rejected
 * with FP8BS_ERR_UNSUPPORTED_SHAPE.  The call allocates nothing.  Its first
 * call on a device looks up the array's device address (cudaGetSymbolAddress),
 * so make that first call before any stream capture.  Each call clears the
 * array's status word and counters on `stream` before the kernel runs; every
 * call shares the one array, so calls that can overlap on the GPU (different
 * streams without ordering) race and must not be issued.  Device-side
 * time-outs are recorded in the shared array and are not reported back.
 * FP8BS_FLAG_OVERLAP_PREV is accepted but gives no overlap here: the kernel's
 * programmatic dependency is on the clearing step this call enqueues, not on
 * the caller's previous kernel.
 * Arguments and result as fp8_blockscaled_gemm_fused, with 1 <= M <= 64.
 */
FP8BS_API fp8bs_status fp8_blockscaled_gemm_fused_noalloc(const void *x, int ldx,
                                                const uint8_t *wq, const float *ws,
                                                void *y, int M, int N, int K,
                                                unsigned flags, void *stream);

/*
 * Native block-scaled (MX) variant ["Kernel-Level Optimisations for LLM
 * Inference and Training", "Writing your own kernel": the block-scaled and
 * MX formats that Blackwell tensor cores scale in hardware].  A different
 * numeric contract from the 128x128 fp32 block scales above: every 32
 * consecutive values along K of a weight row or token share one power-of-two
 * scale 2^e, stored as the byte e + 127 (UE8M0), with
 *   e = floor(log2(amax of the 32 values)) - 8, clamped to [-127, 127]
 *       (0 for a block of zeros; 448 = 1.75 * 2^8 is E4M3's largest value)
 *   code = e4m3_rn_satfinite(v / 2^e)   (exact scaling; values up to 2^9
 *                                         saturate at 448)
 * and Y = bf16_rn( sum over 32-blocks b of 2^(ea[m,b] + ew[n,b]) * sum_{k in b}
 * dec(aq[m,k]) * dec(wq[n,k]) ), the scales applied by the tensor core
 * (tcgen05.mma kind::mxf8f6f4 block_scale) with one fp32 accumulation over
 * each CTA's share of K, so no per-block promotion runs on CUDA cores.
 *
 * Scale bytes are stored in 512-byte atoms, the layout the tensor core's
 * scale-factor copy reads: per 128 rows (weight rows, or tokens) and 128 K,
 * the byte of row r (0..127) and 32-wide K block j (0..3) is at offset
 *   16 * (r % 32) + 4 * (r / 32) + j.
 *
 * fp8_mx_quant_weights: w fp32|bf16 [N][K] (16-byte aligned) ->
 *   wq: codes in the tiled layout of fp8_quant_weight_blocks_tiled,
 *       ceil(N/128) * 128 * K bytes, rows past N zero;
 *   ws_atoms: ceil(N/128) * (K/128) atoms, atom (nb, kb) at
 *       (nb * (K/128) + kb) * 512, rows past N zero.  Both 16-byte aligned.
 * fp8_mx_quant_act: x bf16, M rows (1..512), row stride ldx (>= K, % 8 == 0),
 *   16-byte aligned -> xq u8 [M][K] (16-byte aligned), xs_atoms:
 *   ceil(M/128) * (K/128) atoms, atom (tt, kb) of tokens tt*128.. at
 *   (tt * (K/128) + kb) * 512, token rows past M written as zero.  flags: 0
 *   or FP8BS_FLAG_OVERLAP_PREV (programmatic dependent launch; x is read
 *   after the previous kernel completes).
 * fp8_mx_gemm: y bf16 [M][N] from those operands, 1 <= M <= 512, K % 128 == 0;
 *   same swap-AB / TMA / split-K pipeline and the same workspace contract as
 *   fp8_blockscaled_gemm (size from fp8_mx_gemm_workspace_size).  flags: 0
 *   or FP8BS_FLAG_OVERLAP_PREV (the weights and their atoms may be streamed
 *   before the previous kernel completes).  Bitwise reproducible.
 */
FP8BS_API fp8bs_status fp8_mx_quant_weights(const void *w, fp8bs_dtype wtype, int N, int K, uint8_t *wq,
                                            uint8_t *ws_atoms, void *stream);
FP8BS_API fp8bs_status fp8_mx_quant_act(const void *x, int M, int K, int ldx, uint8_t *xq, uint8_t *xs_atoms,
                                        unsigned flags, void *stream);
FP8BS_API fp8bs_status fp8_mx_gemm_workspace_size(int M, int N, int K, size_t *bytes);
FP8BS_API fp8bs_status fp8_mx_gemm(const uint8_t *aq, const uint8_t *as_atoms, const uint8_t *wq,
                                   const uint8_t *ws_atoms, void *y, int M, int N, int K, void *workspace,
                                   size_t workspace_bytes, unsigned flags, void *stream);

/*
 * 16-bit comparison GEMM for the output layer [P2 "The output layer, which
 * did run": the layer "still 16-bit" before conversion]:
 *   y[m*N + n] = bf16_rn( sum_k x[m,k] * w[n,k] )   (fp32 accumulation)
 * Same swap-AB / TMA / split-K pipeline with bf16 tensor-core MMAs and no
 * block scales.
 * x: bf16 [M][K], w: bf16 [N][K], both 16-byte aligned; y: bf16 [M][N].
 * 1 <= M <= 512, N >= 1, K >= 64, K % 64 == 0.
 */
FP8BS_API fp8bs_status bf16_gemm_ref_workspace_size(int M, int N, int K, size_t *bytes);
/*
 * Copy a bf16 weight matrix [N][K] (K % 64 == 0) into the tiled layout for
 * bf16_gemm_ref with FP8BS_FLAG_WEIGHTS_TILED: tile (nb, kb) of 128 rows x 64
 * elements occupies bytes [(nb*(K/64) + kb) * 16384, +16384), row r at
 * offset r*128; rows past N are zeros.  wt holds ceil(N/128)*128*K*2 bytes.
 * Both pointers 16-byte aligned.
 */
FP8BS_API fp8bs_status bf16_pack_weights_tiled(const void *w, int N, int K, void *wt, void *stream);
FP8BS_API fp8bs_status bf16_gemm_ref(const void *x, const void *w, void *y,
                           int M, int N, int K,
                           void *workspace, size_t workspace_bytes,
                           unsigned flags, void *stream);

/*
 * Device-side failure report.  Every wait inside the GEMM kernels is bounded
 * (about one second); a kernel that gives up records a code in the first
 * word of its workspace, releases its tensor memory and returns.  This call
 * synchronises the device, copies that word to *code (0 = none) and, when
 * clear != 0, resets it.  Returns FP8BS_ERR_DEVICE_TIMEOUT when the word is
 * non-zero, FP8BS_OK otherwise.
 */
FP8BS_API fp8bs_status fp8bs_workspace_status(void *workspace, int clear, int *code);

/*
 * The schedule the FP8 GEMMs choose for M tokens (the plan above is its
 * M <= 64 case), exposed for inspection and tests.  Writes the token-tile
 * width (*npad), the number of token tiles, the CTA count, the work-unit
 * count (units = token tiles * ceil(N/128) * K/128, the K block fastest,
 * then the 128-row weight tile) and whether K is split across CTAs
 * (*split = 1: the fixed-order exchange runs; 0: every CTA owns whole
 * (token tile, weight tile) pairs).  num_sms <= 0 means "the current
 * device".  Nothing is launched.  (fp8_mx_gemm follows the same rules
 * except that above 64 tokens its token tile is always 128 wide: a token
 * scale atom covers 128 tokens.)
 */
FP8BS_API fp8bs_status fp8bs_gemm_schedule(int M, int N, int K, int num_sms, int *npad, int *token_tiles,
                                           int *ctas, long long *units, int *split);

/*
 * The route fp8_blockscaled_gemm_fused takes for this shape and `flags`:
 * *prologue = 1 when every CTA casts its own activation rows in the GEMM
 * kernel's prologue (one kernel; only with FP8BS_FLAG_PROLOGUE_CAST, where
 * the cache fits), 0 when the cast runs as its own kernel into the workspace
 * before the pre-quantised GEMM (two kernels).  num_sms <= 0 means "the
 * current device".  The choice depends only on (M, N, K, SM count, flags).
 * Nothing is launched.  Flags other than the fused entry points' are
 * rejected (FP8BS_ERR_INVALID_ARG).
 */
FP8BS_API fp8bs_status fp8bs_fused_route(int M, int N, int K, int num_sms, unsigned flags, int *prologue);

/*
 * The K-split schedule the GEMMs use, exposed for inspection and tests.
 * Work unit = (128-row weight tile, 128-wide K block) [(tile, 64-wide K
 * block) for bf16_gemm_ref, bf16 = 1]; units are ordered tile-major and
 * split into `ctas` contiguous ranges of equal size +-1, one per SM (fewer
 * when there are fewer units).  num_sms <= 0 means "the current device".
 * Writes the CTA count, the unit count and, for CTA `cta` (when >= 0), its
 * first unit and one-past-last unit.
 */
FP8BS_API fp8bs_status fp8bs_split_plan(int N, int K, int bf16, int num_sms, int cta,
                              int *ctas, long long *units,
                              long long *unit_begin, long long *unit_end);

#ifdef __cplusplus
}
#endif

#endif /* FP8BS_H */
