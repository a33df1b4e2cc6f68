// internal.h -- host-side plumbing shared by the translation units of
// libfp8bs.so (not part of the public ABI).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

#include "fp8bs.h"

namespace fp8bs {

struct DeviceInfo {
    int device = -1;
    int sms = 0;
    int cc_major = 0, cc_minor = 0;
    unsigned long long *runs = nullptr; // this device's kernel launch counters (runs.cu)
};

// Current device's cached attributes; status FP8BS_ERR_CUDA when there is no
// usable device, FP8BS_ERR_UNSUPPORTED_DEVICE when it is not sm_103.
fp8bs_status current_device(DeviceInfo *out);

// One-time per (kernel, device) opt-in to more than 48 KB of dynamic shared
// memory.  `done_mask` is the caller's static per-kernel bit mask of devices.
fp8bs_status ensure_smem_attr(const void *kernel, int bytes, int device, unsigned long long *done_mask);

// 2-D tensor map for a row-major [rows][cols] matrix, box = box_cols x
// box_rows elements, 128-byte swizzle unless told otherwise, zero fill outside
// the matrix on loads (stores outside it are dropped).
fp8bs_status make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                          uint64_t rows, uint64_t cols, uint64_t row_stride_bytes, uint32_t box_cols,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B);

fp8bs_status launch_status(cudaError_t e);

// Largest token count of the GEMMs.
constexpr int kMaxTokens = 512;

// Token-tile width for M <= 64 rows (16, 32, 48 or 64); gemm_shape picks the
// tiles of larger M.
inline int token_pad(int M)
{
    return M <= 16 ? 16 : M <= 32 ? 32 : M <= 48 ? 48 : M <= 64 ? 64 : M <= 128 ? 128 : 256;
}

// Workspace layout shared by the GEMM launchers:
//   [0, 256)                status word (+ padding)
//   [256, 1024)             greedy choice: 64 64-bit keys, then the CTA counter
//   [1024, 1024 + C)        ttiles * ntiles 32-bit arrival counters, C rounded up to 256
//   slots                   ttiles * 2 * ctas slots of NPAD * 128 fp32 partials
//   act, act_scale          M x K codes and M x K/128 scales, used only when the
//                           fused entry point quantises in a separate kernel
struct WorkspaceLayout {
    size_t greedy_off, counters_off, slots_off, act_off, act_scale_off, total;
};
struct GemmShape;
WorkspaceLayout workspace_layout(const GemmShape &sh, int M, int K);

struct GemmLaunch {
    int mode;                 // GemmMode (0 FP8, 1 FP8 fused cast, 2 bf16, 3 MX)
    int M, N, K;
    const void *a;            // mode 0: Aq u8 [M][K]; mode 1: X bf16 [M][ldx]; mode 2: X bf16 [M][K]
    int lda;                  // row stride of `a` in elements
    const float *as;          // mode 0
    const void *w;            // mode 0/1: Wq u8 [N][K]; mode 2: W bf16 [N][K]
    const float *ws;          // mode 0/1
    const uint8_t *sfa;       // mode 3: weight scale atoms
    const uint8_t *sfb;       // mode 3: activation scale atoms
    void *y;
    void *workspace;
    size_t workspace_bytes;
    unsigned flags;
    cudaStream_t stream;
    int test_skip_unit = -1;  // -1 normally
    int test_bad_unit = -1;   // -1 normally (FP8BS_DEBUG test hook)
    unsigned long long timeout_ns;
    int *token;               // greedy choice per token, or nullptr (then y must be set)
    float *logit;             // its logit, or nullptr
    int sms;                  // SM count the schedule is planned for (0: the device's)
};

// Shape and SM count -> schedule; shared by launch and size queries.
struct GemmShape {
    int kg = 0, ntiles = 0, ctas = 0, npad = 0;
    int m = 0;       // tokens (M)
    int ttiles = 0;  // token tiles
    bool split = true; // K is split across CTAs (exchange slots needed)
    long long units = 0;
};
GemmShape gemm_shape(int mode, int M, int N, int K, int sms);

// True when the fused entry point casts the activations in the GEMM
// prologue for this schedule and flags (FP8BS_FLAG_PROLOGUE_CAST, and the
// cache fits); false when it runs the separate cast kernel.
bool fused_prologue_route(const GemmShape &sh, unsigned flags);

// Device address of the current device's kernel launch counters
// (FP8BS_RUNS_SLOTS 64-bit words), looked up once per device; nullptr when
// the lookup failed.
unsigned long long *run_counters(int device);

fp8bs_status launch_gemm_fp8(const GemmLaunch &L, const DeviceInfo &dev);
fp8bs_status launch_gemm_fused(const GemmLaunch &L, const DeviceInfo &dev);
fp8bs_status launch_gemm_bf16(const GemmLaunch &L, const DeviceInfo &dev);
fp8bs_status launch_gemm_mx(const GemmLaunch &L, const DeviceInfo &dev);
fp8bs_status launch_mx_quant_weights(const void *w, int wtype, int N, int K, uint8_t *wq, uint8_t *sf,
                                     cudaStream_t stream, const DeviceInfo &dev);
fp8bs_status launch_mx_quant_act(const void *x, int M, int K, int ldx, uint8_t *xq, uint8_t *sf, bool pdl,
                                 cudaStream_t stream, const DeviceInfo &dev);

fp8bs_status launch_quant_act(const void *x, int M, int K, int ldx, uint8_t *xq, float *xs, bool pdl,
                              cudaStream_t stream, const DeviceInfo &dev);
fp8bs_status launch_quant_weight(const void *w, int wtype, int N, int K, uint8_t *wq, float *ws, bool tiled,
                                 cudaStream_t stream, const DeviceInfo &dev);
fp8bs_status launch_pack_bf16_tiled(const void *w, int N, int K, void *wt, cudaStream_t stream,
                                    const DeviceInfo &dev);

constexpr unsigned long long kDefaultTimeoutNs = 1000000000ull; // one second

} // namespace fp8bs
