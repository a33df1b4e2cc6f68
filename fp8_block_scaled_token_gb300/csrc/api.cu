// api.cu -- the extern "C" entry points of libfp8bs.so: argument checks (all
// on the host, before anything is enqueued), the per-device attribute cache,
// tensor-map encoding, and dispatch to the kernels.  No entry point falls
// back to another implementation: a failure is always a returned status.
#include <atomic>
#include <cstring>
#include <mutex>

#include "fp8bs_testing.h"
#include "internal.h"
#include "plan.cuh"

namespace fp8bs {

namespace {

constexpr int kMaxDevices = 64;
std::mutex g_dev_mutex;
bool g_dev_ready[kMaxDevices];
DeviceInfo g_dev[kMaxDevices];
fp8bs_status g_dev_status[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                   const cuuint64_t *, const cuuint32_t *, const cuuint32_t *,
                                   CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                                   CUtensorMapFloatOOBfill);
std::once_flag g_encode_once;
EncodeTiledFn g_encode = nullptr;

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

} // namespace

fp8bs_status launch_status(cudaError_t e)
{
    if (e == cudaSuccess)
        return FP8BS_OK;
    (void)cudaGetLastError(); // the error was reported; do not leave it sticky for the caller
    return FP8BS_ERR_CUDA;
}

fp8bs_status current_device(DeviceInfo *out)
{
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        (void)cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    if (!__atomic_load_n(&g_dev_ready[dev], __ATOMIC_ACQUIRE)) {
        // First call on this device: query and cache its attributes.  A
        // failed query is not cached, so a later call can retry.
        std::lock_guard<std::mutex> lock(g_dev_mutex);
        if (!g_dev_ready[dev]) {
            DeviceInfo d;
            d.device = dev;
            if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
                cudaDeviceGetAttribute(&d.cc_minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess) {
                (void)cudaGetLastError();
                return FP8BS_ERR_CUDA;
            }
            fp8bs_status st = FP8BS_OK;
            if (d.cc_major != 10 || d.cc_minor != 3) {
                st = FP8BS_ERR_UNSUPPORTED_DEVICE;
            } else {
                d.runs = run_counters(dev);
                if (!d.runs)
                    return FP8BS_ERR_CUDA;
            }
            g_dev[dev] = d;
            g_dev_status[dev] = st;
            __atomic_store_n(&g_dev_ready[dev], true, __ATOMIC_RELEASE);
        }
    }
    *out = g_dev[dev];
    return g_dev_status[dev];
}

fp8bs_status ensure_smem_attr(const void *kernel, int bytes, int device, unsigned long long *done_mask)
{
    const unsigned long long bit = 1ull << device;
    if (__atomic_load_n(done_mask, __ATOMIC_ACQUIRE) & bit)
        return FP8BS_OK;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    __atomic_fetch_or(done_mask, bit, __ATOMIC_ACQ_REL);
    return FP8BS_OK;
}

fp8bs_status make_tmap_2d(CUtensorMap *map, const void *base, CUtensorMapDataType dtype, int elem_bytes,
                          uint64_t rows, uint64_t cols, uint64_t row_stride_bytes, uint32_t box_cols,
                          uint32_t box_rows, CUtensorMapSwizzle swizzle)
{
    std::call_once(g_encode_once, []() {
        void *fn = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        else
            (void)cudaGetLastError();
    });
    if (!g_encode)
        return FP8BS_ERR_CUDA;
    (void)elem_bytes;
    const cuuint64_t dims[2] = {cols, rows};
    const cuuint64_t strides[1] = {row_stride_bytes};
    const cuuint32_t box[2] = {box_cols, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    const CUresult r = g_encode(map, dtype, 2, const_cast<void *>(base), dims, strides, box, estr,
                                CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle,
                                CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? FP8BS_OK : FP8BS_ERR_CUDA;
}

WorkspaceLayout workspace_layout(const GemmShape &sh, int M, int K)
{
    auto up256 = [](size_t b) { return (b + 255) / 256 * 256; };
    WorkspaceLayout w;
    w.greedy_off = 256;
    w.counters_off = 1024;
    w.slots_off = w.counters_off + up256(static_cast<size_t>(sh.ttiles) * sh.ntiles * 4);
    w.act_off = w.slots_off + (sh.split ? static_cast<size_t>(2) * sh.ctas * sh.npad * 128 * 4 : 0);
    w.act_scale_off = w.act_off + up256(static_cast<size_t>(M) * K);
    w.total = w.act_scale_off + up256(static_cast<size_t>(M) * (K / 128) * 4);
    return w;
}

GemmShape gemm_shape(int mode, int M, int N, int K, int sms)
{
    GemmShape s{};
    s.m = M; // read by the fused route choice whatever the schedule below
    s.kg = mode == 2 ? K / 64 : K / 128;
    s.ntiles = (N + 127) / 128;
    s.units = static_cast<long long>(s.ntiles) * s.kg;
    s.npad = token_pad(M);
    s.ttiles = 1;
    s.split = true;
    if (M <= 64) {
        // Decode: the K dimension is split across every SM (stream-K).
        s.ctas = plan_ctas(s.units, sms);
        return s;
    }
    // Larger M.  The work units are (token tile, weight tile, K block), the
    // K block fastest.  With at least as many (token tile, weight tile) pairs
    // of 128 tokens as SMs, stream-K over all of them: every CTA gets the
    // same number of units and shares at most the two pairs at its ends.
    {
        const int tiles_m = (M + 127) / 128;
        if (static_cast<long long>(s.ntiles) * tiles_m >= sms) {
            s.npad = 128;
            s.ttiles = tiles_m;
            s.units = static_cast<long long>(s.ntiles) * tiles_m * s.kg;
            s.ctas = plan_ctas(s.units, sms);
            return s;
        }
    }
    // Fewer pairs than SMs.  One CTA per pair over the whole K (no split, no
    // exchange), with the widest token tile (at most 128) whose pairs fit in
    // one wave, pays off only when those pairs leave few SMs idle for the K
    // length: the idle fraction 1 - pairs/SMs must be at most 16/kg, i.e.
    // pairs * (kg + 16) >= SMs * kg.  Otherwise the idle SMs' share of the
    // bandwidth costs more than the K-split exchange.  Measured on GB300 in
    // chains of layers (M = 128 and 256): 7,168 x 5,120 runs 112 unsplit
    // pairs 3-5% faster than stream-K, while 5,120 x 17,408 (kg = 136) with
    // 80 unsplit pairs is 1.5-1.7x slower than stream-K.  The token tiles of
    // a weight tile read it from L2 after the first.  (256-token tiles
    // promote 15% slower per token than 128-token ones and are not used.)
    for (int tt : {128, 64, 32}) {
        if (mode == 3 && tt != 128)
            break; // MX: the token scale atoms hold 128-token tiles
        const int tiles_m = (M + tt - 1) / tt;
        const long long pairs = static_cast<long long>(s.ntiles) * tiles_m;
        if (pairs <= sms && pairs * (s.kg + 16) >= static_cast<long long>(sms) * s.kg) {
            s.npad = tt;
            s.ttiles = tiles_m;
            s.units = pairs * s.kg;
            s.ctas = static_cast<int>(pairs); // one pair per CTA
            s.split = false;
            return s;
        }
    }
    // Otherwise: stream-K over 128-token pairs.
    s.npad = 128;
    s.ttiles = (M + 127) / 128;
    s.units = static_cast<long long>(s.ntiles) * s.ttiles * s.kg;
    s.ctas = plan_ctas(s.units, sms);
    return s;
}

} // namespace fp8bs

using namespace fp8bs;

namespace {

// Shape limits common to the GEMMs.  Tile coordinates are 32-bit in the
// tensor maps and the kernels.
fp8bs_status check_gemm_shape(int M, int N, int K, int kmult)
{
    if (M < 1 || N < 1 || K < 1)
        return FP8BS_ERR_INVALID_ARG;
    if (M > kMaxTokens || K % kmult != 0 || N > (1 << 30) || K > (1 << 30))
        return FP8BS_ERR_UNSUPPORTED_SHAPE;
    return FP8BS_OK;
}

fp8bs_status check_flags(unsigned flags, unsigned allowed)
{
    return (flags & ~allowed) ? FP8BS_ERR_INVALID_ARG : FP8BS_OK;
}

constexpr unsigned kGemmFlags = FP8BS_FLAG_OVERLAP_PREV | FP8BS_FLAG_WEIGHTS_TILED;
constexpr unsigned kFusedFlags = kGemmFlags | FP8BS_FLAG_PROLOGUE_CAST; // the fused entry points

fp8bs_status quant_weight_common(const void *w, fp8bs_dtype wtype, int N, int K, uint8_t *wq, float *ws,
                                 bool tiled, void *stream)
{
    if (!w || !wq || !ws || N < 1 || K < 1 || (wtype != FP8BS_F32 && wtype != FP8BS_BF16))
        return FP8BS_ERR_INVALID_ARG;
    if (K % 128 != 0 || N > (1 << 30) || K > (1 << 30) ||
        static_cast<long long>((N + 127) / 128) * (K / 128) > 0x7FFFFFFFll)
        return FP8BS_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w, 16) || !aligned(wq, 16) || !aligned(ws, 4))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo dev;
    fp8bs_status st = current_device(&dev);
    if (st != FP8BS_OK)
        return st;
    return launch_quant_weight(w, wtype, N, K, wq, ws, tiled, static_cast<cudaStream_t>(stream), dev);
}

fp8bs_status gemm_workspace(int mode, int M, int N, int K, size_t *bytes, int sms = 0)
{
    if (sms <= 0) {
        DeviceInfo dev;
        fp8bs_status st = current_device(&dev);
        if (st != FP8BS_OK)
            return st;
        sms = dev.sms;
    }
    const GemmShape sh = gemm_shape(mode, M, N, K, sms);
    *bytes = workspace_layout(sh, M, K).total;
    return FP8BS_OK;
}

fp8bs_status run_gemm(GemmLaunch &L)
{
    DeviceInfo dev;
    fp8bs_status st = current_device(&dev);
    if (st != FP8BS_OK)
        return st;
    if (L.sms <= 0)
        L.sms = dev.sms;
    const GemmShape sh = gemm_shape(L.mode, L.M, L.N, L.K, L.sms);
    if (L.workspace_bytes < workspace_layout(sh, L.M, L.K).total)
        return FP8BS_ERR_WORKSPACE_TOO_SMALL;
    switch (L.mode) {
    case 0:
        return launch_gemm_fp8(L, dev);
    case 1:
        return launch_gemm_fused(L, dev);
    case 3:
        return launch_gemm_mx(L, dev);
    default:
        return launch_gemm_bf16(L, dev);
    }
}

} // namespace

extern "C" {

const char *fp8bs_status_string(fp8bs_status status)
{
    switch (status) {
    case FP8BS_OK:
        return "ok";
    case FP8BS_ERR_INVALID_ARG:
        return "invalid argument (null pointer, size below 1, ldx below K, or unknown flag/dtype)";
    case FP8BS_ERR_UNSUPPORTED_SHAPE:
        return "unsupported shape (GEMM M must be 1..512, 1..64 with the greedy choice, without a workspace or in "
               "the MX variant; K must be a multiple of 128, or 64 for the bf16 GEMM)";
    case FP8BS_ERR_MISALIGNED:
        return "misaligned pointer or row stride";
    case FP8BS_ERR_WORKSPACE_TOO_SMALL:
        return "workspace smaller than the size query returned";
    case FP8BS_ERR_UNSUPPORTED_DEVICE:
        return "unsupported device: this library runs only on compute capability 10.3 (sm_103)";
    case FP8BS_ERR_CUDA:
        return "a CUDA runtime or driver call failed";
    case FP8BS_ERR_DEVICE_TIMEOUT:
        return "a kernel gave up waiting inside its pipeline (device-side timeout)";
    }
    return "unknown status";
}

fp8bs_status fp8_quant_act(const void *x, int M, int K, int ldx, uint8_t *xq, float *xs, unsigned flags,
                           void *stream)
{
    if (!x || !xq || !xs || M < 1 || K < 1 || ldx < K)
        return FP8BS_ERR_INVALID_ARG;
    if (check_flags(flags, FP8BS_FLAG_OVERLAP_PREV) != FP8BS_OK)
        return FP8BS_ERR_INVALID_ARG;
    if (K % 128 != 0 || K > (1 << 30) || static_cast<long long>(M) * (K / 128) > (1ll << 34))
        return FP8BS_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(xq, 4) || !aligned(xs, 4))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo dev;
    fp8bs_status st = current_device(&dev);
    if (st != FP8BS_OK)
        return st;
    return launch_quant_act(x, M, K, ldx, xq, xs, (flags & FP8BS_FLAG_OVERLAP_PREV) != 0,
                            static_cast<cudaStream_t>(stream), dev);
}

fp8bs_status fp8_quant_weight_blocks(const void *w, fp8bs_dtype wtype, int N, int K, uint8_t *wq, float *ws,
                                     void *stream)
{
    return quant_weight_common(w, wtype, N, K, wq, ws, false, stream);
}

fp8bs_status fp8_quant_weight_blocks_tiled(const void *w, fp8bs_dtype wtype, int N, int K, uint8_t *wq,
                                           float *ws, void *stream)
{
    return quant_weight_common(w, wtype, N, K, wq, ws, true, stream);
}

fp8bs_status bf16_pack_weights_tiled(const void *w, int N, int K, void *wt, void *stream)
{
    if (!w || !wt || N < 1 || K < 1)
        return FP8BS_ERR_INVALID_ARG;
    if (K % 64 != 0 || N > (1 << 30) || K > (1 << 30) ||
        static_cast<long long>((N + 127) / 128) * (K / 64) > 0x7FFFFFFFll)
        return FP8BS_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w, 16) || !aligned(wt, 16))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo dev;
    fp8bs_status st = current_device(&dev);
    if (st != FP8BS_OK)
        return st;
    return launch_pack_bf16_tiled(w, N, K, wt, static_cast<cudaStream_t>(stream), dev);
}

fp8bs_status fp8_blockscaled_gemm_workspace_size(int M, int N, int K, size_t *bytes)
{
    if (!bytes)
        return FP8BS_ERR_INVALID_ARG;
    *bytes = 0;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    return gemm_workspace(0, M, N, K, bytes);
}

fp8bs_status bf16_gemm_ref_workspace_size(int M, int N, int K, size_t *bytes)
{
    if (!bytes)
        return FP8BS_ERR_INVALID_ARG;
    *bytes = 0;
    fp8bs_status st = check_gemm_shape(M, N, K, 64);
    if (st != FP8BS_OK)
        return st;
    return gemm_workspace(2, M, N, K, bytes);
}

fp8bs_status fp8_blockscaled_gemm(const uint8_t *aq, const float *as, const uint8_t *wq, const float *ws,
                                  void *y, int M, int N, int K, void *workspace, size_t workspace_bytes,
                                  unsigned flags, void *stream)
{
    if (!aq || !as || !wq || !ws || !y || !workspace)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    if (check_flags(flags, kGemmFlags) != FP8BS_OK)
        return FP8BS_ERR_INVALID_ARG;
    if (!aligned(aq, 16) || !aligned(wq, 16) || !aligned(as, 4) || !aligned(ws, 4) || !aligned(y, 2) ||
        !aligned(workspace, 256))
        return FP8BS_ERR_MISALIGNED;
    GemmLaunch L = {};
    L.mode = 0;
    L.M = M;
    L.N = N;
    L.K = K;
    L.a = aq;
    L.lda = K;
    L.as = as;
    L.w = wq;
    L.ws = ws;
    L.y = y;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.flags = flags;
    L.stream = static_cast<cudaStream_t>(stream);
    L.test_skip_unit = -1;
    L.timeout_ns = kDefaultTimeoutNs;
    return run_gemm(L);
}

fp8bs_status fp8_blockscaled_gemm_fused(const void *x, int ldx, const uint8_t *wq, const float *ws, void *y,
                                        int M, int N, int K, void *workspace, size_t workspace_bytes,
                                        unsigned flags, void *stream)
{
    if (!x || !wq || !ws || !y || !workspace)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    if (ldx < K || check_flags(flags, kFusedFlags) != FP8BS_OK)
        return FP8BS_ERR_INVALID_ARG;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(wq, 16) || !aligned(ws, 4) || !aligned(y, 2) ||
        !aligned(workspace, 256))
        return FP8BS_ERR_MISALIGNED;
    GemmLaunch L = {};
    L.mode = 1;
    L.M = M;
    L.N = N;
    L.K = K;
    L.a = x;
    L.lda = ldx;
    L.w = wq;
    L.ws = ws;
    L.y = y;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.flags = flags;
    L.stream = static_cast<cudaStream_t>(stream);
    L.test_skip_unit = -1;
    L.timeout_ns = kDefaultTimeoutNs;
    return run_gemm(L);
}

fp8bs_status fp8_blockscaled_gemm_fused_greedy(const void *x, int ldx, const uint8_t *wq, const float *ws,
                                               void *y, int M, int N, int K, int32_t *token, float *logit,
                                               void *workspace, size_t workspace_bytes, unsigned flags,
                                               void *stream)
{
    if (!x || !wq || !ws || !token || !workspace)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    if (M > 64)
        return FP8BS_ERR_UNSUPPORTED_SHAPE; // one greedy key per token, at most 64
    if (ldx < K || check_flags(flags, kFusedFlags) != FP8BS_OK)
        return FP8BS_ERR_INVALID_ARG;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(wq, 16) || !aligned(ws, 4) || !aligned(y, 2) ||
        !aligned(token, 4) || !aligned(logit, 4) || !aligned(workspace, 256))
        return FP8BS_ERR_MISALIGNED;
    GemmLaunch L = {};
    L.mode = 1;
    L.M = M;
    L.N = N;
    L.K = K;
    L.a = x;
    L.lda = ldx;
    L.w = wq;
    L.ws = ws;
    L.y = y;
    L.token = token;
    L.logit = logit;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.flags = flags;
    L.stream = static_cast<cudaStream_t>(stream);
    L.test_skip_unit = -1;
    L.timeout_ns = kDefaultTimeoutNs;
    return run_gemm(L);
}

fp8bs_status bf16_gemm_ref(const void *x, const void *w, void *y, int M, int N, int K, void *workspace,
                           size_t workspace_bytes, unsigned flags, void *stream)
{
    if (!x || !w || !y || !workspace)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_gemm_shape(M, N, K, 64);
    if (st != FP8BS_OK)
        return st;
    if (check_flags(flags, kGemmFlags) != FP8BS_OK)
        return FP8BS_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(w, 16) || !aligned(y, 2) || !aligned(workspace, 256))
        return FP8BS_ERR_MISALIGNED;
    GemmLaunch L = {};
    L.mode = 2;
    L.M = M;
    L.N = N;
    L.K = K;
    L.a = x;
    L.lda = K;
    L.w = w;
    L.y = y;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.flags = flags;
    L.stream = static_cast<cudaStream_t>(stream);
    L.test_skip_unit = -1;
    L.timeout_ns = kDefaultTimeoutNs;
    return run_gemm(L);
}

fp8bs_status fp8bs_workspace_status(void *workspace, int clear, int *code)
{
    if (!workspace || !code)
        return FP8BS_ERR_INVALID_ARG;
    *code = 0;
    unsigned word = 0;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(&word, workspace, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess) {
        (void)cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    *code = static_cast<int>(word);
    if (clear && word != 0) {
        const unsigned zero = 0;
        if (cudaMemcpy(workspace, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess) {
            (void)cudaGetLastError();
            return FP8BS_ERR_CUDA;
        }
    }
    return word ? FP8BS_ERR_DEVICE_TIMEOUT : FP8BS_OK;
}

fp8bs_status fp8bs_split_plan(int N, int K, int bf16, int num_sms, int cta, int *ctas, long long *units,
                              long long *unit_begin, long long *unit_end)
{
    if (!ctas || !units || N < 1 || K < 1)
        return FP8BS_ERR_INVALID_ARG;
    if (K % (bf16 ? 64 : 128) != 0)
        return FP8BS_ERR_UNSUPPORTED_SHAPE;
    int sms = num_sms;
    if (sms <= 0) {
        DeviceInfo dev;
        fp8bs_status st = current_device(&dev);
        if (st != FP8BS_OK)
            return st;
        sms = dev.sms;
    }
    const GemmShape sh = gemm_shape(bf16 ? 2 : 0, 1, N, K, sms);
    *ctas = sh.ctas;
    *units = sh.units;
    if (cta >= 0) {
        if (cta >= sh.ctas || !unit_begin || !unit_end)
            return FP8BS_ERR_INVALID_ARG;
        *unit_begin = plan_begin(sh.units, sh.ctas, cta);
        *unit_end = plan_begin(sh.units, sh.ctas, cta + 1);
    }
    return FP8BS_OK;
}

fp8bs_status fp8bs_gemm_schedule(int M, int N, int K, int num_sms, int *npad, int *token_tiles, int *ctas,
                                 long long *units, int *split)
{
    if (!npad || !token_tiles || !ctas || !units || !split)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    int sms = num_sms;
    if (sms <= 0) {
        DeviceInfo dev;
        st = current_device(&dev);
        if (st != FP8BS_OK)
            return st;
        sms = dev.sms;
    }
    const GemmShape sh = gemm_shape(0, M, N, K, sms);
    *npad = sh.npad;
    *token_tiles = sh.ttiles;
    *ctas = sh.ctas;
    *units = sh.units;
    *split = sh.split ? 1 : 0;
    return FP8BS_OK;
}

// ---------------------------------------------------------------- MX variant
fp8bs_status fp8_mx_quant_weights(const void *w, fp8bs_dtype wtype, int N, int K, uint8_t *wq, uint8_t *ws_atoms,
                                  void *stream)
{
    if (!w || !wq || !ws_atoms || N < 1 || K < 1 || (wtype != FP8BS_F32 && wtype != FP8BS_BF16))
        return FP8BS_ERR_INVALID_ARG;
    if (K % 128 != 0 || N > (1 << 30) || K > (1 << 30) ||
        static_cast<long long>((N + 127) / 128) * (K / 128) > 0x7FFFFFFFll)
        return FP8BS_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(w, 16) || !aligned(wq, 16) || !aligned(ws_atoms, 16))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo dev;
    fp8bs_status st = current_device(&dev);
    if (st != FP8BS_OK)
        return st;
    return launch_mx_quant_weights(w, wtype, N, K, wq, ws_atoms, static_cast<cudaStream_t>(stream), dev);
}

fp8bs_status fp8_mx_quant_act(const void *x, int M, int K, int ldx, uint8_t *xq, uint8_t *xs_atoms, unsigned flags,
                              void *stream)
{
    if (!x || !xq || !xs_atoms || M < 1 || K < 1 || ldx < K)
        return FP8BS_ERR_INVALID_ARG;
    if (check_flags(flags, FP8BS_FLAG_OVERLAP_PREV) != FP8BS_OK)
        return FP8BS_ERR_INVALID_ARG;
    if (M > kMaxTokens || K % 128 != 0 || K > (1 << 30))
        return FP8BS_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(xq, 16) || !aligned(xs_atoms, 16))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo dev;
    fp8bs_status st = current_device(&dev);
    if (st != FP8BS_OK)
        return st;
    return launch_mx_quant_act(x, M, K, ldx, xq, xs_atoms, (flags & FP8BS_FLAG_OVERLAP_PREV) != 0,
                               static_cast<cudaStream_t>(stream), dev);
}

fp8bs_status fp8_mx_gemm_workspace_size(int M, int N, int K, size_t *bytes)
{
    if (!bytes)
        return FP8BS_ERR_INVALID_ARG;
    *bytes = 0;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    return gemm_workspace(3, M, N, K, bytes);
}

fp8bs_status fp8_mx_gemm(const uint8_t *aq, const uint8_t *as_atoms, const uint8_t *wq, const uint8_t *ws_atoms,
                         void *y, int M, int N, int K, void *workspace, size_t workspace_bytes, unsigned flags,
                         void *stream)
{
    if (!aq || !as_atoms || !wq || !ws_atoms || !y || !workspace)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    if (check_flags(flags, FP8BS_FLAG_OVERLAP_PREV) != FP8BS_OK)
        return FP8BS_ERR_INVALID_ARG;
    if (!aligned(aq, 16) || !aligned(as_atoms, 16) || !aligned(wq, 16) || !aligned(ws_atoms, 16) ||
        !aligned(y, 2) || !aligned(workspace, 256))
        return FP8BS_ERR_MISALIGNED;
    GemmLaunch L = {};
    L.mode = 3;
    L.M = M;
    L.N = N;
    L.K = K;
    L.a = aq;
    L.lda = K;
    L.w = wq;
    L.sfa = ws_atoms;
    L.sfb = as_atoms;
    L.y = y;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.flags = flags | FP8BS_FLAG_WEIGHTS_TILED; // the MX weight codes are always tiled
    L.stream = static_cast<cudaStream_t>(stream);
    L.timeout_ns = kDefaultTimeoutNs;
    return run_gemm(L);
}

fp8bs_status fp8bs_fused_route(int M, int N, int K, int num_sms, unsigned flags, int *prologue)
{
    if (!prologue || check_flags(flags, kFusedFlags) != FP8BS_OK)
        return FP8BS_ERR_INVALID_ARG;
    *prologue = 0;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    int sms = num_sms;
    if (sms <= 0) {
        DeviceInfo dev;
        st = current_device(&dev);
        if (st != FP8BS_OK)
            return st;
        sms = dev.sms;
    }
    *prologue = fused_prologue_route(gemm_shape(1, M, N, K, sms), flags) ? 1 : 0;
    return FP8BS_OK;
}

} // extern "C"

// Test hook (declared in include/fp8bs_testing.h): the FP8 GEMM with the
// producer told never to fill the stage of unit `skip_unit` of every CTA, so
// the MMA warp's bounded wait on that stage runs out.  Used by the failure
// detection test to check that a time-out is reported through the status
// word and leaves the CUDA context usable.
extern "C" fp8bs_status fp8bs_testhook_gemm_stall(const uint8_t *aq, const float *as, const uint8_t *wq,
                                                  const float *ws, void *y, int M, int N, int K,
                                                  void *workspace, size_t workspace_bytes, int skip_unit,
                                                  unsigned long long timeout_ns, void *stream)
{
    if (!aq || !as || !wq || !ws || !y || !workspace || skip_unit < 0 || timeout_ns == 0 ||
        timeout_ns > 10ull * kDefaultTimeoutNs)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    if (!aligned(aq, 16) || !aligned(wq, 16) || !aligned(as, 4) || !aligned(ws, 4) || !aligned(y, 2) ||
        !aligned(workspace, 256))
        return FP8BS_ERR_MISALIGNED;
    GemmLaunch L = {};
    L.mode = 0;
    L.M = M;
    L.N = N;
    L.K = K;
    L.a = aq;
    L.lda = K;
    L.as = as;
    L.w = wq;
    L.ws = ws;
    L.y = y;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.flags = 0;
    L.stream = static_cast<cudaStream_t>(stream);
    L.test_skip_unit = skip_unit;
    L.timeout_ns = timeout_ns;
    return run_gemm(L);
}

// Test hooks (declared in include/fp8bs_testing.h): the fused layer with its
// schedule planned for another SM count, and the workspace that needs.
extern "C" fp8bs_status fp8bs_testhook_workspace_size_sms(int M, int N, int K, int num_sms, size_t *bytes)
{
    if (!bytes || num_sms < 1 || num_sms > 4096)
        return FP8BS_ERR_INVALID_ARG;
    *bytes = 0;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    return gemm_workspace(1, M, N, K, bytes, num_sms);
}

extern "C" fp8bs_status fp8bs_testhook_gemm_fused_sms(const void *x, int ldx, const uint8_t *wq, const float *ws,
                                                      void *y, int M, int N, int K, void *workspace,
                                                      size_t workspace_bytes, unsigned flags, int num_sms,
                                                      void *stream)
{
    if (!x || !wq || !ws || !y || !workspace || num_sms < 1 || num_sms > 4096)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    if (ldx < K || check_flags(flags, kFusedFlags) != FP8BS_OK)
        return FP8BS_ERR_INVALID_ARG;
    if (!aligned(x, 16) || ldx % 8 != 0 || !aligned(wq, 16) || !aligned(ws, 4) || !aligned(y, 2) ||
        !aligned(workspace, 256))
        return FP8BS_ERR_MISALIGNED;
    GemmLaunch L = {};
    L.mode = 1;
    L.M = M;
    L.N = N;
    L.K = K;
    L.a = x;
    L.lda = ldx;
    L.w = wq;
    L.ws = ws;
    L.y = y;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.flags = flags;
    L.stream = static_cast<cudaStream_t>(stream);
    L.test_skip_unit = -1;
    L.timeout_ns = kDefaultTimeoutNs;
    L.sms = num_sms;
    return run_gemm(L);
}

// Test hook (declared in include/fp8bs_testing.h): the pre-quantised GEMM
// with unit `bad_unit` of every CTA addressed one weight tile past the end.
// Only the FP8BS_DEBUG build accepts it; its device-side checks must catch
// the coordinate, skip the load and report FP8BS_ERR_DEVICE_TIMEOUT-class
// codes in the status word (the unfilled stage's wait then runs out after
// timeout_ns).  A coordinate past the end is safe even if a check missed
// it: the tensor load fills such rows with zeros.
extern "C" fp8bs_status fp8bs_testhook_debug_bad_tile(const uint8_t *aq, const float *as, const uint8_t *wq,
                                                     const float *ws, void *y, int M, int N, int K,
                                                     void *workspace, size_t workspace_bytes, int bad_unit,
                                                     unsigned long long timeout_ns, void *stream)
{
#ifndef FP8BS_DEBUG
    (void)aq, (void)as, (void)wq, (void)ws, (void)y, (void)M, (void)N, (void)K, (void)workspace;
    (void)workspace_bytes, (void)bad_unit, (void)timeout_ns, (void)stream;
    return FP8BS_ERR_INVALID_ARG; // the checks exist only in the FP8BS_DEBUG build
#else
    if (!aq || !as || !wq || !ws || !y || !workspace || bad_unit < 0 || timeout_ns == 0 ||
        timeout_ns > 10ull * kDefaultTimeoutNs)
        return FP8BS_ERR_INVALID_ARG;
    fp8bs_status st = check_gemm_shape(M, N, K, 128);
    if (st != FP8BS_OK)
        return st;
    if (!aligned(aq, 16) || !aligned(wq, 16) || !aligned(as, 4) || !aligned(ws, 4) || !aligned(y, 2) ||
        !aligned(workspace, 256))
        return FP8BS_ERR_MISALIGNED;
    GemmLaunch L = {};
    L.mode = 0;
    L.M = M;
    L.N = N;
    L.K = K;
    L.a = aq;
    L.lda = K;
    L.as = as;
    L.w = wq;
    L.ws = ws;
    L.y = y;
    L.workspace = workspace;
    L.workspace_bytes = workspace_bytes;
    L.flags = 0;
    L.stream = static_cast<cudaStream_t>(stream);
    L.test_bad_unit = bad_unit;
    L.timeout_ns = timeout_ns;
    return run_gemm(L);
#endif
}

// Whether this copy of the library was built with the device-side checks.
extern "C" int fp8bs_testhook_debug_build(void)
{
#ifdef FP8BS_DEBUG
    return 1;
#else
    return 0;
#endif
}
