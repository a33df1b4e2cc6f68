// noalloc.cu -- fp8_blockscaled_gemm_fused_noalloc: the fused layer for
// callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc at all: code that runs inside a CUDA
// graph capture that must not allocate, allocator-less embedded runtimes,
// hooks that execute while an outer framework holds its own memory pool
// locked.  They cannot provide the workspace that fp8_blockscaled_gemm_fused
// needs for its split-K partials and arrival counters.  This entry point uses
// a scratch array that lives in the library itself instead, so the caller
// passes only inputs and outputs.
//
// The scratch is a file-scope __device__ array of kNoallocScratchBytes; every
// GPU that loads the library holds it until the process exits.  Host code may
// not use the array's name as a device address, so its address is looked up
// once per device, with that device current, by cudaGetSymbolAddress and
// handed to the kernels.
#include <mutex>

#include "internal.h"

namespace fp8bs {
namespace {

constexpr size_t kNoallocScratchBytes = 12u << 20; // 12 MiB

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoallocScratchBytes];

constexpr int kMaxDev = 64;
std::mutex g_scratch_mutex;
void *g_scratch_ptr[kMaxDev];

// Device address of the scratch array on `device` (the current device), or
// an error.  A failed lookup is not remembered, so a later call retries.
cudaError_t scratch_address(int device, void **out)
{
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (!g_scratch_ptr[device]) {
        void *ptr = nullptr;
        const cudaError_t e = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
        if (e != cudaSuccess)
            return e;
        if (!ptr)
            return cudaErrorInvalidSymbol;
        g_scratch_ptr[device] = ptr;
    }
    *out = g_scratch_ptr[device];
    return cudaSuccess;
}

} // namespace
} // namespace fp8bs

using namespace fp8bs;

extern "C" fp8bs_status fp8_blockscaled_gemm_fused_noalloc(const void *x, int ldx, const uint8_t *wq,
                                                           const float *ws, void *y, int M, int N, int K,
                                                           unsigned flags, void *stream)
{
    if (!x || !wq || !ws || !y || M < 1 || N < 1 || K < 1 || ldx < K)
        return FP8BS_ERR_INVALID_ARG;
    if (flags & ~(FP8BS_FLAG_OVERLAP_PREV | FP8BS_FLAG_WEIGHTS_TILED | FP8BS_FLAG_PROLOGUE_CAST))
        return FP8BS_ERR_INVALID_ARG;
    if (M > 64 || K % 128 != 0 || N > (1 << 30) || K > (1 << 30))
        return FP8BS_ERR_UNSUPPORTED_SHAPE;
    auto misaligned = [](const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) != 0; };
    if (misaligned(x, 16) || ldx % 8 != 0 || misaligned(wq, 16) || misaligned(ws, 4) || misaligned(y, 2))
        return FP8BS_ERR_MISALIGNED;
    DeviceInfo dev;
    fp8bs_status st = current_device(&dev);
    if (st != FP8BS_OK)
        return st;
    if (dev.device < 0 || dev.device >= kMaxDev)
        return FP8BS_ERR_CUDA;
    constexpr int kFused = 1; // the fused mode of the GEMM kernel
    const GemmShape sh = gemm_shape(kFused, M, N, K, dev.sms);
    const WorkspaceLayout wl = workspace_layout(sh, M, K);
    if (wl.total > kNoallocScratchBytes)
        return FP8BS_ERR_UNSUPPORTED_SHAPE; // needs more scratch than the library holds

    void *scratch = nullptr;
    cudaError_t e = scratch_address(dev.device, &scratch);
    if (e != cudaSuccess)
        return launch_status(e);

    // The status word and arrival counters must start at zero; the array
    // keeps whatever the previous call left there.
    const cudaStream_t s = static_cast<cudaStream_t>(stream);
    e = cudaMemsetAsync(scratch, 0, wl.slots_off, s);
    if (e != cudaSuccess)
        return launch_status(e);

    GemmLaunch L = {};
    L.mode = kFused;
    L.M = M;
    L.N = N;
    L.K = K;
    L.a = x;
    L.lda = ldx;
    L.w = wq;
    L.ws = ws;
    L.y = y;
    L.workspace = scratch;
    L.workspace_bytes = kNoallocScratchBytes;
    L.flags = flags;
    L.stream = s;
    L.test_skip_unit = -1;
    L.timeout_ns = kDefaultTimeoutNs;
    L.sms = dev.sms;
    return launch_gemm_fused(L, dev);
}
