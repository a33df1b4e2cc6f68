// runs.cu -- per-device launch counters of the library's kernels.
//
// Every kernel adds one to its slot when it starts, so a test can check,
// inside the running process, that the kernel it meant to exercise is the
// one that ran ("The profiler said the kernel ran zero times", "Why it never
// ran").  The counters live in one file-scope device array; kernels of other
// translation units receive its device address as a parameter.
#include <mutex>

#include "fp8bs_testing.h"
#include "internal.h"

namespace fp8bs {
namespace {

__device__ __align__(256) unsigned long long g_runs[FP8BS_RUNS_SLOTS];

constexpr int kMaxDev = 64;
std::mutex g_runs_mutex;
unsigned long long *g_runs_ptr[kMaxDev];

} // namespace

unsigned long long *run_counters(int device)
{
    if (device < 0 || device >= kMaxDev)
        return nullptr;
    std::lock_guard<std::mutex> lock(g_runs_mutex);
    if (!g_runs_ptr[device]) {
        // The array's name is a host-side stand-in; the device address comes
        // from the runtime, for the device that is current now.
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_runs) != cudaSuccess) {
            (void)cudaGetLastError();
            return nullptr; // not latched: a later call may retry
        }
        g_runs_ptr[device] = static_cast<unsigned long long *>(p);
    }
    return g_runs_ptr[device];
}

} // namespace fp8bs

using namespace fp8bs;

extern "C" fp8bs_status fp8bs_testhook_kernel_runs(int first, int count, unsigned long long *out)
{
    if (!out || first < 0 || count < 1 || first > FP8BS_RUNS_SLOTS - count)
        return FP8BS_ERR_INVALID_ARG;
    DeviceInfo dev;
    fp8bs_status st = current_device(&dev);
    if (st != FP8BS_OK)
        return st;
    if (!dev.runs)
        return FP8BS_ERR_CUDA;
    if (cudaDeviceSynchronize() != cudaSuccess ||
        cudaMemcpy(out, dev.runs + first, sizeof(unsigned long long) * count, cudaMemcpyDeviceToHost) !=
            cudaSuccess) {
        (void)cudaGetLastError();
        return FP8BS_ERR_CUDA;
    }
    return FP8BS_OK;
}
