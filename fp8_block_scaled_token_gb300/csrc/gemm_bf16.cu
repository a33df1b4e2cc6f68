// gemm_bf16.cu -- instantiation of the small-M GEMM for mode kModeBf16.
#include "gemm_launch.cuh"

namespace fp8bs {

fp8bs_status launch_gemm_bf16(const GemmLaunch &L, const DeviceInfo &dev)
{
    return launch_gemm_mode<kModeBf16>(L, dev);
}

} // namespace fp8bs
