// gemm_fused.cu -- instantiation of the small-M GEMM for mode kModeFp8Fused.
#include "gemm_launch.cuh"

namespace fp8bs {

fp8bs_status launch_gemm_fused(const GemmLaunch &L, const DeviceInfo &dev)
{
    return launch_gemm_mode<kModeFp8Fused>(L, dev);
}

} // namespace fp8bs
