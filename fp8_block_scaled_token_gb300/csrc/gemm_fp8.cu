// gemm_fp8.cu -- instantiation of the small-M GEMM for mode kModeFp8.
#include "gemm_launch.cuh"

namespace fp8bs {

fp8bs_status launch_gemm_fp8(const GemmLaunch &L, const DeviceInfo &dev)
{
    return launch_gemm_mode<kModeFp8>(L, dev);
}

} // namespace fp8bs
