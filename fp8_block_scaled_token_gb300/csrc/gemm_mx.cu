// gemm_mx.cu -- instantiation of the small-M GEMM for mode kModeMx (E4M3
// operands with 1x32 power-of-two scales applied by the tensor core).
#include "gemm_launch.cuh"

namespace fp8bs {

fp8bs_status launch_gemm_mx(const GemmLaunch &L, const DeviceInfo &dev)
{
    return launch_gemm_mode<kModeMx>(L, dev);
}

} // namespace fp8bs
