// gemm_greedy.cu -- the GEMM kernels with the greedy-choice epilogue, for
// both FP8 modes, compiled apart from the plain ones so the build stays
// parallel.
#include "gemm_launch.cuh"

namespace fp8bs {

template fp8bs_status launch_gemm_greedy<kModeFp8, true>(const GemmLaunch &, const DeviceInfo &, const GemmShape &);
template fp8bs_status launch_gemm_greedy<kModeFp8Fused, true>(const GemmLaunch &, const DeviceInfo &,
                                                              const GemmShape &);

} // namespace fp8bs
