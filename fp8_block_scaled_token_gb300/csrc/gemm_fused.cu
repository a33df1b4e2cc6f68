// gemm_fused.cu -- the FP8 GEMM with the activation cast fused into the
// kernel prologue.  When the CTA's activation slice does not fit the
// shared-memory cache (large M x K), the cast runs as its own kernel into the
// workspace and the pre-quantised GEMM follows on the same stream.
#include "gemm_launch.cuh"

namespace fp8bs {

bool fused_prologue_route(const GemmShape &sh, unsigned flags)
{
    return (flags & FP8BS_FLAG_PROLOGUE_CAST) != 0 && fused_cache_fits<kModeFp8Fused>(sh);
}

fp8bs_status launch_gemm_fused(const GemmLaunch &L, const DeviceInfo &dev)
{
    const GemmShape sh = gemm_shape(kModeFp8Fused, L.M, L.N, L.K, L.sms > 0 ? L.sms : dev.sms);
    if (fused_prologue_route(sh, L.flags))
        return launch_gemm_mode<kModeFp8Fused>(L, dev);
    const WorkspaceLayout wl = workspace_layout(sh, L.M, L.K);
    uint8_t *aq = static_cast<uint8_t *>(L.workspace) + wl.act_off;
    float *as = reinterpret_cast<float *>(static_cast<uint8_t *>(L.workspace) + wl.act_scale_off);
    fp8bs_status st = launch_quant_act(L.a, L.M, L.K, L.lda, aq, as, (L.flags & FP8BS_FLAG_OVERLAP_PREV) != 0,
                                       L.stream, dev);
    if (st != FP8BS_OK)
        return st;
    GemmLaunch G = L;
    G.mode = kModeFp8;
    G.a = aq;
    G.lda = L.K;
    G.as = as;
    G.flags = L.flags | FP8BS_FLAG_OVERLAP_PREV; // ordered after the cast by the dependency wait
    return launch_gemm_fp8(G, dev);
}

} // namespace fp8bs
