// gemm_launch.cuh -- host launch of gemm_small_m_kernel for one mode; each
// gemm_*.cu translation unit instantiates it for its mode so the four token
// widths of the three modes compile in parallel.
#pragma once

#include "gemm_kernel.cuh"
#include "internal.h"

namespace fp8bs {

constexpr int kSmemLimit = 227 * 1024;      // dynamic shared memory per CTA
constexpr int kRingBudget = 200 * 1024;     // ring of a kernel that has the SM to itself
constexpr int kSharedRingBudget = 100 * 1024; // ring of a kernel that runs two CTAs per SM
constexpr int kActCacheBudget = 96 * 1024;  // fused: activation cache + scales
// fused, FP8BS_FLAG_PROLOGUE_CAST: the prologue cast is taken only up to this
// many (K block, token) rows per CTA.  It can only start once the previous
// kernel has produced the activations, and every CTA repeats it for its own
// K blocks, while the separate kernel casts each row once and the GEMM
// (two CTAs per SM at 16 tokens) streams weights meanwhile.  Measured on
// GB300, the separate cast was the faster route for every shape tried, from
// 2 to 88 rows per CTA (5,120^2 at M = 8: 13.9 us with the prologue, 11.9 us
// without; 1 to 16 tokens, 2 to 16 rows: 3-10 % in chains), hence opt-in.
constexpr int kPrologueMaxRows = 16;

// Ring depth and activation-cache size of a launch; act_chunks < 0 means the
// fused kernel's cache would not fit (the caller then quantises separately).
template <int NPAD, int MODE>
void gemm_smem_plan(const GemmShape &sh, int &stages, int &act_chunks, bool greedy = false)
{
    using C = GemmCfg<NPAD, MODE>;
    const int ybytes = greedy ? 0 : C::kYStageBytes;
    act_chunks = 0;
    int ring = C::kMinBlocks == 2 ? kSharedRingBudget : kRingBudget;
    if (MODE == kModeFp8Fused) {
        const long long per_cta = (sh.units + sh.ctas - 1) / sh.ctas;
        act_chunks = static_cast<int>(per_cta < sh.kg ? per_cta : sh.kg);
        if (act_chunks * (C::kBBytes + C::kActScaleBytes) > kActCacheBudget ||
            act_chunks * sh.m > kPrologueMaxRows) {
            act_chunks = -1;
            stages = 0;
            return;
        }
        ring = kSmemLimit - C::smem_bytes(0, act_chunks, 0);
    }
    if (ybytes > 0 && ring > kSmemLimit - C::smem_bytes(0, 0, ybytes))
        ring = kSmemLimit - C::smem_bytes(0, 0, ybytes); // room for the Y staging tile
    stages = ring / C::kStageBytes;
    if (stages > C::kMaxStages)
        stages = C::kMaxStages;
}

template <int NPAD, int MODE, bool GREEDY>
fp8bs_status launch_gemm_npad(const GemmLaunch &L, const DeviceInfo &dev, const GemmShape &sh)
{
    using C = GemmCfg<NPAD, MODE>;
    static unsigned long long attr_done = 0;
    auto kernel = gemm_small_m_kernel<NPAD, MODE, GREEDY>;
    int stages = 0, act_chunks = 0;
    gemm_smem_plan<NPAD, MODE>(sh, stages, act_chunks, GREEDY);
    if (act_chunks < 0 || stages < 2)
        return FP8BS_ERR_UNSUPPORTED_SHAPE; // not reached: the fused launcher checks first
    if ((NPAD == 16 || MODE == kModeFp8Fused || GREEDY) && sh.ttiles != 1)
        return FP8BS_ERR_UNSUPPORTED_SHAPE; // not reached: these serve one token tile only
    const int smem = C::smem_bytes(stages, act_chunks, GREEDY ? 0 : C::kYStageBytes);
    fp8bs_status st = ensure_smem_attr(reinterpret_cast<const void *>(kernel), kSmemLimit, dev.device, &attr_done);
    if (st != FP8BS_OK)
        return st;

    CUtensorMap tm_w, tm_b;
    const bool tiled = (L.flags & FP8BS_FLAG_WEIGHTS_TILED) != 0;
    // Tiled weights are addressed as a [ntiles * kg * 128 rows][128 bytes] matrix.
    const uint64_t tiled_rows = static_cast<uint64_t>(sh.ntiles) * sh.kg * 128;
    if (MODE == kModeBf16) {
        if (tiled)
            st = make_tmap_2d(&tm_w, L.w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, tiled_rows, 64, 128, 64, 128);
        else
            st = make_tmap_2d(&tm_w, L.w, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(L.N),
                              static_cast<uint64_t>(L.K), static_cast<uint64_t>(L.K) * 2, 64, 128);
        if (st == FP8BS_OK)
            st = make_tmap_2d(&tm_b, L.a, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(L.M),
                              static_cast<uint64_t>(L.K), static_cast<uint64_t>(L.lda) * 2, 64, NPAD);
    } else {
        if (tiled)
            st = make_tmap_2d(&tm_w, L.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, tiled_rows, 128, 128, 128, 128);
        else
            st = make_tmap_2d(&tm_w, L.w, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(L.N),
                              static_cast<uint64_t>(L.K), static_cast<uint64_t>(L.K), 128, 128);
        if (st == FP8BS_OK) {
            if (MODE == kModeFp8 || MODE == kModeMx)
                st = make_tmap_2d(&tm_b, L.a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, static_cast<uint64_t>(L.M),
                                  static_cast<uint64_t>(L.K), static_cast<uint64_t>(L.lda), 128, NPAD);
            else
                tm_b = tm_w; // unused by the fused kernel
        }
    }
    if (st != FP8BS_OK)
        return st;
    // Y by TMA store (plain FP8 and MX layers): the tensor map needs a
    // 16-byte aligned base and a row pitch that is a multiple of 16 bytes;
    // otherwise the epilogue stores rows itself.
    CUtensorMap tm_y = tm_w; // not read unless y_tma
    int y_tma = 0;
    if (C::kYTma && !GREEDY && L.y != nullptr && reinterpret_cast<uintptr_t>(L.y) % 16 == 0 && L.N % 8 == 0) {
        st = make_tmap_2d(&tm_y, L.y, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, static_cast<uint64_t>(L.M),
                          static_cast<uint64_t>(L.N), static_cast<uint64_t>(L.N) * 2, C::kTileRows, NPAD,
                          CU_TENSOR_MAP_SWIZZLE_NONE);
        if (st != FP8BS_OK)
            return st;
        y_tma = 1;
    }

    const WorkspaceLayout wl = workspace_layout(sh, L.M, L.K);
    uint8_t *wsb = static_cast<uint8_t *>(L.workspace);
    GemmParams p;
    p.M = L.M;
    p.N = L.N;
    p.K = L.K;
    p.kg = sh.kg;
    p.ntiles = sh.ntiles;
    p.ttiles = sh.ttiles;
    p.units = sh.units;
    p.ctas = sh.ctas;
    p.stages = stages;
    p.act_chunks = act_chunks;
    p.as = L.as;
    p.ws = L.ws;
    p.sfa = L.sfa;
    p.sfb = L.sfb;
    p.x = static_cast<const uint16_t *>(MODE == kModeFp8Fused ? L.a : nullptr);
    p.ldx = L.lda;
    p.y = static_cast<uint16_t *>(L.y);
    p.status = reinterpret_cast<unsigned *>(wsb);
    p.counters = reinterpret_cast<unsigned *>(wsb + wl.counters_off);
    p.slots = reinterpret_cast<float *>(wsb + wl.slots_off);
    p.prefetch_before_wait = (L.flags & FP8BS_FLAG_OVERLAP_PREV) ? 1 : 0;
    p.w_tiled = tiled ? 1 : 0;
    p.y_tma = y_tma;
    p.test_skip_unit = L.test_skip_unit;
    p.test_bad_unit = L.test_bad_unit;
    p.timeout_ns = L.timeout_ns;
    p.token = L.token;
    p.logit = L.logit;
    p.best = reinterpret_cast<unsigned long long *>(wsb + wl.greedy_off);
    p.done = reinterpret_cast<unsigned *>(wsb + wl.greedy_off + 64 * 8);
    p.runs = dev.runs;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(sh.ctas), 1, 1);
    cfg.blockDim = dim3(C::kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = L.stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = (L.flags & FP8BS_FLAG_OVERLAP_PREV) ? 1 : 0;
    return launch_status(cudaLaunchKernelEx(&cfg, kernel, tm_w, tm_b, tm_y, p));
}

// True when the fused kernel's activation cache fits for this shape.
template <int MODE> bool fused_cache_fits(const GemmShape &sh)
{
    int stages = 0, act_chunks = 0;
    if (sh.m > 64 || sh.ttiles > 1)
        return false; // the prologue cast serves one token tile of at most 64
    switch (sh.npad) {
    case 16:
        gemm_smem_plan<16, MODE>(sh, stages, act_chunks);
        break;
    case 32:
        gemm_smem_plan<32, MODE>(sh, stages, act_chunks);
        break;
    case 48:
        gemm_smem_plan<48, MODE>(sh, stages, act_chunks);
        break;
    default:
        gemm_smem_plan<64, MODE>(sh, stages, act_chunks);
        break;
    }
    return act_chunks >= 0 && stages >= 2;
}

template <int MODE, bool GREEDY>
fp8bs_status launch_gemm_greedy(const GemmLaunch &L, const DeviceInfo &dev, const GemmShape &sh)
{
    // 128-token tiles exist for the plain (non-fused, non-greedy) GEMMs and
    // MX only; the callers reject larger M before they get here.
    if constexpr (MODE != kModeFp8Fused && !GREEDY) {
        if (sh.npad == 128)
            return launch_gemm_npad<128, MODE, GREEDY>(L, dev, sh);
    }
    switch (sh.npad) {
    case 16:
        return launch_gemm_npad<16, MODE, GREEDY>(L, dev, sh);
    case 32:
        return launch_gemm_npad<32, MODE, GREEDY>(L, dev, sh);
    case 48:
        return launch_gemm_npad<48, MODE, GREEDY>(L, dev, sh);
    case 64:
        return launch_gemm_npad<64, MODE, GREEDY>(L, dev, sh);
    default:
        return FP8BS_ERR_UNSUPPORTED_SHAPE;
    }
}

// The greedy instantiations compile in their own translation unit (gemm_greedy.cu).
extern template fp8bs_status launch_gemm_greedy<kModeFp8, true>(const GemmLaunch &, const DeviceInfo &,
                                                                const GemmShape &);
extern template fp8bs_status launch_gemm_greedy<kModeFp8Fused, true>(const GemmLaunch &, const DeviceInfo &,
                                                                     const GemmShape &);

template <int MODE>
fp8bs_status launch_gemm_mode(const GemmLaunch &L, const DeviceInfo &dev)
{
    const GemmShape sh = gemm_shape(MODE, L.M, L.N, L.K, L.sms > 0 ? L.sms : dev.sms);
    if constexpr (MODE == kModeFp8 || MODE == kModeFp8Fused) {
        if (L.token != nullptr)
            return launch_gemm_greedy<MODE, true>(L, dev, sh);
    }
    return launch_gemm_greedy<MODE, false>(L, dev, sh);
}

} // namespace fp8bs
