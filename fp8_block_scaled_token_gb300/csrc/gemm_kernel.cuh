// gemm_kernel.cuh -- swap-AB, K-split GEMM for small M on sm_103a.
//
// Y[M,N] = dequant(Aq[M,K]) . dequant(Wq[N,K])^T with W in 128x128 fp32
// block scales and A in 1x128 fp32 group scales ("A 23% faster GPU kernel, and
// a model that did not move", "Why this shape is hard"), plus the same
// pipeline for the 16-bit output-layer baseline ("The profiler said the kernel
// ran zero times", "The output layer, which did run").
//
// Work is cut into units of one 128-wide K block of one (token tile, weight
// tile) pair; each CTA takes a contiguous range of units (stream-K), so a
// pair may be split across CTAs and is then summed in a fixed order.
//
// Design (warp-specialised; two CTAs per SM for the 16-token tile):
//   warp 0      TMA producer: streams 128-row x 128-byte weight tiles (and,
//               when the activations are pre-quantised or bf16, the token
//               tile of the same K block) into an S-stage shared-memory ring,
//               128-byte swizzled, no multicast.
//   warp 1      MMA issuer: per 128-wide K block, four tcgen05.mma with the
//               weights as the 128-row A operand and the tokens (padded to
//               NPAD = 16/32/48/64/128) as the B operand, fp32 accumulator in
//               tensor memory (8 buffers for the 16-token tile, 4 otherwise,
//               so the epilogue rarely stalls it; 2 whole-segment sums for
//               the MX 128-token tile).
//   warps 2-5   promotion / epilogue (warps 2-9 from 64 tokens, two groups
//               splitting the token columns): one thread per weight row reads
//               its accumulator row (tcgen05.ld), multiplies by
//               s_w[tile,kb] * s_a[m,kb] and adds into fp32 registers; at the
//               end of a pair it stores bf16 Y (the 128-token tile through a
//               shared-memory tile and one TMA store where Y's alignment
//               allows), or hands its partial to the
//               fixed-order K-split reduction (whose last contributor gathers
//               the partials, by bulk copy into the idle ring from 32 tokens
//               up).
//   greedy (optional, the output layer): while storing a finished tile the
//               epilogue warps also pick, per token, the tile's largest bf16
//               logit (lowest column on ties); each CTA folds its tiles in
//               shared memory and publishes one 64-bit key per token with a
//               device-scope atomic max, and the last CTA to finish writes
//               the chosen columns and clears the keys for the next call.
//   fused only: warps 2-9 first quantise, in the kernel prologue, the token
//               rows of every K block this CTA will use into an activation
//               cache in shared memory (E4M3 codes in the swizzled B-operand
//               layout, plus the per-token scales).  The ring then carries
//               weights only, and the MMA reads its B operand from the cache.
//
// Shared memory: [1 KB barriers and flags][ring: S stages][Y staging tile
// (128-token tile)][activation cache][activation scales][per-warp scale
// products]; S and the cache size are chosen per launch.
//
// Every wait is bounded; on time-out the CTA records a code in the status
// word, drains what it has in flight, frees its tensor memory and returns.
#pragma once

#include <cuda_bf16.h>
#include <type_traits>

#include "fp8bs_testing.h"
#include "plan.cuh"
#include "ptx.cuh"
#include "quant_math.cuh"


// Columns per TMEM load in the promotion step: 32 where the token columns are
// split over two epilogue groups (64 tokens and up), the next 32 in flight
// while the first are promoted (decode pass at 128 / 512 tokens 1.0 / 1.7 %
// faster than four 16-column loads each with its own wait; the same pipeline
// over 16-column loads gained nothing, one 64-column load per unit lost:
// 180 -> 204 ns of promotion per unit at 128 tokens); 64 for a single group
// of 128 columns, 32 where the columns allow, else 16.
#define FP8BS_TMEM_LD_COLS(cols, groups)                                                                     \
    (((groups) != 1) ? 32 : ((cols) >= 128) ? 64 : ((cols) % 32 == 0) ? 32 : 16)

namespace fp8bs {

enum GemmMode : int {
    kModeFp8 = 0,      // pre-quantised activations (Aq, s_a) read by TMA
    kModeFp8Fused = 1, // bf16 activations quantised in the kernel prologue
    kModeBf16 = 2,     // bf16 x bf16, no block scales
    kModeMx = 3,       // E4M3 x E4M3 with one UE8M0 scale per 32 K per row, applied by the tensor core
};

struct GemmParams {
    int M, N, K;
    int kg;          // K blocks per tile (K/128 for FP8, K/64 for bf16)
    int ntiles;      // ceil(N / 128) weight tiles
    int ttiles;      // token tiles
    long long units; // token tiles * ntiles * kg: unit u is K block u % kg of
                     // pair u / kg = (token tile, weight tile), weight tile fastest
    int ctas;
    int stages;      // ring depth, <= kMaxStages
    int act_chunks;  // fused: K blocks in the activation cache (>= distinct K blocks of any CTA)
    const float *as;         // FP8: s_a [M][K/128] (M <= 16) or [K/128][M] (M > 16)
    const float *ws;         // FP8: s_w [ntiles][K/128]
    const uint8_t *sfa;      // MX: weight scale atoms [ntiles][K/128][512]
    const uint8_t *sfb;      // MX: activation scale atoms [K/128][512]
    const uint16_t *x;       // fused: bf16 activations [M][ldx]
    int ldx;
    uint16_t *y;             // bf16 [M][N]
    unsigned *status;        // workspace word 0
    unsigned *counters;      // [ntiles] arrival counters, zero between calls
    float *slots;            // [2 * ctas][NPAD * 128] fp32 partials
    int prefetch_before_wait;// weights may be fetched before the previous grid completes
    int w_tiled;             // weights in the tiled layout (one contiguous 16 KB run per tile)
    int y_tma;               // Y tiles leave through shared memory and a TMA store
    int test_skip_unit;      // -1, or a unit whose stage the producer never fills
    int test_bad_unit;       // -1, or a unit the producer addresses one weight tile past the end
                             // (the FP8BS_DEBUG build's checks must catch it)
    unsigned long long timeout_ns;
    // greedy token choice (kernels instantiated with GREEDY only)
    int *token;                  // [M] chosen column per token
    float *logit;                // [M] its logit, or nullptr
    unsigned long long *best;    // workspace: [64] keys, zero between calls
    unsigned *done;              // workspace: CTAs finished, zero between calls
    unsigned long long *runs;    // per-device launch counters (slot per instantiation)
};

// Order-preserving 32-bit key of a finite float (larger value, larger key;
// +0 and -0 get the same key).  Key 0 is below every finite value.
__device__ __forceinline__ uint32_t logit_key(float v)
{
    uint32_t b = __float_as_uint(v);
    if (b == 0x80000000u)
        b = 0u;
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t k)
{
    return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

template <int NPAD, int MODE> struct GemmCfg {
    static_assert((NPAD % 16 == 0 && NPAD >= 16 && NPAD <= 64) || NPAD == 128 || NPAD == 256, "token tile");
    static constexpr int kTileRows = 128;                   // weight rows per tile (MMA M)
    static constexpr int kRowBytes = 128;                   // K bytes per row per unit
    static constexpr int kChunkElems = MODE == kModeBf16 ? 64 : 128;
    static constexpr int kWBytes = kTileRows * kRowBytes;   // 16 KB
    static constexpr int kBBytes = NPAD * kRowBytes;        // 2..32 KB token tile
    // MX: the stage also carries the unit's two 512-byte scale-factor atoms
    // (weights, tokens), copied into tensor memory by the MMA thread.
    static constexpr bool kMx = MODE == kModeMx;
    static constexpr int kSfBytes = kMx ? 1024 : 0;
    static constexpr int kStageBytes = kWBytes + (MODE == kModeFp8Fused ? 0 : kBBytes) + kSfBytes;
    // bf16 and MX accumulate a whole tile segment in tensor memory (no
    // per-K-block scale to apply on CUDA cores).
    static constexpr bool kTileAcc = MODE == kModeBf16 || kMx;
    static constexpr int kMaxStages = 12;
    // Accumulators in tensor memory (512 fp32 columns per SM, two CTAs of
    // the 16-token tile sharing them): eight for the 16-token tile, so the
    // MMA runs up to eight units ahead of an epilogue that stalls (for
    // instance ~1.3 us on a release-ordered arrival issued while every SM
    // streams weights); four otherwise.  Measured on the decode pass (two
    // libraries alternating in one process, three boxes): eight against four
    // 1.2-1.6 % faster at M = 1 and 8; sixteen 0.3 % slower than eight; eight
    // for the 32- to 64-token tiles within +-0.7 % (not taken).
    // (MX at 128 tokens: two, each a whole tile segment's sum, so that they
    // and the scale-factor columns fit the 512 columns.)
    static constexpr int kAcc = NPAD == 16 ? 8 : (NPAD == 256 || (MODE == kModeMx && NPAD == 128)) ? 2 : 4;
    // MX: after the accumulators, 8 columns of scale factors per ring stage
    // (4 for the weight atom, 4 for the token atom).
    static constexpr int kSfCol = kAcc * NPAD;
    static constexpr int kTmemNeed = kAcc * NPAD + (kMx ? kMaxStages * 8 : 0);
    static_assert(kTmemNeed <= 512, "tensor memory has 512 columns");
    static constexpr int kTmemCols =
        kTmemNeed <= 32 ? 32 : kTmemNeed <= 64 ? 64 : kTmemNeed <= 128 ? 128 : kTmemNeed <= 256 ? 256 : 512;
    static constexpr int kQuantWarps = MODE == kModeFp8Fused ? 4 : 0;
    // Up to 16 tokens the non-fused kernels run two CTAs per SM (a ~100 KB
    // ring each): the next GEMM's CTA, launched early by programmatic
    // dependent launch, then shares the SM and streams its weights while this
    // one finishes.  Measured on GB300 this beats one CTA per SM with a
    // 200 KB ring for every layer shape of the workloads at M <= 16.  At
    // M = 32 and 48 it loses by 5% and 11% over a whole decode pass (cast
    // kernels included), although it wins by 2-5% in a chain of
    // pre-quantised layers.
    static constexpr int kMinBlocks = (MODE != kModeFp8Fused && NPAD == 16) ? 2 : 1;
    // From 64 tokens up the columns of a token tile are split over two groups
    // of four epilogue warps: twice the threads promote each unit, which the
    // wider tiles need more than a second resident CTA (measured in a chain
    // of layers: 64-token tiles 7-16% faster than with one group, 128-token
    // tiles 1-13%), and a thread keeps at most 128 accumulators in registers.
    static constexpr int kColGroups = NPAD >= 64 ? 2 : 1;
    static constexpr int kCols = NPAD / kColGroups;         // token columns per epilogue thread
    static constexpr int kEpiWarps = 4 * kColGroups;
    // From 32 tokens up, the per-unit scale products s_w * s_a[m] of a
    // warp's token columns are formed by the warp itself (each lane one or
    // two tokens, their scales one coalesced load apiece from the
    // K-block-major activation scales) into its own shared-memory slot and
    // read back four per load, which removes a shuffle and a multiply per
    // token per weight row.  A __syncwarp publishes them: no barrier across
    // the epilogue warps in the per-unit loop (measured against products
    // formed once per token and published by such a barrier: 128-token tiles
    // 6-11% faster per layer, 32- and 64-token tiles 2%).  The 16-token tile
    // (decode) keeps the per-lane scales and shuffles: there the extra
    // shared-memory round trip on the per-unit critical path cost ~0.2 us.
    // The activation-scale layout goes with M: token-major [M][K/128] up to
    // 16 tokens, K-block-major [K/128][M] above (the cast writes it so); the
    // schedule gives exactly those M the 16-token tile, so each
    // instantiation reads one fixed layout (a run-time choice in this loop
    // cost 3 % at decode sizes).
    static constexpr bool kProducts = NPAD >= 32 && !kTileAcc;
    static constexpr int kProdPerLane = (kCols + 31) / 32; // token columns per lane
    static constexpr int kProdBytes = kProducts ? kEpiWarps * 2 * kCols * 4 : 0; // per warp, by unit parity
    static constexpr int kThreads = 32 * (2 + kEpiWarps + kQuantWarps);
    // Registers per thread.  An SM's register file is four 16,384-register
    // banks, one per scheduler, and a CTA's warps are spread over the four:
    // with W resident warps a bank holds ceil(W / 4) of them, so a thread may
    // have at most 16,384 / (32 * ceil(W / 4)) (rounded down to 8, at most
    // 255).  With two CTAs per SM the cap is lower, 160: next to two GEMM
    // CTAs (three 5,120-register warps per bank) the activation cast's
    // 4-warp CTA (one 1,024-register warp per bank at 32 registers) still
    // fits, so the next GEMM's early CTA is not kept off an SM where a cast
    // CTA landed (decode pass 5.31 -> 5.27 ms at M = 8).
    static constexpr int kWarpsPerBank = (kMinBlocks * (kThreads / 32) + 3) / 4;
    static constexpr int kRegSplit = (16384 / (32 * kWarpsPerBank)) & ~7;
    static constexpr int kMaxRegs = kMinBlocks == 2 ? 160 : kRegSplit > 255 ? 255 : kRegSplit;
    static_assert(kMaxRegs <= kRegSplit || kRegSplit > 255, "the CTAs must fit in the register file");
    // Plain FP8 and MX layers (not the greedy output layer): a finished Y
    // tile (128 weight rows x NPAD tokens, bf16) is staged in shared memory as
    // [token][row] and written by one TMA store, instead of up to 64
    // two-byte stores per thread (1.7 us per whole tile at 512 tokens, the
    // promotion's time for ~10 units; on the last contributor's critical path
    // below 128 tokens).  For the 128-token tile the 32 KB cost the ring its
    // sixth stage (1.5 % on its own); the 16-token tile's 4 KB fit beside
    // its two CTAs' rings.  Net, decode pass: 1 / 4 / 8 / 16 tokens 0.4 /
    // 0.4 / 0.9 / 1.5 % faster, 32 / 48 / 64 tokens 1.9 / 2.4 / 1.5 %, 128 /
    // 256 / 512 tokens 2.0-2.2 %.
    static constexpr bool kYTma = MODE == kModeFp8 || MODE == kModeMx;
    static constexpr int kYStageBytes = kYTma ? kTileRows * NPAD * 2 : 0;
    static constexpr int kHeader = 1024;                    // barriers and flags
    // the mbarriers, the TMEM address and two flags end below the greedy keys at 512
    static_assert((2 * kMaxStages + 2 * kAcc + 3) * 8 + 12 <= 512, "header layout");
    static constexpr int kMmaSteps = kRowBytes / 32;        // 32 bytes of K per tcgen05.mma
    static constexpr int kActScaleBytes = NPAD * 4;         // per cached K block
    static constexpr uint32_t kIdesc =
        MODE == kModeBf16 ? idesc_bf16_f32(kTileRows, NPAD) : idesc_e4m3_f32(kTileRows, NPAD);
    static_assert(kStageBytes % 1024 == 0 && kBBytes % 1024 == 0, "swizzle atoms must stay 1024-byte aligned");

    // Dynamic shared memory of a launch (+1024 for aligning the base).
    // (ystage_bytes: kYStageBytes, or 0 for an instantiation that does not stage Y)
    static constexpr int smem_bytes(int stages, int act_chunks, int ystage_bytes)
    {
        return 1024 + kHeader + stages * kStageBytes + ystage_bytes + act_chunks * (kBBytes + kActScaleBytes) +
               kProdBytes;
    }
};

// GREEDY: the greedy-choice epilogue is compiled in (a separate instantiation,
// so the plain layer carries none of its code).
template <int NPAD, int MODE, bool GREEDY>
__global__ void __maxnreg__((GemmCfg<NPAD, MODE>::kMaxRegs))
    gemm_small_m_kernel(const __grid_constant__ CUtensorMap tm_w, const __grid_constant__ CUtensorMap tm_b,
                        const __grid_constant__ CUtensorMap tm_y, const GemmParams p)
{
    using C = GemmCfg<NPAD, MODE>;
    static_assert(!GREEDY || NPAD <= 64, "the greedy choice keeps one key per token for at most 64 tokens");
    static_assert(MODE != kModeFp8Fused || NPAD <= 64, "the fused cast serves at most 64 tokens");
    static_assert(MODE != kModeMx || ((NPAD <= 64 || NPAD == 128) && !GREEDY),
                  "the MX layer: tiles of up to 64 tokens, or 128-token tiles (whose atoms hold 128 tokens)");
    // Instantiations that only ever run one token tile (the 16-token decode
    // tile, the fused cast and the greedy choice serve at most 64 tokens):
    // pair index == weight tile, and no token-tile stepping is compiled in.
    constexpr bool kOneTT = NPAD == 16 || MODE == kModeFp8Fused || GREEDY;
    constexpr bool kYStage = C::kYTma && !GREEDY; // Y through the staging tile and TMA
    // Under programmatic dependent launch the next grid is released once
    // this CTA's producer has six weight loads left to issue, not at its
    // start: the next layer's CTAs then fetch their first ring pass while this
    // grid finishes instead of while it streams (decode pass, M = 1 to 64:
    // 0.2-0.9 % faster than a release at the start; a release after the last
    // load was 4 % slower at M = 16, three loads early 0.6 % slower there).
    constexpr int kTriggerLead = 6;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t *smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    uint64_t *empty = full + C::kMaxStages;
    uint64_t *tfull = empty + C::kMaxStages;
    uint64_t *tempty = tfull + C::kAcc;
    uint64_t *mma_done = tempty + C::kAcc;
    uint64_t *act_ready = mma_done + 1;
    uint64_t *red_ready = act_ready + 1; // bulk copies of the exchange slots (last segment)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(red_ready + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    volatile int *last_flag = abort_flag + 1;
    unsigned long long *cta_best = reinterpret_cast<unsigned long long *>(smem + 512); // [64] greedy keys
    const int S = p.stages;
    uint8_t *ring = smem + C::kHeader;
    uint16_t *ystage = reinterpret_cast<uint16_t *>(ring + S * C::kStageBytes); // [NPAD][128] bf16
    uint8_t *act_cache = ring + S * C::kStageBytes + (kYStage ? C::kYStageBytes : 0);
    float *act_scale = reinterpret_cast<float *>(act_cache + p.act_chunks * C::kBBytes);
    float *prod = act_scale + p.act_chunks * NPAD; // [epilogue warp][2][kCols] s_w * s_a

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = blockIdx.x;
    const long long u0 = plan_begin(p.units, p.ctas, cta);
    const int nunits = static_cast<int>(plan_begin(p.units, p.ctas, cta + 1) - u0);
    const int kg = p.kg;
    // The CTA's units cover the cyclic run of K blocks starting at kb0; the
    // activation-cache slot of its i-th unit is i mod kg.
    const int kb0 = static_cast<int>(u0 % kg);

    if (threadIdx.x == 0) {
        if (blockIdx.x == 0)
            atomicAdd(p.runs + FP8BS_RUNS_GEMM(MODE, NPAD, GREEDY ? 1 : 0), 1ull); // this instantiation ran
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int a = 0; a < C::kAcc; ++a) {
            mbar_init(&tfull[a], 1);
            mbar_init(&tempty[a], C::kEpiWarps);
        }
        mbar_init(mma_done, 1);
        mbar_init(act_ready, 1);
        mbar_init(red_ready, 1);
        *abort_flag = 0;
        *last_flag = 0;
    }
    if (threadIdx.x < 64)
        cta_best[threadIdx.x] = 0ull;
    if (threadIdx.x == 0) {
        fence_mbar_init();
        fence_proxy_async_smem();
    }
    if (warp == 0 && lane == 0) {
        prefetch_tmap(&tm_w);
        if (MODE != kModeFp8Fused)
            prefetch_tmap(&tm_b);
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, C::kTmemCols);
        tmem_relinquish();
    }
    if (MODE == kModeFp8Fused) {
        // Token rows >= M of every cached B tile, and their scales, stay zero.
        const int n16 = p.act_chunks * ((C::kBBytes + C::kActScaleBytes) / 16);
        for (int i = threadIdx.x; i < n16; i += C::kThreads)
            reinterpret_cast<uint4 *>(act_cache)[i] = make_uint4(0, 0, 0, 0);
    }
    tc_fence_before_sync();
    __syncthreads();
    tc_fence_after_sync();
    const uint32_t tmem_base = *tmem_slot;

    if (warp == 0) {
        // ------------------------------------------------ TMA producer
        if (lane == 0) {
            const uint64_t pol_w = l2_policy_evict_first();
            const uint64_t pol_b = l2_policy_evict_last();
            const uint32_t tx = C::kStageBytes;
            uint32_t armed_mask = 0, armed_parity = 0;
            const int pre = p.prefetch_before_wait ? (nunits < S ? nunits : S) : 0;
            // Per-unit state (K block, weight tile, first token row) advances
            // by increments from the CTA's first unit: no divisions in these
            // single-thread loops, whose latency sets the issue rate.
            const int pair_first = static_cast<int>(u0 / kg);
            const int wt_first = kOneTT ? pair_first : pair_first % p.ntiles;
            const int trow_first = kOneTT ? 0 : (pair_first / p.ntiles) * NPAD;
            int kb = kb0, wt = wt_first, trow = trow_first;
            auto step = [&](int &k, int &w, int &t) {
                if (++k == kg) {
                    k = 0;
                    ++w;
                    if (!kOneTT && w == p.ntiles) {
                        w = 0;
                        t += NPAD;
                    }
                }
            };
            // Coordinates of one unit's loads lie inside their tensors (the
            // FP8BS_DEBUG build checks them; weight rows past N are zero-filled).
            auto unit_ok = [&](int stage, int k, int w, int t) {
                return FP8BS_CHECK(stage >= 0 && stage < S && S <= C::kMaxStages && k >= 0 && k < kg && w >= 0 &&
                                   w < p.ntiles && t >= 0 && t < p.M);
            };
#ifdef FP8BS_DEBUG
            // test hook: unit test_bad_unit addresses one tile past the last
            auto bad = [&](int i, int w) { return i == p.test_bad_unit ? p.ntiles : w; };
#else
            auto bad = [](int, int w) { return w; };
#endif
            // Weights for the first ring pass, possibly before the previous grid is done.
            for (int i = 0; i < pre; ++i, step(kb, wt, trow)) {
                if (i == p.test_skip_unit || !unit_ok(i, kb, bad(i, wt), trow))
                    continue;
                mbar_arrive_expect_tx(&full[i], tx);
                armed_mask |= 1u << i;
                const int wb = bad(i, wt);
                const int wx = p.w_tiled ? 0 : kb * C::kChunkElems;
                const int wy = p.w_tiled ? (wb * kg + kb) * C::kTileRows : wb * C::kTileRows;
                tma_load_2d(ring + i * C::kStageBytes, &tm_w, &full[i], wx, wy, pol_w);
                if constexpr (C::kMx)
                    bulk_load_1d(ring + i * C::kStageBytes + C::kWBytes + C::kBBytes,
                                 p.sfa + (static_cast<long long>(wt) * kg + kb) * 512, 512, &full[i], pol_w);
            }
            grid_dependency_wait();
            if (MODE != kModeFp8Fused) {
                int kb_b = kb0, wt_b = wt_first, trow_b = trow_first;
                for (int i = 0; i < pre; ++i, step(kb_b, wt_b, trow_b)) {
                    if (i == p.test_skip_unit || !(armed_mask & (1u << i)))
                        continue;
                    tma_load_2d(ring + i * C::kStageBytes + C::kWBytes, &tm_b, &full[i], kb_b * C::kChunkElems,
                                trow_b, pol_b);
                    if constexpr (C::kMx) // token atoms [128-token tile][K block]
                        bulk_load_1d(ring + i * C::kStageBytes + C::kWBytes + C::kBBytes + 512,
                                     p.sfb + (static_cast<long long>(trow_b / 128) * kg + kb_b) * 512, 512, &full[i],
                                     pol_b);
                }
            }
            int s = pre % S;
            uint32_t ph = static_cast<uint32_t>(pre / S) & 1u;
            bool triggered = false;
            for (int i = pre; i < nunits; ++i) {
                if (!triggered && i >= nunits - kTriggerLead) {
                    grid_launch_dependents();
                    triggered = true;
                }
                if (!mbar_wait(&empty[s], ph ^ 1u, abort_flag, p.status, kErrTimeoutProducer, p.timeout_ns))
                    break;
                if (i != p.test_skip_unit && unit_ok(s, kb, bad(i, wt), trow)) {
                    mbar_arrive_expect_tx(&full[s], tx);
                    armed_mask |= 1u << s;
                    armed_parity = (armed_parity & ~(1u << s)) | (ph << s);
                    const int wb = bad(i, wt);
                    const int wx = p.w_tiled ? 0 : kb * C::kChunkElems;
                    const int wy = p.w_tiled ? (wb * kg + kb) * C::kTileRows : wb * C::kTileRows;
                    tma_load_2d(ring + s * C::kStageBytes, &tm_w, &full[s], wx, wy, pol_w);
                    if (MODE != kModeFp8Fused)
                        tma_load_2d(ring + s * C::kStageBytes + C::kWBytes, &tm_b, &full[s], kb * C::kChunkElems,
                                    trow, pol_b);
                    if constexpr (C::kMx) {
                        uint8_t *sf = ring + s * C::kStageBytes + C::kWBytes + C::kBBytes;
                        bulk_load_1d(sf, p.sfa + (static_cast<long long>(wt) * kg + kb) * 512, 512, &full[s], pol_w);
                        bulk_load_1d(sf + 512, p.sfb + (static_cast<long long>(trow / 128) * kg + kb) * 512, 512,
                                     &full[s], pol_b);
                    }
                }
                if (++s == S) {
                    s = 0;
                    ph ^= 1u;
                }
                step(kb, wt, trow);
            }
            if (!triggered)
                grid_launch_dependents(); // every weight load of this CTA is issued
            // Nothing may still be landing in shared memory when the CTA exits:
            // wait (bounded) for the last phase armed on every stage.
            for (int s = 0; s < S; ++s) {
                if (!(armed_mask & (1u << s)))
                    continue;
                const uint32_t ph = (armed_parity >> s) & 1u;
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_test(&full[s], ph)) {
                    if (globaltimer_ns() - t0 > p.timeout_ns) {
                        atomicOr(p.status, kErrTimeoutDrain);
                        break;
                    }
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------ MMA issuer
        if (lane == 0) {
            int acc = 0;
            uint32_t acc_ph = 0;
            bool ok = true;
            if (MODE == kModeFp8Fused)
                ok = mbar_wait(act_ready, 0, abort_flag, p.status, kErrTimeoutMma, p.timeout_ns);
            int s = 0, kb = kb0, slot = 0;
            uint32_t ph = 0;
            for (int i = 0; ok && i < nunits; ++i) {
                if (i > 0) {
                    if (++s == S) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++kb == kg)
                        kb = 0;
                    if (++slot == kg)
                        slot = 0;
                }
                const bool seg_start = (i == 0) || (kb == 0);
                const bool seg_end = (i == nunits - 1) || (kb == kg - 1);
                // FP8: every K block gets a fresh accumulator (its scale differs);
                // bf16: one accumulator per tile segment.
                const bool fresh = !C::kTileAcc || seg_start;
                const bool publish = !C::kTileAcc || seg_end;
                if (fresh && !mbar_wait(&tempty[acc], acc_ph ^ 1u, abort_flag, p.status, kErrTimeoutMma,
                                        p.timeout_ns))
                    break;
                if (!mbar_wait(&full[s], ph, abort_flag, p.status, kErrTimeoutMma, p.timeout_ns))
                    break;
                if (MODE == kModeFp8Fused && !FP8BS_CHECK(slot < p.act_chunks))
                    break;
                tc_fence_after_sync();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * NPAD);
                const uint64_t a_desc = sw128_kmajor_desc(smem_u32(ring + s * C::kStageBytes));
                const uint8_t *b_tile = MODE == kModeFp8Fused ? act_cache + slot * C::kBBytes
                                                              : ring + s * C::kStageBytes + C::kWBytes;
                const uint64_t b_desc = sw128_kmajor_desc(smem_u32(b_tile));
                if constexpr (C::kMx) {
                    // this unit's scale factors to tensor memory (per-stage
                    // columns: the copy is ordered before the MMAs below,
                    // and a stage's columns are rewritten only after the
                    // MMAs that read them have completed)
                    const uint32_t sf = tmem_base + static_cast<uint32_t>(C::kSfCol + s * 8);
                    const uint32_t sf_smem = smem_u32(ring + s * C::kStageBytes + C::kWBytes + C::kBBytes);
                    tmem_cp_sf_atom(sf, sf_atom_desc(sf_smem));
                    tmem_cp_sf_atom(sf + 4, sf_atom_desc(sf_smem + 512));
#pragma unroll
                    for (int k = 0; k < C::kMmaSteps; ++k)
                        mma_mxf8f6f4(d_tmem, a_desc + 2 * k, b_desc + 2 * k,
                                     idesc_mx_e4m3(C::kTileRows, NPAD, static_cast<uint32_t>(k), static_cast<uint32_t>(k)),
                                     sf, sf + 4, (k > 0 || !fresh) ? 1u : 0u);
                } else {
#pragma unroll
                    for (int k = 0; k < C::kMmaSteps; ++k) {
                        const uint32_t accumulate = (k > 0 || !fresh) ? 1u : 0u;
                        if (MODE == kModeBf16)
                            mma_f16(d_tmem, a_desc + 2 * k, b_desc + 2 * k, C::kIdesc, accumulate);
                        else
                            mma_f8f6f4(d_tmem, a_desc + 2 * k, b_desc + 2 * k, C::kIdesc, accumulate);
                    }
                }
                mma_commit(&empty[s]);
                if (publish) {
                    mma_commit(&tfull[acc]);
                    if (++acc == C::kAcc) {
                        acc = 0;
                        acc_ph ^= 1u;
                    }
                }
            }
            // Every MMA this thread issued must be complete before the
            // tensor memory is released.
            mma_commit(mma_done);
            const uint64_t t0 = globaltimer_ns();
            while (!mbar_test(mma_done, 0)) {
                if (globaltimer_ns() - t0 > p.timeout_ns) {
                    atomicOr(p.status, kErrTimeoutDrain);
                    break;
                }
            }
        }
    } else {
        if constexpr (MODE == kModeFp8Fused) {
            grid_dependency_wait();
            // -------------------------------------------- prologue: activation cast
            // Warps 2-9 quantise every (cached K block, token) row once: item
            // j = chunk * M + m, eight consecutive items per warp at a time so
            // their loads, reductions and divisions overlap.
            const int qw = warp - 2;
            constexpr int kQW = C::kEpiWarps + C::kQuantWarps;
            const int total = p.act_chunks * p.M;
            // Items go round-robin over the warps (item j to warp j % kQW), and
            // each warp takes its items eight at a time.  First ask for every
            // row this warp will read to be brought into L1.
            for (int j = qw + kQW * lane; j < total; j += kQW * 32) {
                const int c = j / p.M, m = j - c * p.M;
                const int kbj = kb0 + c < kg ? kb0 + c : kb0 + c - kg;
                const uint16_t *row_ptr = p.x + static_cast<long long>(m) * p.ldx + kbj * 128;
                prefetch_l1(row_ptr);
                prefetch_l1(row_ptr + 64);
            }
            // One batch: this warp's items j0, j0 + kQW, ... (n of them; n == 8
            // except in the last batch).  Full batches take a straight-line
            // path so the eight items' loads, reductions and conversions
            // overlap; only the tail guards each item.
            auto cast_batch = [&](int j0, int n, auto full_batch) {
                constexpr bool kFull = decltype(full_batch)::value;
                uint2 raw[8];
                int cs[8], ms[8];
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    const int j = j0 + b * kQW;
                    cs[b] = j / p.M;
                    ms[b] = j - cs[b] * p.M;
                    raw[b] = make_uint2(0u, 0u);
                    if (kFull || b < n) {
                        const int kbj = kb0 + cs[b] < kg ? kb0 + cs[b] : kb0 + cs[b] - kg;
                        if (FP8BS_CHECK(ms[b] >= 0 && ms[b] < p.M && kbj >= 0 && kbj < kg))
                            raw[b] = *reinterpret_cast<const uint2 *>(p.x + static_cast<long long>(ms[b]) * p.ldx +
                                                                      kbj * 128 + lane * 4);
                    }
                }
                float v[8][4], am[8];
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    v[b][0] = bf16_lo(raw[b].x);
                    v[b][1] = bf16_hi(raw[b].x);
                    v[b][2] = bf16_lo(raw[b].y);
                    v[b][3] = bf16_hi(raw[b].y);
                    am[b] = warp_max(abs_max4(v[b][0], v[b][1], v[b][2], v[b][3]));
                }
#pragma unroll
                for (int b = 0; b < 8; ++b) {
                    if ((kFull || b < n) && FP8BS_CHECK(cs[b] >= 0 && cs[b] < p.act_chunks && ms[b] < NPAD)) {
                        const int m = ms[b];
                        const float sc = group_scale(am[b]);
                        const uint32_t codes = quantize4(v[b][0], v[b][1], v[b][2], v[b][3], sc);
                        // row m, bytes 4*lane..4*lane+3 of its 128-byte row; the
                        // 16-byte chunk index is XOR-ed with (row mod 8) as TMA's
                        // 128-byte swizzle does.
                        const uint32_t off = static_cast<uint32_t>(m * 128 + ((((lane >> 2) ^ (m & 7)) & 7) << 4) +
                                                                   ((lane & 3) << 2));
                        *reinterpret_cast<uint32_t *>(act_cache + cs[b] * C::kBBytes + off) = codes;
                        if (lane == 0)
                            act_scale[cs[b] * NPAD + m] = sc;
                    }
                }
            };
            const int mine = total > qw ? (total - qw + kQW - 1) / kQW : 0; // items of this warp
            for (int t = 0; t < mine; t += 8) {
                const int j0 = qw + t * kQW;
                if (t + 8 <= mine)
                    cast_batch(j0, 8, std::true_type{});
                else
                    cast_batch(j0, mine - t, std::false_type{});
            }
            fence_proxy_async_smem(); // codes are read by the tensor core
            named_bar_sync(2, 32 * kQW);
            if (warp == 2 && lane == 0)
                mbar_arrive(act_ready);
        }
        if (warp < 2 + C::kEpiWarps) {
            // -------------------------------------------- promotion / epilogue
            const int quarter = warp & 3;             // TMEM lanes this warp may read
            const int row = quarter * 32 + lane;      // weight row within the tile
            const uint32_t lane_addr = static_cast<uint32_t>(quarter * 32) << 16;
            // This thread's token columns: col0.. of the token tile, tokens
            // tok0.. of the layer (per pair); mcnt of them exist (may exceed kCols).
            const int col0 = ((warp - 2) >> 2) * C::kCols;
            const int pair_start = static_cast<int>(u0 / kg);
            int wt = kOneTT ? pair_start : pair_start % p.ntiles;  // weight tile
            int ttile = kOneTT ? 0 : pair_start / p.ntiles;        // token tile
            int tok0 = ttile * NPAD + col0;
            int mcnt = p.M - tok0;
            float *const slots_y = p.slots;
            unsigned *const counters_y = p.counters;
            float acc[C::kCols];
#pragma unroll
            for (int m = 0; m < C::kCols; ++m)
                acc[m] = 0.0f;
            int accb = 0;
            uint32_t acc_ph = 0;
            int seg_first_kb = 0;
            bool bulk_issued = false; // warp 2 lane 0: slot copies into the ring
            int tile = static_cast<int>(u0 / kg), kb = kb0, slot = 0;
            // Reduction plans of the (at most two) tiles this CTA may share:
            // the tile its range starts in and the one it ends in.  Worked out
            // once here, off the critical path, so the end-of-tile exchange
            // does no 64-bit division.  Contributors are the consecutive CTAs
            // c_first..c_last; each uses slot 2c, except that c_first uses
            // 2c+1 when its range began in an earlier tile.
            struct SplitPlan {
                int c_first, c_last, slot_first;
            };
            auto make_plan = [&](int t) {
                const long long tf = static_cast<long long>(t) * kg;
                SplitPlan sp;
                sp.c_first = plan_owner(p.units, p.ctas, tf);
                sp.c_last = plan_owner(p.units, p.ctas, tf + kg - 1);
                sp.slot_first = 2 * sp.c_first + (plan_begin(p.units, p.ctas, sp.c_first) == tf ? 0 : 1);
                return sp;
            };
            const int tile_a = tile;
            const int tile_b = static_cast<int>((u0 + nunits - 1) / kg);
            const SplitPlan plan_a = make_plan(tile_a);
            const SplitPlan plan_b = tile_b != tile_a ? make_plan(tile_b) : plan_a;
            // Final values of weight row n for every token: round to bf16,
            // store Y (when asked for) and fold the greedy choice.
            auto finish_row = [&](int n) {
                const bool in_n = n < p.N;
#pragma unroll
                for (int m = 0; m < C::kCols; ++m) {
                    if (m < mcnt) {
                        const __nv_bfloat16 h = __float2bfloat16_rn(acc[m]);
                        if (in_n && p.y != nullptr)
                            p.y[static_cast<long long>(tok0 + m) * p.N + n] = __bfloat16_as_ushort(h);
                        if constexpr (GREEDY) {
                            const uint32_t key = in_n ? logit_key(__bfloat162float(h)) : 0u;
                            const uint32_t kmax = __reduce_max_sync(0xffffffffu, key);
                            const uint32_t nmin =
                                __reduce_min_sync(0xffffffffu, key == kmax ? static_cast<uint32_t>(n) : 0xffffffffu);
                            if (lane == 0)
                                atomicMax(&cta_best[col0 + m],
                                          (static_cast<unsigned long long>(kmax) << 32) | (0xffffffffu - nmin));
                        }
                    }
                }
            };
            // Final values of the tile (weight tile wt, token tile ttile): by TMA
            // from the staging tile where the launch set it up, else per row.
            // Every epilogue warp calls it (it holds named barriers).
            bool y_pending = false; // warp 2 lane 0: a TMA store may still read the staging tile
            auto store_y = [&](int n) {
                if constexpr (kYStage) {
                    if (p.y_tma) {
                        if (warp == 2 && lane == 0 && y_pending)
                            bulk_wait_read_all(); // the previous tile's store is done with the buffer
                        named_bar_sync(1, 32 * C::kEpiWarps);
#pragma unroll
                        for (int m = 0; m < C::kCols; ++m)
                            ystage[(col0 + m) * C::kTileRows + row] = __bfloat16_as_ushort(__float2bfloat16_rn(acc[m]));
                        fence_proxy_async_smem(); // generic writes, read by the TMA unit
                        named_bar_sync(1, 32 * C::kEpiWarps);
                        if (warp == 2 && lane == 0 && FP8BS_CHECK(wt >= 0 && wt < p.ntiles && ttile >= 0 && ttile < p.ttiles)) {
                            tma_store_2d(&tm_y, ystage, wt * C::kTileRows, ttile * NPAD); // rows >= M, cols >= N clipped
                            bulk_commit_group();
                            y_pending = true;
                        }
                        return;
                    }
                }
                finish_row(n);
            };
            // Scales of the next unit to promote, loaded one unit ahead by
            // every lane for its token columns col0 + lane + 32 q of the tile
            // (the activation scales are K-block-major above 16 tokens: the
            // lanes' loads are consecutive words).
            float nx_sw = 0.0f, nx_sa[C::kProdPerLane];
#pragma unroll
            for (int q = 0; q < C::kProdPerLane; ++q)
                nx_sa[q] = 0.0f;
            auto load_scales = [&](int wtl, int ttl, int kbb, int sl) {
                if (!FP8BS_CHECK(wtl >= 0 && wtl < p.ntiles && kbb >= 0 && kbb < kg &&
                                 (MODE != kModeFp8Fused || (sl >= 0 && sl < p.act_chunks))))
                    return;
                nx_sw = p.ws[static_cast<long long>(wtl) * kg + kbb];
#pragma unroll
                for (int q = 0; q < C::kProdPerLane; ++q) {
                    const int t = col0 + lane + 32 * q; // column within the token tile
                    const bool col_ok = lane + 32 * q < C::kCols;
                    if (MODE == kModeFp8) {
                        // 32 tokens and wider: M > 16, K-block-major scales
                        const int tok = ttl * NPAD + t;
                        nx_sa[q] = (col_ok && tok < p.M) ? p.as[static_cast<long long>(kbb) * p.M + tok] : 0.0f;
                    } else {
                        nx_sa[q] = col_ok ? act_scale[sl * NPAD + t] : 0.0f; // zero for rows >= M
                    }
                }
            };
            float *const wprod = prod + (warp - 2) * 2 * C::kCols; // this warp's [2][kCols]
            // 16-token tile: the weight-block scale of the next unit and
            // (pre-quantised activations) each lane's token scale, loaded one
            // unit ahead so no global load sits between a finished MMA and
            // its promotion.
            constexpr bool kLaneScales = !C::kProducts && !C::kTileAcc;
            float nx16_sw = 1.0f, nx16_sa = 0.0f;
            auto load_scales16 = [&](int wtl, int kbb) {
                if (!FP8BS_CHECK(wtl >= 0 && wtl < p.ntiles && kbb >= 0 && kbb < kg))
                    return;
                nx16_sw = p.ws[static_cast<long long>(wtl) * kg + kbb];
                if (MODE == kModeFp8 && lane < mcnt)
                    nx16_sa = p.as[static_cast<long long>(tok0 + lane) * kg + kbb]; // M <= 16: token-major
            };
            // Everything above is local set-up (split plans, unit state); the
            // first read of data the previous grid may write comes next, so
            // the dependency wait sits here (decode layer 11.57 -> 11.32 us).
            if constexpr (MODE != kModeFp8Fused)
                grid_dependency_wait();
            if (C::kProducts && nunits > 0)
                load_scales(wt, ttile, kb, slot);
            if (kLaneScales && nunits > 0)
                load_scales16(wt, kb);
            for (int i = 0; i < nunits; ++i) {
                if (i > 0) {
                    if (++kb == kg) {
                        kb = 0;
                        ++tile;
                        ++wt;
                        if (!kOneTT && wt == p.ntiles) {
                            wt = 0;
                            ++ttile;
                            tok0 += NPAD;
                            mcnt -= NPAD;
                        }
                    }
                    if (++slot == kg)
                        slot = 0;
                }
                const bool seg_start = (i == 0) || (kb == 0);
                const bool seg_end = (i == nunits - 1) || (kb == kg - 1);
                if (seg_start)
                    seg_first_kb = kb;
                if (!C::kTileAcc || seg_end) {
                    // Each lane forms s_w * s_a of its token columns for this
                    // unit from the scales it loaded one unit ahead, and
                    // loads the next unit's; the __syncwarp publishes the
                    // warp's products (double-buffered by unit parity: a
                    // buffer is rewritten only after every lane has passed
                    // the next unit's __syncwarp).
                    float *pr = wprod + (i & 1) * C::kCols;
                    if constexpr (C::kProducts) {
#pragma unroll
                        for (int q = 0; q < C::kProdPerLane; ++q)
                            if (lane + 32 * q < C::kCols)
                                pr[lane + 32 * q] = nx_sw * nx_sa[q];
                        __syncwarp();
                        if (i + 1 < nunits) {
                            const bool wrap = kb + 1 == kg;
                            const bool wrap_w = !kOneTT && wrap && wt + 1 == p.ntiles;
                            load_scales(wrap ? (wrap_w ? 0 : wt + 1) : wt, wrap_w ? ttile + 1 : ttile, wrap ? 0 : kb + 1,
                                        slot + 1 == kg ? 0 : slot + 1);
                        }
                    }
                    // 16-token tile: each lane holds the scale of token `lane`
                    // (pre-quantised) and shuffles it to the others.
                    float sw = 1.0f, sa_l = 0.0f;
                    if constexpr (kLaneScales) {
                        sw = nx16_sw;
                        sa_l = nx16_sa;
                        if (i + 1 < nunits)
                            load_scales16(kb + 1 == kg ? wt + 1 : wt, kb + 1 == kg ? 0 : kb + 1);
                    }
                    const bool slot_ok = MODE != kModeFp8Fused || FP8BS_CHECK(slot >= 0 && slot < p.act_chunks);
                    const float *sa_c = act_scale + (MODE == kModeFp8Fused && slot_ok ? slot * NPAD : 0) + col0;
                    mbar_wait(&tfull[accb], acc_ph, abort_flag, p.status, kErrTimeoutEpilogue, p.timeout_ns);
                    // No barrier here: a thread whose wait gave up
                    // (abort) carries on through the remaining units and the
                    // exchange with whatever the accumulator holds: every
                    // later wait gives up after its next look at the abort
                    // flag, every access stays in bounds, and every epilogue
                    // warp still meets every named barrier of the exchange;
                    // the status word reports the failure.
                    tc_fence_after_sync();
                    const uint32_t taddr = tmem_base + lane_addr + static_cast<uint32_t>(accb * NPAD + col0);
                    // TMEM loads of kLd columns (FP8BS_TMEM_LD_COLS)
                    constexpr int kLd = FP8BS_TMEM_LD_COLS(C::kCols, C::kColGroups);
                    static_assert(C::kCols % kLd == 0, "whole loads only");
                    constexpr int kNLd = C::kCols / kLd;
                    // promotion of chunk c (columns c * kLd ..) from its registers
                    auto promote = [&](int c, const uint32_t (&r)[kLd]) {
                        float sc[kLd];
                        if constexpr (C::kProducts) {
#pragma unroll
                            for (int q = 0; q < kLd / 4; ++q)
                                *reinterpret_cast<float4 *>(&sc[4 * q]) = reinterpret_cast<const float4 *>(pr + c * kLd)[q];
                        } else if constexpr (!C::kTileAcc) {
#pragma unroll
                            for (int j = 0; j < kLd; ++j)
                                sc[j] = sw * (MODE == kModeFp8Fused ? sa_c[c * kLd + j]
                                                                    : __shfl_sync(0xffffffffu, sa_l, (c * kLd + j) & 31));
                        }
                        if constexpr (C::kTileAcc) {
#pragma unroll
                            for (int j = 0; j < kLd; ++j)
                                acc[c * kLd + j] = __uint_as_float(r[j]);
                        } else {
                            // two columns per packed multiply-add
#pragma unroll
                            for (int j = 0; j < kLd; j += 2)
                                fma2(acc[c * kLd + j], acc[c * kLd + j + 1], sc[j], sc[j + 1], __uint_as_float(r[j]),
                                     __uint_as_float(r[j + 1]));
                        }
                    };
                    if constexpr (kLd < 64 && kNLd > 1) {
                        // chunk c + 1 in flight while chunk c is promoted
                        uint32_t ra[kLd], rb[kLd];
                        tmem_issue(taddr, ra);
                        tmem_wait(ra);
#pragma unroll
                        for (int c = 0; c < kNLd; ++c) {
                            uint32_t(&cur)[kLd] = (c & 1) ? rb : ra;
                            uint32_t(&nxt)[kLd] = (c & 1) ? ra : rb;
                            if (c + 1 < kNLd)
                                tmem_issue(taddr + (c + 1) * kLd, nxt);
                            promote(c, cur);
                            if (c + 1 < kNLd)
                                tmem_wait(nxt);
                        }
                    } else {
#pragma unroll
                        for (int c = 0; c < kNLd; ++c) {
                            uint32_t r[kLd];
                            if constexpr (kLd == 64)
                                tmem_load64(taddr + c * kLd, r);
                            else if constexpr (kLd == 32)
                                tmem_load32(taddr + c * kLd, r);
                            else
                                tmem_load16(taddr + c * kLd, r);
                            promote(c, r);
                        }
                    }
                    tc_fence_before_sync();
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(&tempty[accb]);
                    if (++accb == C::kAcc) {
                        accb = 0;
                        acc_ph ^= 1u;
                    }
                }
                if (!seg_end)
                    continue;
                // ---- tile segment complete: store or reduce
                const int n = wt * C::kTileRows + row;
                const bool whole_tile = (seg_first_kb == 0) && (kb == kg - 1);
                if (whole_tile) {
                    store_y(n);
                } else {
                    // K-split tile: publish this CTA's partial, and the last
                    // contributor to arrive sums all of them in contributor order.
                    const SplitPlan &pl = tile == tile_a ? plan_a : plan_b;
                    const int c_first = pl.c_first, c_last = pl.c_last;
                    auto slot_of = [&](int c) { return c == c_first ? pl.slot_first : 2 * c; };
                    const bool ex_ok = FP8BS_CHECK(c_first >= 0 && c_first <= cta && cta <= c_last && c_last < p.ctas &&
                                                   slot_of(cta) < 2 * p.ctas && tile >= 0 &&
                                                   tile < p.ttiles * p.ntiles);
                    float *mine = slots_y + static_cast<long long>(slot_of(cta)) * (NPAD * 128) + col0 * 128;
#pragma unroll
                    for (int m = 0; m < C::kCols; ++m)
                        if (m < mcnt && ex_ok)
                            __stcg(mine + m * 128 + row, acc[m]);
                    named_bar_sync(1, 32 * C::kEpiWarps);
                    if (warp == 2 && lane == 0) {
                        // one release for the whole epilogue group's stores (ordered
                        // by the barrier above); acquire for the others' partials
                        const unsigned prev = ex_ok ? atomic_add_acq_rel_gpu(&counters_y[tile], 1u) : 0u;
                        *last_flag = (ex_ok && prev == static_cast<unsigned>(c_last - c_first)) ? 1 : 0;
                    }
                    named_bar_sync(1, 32 * C::kEpiWarps);
                    if (*last_flag) {
#pragma unroll
                        for (int m = 0; m < C::kCols; ++m)
                            acc[m] = 0.0f;
                        // From 32 tokens up, at the range's last segment: every
                        // unit's MMAs are done, so the weight ring is idle and
                        // each contributor's whole slot (16 to 64 KB) comes in
                        // with one bulk copy, all in one round trip; the sums
                        // then read shared memory, in contributor order as
                        // below.  (Through registers a thread keeps two to six
                        // contributors' 8 to 32 columns in flight at a time:
                        // several sequential round trips per tile.  The 16-token
                        // tile's partials take one round trip that way.)
                        constexpr int kSlotBytes = NPAD * 128 * 4;
                        const int ncon = c_last - c_first + 1;
                        const bool bulk = NPAD >= 32 && i == nunits - 1 &&
                                          static_cast<long long>(ncon) * kSlotBytes <= static_cast<long long>(S) * C::kStageBytes;
                        if (bulk) {
                            if (warp == 2 && lane == 0) {
                                fence_proxy_async_global(); // the partials were stored by generic writes
                                mbar_arrive_expect_tx(red_ready, static_cast<uint32_t>(ncon * kSlotBytes));
                                const uint64_t pol = l2_policy_evict_first();
                                for (int j = 0; j < ncon; ++j)
                                    if (FP8BS_CHECK(slot_of(c_first + j) < 2 * p.ctas))
                                        bulk_load_1d(ring + j * kSlotBytes,
                                                     slots_y + static_cast<long long>(slot_of(c_first + j)) * (NPAD * 128),
                                                     kSlotBytes, red_ready, pol);
                                bulk_issued = true;
                            }
                            mbar_wait(red_ready, 0, abort_flag, p.status, kErrTimeoutEpilogue, p.timeout_ns);
                            const float *sm = reinterpret_cast<const float *>(ring) + col0 * 128 + row;
                            for (int j = 0; j < ncon; ++j)
#pragma unroll
                                for (int m = 0; m < C::kCols; m += 2)
                                    // packed adds, token pairs (column m + 1 >= M is never stored):
                                    // decode pass at 32 / 64 tokens 1.3 / 0.9 % faster; in the
                                    // register path below they cost the 16-token tile 2.8 %
                                    if (m < mcnt)
                                        add2(acc[m], acc[m + 1], sm[j * (NPAD * 128) + m * 128],
                                             sm[j * (NPAD * 128) + (m + 1) * 128]);
                        }
                        // Otherwise issue every contributor's loads for a chunk of
                        // tokens at once (one L2 round trip per chunk), then add
                        // them in contributor order.
                        constexpr int kMaxC = NPAD > 64 ? 2 : 6;
                        constexpr int kMC = NPAD <= 16 ? 16 : NPAD > 64 ? 32 : 8;
                        for (int c0 = bulk ? c_last + 1 : c_first; c0 <= c_last; c0 += kMaxC) {
                            const int nc = c_last - c0 + 1 < kMaxC ? c_last - c0 + 1 : kMaxC;
                            const float *src[kMaxC];
#pragma unroll
                            for (int j = 0; j < kMaxC; ++j)
                                src[j] = slots_y + static_cast<long long>(slot_of(c0 + (j < nc ? j : 0))) * (NPAD * 128) +
                                         col0 * 128 + row;
#pragma unroll
                            for (int mc = 0; mc < C::kCols; mc += kMC) {
                                if (mc >= mcnt)
                                    break;
                                float v[kMaxC][kMC];
#pragma unroll
                                for (int j = 0; j < kMaxC; ++j)
#pragma unroll
                                    for (int q = 0; q < kMC; ++q)
                                        v[j][q] = (j < nc && mc + q < mcnt) ? __ldcg(src[j] + (mc + q) * 128) : 0.0f;
#pragma unroll
                                for (int j = 0; j < kMaxC; ++j)
#pragma unroll
                                    for (int q = 0; q < kMC; ++q)
                                        if (j < nc)
                                            acc[mc + q] += v[j][q];
                            }
                        }
                        store_y(n);
                        if (warp == 2 && lane == 0)
                            counters_y[tile] = 0u; // ready for the next call
                    }
                    named_bar_sync(1, 32 * C::kEpiWarps);
                }
#pragma unroll
                for (int m = 0; m < C::kCols; ++m)
                    acc[m] = 0.0f;
            }
            if (y_pending)
                bulk_wait_all(); // Y written before the CTA exits
            // The slot copies must have landed before the CTA exits, also when
            // the wait above gave up (abort): a bounded wait of the thread that
            // issued them.
            if (bulk_issued) {
                const uint64_t t0 = globaltimer_ns();
                while (!mbar_test(red_ready, 0)) {
                    if (globaltimer_ns() - t0 > p.timeout_ns) {
                        atomicOr(p.status, kErrTimeoutEpilogue);
                        break;
                    }
                }
            }
            if constexpr (GREEDY) {
                // ---- greedy: publish this CTA's keys; the last CTA finishes
                named_bar_sync(1, 32 * C::kEpiWarps); // every warp's shared-memory folds are done
                if (warp == 2) {
                    for (int m = lane; m < p.M; m += 32)
                        atomicMax(&p.best[m], cta_best[m]);
                    __threadfence();
                    __syncwarp();
                    unsigned prev = 0;
                    if (lane == 0)
                        prev = atomic_add_acq_rel_gpu(p.done, 1u);
                    prev = __shfl_sync(0xffffffffu, prev, 0);
                    if (prev == static_cast<unsigned>(p.ctas - 1)) {
                        __threadfence();
                        for (int m = lane; m < p.M; m += 32) {
                            const unsigned long long k = atomicExch(&p.best[m], 0ull); // read and clear
                            p.token[m] = static_cast<int>(0xffffffffu - static_cast<uint32_t>(k));
                            if (p.logit != nullptr)
                                p.logit[m] = key_logit(static_cast<uint32_t>(k >> 32));
                        }
                        if (lane == 0)
                            *p.done = 0u;
                    }
                }
            }
        }
    }

    __syncwarp();
    tc_fence_before_sync();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after_sync();
        tmem_dealloc(tmem_base, C::kTmemCols);
    }
}

} // namespace fp8bs
