// quant.cu -- E4M3 quantisation kernels.
//
// quant_act_kernel: the run-time cast of the activations to FP8, one fp32
// scale per token per 128 consecutive K ("The profiler said the kernel ran
// zero times", "What the trace showed": casting inputs to FP8).  One warp per
// 128-element group; each lane converts four values.
//
// quant_weight_kernel: one fp32 scale per 128x128 weight block ("A 23% faster
// GPU kernel, and a model that did not move", "Why this shape is hard"; "The
// profiler said the kernel ran zero times", "The output layer, which did
// run").  One CTA per block; each warp reads 16 full rows (512 contiguous
// bytes of fp32 per row per instruction), so loads and stores are coalesced
// and the block stays in registers between the max and the conversion.
#include <cuda_bf16.h>

#include "fp8bs_testing.h"
#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8bs {

// Activation cast: one warp per (token, 128-wide K group), four per CTA.  A
// CTA this small (4,096 registers) fits on an SM beside the two CTAs of the
// 16-token GEMM, so under programmatic dependent launch it never keeps the
// next GEMM's early CTA off that SM.
constexpr int kCastThreads = 128;

// kKMajor (M > 16): the scales are written K-block-major ([K/128][M], the
// layout the GEMM reads above 16 tokens) rather than token-major
// ([M][K/128]); a separate instantiation each, so the token-major one's code
// is the same as if the other did not exist.
template <bool kKMajor>
__global__ void __launch_bounds__(kCastThreads) quant_act_kernel(const uint16_t *__restrict__ x, int M, int K, int ldx,
                                                        uint8_t *__restrict__ xq, float *__restrict__ xs,
                                                        unsigned long long *runs)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        atomicAdd(runs + FP8BS_RUNS_QUANT_ACT, 1ull);
    grid_launch_dependents();
    grid_dependency_wait();
    const int kg = K / 128;
    const long long group = static_cast<long long>(blockIdx.x) * (kCastThreads / 32) + (threadIdx.x >> 5);
    if (group >= static_cast<long long>(M) * kg)
        return; // whole warp
    const int lane = threadIdx.x & 31;
    // groups in the order of the scales they write: a CTA's warps then store
    // consecutive scale words
    const int m = static_cast<int>(kKMajor ? group % M : group / kg);
    const int g = static_cast<int>(kKMajor ? group / M : group % kg);
    const uint2 raw = *reinterpret_cast<const uint2 *>(x + static_cast<long long>(m) * ldx + g * 128 + lane * 4);
    uint32_t codes;
    const float s = quant_group_warp(raw, codes);
    *reinterpret_cast<uint32_t *>(xq + static_cast<long long>(m) * K + g * 128 + lane * 4) = codes;
    if (lane == 0)
        xs[kKMajor ? static_cast<long long>(g) * M + m : static_cast<long long>(m) * kg + g] = s;
}

// kTiled: write the codes of block (nb, kb) as one contiguous 16 KB run
// (row r of the block at r*128), rows past N as zeros.
template <bool kBf16, bool kTiled>
__global__ void __launch_bounds__(256) quant_weight_kernel(const void *__restrict__ w, int N, int K,
                                                           uint8_t *__restrict__ wq, float *__restrict__ ws,
                                                           unsigned long long *runs)
{
    __shared__ float warp_amax[8];
    if (blockIdx.x == 0 && threadIdx.x == 0)
        atomicAdd(runs + FP8BS_RUNS_QUANT_WEIGHT, 1ull);
    const int kg = K / 128;
    const long long blk = blockIdx.x;
    const int nb = static_cast<int>(blk / kg), kb = static_cast<int>(blk % kg);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r0 = nb * 128 + warp * 16;
    float v[16][4];
    float amax = 0.0f;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int r = r0 + j;
        if (r < N) {
            const long long off = static_cast<long long>(r) * K + kb * 128 + lane * 4;
            if (kBf16) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(w) + off);
                v[j][0] = bf16_lo(raw.x);
                v[j][1] = bf16_hi(raw.x);
                v[j][2] = bf16_lo(raw.y);
                v[j][3] = bf16_hi(raw.y);
            } else {
                const float4 f = *reinterpret_cast<const float4 *>(static_cast<const float *>(w) + off);
                v[j][0] = f.x;
                v[j][1] = f.y;
                v[j][2] = f.z;
                v[j][3] = f.w;
            }
        } else {
            v[j][0] = v[j][1] = v[j][2] = v[j][3] = 0.0f;
        }
        amax = fmaxf(amax, abs_max4(v[j][0], v[j][1], v[j][2], v[j][3]));
    }
    amax = warp_max(amax);
    if (lane == 0)
        warp_amax[warp] = amax;
    __syncthreads();
    amax = warp_amax[0];
#pragma unroll
    for (int i = 1; i < 8; ++i)
        amax = fmaxf(amax, warp_amax[i]);
    const float s = group_scale(amax);
#pragma unroll
    for (int j = 0; j < 16; ++j) {
        const int r = r0 + j;
        if (kTiled) {
            const long long off = blk * 16384 + static_cast<long long>(warp * 16 + j) * 128 + lane * 4;
            *reinterpret_cast<uint32_t *>(wq + off) =
                r < N ? quantize4(v[j][0], v[j][1], v[j][2], v[j][3], s) : 0u;
        } else if (r < N) {
            const long long off = static_cast<long long>(r) * K + kb * 128 + lane * 4;
            *reinterpret_cast<uint32_t *>(wq + off) = quantize4(v[j][0], v[j][1], v[j][2], v[j][3], s);
        }
    }
    if (threadIdx.x == 0)
        ws[blk] = s;
}

fp8bs_status launch_quant_act(const void *x, int M, int K, int ldx, uint8_t *xq, float *xs, bool pdl,
                              cudaStream_t stream, const DeviceInfo &dev)
{
    const long long groups = static_cast<long long>(M) * (K / 128);
    cudaLaunchConfig_t cfg = {};
    constexpr int kGroupsPerCta = kCastThreads / 32;
    cfg.gridDim = dim3(static_cast<unsigned>((groups + kGroupsPerCta - 1) / kGroupsPerCta), 1, 1);
    cfg.blockDim = dim3(kCastThreads, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return launch_status(cudaLaunchKernelEx(&cfg, M > 16 ? quant_act_kernel<true> : quant_act_kernel<false>,
                                            static_cast<const uint16_t *>(x), M, K, ldx,
                                            xq, xs, dev.runs));
}

// bf16 [N][K] -> tiled: tile (nb, kb) of 128 rows x 64 elements is one
// contiguous 16 KB run, row r at r*128 bytes, rows past N zero.
__global__ void __launch_bounds__(256) pack_bf16_tiled_kernel(const uint8_t *__restrict__ w, int N, int K,
                                                              uint8_t *__restrict__ wt, unsigned long long *runs)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        atomicAdd(runs + FP8BS_RUNS_PACK_BF16, 1ull);
    const int kg = K / 64;
    const long long blk = blockIdx.x;
    const int nb = static_cast<int>(blk / kg), kb = static_cast<int>(blk % kg);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const int idx = j * 256 + threadIdx.x; // 1024 16-byte pieces per tile
        const int r = idx >> 3, c = idx & 7;
        const int row = nb * 128 + r;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (row < N)
            v = *reinterpret_cast<const uint4 *>(w + static_cast<long long>(row) * K * 2 + kb * 128 + c * 16);
        *reinterpret_cast<uint4 *>(wt + blk * 16384 + r * 128 + c * 16) = v;
    }
}

fp8bs_status launch_pack_bf16_tiled(const void *w, int N, int K, void *wt, cudaStream_t stream,
                                    const DeviceInfo &dev)
{
    const long long blocks = static_cast<long long>((N + 127) / 128) * (K / 64);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    return launch_status(cudaLaunchKernelEx(&cfg, pack_bf16_tiled_kernel, static_cast<const uint8_t *>(w), N, K,
                                            static_cast<uint8_t *>(wt), dev.runs));
}

fp8bs_status launch_quant_weight(const void *w, int wtype, int N, int K, uint8_t *wq, float *ws, bool tiled,
                                 cudaStream_t stream, const DeviceInfo &dev)
{
    const long long blocks = static_cast<long long>((N + 127) / 128) * (K / 128);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    if (wtype == FP8BS_BF16)
        return launch_status(cudaLaunchKernelEx(&cfg, tiled ? quant_weight_kernel<true, true> : quant_weight_kernel<true, false>,
                                                w, N, K, wq, ws, dev.runs));
    return launch_status(cudaLaunchKernelEx(&cfg, tiled ? quant_weight_kernel<false, true> : quant_weight_kernel<false, false>,
                                            w, N, K, wq, ws, dev.runs));
}

} // namespace fp8bs
