// mx.cu -- microscaling (MX) E4M3 quantisation: one power-of-two scale per
// 32 consecutive values along K, the format whose products the Blackwell
// tensor core scales by itself (kind::mxf8f6f4).  "Kernel-Level
// Optimisations for LLM Inference and Training", "Writing your own kernel",
// names the block-scaled MX formats; the conversion is the one of the OCP
// microscaling specification:
//   e     = floor(log2(amax)) - 8, clamped to [-127, 127]  (0 for a zero block;
//           8 is the exponent of E4M3's largest value, 448 = 1.75 * 2^8)
//   scale = 2^e, stored as the byte e + 127 (UE8M0)
//   code  = E4M3 round-to-nearest-even, saturating, of v / 2^e (exact: a
//           power-of-two scaling), so block values up to 2^9 saturate at 448.
//
// Both kernels write the scale bytes in the 512-byte atoms the GEMM copies
// into tensor memory (ptx.cuh): per 128 rows and 128 K, the byte of row r
// and 32-wide K block j at 16 * (r % 32) + 4 * (r / 32) + j.
#include "fp8bs_testing.h"
#include "internal.h"
#include "ptx.cuh"
#include "quant_math.cuh"

namespace fp8bs {

// Shared exponent of one block from its largest magnitude (amax >= 0).
__device__ __forceinline__ int mx_shared_exponent(float amax)
{
    const uint32_t b = __float_as_uint(amax);
    const int E = static_cast<int>(b >> 23); // biased exponent (sign bit clear)
    if (E == 0)
        return b == 0 ? 0 : -127; // zero block; subnormal amax has floor(log2) <= -127
    const int e = E - 127 - 8;    // E <= 254 for finite input, so e <= 119
    return e < -127 ? -127 : e;
}

// 2^-e as a float, exact for e in [-127, 119].
__device__ __forceinline__ float mx_inv_scale(int e)
{
    return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

__device__ __forceinline__ int sf_atom_offset(int r, int j)
{
    return 16 * (r & 31) + 4 * (r >> 5) + j;
}

// One 128-value row segment held by a warp, lane l holding values 4l..4l+3:
// the four MX blocks are lanes 0-7, 8-15, 16-23, 24-31.  Returns this lane's
// four codes and, in *byte, its block's scale byte.
__device__ __forceinline__ uint32_t mx_quant_row128(float a, float b, float c, float d, uint32_t *byte)
{
    float m = abs_max4(a, b, c, d);
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 1));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 2));
    m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
    const int e = mx_shared_exponent(m);
    const float inv = mx_inv_scale(e);
    *byte = static_cast<uint32_t>(e + 127);
    return e4m3x4(a * inv, b * inv, c * inv, d * inv);
}

// Weights: one CTA per 128-row x 128-K tile, each warp 16 rows.  Codes in
// the tiled layout (tile (nb, kb) one contiguous 16 KB run, row r at r*128),
// scales as one atom per tile; rows past N are zero codes and zero bytes.
template <bool kBf16>
__global__ void __launch_bounds__(256) mx_quant_weight_kernel(const void *__restrict__ w, int N, int K,
                                                              uint8_t *__restrict__ wq, uint8_t *__restrict__ sf,
                                                              unsigned long long *runs)
{
    if (blockIdx.x == 0 && threadIdx.x == 0)
        atomicAdd(runs + FP8BS_RUNS_MX_QUANT_WEIGHT, 1ull);
    const int kg = K / 128;
    const long long blk = blockIdx.x;
    const int nb = static_cast<int>(blk / kg), kb = static_cast<int>(blk % kg);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 4
    for (int j = 0; j < 16; ++j) {
        const int r = warp * 16 + j;
        const int n = nb * 128 + r;
        float v0 = 0.0f, v1 = 0.0f, v2 = 0.0f, v3 = 0.0f;
        if (n < N) {
            const long long off = static_cast<long long>(n) * K + kb * 128 + lane * 4;
            if (kBf16) {
                const uint2 raw = *reinterpret_cast<const uint2 *>(static_cast<const uint16_t *>(w) + off);
                v0 = bf16_lo(raw.x);
                v1 = bf16_hi(raw.x);
                v2 = bf16_lo(raw.y);
                v3 = bf16_hi(raw.y);
            } else {
                const float4 f = *reinterpret_cast<const float4 *>(static_cast<const float *>(w) + off);
                v0 = f.x;
                v1 = f.y;
                v2 = f.z;
                v3 = f.w;
            }
        }
        uint32_t byte;
        const uint32_t codes = mx_quant_row128(v0, v1, v2, v3, &byte);
        *reinterpret_cast<uint32_t *>(wq + blk * 16384 + r * 128 + lane * 4) = n < N ? codes : 0u;
        if ((lane & 7) == 0)
            sf[blk * 512 + sf_atom_offset(r, lane >> 3)] = static_cast<uint8_t>(n < N ? byte : 0u);
    }
}

// Activations: one CTA of four warps per (128-wide K group, 128-token tile,
// 16-row slice of the tile) (a CTA small enough to sit beside the two CTAs of
// the 16-token GEMM).  Warp w takes rows w, w+4, ... of its slice, loads all
// four before converting any, and writes each row's four scale bytes as the
// one atom word they form (word 4 (r % 32) + r / 32), zero for rows >= M; the
// last slice's CTA also zeroes the words of the rows past every slice (a tile
// of fewer than 128 tokens has fewer slices).  Codes row-major [M][K]; atoms
// [token tile][K group].
constexpr int kMxCastWarps = 4;
constexpr int kMxSliceRows = 16;                                   // rows per CTA
constexpr int kMxRowsPerWarp = kMxSliceRows / kMxCastWarps;        // loaded together

__global__ void __maxnreg__(32) mx_quant_act_kernel(const uint16_t *__restrict__ x, int M, int K, int ldx,
                                                           uint8_t *__restrict__ xq, uint8_t *__restrict__ sf,
                                                           unsigned long long *runs)
{
    if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0)
        atomicAdd(runs + FP8BS_RUNS_MX_QUANT_ACT, 1ull);
    grid_launch_dependents();
    grid_dependency_wait();
    const int g = blockIdx.x, tt = blockIdx.y, slice = blockIdx.z;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    uint8_t *atom = sf + (static_cast<long long>(tt) * (K / 128) + g) * 512;
    uint32_t *const words = reinterpret_cast<uint32_t *>(atom);
    const int r0 = slice * kMxSliceRows + warp; // this warp's rows r0, r0 + 4, ... of the tile
    uint2 raw[kMxRowsPerWarp];
#pragma unroll
    for (int i = 0; i < kMxRowsPerWarp; ++i) {
        const int m = tt * 128 + r0 + kMxCastWarps * i;
        raw[i] = make_uint2(0u, 0u);
        if (m < M) // whole warp
            raw[i] = *reinterpret_cast<const uint2 *>(x + static_cast<long long>(m) * ldx + g * 128 + lane * 4);
    }
#pragma unroll
    for (int i = 0; i < kMxRowsPerWarp; ++i) {
        const int r = r0 + kMxCastWarps * i;
        const int m = tt * 128 + r;
        uint32_t word = 0u;
        if (m < M) { // whole warp
            uint32_t byte;
            const uint32_t codes =
                mx_quant_row128(bf16_lo(raw[i].x), bf16_hi(raw[i].x), bf16_lo(raw[i].y), bf16_hi(raw[i].y), &byte);
            *reinterpret_cast<uint32_t *>(xq + static_cast<long long>(m) * K + g * 128 + lane * 4) = codes;
            // the bytes of K blocks 0-3 sit in lanes 0, 8, 16, 24
            word = byte | (__shfl_sync(0xffffffffu, byte, 8) << 8) | (__shfl_sync(0xffffffffu, byte, 16) << 16) |
                   (__shfl_sync(0xffffffffu, byte, 24) << 24);
        }
        if (lane == 0)
            words[sf_atom_offset(r, 0) >> 2] = word;
    }
    // words of the rows no slice covers (a tile of fewer than 128 tokens):
    // word w holds row 32 (w % 4) + w / 4
    static_assert(32 * kMxCastWarps == 128, "one atom word per thread");
    const int wrow = 32 * static_cast<int>(threadIdx.x & 3) + static_cast<int>(threadIdx.x >> 2);
    if (slice == static_cast<int>(gridDim.z) - 1 && wrow >= (slice + 1) * kMxSliceRows)
        words[threadIdx.x] = 0u;
}

fp8bs_status launch_mx_quant_weights(const void *w, int wtype, int N, int K, uint8_t *wq, uint8_t *sf,
                                     cudaStream_t stream, const DeviceInfo &dev)
{
    const long long blocks = static_cast<long long>((N + 127) / 128) * (K / 128);
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(blocks), 1, 1);
    cfg.blockDim = dim3(256, 1, 1);
    cfg.stream = stream;
    if (wtype == FP8BS_BF16)
        return launch_status(cudaLaunchKernelEx(&cfg, mx_quant_weight_kernel<true>, w, N, K, wq, sf, dev.runs));
    return launch_status(cudaLaunchKernelEx(&cfg, mx_quant_weight_kernel<false>, w, N, K, wq, sf, dev.runs));
}

fp8bs_status launch_mx_quant_act(const void *x, int M, int K, int ldx, uint8_t *xq, uint8_t *sf, bool pdl,
                                 cudaStream_t stream, const DeviceInfo &dev)
{
    cudaLaunchConfig_t cfg = {};
    const int tile_rows = M < 128 ? M : 128;
    cfg.gridDim = dim3(static_cast<unsigned>(K / 128), static_cast<unsigned>((M + 127) / 128),
                       static_cast<unsigned>((tile_rows + kMxSliceRows - 1) / kMxSliceRows));
    cfg.blockDim = dim3(32 * kMxCastWarps, 1, 1);
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = pdl ? 1 : 0;
    return launch_status(cudaLaunchKernelEx(&cfg, mx_quant_act_kernel, static_cast<const uint16_t *>(x), M, K, ldx,
                                            xq, sf, dev.runs));
}

} // namespace fp8bs
