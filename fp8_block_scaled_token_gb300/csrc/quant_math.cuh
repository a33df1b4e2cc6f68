// quant_math.cuh -- the E4M3 group quantisation step, shared by the
// standalone activation-quantisation kernel, the weight-block kernel and the
// fused GEMM prologue so that all three write identical bytes.
//
// Per group (1x128 activations or 128x128 weights):
//   scale = amax == 0 ? 1 : fl32(amax / 448)      (IEEE fp32 division)
//   code  = e4m3 round-to-nearest-even, saturating, of fl32(x / scale)
// ("The profiler said the kernel ran zero times", "What the trace showed":
// inputs are cast to FP8 at run time; "A 23% faster GPU kernel, and a model
// that did not move", "Why this shape is hard": one scale per 128x128 weight
// block; E4M3 per "Kernel-Level Optimisations for LLM Inference and
// Training", "Quantisation kernels".)
#pragma once

#include <cstdint>

namespace fp8bs {

constexpr float kE4M3Max = 448.0f;

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xFFFF0000u); }

__device__ __forceinline__ float group_scale(float amax)
{
    return amax == 0.0f ? 1.0f : __fdiv_rn(amax, kE4M3Max);
}

// Four fp32 values -> four E4M3 bytes, a in the lowest byte.  The hardware
// conversion rounds to nearest even and saturates to +-448.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d)
{
    uint16_t lo, hi;
    // cvt ...e4m3x2.f32 d, hi_src, lo_src: the first source lands in the upper byte.
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(lo) : "f"(b), "f"(a));
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(hi) : "f"(d), "f"(c));
    return static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
}

__device__ __forceinline__ float abs_max4(float a, float b, float c, float d)
{
    return fmaxf(fmaxf(fabsf(a), fabsf(b)), fmaxf(fabsf(c), fabsf(d)));
}

__device__ __forceinline__ float warp_max(float v)
{
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
        v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ uint32_t quantize4(float a, float b, float c, float d, float scale)
{
    return e4m3x4(__fdiv_rn(a, scale), __fdiv_rn(b, scale), __fdiv_rn(c, scale), __fdiv_rn(d, scale));
}

// One 128-wide activation group held by a warp, 4 consecutive bf16 per lane
// (lane l holds elements 4l..4l+3 as two packed 32-bit words).  Returns the
// group scale (same on every lane) and this lane's four codes.
__device__ __forceinline__ float quant_group_warp(uint2 raw, uint32_t &codes)
{
    const float a = bf16_lo(raw.x), b = bf16_hi(raw.x), c = bf16_lo(raw.y), d = bf16_hi(raw.y);
    const float s = group_scale(warp_max(abs_max4(a, b, c, d)));
    codes = quantize4(a, b, c, d, s);
    return s;
}

} // namespace fp8bs
