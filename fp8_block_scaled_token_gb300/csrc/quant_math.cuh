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

// Maximum over the warp of a non-negative float (an absolute value).  For
// non-negative IEEE values the unsigned bit patterns order like the values,
// so one unsigned warp reduction gives the exact maximum.
__device__ __forceinline__ float warp_max(float v)
{
    return __uint_as_float(__reduce_max_sync(0xffffffffu, __float_as_uint(v)));
}

// Codes of four values of one group: e4m3 of the correctly rounded fp32
// quotient x / scale.
//
// Fast path: q = x * rcp(scale) is within a few fp32 ulps of x / scale, and
// the interval [q - |q|e, q + |q|e] with e = 2^-19 contains both the exact
// quotient and its fp32 rounding.  E4M3 rounding is monotonic, so when both
// ends of the interval convert to the same code, every value inside it does,
// and that code is exactly the one of the correctly rounded quotient.  Only
// when an E4M3 rounding boundary falls inside the interval (about one value
// in 2^15) is the IEEE division done.  A subnormal scale (all |x| below
// 448 * 2^-126) always takes the exact path.
__device__ __forceinline__ uint32_t quantize4(float a, float b, float c, float d, float scale)
{
    if (scale < 1.17549435e-38f) // subnormal scale: reciprocal not accurate enough
        return e4m3x4(__fdiv_rn(a, scale), __fdiv_rn(b, scale), __fdiv_rn(c, scale), __fdiv_rn(d, scale));
    float r;
    asm("rcp.approx.f32 %0, %1;" : "=f"(r) : "f"(scale));
    const float qa = a * r, qb = b * r, qc = c * r, qd = d * r;
    constexpr float kE = 1.0f / 524288.0f; // 2^-19
    const float ea = fabsf(qa) * kE, eb = fabsf(qb) * kE, ec = fabsf(qc) * kE, ed = fabsf(qd) * kE;
    const uint32_t lo = e4m3x4(qa - ea, qb - eb, qc - ec, qd - ed);
    const uint32_t hi = e4m3x4(qa + ea, qb + eb, qc + ec, qd + ed);
    if (lo == hi)
        return lo;
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
