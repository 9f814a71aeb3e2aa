// e4m3 block-quantisation codec shared by the quantiser kernels and the FP8
// GEMM epilogue, so both take every code decision the same way.
//
// "Lower latency and higher throughput with multi-node DeepSeek deployment"
// (Perplexity blog), §Quantization: one scale per block; here a block's scale
// is amax/448 in fp32 (448 = largest finite e4m3) or, in the second format, the
// smallest power of two that brings amax to 448 or below; 1 for an all-zero
// block.  A value's code is round-to-nearest-even of fl32(v / scale), saturated.
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace moe {
namespace fp8 {

__device__ __forceinline__ uint32_t e4m3(float v) {
    return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float block_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

// The power-of-two scale format: the smallest 2^e with amax / 2^e <= 448 (1 for
// an all-zero block, e >= -127), found from amax's bits.  With amax =
// (1 + m / 2^23) * 2^(E - 127) and 448 = 1.75 * 2^8: e = E - 135 when the
// significand is at most 1.75, else E - 134.  Division by it is exact.
__device__ __forceinline__ float block_scale_pow2(float amax) {
    if (!(amax > 0.0f)) return 1.0f;
    const uint32_t b = __float_as_uint(amax);
    const int E = (int)(b >> 23);
    int e = E == 0 ? -127 : ((b & 0x7FFFFFu) <= 0x600000u ? E - 135 : E - 134);
    if (e < -127) e = -127;
    return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(0x00400000u);  // 2^-127
}
__device__ __forceinline__ float scale_for(float amax, bool pow2) {
    return pow2 ? block_scale_pow2(amax) : block_scale(amax);
}

// Four codes packed with v0 in the low byte, exactly as four e4m3() calls would pack them
// (two values per conversion).
__device__ __forceinline__ uint32_t e4m3x4(float v0, float v1, float v2, float v3) {
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v0, v1), __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v2, v3), __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

// fl32(v / s), the quotient a code is taken from, with one division per block instead of one per
// value: rs = fl32(1 / s) is the block's correctly rounded reciprocal.
//
// A power-of-two s: v * rs is the same real number as v / s, so it rounds the same.  Otherwise
// Markstein's correction (P. Markstein, "Computation of elementary functions on the IBM RISC
// System/6000 processor", IBM J. Res. Develop. 34(1), 1990): when y is within half an ulp of 1/s
// and q within one ulp of v/s, the residual r = v - s*q is exact in one fma and fl32(q + r*y) is
// fl32(v / s).  q0 = fl32(v * rs) can be up to 1.5 ulp off, so one step first brings it within an
// ulp (its residual may round, which moves the step's result by far less than an ulp), and the
// second step is the exact one.  That needs every step free of overflow and of underflow that
// loses bits: s in [2^-80, 2^100] (quotient_ok), |v| <= 448 s (every value of the block whose amax
// gave s), and |v| >= 2^-102, below which v / s < 2^-22 and both roundings give the code 0 all the
// same.  The caller divides when quotient_ok(s) is false.
__device__ __forceinline__ bool quotient_ok(float s) { return s >= 0x1p-80f && s <= 0x1p100f; }
__device__ __forceinline__ float quotient(float v, float s, float rs) {
    const float q0 = __fmul_rn(v, rs);
    const float q1 = __fmaf_rn(__fmaf_rn(-s, q0, v), rs, q0);
    return __fmaf_rn(__fmaf_rn(-s, q1, v), rs, q1);
}
// Exponent byte (UE8M0: 2^(byte - 127)) of a power-of-two scale, as block-scaled
// tensor-core instructions take it.
__device__ __forceinline__ uint32_t ue8m0(float pow2_scale) {
    const uint32_t b = __float_as_uint(pow2_scale);
    return b >= 0x00800000u ? b >> 23 : 0u;  // 2^-127 (the one subnormal scale) is byte 0
}

}  // namespace fp8
}  // namespace moe
