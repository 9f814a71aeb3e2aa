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
// Exponent byte (UE8M0: 2^(byte - 127)) of a power-of-two scale, as block-scaled
// tensor-core instructions take it.
__device__ __forceinline__ uint32_t ue8m0(float pow2_scale) {
    const uint32_t b = __float_as_uint(pow2_scale);
    return b >= 0x00800000u ? b >> 23 : 0u;  // 2^-127 (the one subnormal scale) is byte 0
}

}  // namespace fp8
}  // namespace moe
