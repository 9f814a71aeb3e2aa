// e4m3 block-quantisation codec shared by the quantiser kernels and the FP8
// GEMM epilogue, so both take every code decision the same way.
//
// "Lower latency and higher throughput with multi-node DeepSeek deployment"
// (Perplexity blog), §Quantization: one fp32 scale per block; here a block's
// scale is amax/448 (448 = largest finite e4m3), 1 for an all-zero block, and
// a value's code is round-to-nearest-even of fl32(v / scale), saturated.
#pragma once

#include <cuda_fp8.h>

#include <cstdint>

namespace moe {
namespace fp8 {

__device__ __forceinline__ uint32_t e4m3(float v) {
    return (uint32_t)__nv_cvt_float_to_fp8(v, __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float block_scale(float amax) { return amax > 0.0f ? amax / 448.0f : 1.0f; }

}  // namespace fp8
}  // namespace moe
