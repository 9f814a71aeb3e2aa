// FP8 (e4m3) block quantisation.
//
// "Lower latency and higher throughput with multi-node DeepSeek deployment"
// (Perplexity blog), §Quantization: DeepSeek-V3/R1 quantises per block, with
// scales per 128-element vector for activations (computed on the fly) and per
// 128x128 tile for weights (static).  A block's scale is amax/448 in fp32, or
// the smallest power of two bringing amax to 448 or below in the power-of-two
// format (1 for an all-zero block); each value becomes the e4m3 code of
// fl32(v / scale), rounded to nearest even and saturated at +-448.
#include "fp8_codec.cuh"
#include "moe_internal.cuh"

namespace moe {
namespace {

using fp8::e4m3;
using fp8::scale_for;

__device__ __forceinline__ float to_f(__nv_bfloat16 v) { return __bfloat162float(v); }
__device__ __forceinline__ float to_f(float v) { return v; }

__device__ __forceinline__ void load8(const __nv_bfloat16* p, float (&v)[8]) {
    const uint4 u = __ldg(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        v[2 * i] = __uint_as_float(w[i] << 16);
        v[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}
__device__ __forceinline__ void load8(const float* p, float (&v)[8]) {
    const float4 a = __ldg(reinterpret_cast<const float4*>(p)), b = __ldg(reinterpret_cast<const float4*>(p) + 1);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
}

// Half a warp per (row, 128-column block), eight values per lane, so a warp
// takes two blocks of one row per step with one 16-byte load per lane (8 bf16).
// Rows whose width is not a multiple of 8 take the guarded scalar path.
template <typename T>
__global__ void __launch_bounds__(256)
quantize_rows_kernel(const T* __restrict__ a, int64_t rows, int cols, int kb, int ld_scales,
                     uint8_t* __restrict__ codes, float* __restrict__ scales, bool pow2) {
    const int lane = threadIdx.x & 31, hl = lane & 15;
    const int kb2 = (kb + 1) / 2;  // block pairs per row
    pdl_trigger();  // launched after another kernel: the next one may be scheduled
    pdl_wait();     // before any read of what earlier work on the stream wrote

    const bool vec = (cols & 7) == 0;
    const int64_t nw = (int64_t)gridDim.x * (blockDim.x / 32);
    for (int64_t item = (int64_t)blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5); item < rows * kb2;
         item += nw) {
        const int64_t r = item / kb2;
        const int b = (int)(item - r * kb2) * 2 + (lane >> 4);
        const int c0 = b * 128 + hl * 8;
        const T* row = a + r * cols;
        float v[8];
        if (vec && b < kb && c0 + 8 <= cols) {
            load8(row + c0, v);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = b < kb && c0 + i < cols ? to_f(row[c0 + i]) : 0.0f;
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
#pragma unroll
        for (int off = 8; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
        if (b >= kb) continue;  // the second half of the last pair of an odd block count
        const float s = scale_for(amax, pow2);
        // fl32(v / s) for each value: one division per block (fp8_codec.cuh)
        const float rs = 1.0f / s;
        if (pow2) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], rs);
        } else if (fp8::quotient_ok(s)) {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = fp8::quotient(v[i], s, rs);
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = v[i] / s;
        }
        uint8_t* crow = codes + r * cols;
        if (vec && c0 + 8 <= cols) {
            uint2 packed;
            packed.x = fp8::e4m3x4(v[0], v[1], v[2], v[3]);
            packed.y = fp8::e4m3x4(v[4], v[5], v[6], v[7]);
            *reinterpret_cast<uint2*>(crow + c0) = packed;
        } else {
            for (int i = 0; i < 8; ++i)
                if (c0 + i < cols) crow[c0 + i] = (uint8_t)e4m3(v[i]);
        }
        if (hl == 0) scales[r * ld_scales + b] = s;
    }
}

// One block per 128x128 tile of a [G][rows][cols] matrix.
template <typename T>
__global__ void __launch_bounds__(256)
quantize_tiles_kernel(const T* __restrict__ w, int rows, int cols, int nb, int kb, uint8_t* __restrict__ codes,
                      float* __restrict__ scales, bool pow2) {
    __shared__ float red[8];
    const int64_t tile = blockIdx.x;
    const int64_t g = tile / ((int64_t)nb * kb);
    const int bn = (int)((tile / kb) % nb), bk = (int)(tile % kb);
    const int r0 = bn * 128, c0 = bk * 128;
    const int r1 = min(rows, r0 + 128), c1 = min(cols, c0 + 128);
    const T* base = w + g * rows * (int64_t)cols;
    float amax = 0.0f;
    for (int i = threadIdx.x; i < 128 * 128; i += blockDim.x) {
        const int r = r0 + i / 128, c = c0 + i % 128;
        if (r < r1 && c < c1) amax = fmaxf(amax, fabsf(to_f(base[(int64_t)r * cols + c])));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
    __syncthreads();
    amax = red[0];
    for (int i = 1; i < (int)(blockDim.x >> 5); ++i) amax = fmaxf(amax, red[i]);
    const float s = scale_for(amax, pow2);
    uint8_t* cbase = codes + g * rows * (int64_t)cols;
    for (int i = threadIdx.x; i < 128 * 128; i += blockDim.x) {
        const int r = r0 + i / 128, c = c0 + i % 128;
        if (r < r1 && c < c1) cbase[(int64_t)r * cols + c] = (uint8_t)e4m3(to_f(base[(int64_t)r * cols + c]) / s);
    }
    if (threadIdx.x == 0) scales[(g * nb + bn) * kb + bk] = s;
}

}  // namespace

moe_status_t launch_quantize_rows_fp8(const void* a, moe_dtype_t dt, int64_t rows, int cols, uint8_t* codes,
                                      float* scales, int ld_scales, cudaStream_t s, bool pow2, bool pdl) {
    if (rows == 0) return MOE_OK;
    const int kb = (cols + 127) / 128;
    const int64_t items = rows * ((kb + 1) / 2);  // one warp per pair of blocks
    const int grid = (int)std::min<int64_t>(ceil_div(items, 8), (int64_t)sm_count() * 16);
    if (dt == MOE_BF16) {
        const __nv_bfloat16* ab = static_cast<const __nv_bfloat16*>(a);
        if (pdl)
            MOE_CUDA_TRY(launch_pdl(quantize_rows_kernel<__nv_bfloat16>, dim3(grid), dim3(256), 0, s, ab, rows, cols,
                                    kb, ld_scales, codes, scales, pow2));
        else
            quantize_rows_kernel<__nv_bfloat16><<<grid, 256, 0, s>>>(ab, rows, cols, kb, ld_scales, codes, scales, pow2);
    } else {
        const float* af = static_cast<const float*>(a);
        if (pdl)
            MOE_CUDA_TRY(launch_pdl(quantize_rows_kernel<float>, dim3(grid), dim3(256), 0, s, af, rows, cols, kb,
                                    ld_scales, codes, scales, pow2));
        else
            quantize_rows_kernel<float><<<grid, 256, 0, s>>>(af, rows, cols, kb, ld_scales, codes, scales, pow2);
    }
    MOE_CUDA_TRY(cudaGetLastError());
    note_launch();
    return MOE_OK;
}

moe_status_t launch_quantize_tiles_fp8(const void* w, moe_dtype_t dt, int G, int rows, int cols, uint8_t* codes,
                                       float* scales, cudaStream_t s, bool pow2) {
    const int nb = (rows + 127) / 128, kb = (cols + 127) / 128;
    const int64_t tiles = (int64_t)G * nb * kb;
    if (tiles == 0) return MOE_OK;
    if (dt == MOE_BF16)
        quantize_tiles_kernel<__nv_bfloat16><<<(unsigned)tiles, 256, 0, s>>>(static_cast<const __nv_bfloat16*>(w),
                                                                             rows, cols, nb, kb, codes, scales, pow2);
    else
        quantize_tiles_kernel<float><<<(unsigned)tiles, 256, 0, s>>>(static_cast<const float*>(w), rows, cols, nb, kb,
                                                                     codes, scales, pow2);
    note_launch();
    return last_launch_status();
}

}  // namespace moe
