// Finalize-routing: un-permute, top-k weighted sum, plus the shared expert.
//
// "DeepSeek-R1 prefill inference optimisation on Atlas A3" (cann-recipes-infer),
// §MoE deployment strategy, Double-Routing step 8: finalize-routing restores
// the original token order through expanded_src_to_dst_row, multiplies by
// scales=topk_weight and adds the shared expert output given as skip1, in one
// operation.  "Lower latency and higher throughput with multi-node DeepSeek
// deployment" (Perplexity blog), §Expert Parallelism: routed outputs are summed
// with weights and the shared expert's output is added.
//
// One block per token (grid-stride); each thread owns 16-byte vectors of the
// hidden dimension, issues the k row loads of a group of 8 before using any of
// them, accumulates in fp32 in slot order (skip first) and rounds once.
// HBM-bound: T*k*H*b read + T*H*b skip read + T*H*b written.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 128;

template <typename T>
struct Vec;
template <>
struct Vec<float> {
    static constexpr int N = 4;
    __device__ static void unpack(const uint4& u, float* f) {
        f[0] = __uint_as_float(u.x);
        f[1] = __uint_as_float(u.y);
        f[2] = __uint_as_float(u.z);
        f[3] = __uint_as_float(u.w);
    }
    __device__ static uint4 pack(const float* f) {
        return make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]),
                          __float_as_uint(f[3]));
    }
};
template <>
struct Vec<__nv_bfloat16> {
    static constexpr int N = 8;
    __device__ static void unpack(const uint4& u, float* f) {
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            f[2 * i] = __uint_as_float(w[i] << 16);
            f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
        }
    }
    __device__ static uint4 pack(const float* f) {
        uint32_t w[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            __nv_bfloat162 b = __floats2bfloat162_rn(f[2 * i], f[2 * i + 1]);
            w[i] = *reinterpret_cast<uint32_t*>(&b);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <typename T>
__global__ void __launch_bounds__(kThreads)
finalize_kernel(const uint4* __restrict__ y, int64_t y_rows, const uint4* __restrict__ skip,
                const float* __restrict__ w, const int32_t* __restrict__ row_idx, int Tn, int nvec, int k,
                uint4* __restrict__ out, uint32_t* status) {
    constexpr int N = Vec<T>::N;
    __shared__ int rows[32];
    __shared__ float wts[32];
    pdl_trigger();  // launched after another kernel: the next one may be scheduled
    pdl_wait();     // before any read of what earlier work on the stream wrote
    for (int t = blockIdx.x; t < Tn; t += gridDim.x) {
        if (threadIdx.x < k) {
            const int r = row_idx[(size_t)t * k + threadIdx.x];
            const bool ok = r >= 0 && r < y_rows;
            if (!ok) set_status(status, MOE_DEVERR_BAD_ROW_INDEX);
            rows[threadIdx.x] = ok ? r : -1;
            wts[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
        }
        __syncthreads();
        for (int v = threadIdx.x; v < nvec; v += kThreads) {
            float acc[N];
            if (skip) {
                Vec<T>::unpack(__ldcs(skip + (size_t)t * nvec + v), acc);
            } else {
#pragma unroll
                for (int i = 0; i < N; ++i) acc[i] = 0.f;
            }
            for (int j0 = 0; j0 < k; j0 += 8) {
                uint4 val[8];
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + u;
                    if (j < k && rows[j] >= 0) val[u] = __ldcs(y + (size_t)rows[j] * nvec + v);
                }
#pragma unroll
                for (int u = 0; u < 8; ++u) {
                    const int j = j0 + u;
                    if (j < k && rows[j] >= 0) {
                        float f[N];
                        Vec<T>::unpack(val[u], f);
                        const float wj = wts[j];
#pragma unroll
                        for (int i = 0; i < N; ++i) acc[i] = fmaf(wj, f[i], acc[i]);
                    }
                }
            }
            out[(size_t)t * nvec + v] = Vec<T>::pack(acc);
        }
        __syncthreads();
    }
}

}  // namespace

moe_status_t launch_finalize(const void* y, int64_t y_rows, const void* skip, const float* w,
                             const int32_t* row_idx, moe_dtype_t dt, int T, int H, int k, void* out,
                             uint32_t* status, cudaStream_t s) {
    if (T == 0) return MOE_OK;
    const int nvec = (int)((size_t)H * dt_size(dt) / 16);
    const int grid = (int)std::min<int64_t>(T, (int64_t)sm_count() * 16);
    if (dt == MOE_BF16)
        MOE_CUDA_TRY(launch_pdl(finalize_kernel<__nv_bfloat16>, dim3(grid), dim3(kThreads), 0, s,
                                static_cast<const uint4*>(y), y_rows, static_cast<const uint4*>(skip), w, row_idx, T,
                                nvec, k, static_cast<uint4*>(out), status));
    else
        MOE_CUDA_TRY(launch_pdl(finalize_kernel<float>, dim3(grid), dim3(kThreads), 0, s, static_cast<const uint4*>(y),
                                y_rows, static_cast<const uint4*>(skip), w, row_idx, T, nvec, k,
                                static_cast<uint4*>(out), status));
    note_launch();
    return MOE_OK;
}

}  // namespace moe
