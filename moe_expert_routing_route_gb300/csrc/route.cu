// Top-k routing, one warp per token.
//
// "Lower latency and higher throughput with multi-node DeepSeek deployment"
// (Perplexity blog), §MoE Router: the router is a top-k over the scores that
// also tracks the indices of the selected elements; §Expert Parallelism: each
// token is sent to k distinct routed experts whose outputs are summed with
// weights.  The page's router is a sort in Triton; here a token's E scores sit
// in the registers of one warp (E/32 per lane) and k rounds of a warp-wide
// argmax pick the experts in descending order, ties to the lower expert id.
//
// Weights: softmax over the E scores evaluated at the selected experts; with
// renormalisation the full-softmax denominator cancels and only the k selected
// exponentials are summed.  Scores are s_e = logit + bias (one fp32 add).
#include "moe_internal.cuh"

#include <climits>

namespace moe {
namespace {

constexpr int kWarps = 8;

// Strict total order on (score, id): higher score first, then lower id.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

template <int VPL>
__global__ void __launch_bounds__(kWarps * 32)
route_topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E, int k,
                  int renorm, int32_t* __restrict__ ids, float* __restrict__ w) {
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    if (t >= T) return;  // whole warp leaves together
    const float* row = logits + (size_t)t * E;

    float v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = i * 32 + lane;
        if (e < E) {
            const float b = bias ? __ldg(bias + e) : 0.0f;
            v[i] = __ldg(row + e) + b;
        } else {
            v[i] = -INFINITY;
        }
    }

    uint32_t taken = 0;
    int my_id = 0;
    float my_v = 0.f, top = 0.f;
    for (int j = 0; j < k; ++j) {
        float bv = -INFINITY;
        int bi = INT_MAX;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = i * 32 + lane;
            if (!((taken >> i) & 1u) && e < E && better(v[i], e, bv, bi)) {
                bv = v[i];
                bi = e;
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
            const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
            if (better(ov, oi, bv, bi)) {
                bv = ov;
                bi = oi;
            }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (j == 0) top = bv;
        if (lane == j) {
            my_id = bi;
            my_v = bv;
        }
    }

    const float ex = lane < k ? expf(my_v - top) : 0.0f;
    float denom;
    if (renorm) {
        denom = ex;
    } else {
        denom = 0.f;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (i * 32 + lane < E) denom += expf(v[i] - top);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) denom += __shfl_xor_sync(0xffffffffu, denom, off);

    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        w[(size_t)t * k + lane] = ex / denom;
    }
}

template <int VPL>
cudaError_t launch(const float* logits, const float* bias, int T, int E, int k, int renorm, int32_t* ids,
                   float* w, cudaStream_t s) {
    const int blocks = (int)ceil_div(T, kWarps);
    route_topk_kernel<VPL><<<blocks, kWarps * 32, 0, s>>>(logits, bias, T, E, k, renorm, ids, w);
    return cudaGetLastError();
}

}  // namespace

moe_status_t launch_route_topk(const float* logits, const float* bias, int T, int E, int k, int renorm,
                               int32_t* ids, float* w, cudaStream_t s) {
    if (T == 0) return MOE_OK;
    cudaError_t err;
    if (E <= 32) err = launch<1>(logits, bias, T, E, k, renorm, ids, w, s);
    else if (E <= 64) err = launch<2>(logits, bias, T, E, k, renorm, ids, w, s);
    else if (E <= 128) err = launch<4>(logits, bias, T, E, k, renorm, ids, w, s);
    else if (E <= 256) err = launch<8>(logits, bias, T, E, k, renorm, ids, w, s);
    else if (E <= 512) err = launch<16>(logits, bias, T, E, k, renorm, ids, w, s);
    else err = launch<32>(logits, bias, T, E, k, renorm, ids, w, s);
    note_launch();
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
