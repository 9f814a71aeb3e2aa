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
//
// Group-limited routing (the same page: flat routing is DeepSeek routing with
// one group of all experts): the E experts form n_group contiguous groups;
// lane g scores group g from a shared-memory copy of the token's scores (the
// largest score, or the largest two added in fp32), topk_group rounds of the
// warp argmax keep the best groups, and the experts of the other groups are
// excluded before the top-k rounds.
//
// The gate GEMM may hand over its logits as K-sliced partial sums; they are
// added here in slice order while loading (deterministic, no extra kernel).
#include "moe_internal.cuh"

#include <climits>

namespace moe {
namespace {

constexpr int kWarps = 8;

// Strict total order on (score, id): higher score first, then lower id.
__device__ __forceinline__ bool better(float a, int ia, float b, int ib) {
    return a > b || (a == b && ia < ib);
}

struct Grouping {
    int n_group;     // 1 = flat top-k
    int topk_group;  // groups kept
    int rule;        // 0: group score = max score; 1: sum of the two largest scores
};

// Warp-wide argmax over (value, index) pairs; every lane ends with the winner.
__device__ __forceinline__ void warp_argmax(float& bv, int& bi) {
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (better(ov, oi, bv, bi)) {
            bv = ov;
            bi = oi;
        }
    }
}

template <int VPL>
__global__ void __launch_bounds__(kWarps * 32)
route_topk_kernel(const float* logits, const float* __restrict__ bias, int T, int E, int k, Grouping grp,
                  int renorm, int nsplit, int64_t slice_stride, int32_t* __restrict__ ids, float* __restrict__ w) {
    extern __shared__ float sh_scores[];  // [kWarps][E], grouped routing only
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * kWarps + (threadIdx.x >> 5);
    pdl_trigger();  // the init-routing histogram may be scheduled; it waits for these ids
    pdl_wait();     // the logits come from the gate GEMM
    if (t >= T) return;  // whole warp leaves together
    const float* row = logits + (size_t)t * E;

    float v[VPL];
#pragma unroll
    for (int i = 0; i < VPL; ++i) v[i] = i * 32 + lane < E ? row[i * 32 + lane] : 0.0f;
    if (nsplit > 1) {
        // K slices of the gate GEMM, added in slice order; each round issues all
        // of a lane's loads before any add, and the sums go back to slice 0 last
        for (int q = 1; q < nsplit; ++q) {
            const float* sl = row + (size_t)q * slice_stride;
            float p[VPL];
#pragma unroll
            for (int i = 0; i < VPL; ++i) p[i] = i * 32 + lane < E ? sl[i * 32 + lane] : 0.0f;
#pragma unroll
            for (int i = 0; i < VPL; ++i) v[i] += p[i];
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (i * 32 + lane < E) const_cast<float*>(row)[i * 32 + lane] = v[i];
    }
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        const int e = i * 32 + lane;
        v[i] = e < E ? v[i] + (bias ? __ldg(bias + e) : 0.0f) : -INFINITY;
    }

    uint32_t taken = 0;  // bit i: register slot i is no longer a candidate
    if (grp.n_group > 1) {
        float* sc = sh_scores + (threadIdx.x >> 5) * E;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (i * 32 + lane < E) sc[i * 32 + lane] = v[i];
        __syncwarp();
        const int gs = E / grp.n_group;
        float gscore = -INFINITY;
        if (lane < grp.n_group) {
            float m1 = -INFINITY, m2 = -INFINITY;  // largest and second largest, in expert order
            for (int e = lane * gs; e < (lane + 1) * gs; ++e) {
                const float x = sc[e];
                if (x > m1) {
                    m2 = m1;
                    m1 = x;
                } else if (x > m2) {
                    m2 = x;
                }
            }
            gscore = grp.rule == 1 ? m1 + m2 : m1;
        }
        uint32_t kept = 0;
        bool gtaken = false;
        for (int r = 0; r < grp.topk_group; ++r) {
            const bool cand = lane < grp.n_group && !gtaken;
            float bv = cand ? gscore : -INFINITY;
            int bi = cand ? lane : INT_MAX;
            warp_argmax(bv, bi);
            if (bi == lane) gtaken = true;
            kept |= 1u << bi;
        }
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            const int e = i * 32 + lane;
            if (e < E && !((kept >> (e / gs)) & 1u)) taken |= 1u << i;
        }
    }

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
        warp_argmax(bv, bi);
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (j == 0) top = bv;
        if (lane == j) {
            my_id = bi;
            my_v = bv;
        }
    }

    // The shift of the exponentials only sets their range.  Renormalised weights
    // involve the selected experts alone: shift by the best of them.  Otherwise
    // the denominator runs over all E: shift by the largest score overall (the
    // same expert unless grouping excluded it).
    if (grp.n_group > 1 && !renorm) {
        float vmax = -INFINITY;
#pragma unroll
        for (int i = 0; i < VPL; ++i)
            if (i * 32 + lane < E) vmax = fmaxf(vmax, v[i]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) vmax = fmaxf(vmax, __shfl_xor_sync(0xffffffffu, vmax, off));
        top = vmax;
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
cudaError_t launch(const float* logits, const float* bias, int T, int E, int k, Grouping grp, int renorm,
                   int nsplit, int64_t slice_stride, int32_t* ids, float* w, cudaStream_t s) {
    const int blocks = (int)ceil_div(T, kWarps);
    const size_t smem = grp.n_group > 1 ? (size_t)kWarps * E * sizeof(float) : 0;
    return launch_pdl(route_topk_kernel<VPL>, dim3(blocks), dim3(kWarps * 32), smem, s, logits, bias, T, E, k, grp,
                      renorm, nsplit, slice_stride, ids, w);
}

}  // namespace

moe_status_t launch_route_topk(const float* logits, const float* bias, int T, int E, int k, int renorm,
                               int32_t* ids, float* w, cudaStream_t s, int n_group, int topk_group, int rule,
                               int nsplit, int64_t slice_stride) {
    if (T == 0) return MOE_OK;
    const Grouping grp{n_group > 1 ? n_group : 1, topk_group, rule};
    const int ns = nsplit > 1 ? nsplit : 1;
    const int64_t ss = slice_stride > 0 ? slice_stride : (int64_t)T * E;
    cudaError_t err;
    if (E <= 32) err = launch<1>(logits, bias, T, E, k, grp, renorm, ns, ss, ids, w, s);
    else if (E <= 64) err = launch<2>(logits, bias, T, E, k, grp, renorm, ns, ss, ids, w, s);
    else if (E <= 128) err = launch<4>(logits, bias, T, E, k, grp, renorm, ns, ss, ids, w, s);
    else if (E <= 256) err = launch<8>(logits, bias, T, E, k, grp, renorm, ns, ss, ids, w, s);
    else if (E <= 512) err = launch<16>(logits, bias, T, E, k, grp, renorm, ns, ss, ids, w, s);
    else err = launch<32>(logits, bias, T, E, k, grp, renorm, ns, ss, ids, w, s);
    note_launch();
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

}  // namespace moe
