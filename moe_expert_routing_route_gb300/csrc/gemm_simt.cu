// fp32 GEMMs on the FFMA pipes: the gate GEMM and the grouped expert FFN for
// fp32 layers.  tcgen05 has no exact-fp32 kind (tf32 would miss a 1e-5 relative
// tolerance), so fp32 layers take this path; bf16 layers take gemm_tc.cu.
//
// "Lower latency and higher throughput with multi-node DeepSeek deployment"
// (Perplexity blog), §Roofline / GroupGEMM: g groups, group i computes
// [m_i,k]x[k,n]; §Quantization: kernels read the routing counts on the device
// instead of sizing work by the buffers' upper bound -- each block maps its
// slot to (expert, row tile) from the offsets, slots past the populated tiles
// exit at once.
//
// C[r, :] = A[r, :] B_g^T for the rows r of group g (B_g = rows [g*Nb, g*Nb+Nb)
// of B, reduction dimension contiguous in both operands).  64x64 tiles, 256
// threads, 4x4 outputs per thread, K in steps of 16 through shared memory.
// The SwiGLU variant reads the packed gate/up weights (blocks of 128 gate rows
// followed by the 128 matching up rows) and writes h = silu(gate) * up.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <bool SWIGLU>
__global__ void __launch_bounds__(256)
simt_grouped_kernel(const float* __restrict__ A, int M, int K, const int32_t* __restrict__ offsets, int G,
                    const float* __restrict__ B, int Nb, int N, float* __restrict__ C, int64_t ldc,
                    uint32_t* status) {
    __shared__ float As[BK][BM + 4];
    __shared__ float Bs[BK][BN + 4];
    __shared__ float Us[SWIGLU ? BK : 1][BN + 4];
    __shared__ int sh_g, sh_r0, sh_r1;
    pdl_trigger();  // launched after another kernel: the next one may be scheduled
    pdl_wait();     // before any read of what earlier work on the stream wrote

    if (threadIdx.x == 0) {
        // slot blockIdx.y -> (group, row tile) from the device-side offsets
        int slot = blockIdx.y, g = -1, r0 = 0, r1 = 0;
        if (!offsets) {
            if (slot * BM < M) { g = 0; r0 = slot * BM; r1 = min(M, r0 + BM); }
        } else {
            for (int q = 0; q < G; ++q) {
                const int a = offsets[q], b = offsets[q + 1];
                if (a < 0 || b < a || b > M) { set_status(status, MOE_DEVERR_BAD_OFFSETS); break; }
                const int tiles = (b - a + BM - 1) / BM;
                if (slot < tiles) { g = q; r0 = a + slot * BM; r1 = min(b, r0 + BM); break; }
                slot -= tiles;
            }
        }
        sh_g = g; sh_r0 = r0; sh_r1 = r1;
    }
    __syncthreads();
    const int g = sh_g;
    if (g < 0) return;
    const int r0 = sh_r0, r1 = sh_r1;
    const int c0 = blockIdx.x * BN;  // first output column of this tile
    if (c0 >= N) return;

    const int tx = threadIdx.x & 15, ty = threadIdx.x >> 4;
    float acc[4][4] = {}, accu[4][4] = {};

    // B row of output column c (within group g)
    auto brow = [&](int c, bool up) -> int64_t {
        if (!SWIGLU) return (int64_t)g * Nb + c;
        return (int64_t)g * Nb + (c / 128) * 256 + (up ? 128 : 0) + (c & 127);
    };

    // each thread stages 4 elements of A, B (and U) per k-tile; the next tile's
    // loads are issued before the current tile's FMAs, so their latency overlaps
    constexpr int PER = BM * BK / 256;
    float ra[PER], rb[PER], ru[PER];
    auto fetch = [&](int k0) {
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int i = threadIdx.x + q * 256;
            const int r = i / BK, kk = i % BK;
            const int row = r0 + r, kc = k0 + kk, c = c0 + r;
            ra[q] = (row < r1 && kc < K) ? A[(int64_t)row * K + kc] : 0.f;
            rb[q] = (c < N && kc < K) ? B[brow(c, false) * K + kc] : 0.f;
            if (SWIGLU) ru[q] = (c < N && kc < K) ? B[brow(c, true) * K + kc] : 0.f;
        }
    };
    fetch(0);
    for (int k0 = 0; k0 < K; k0 += BK) {
#pragma unroll
        for (int q = 0; q < PER; ++q) {
            const int i = threadIdx.x + q * 256;
            const int r = i / BK, kk = i % BK;
            As[kk][r] = ra[q];
            Bs[kk][r] = rb[q];
            if (SWIGLU) Us[kk][r] = ru[q];
        }
        __syncthreads();
        if (k0 + BK < K) fetch(k0 + BK);
#pragma unroll
        for (int kk = 0; kk < BK; ++kk) {
            float a[4], b[4], u[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                a[i] = As[kk][ty * 4 + i];
                b[i] = Bs[kk][tx * 4 + i];
                if (SWIGLU) u[i] = Us[kk][tx * 4 + i];
            }
#pragma unroll
            for (int i = 0; i < 4; ++i)
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
                    if (SWIGLU) accu[i][j] = fmaf(a[i], u[j], accu[i][j]);
                }
        }
        __syncthreads();
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const int row = r0 + ty * 4 + i;
        if (row >= r1) continue;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int c = c0 + tx * 4 + j;
            if (c >= N) continue;
            float v = acc[i][j];
            if (SWIGLU) v = v / (1.0f + expf(-v)) * accu[i][j];
            C[(int64_t)row * ldc + c] = v;
        }
    }
}

int row_slots(int M, int G, bool grouped) {
    return (int)ceil_div(M, BM) + (grouped ? G : 0);
}

}  // namespace

moe_status_t launch_simt_gate(const float* x, const float* wr, int T, int H, int E, float* logits,
                              cudaStream_t s) {
    if (T == 0) return MOE_OK;
    dim3 grid((unsigned)ceil_div(E, BN), (unsigned)row_slots(T, 1, false));
    MOE_CUDA_TRY(launch_pdl(simt_grouped_kernel<false>, grid, dim3(256), 0, s, x, T, H, nullptr, 1, wr, E, E, logits,
                            (int64_t)E, nullptr));
    note_launch();
    return MOE_OK;
}

moe_status_t launch_simt_grouped_ffn_up(const float* a, int M, int H, const int32_t* offsets, int G,
                                        const float* w13_packed, int Ip, int I, float* h, uint32_t* status,
                                        cudaStream_t s, bool pdl) {
    if (M == 0) return MOE_OK;
    dim3 grid((unsigned)ceil_div(I, BN), (unsigned)row_slots(M, G, offsets != nullptr));
    if (pdl)
        MOE_CUDA_TRY(launch_pdl(simt_grouped_kernel<true>, grid, dim3(256), 0, s, a, M, H, offsets, G, w13_packed,
                                2 * Ip, I, h, (int64_t)I, status));
    else
        simt_grouped_kernel<true><<<grid, 256, 0, s>>>(a, M, H, offsets, G, w13_packed, 2 * Ip, I, h, I, status);
    MOE_CUDA_TRY(cudaGetLastError());
    note_launch();
    return MOE_OK;
}

moe_status_t launch_simt_grouped_down(const float* h, int M, int I, const int32_t* offsets, int G,
                                      const float* w2, int H, float* y, uint32_t* status, cudaStream_t s,
                                      bool pdl) {
    if (M == 0) return MOE_OK;
    dim3 grid((unsigned)ceil_div(H, BN), (unsigned)row_slots(M, G, offsets != nullptr));
    if (pdl)
        MOE_CUDA_TRY(launch_pdl(simt_grouped_kernel<false>, grid, dim3(256), 0, s, h, M, I, offsets, G, w2, H, H, y,
                                (int64_t)H, status));
    else
        simt_grouped_kernel<false><<<grid, 256, 0, s>>>(h, M, I, offsets, G, w2, H, H, y, H, status);
    MOE_CUDA_TRY(cudaGetLastError());
    note_launch();
    return MOE_OK;
}

}  // namespace moe
