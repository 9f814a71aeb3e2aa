// Init-routing: the expand-and-sort permutation of the token rows.
//
// "DeepSeek-R1 prefill inference optimisation on Atlas A3" (cann-recipes-infer),
// §MoE deployment strategy, Double-Routing step 1: expand every token k times,
// sort the copies by expert, and return expanded_x, expanded_row_idx (which
// restores the original order) and tokens_per_expert.  "Lower latency and
// higher throughput with multi-node DeepSeek deployment" (Perplexity blog),
// §MoE Router: dense dispatch needs the routing aggregated per expert.
//
// The sort is a stable counting sort in two small kernels plus one copy, chained
// with programmatic dependent launch (each kernel's blocks are resident and
// waiting when the previous kernel finishes):
//   hist    one block per chunk of kChunk source rows -> per-chunk histogram
//           hist[c][e] (chunk-major: coalesced writes)
//   scatter one block per chunk.  Each block first derives from the histograms
//           what a scan would give it: every expert's total (block 0 writes
//           tokens_per_expert and expert_offsets, the exclusive scan of the
//           totals) and the first destination row of this chunk's copies per
//           expert.  Then each warp ranks its 128 rows in source order
//           (__match_any_sync groups the lanes with the same expert, the rank
//           inside the group keeps source order), and the warps' per-expert
//           counts are prefix-summed in warp order: stable overall
//   copy    x is read once (16-byte vectors) and each row is written to its
//           k destinations (HBM-bound: T*H*b read + T*k*H*b written)
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kChunk = 1024;      // source rows per chunk (one block)
constexpr int kChunkThreads = 256;
constexpr int kChunkWarps = kChunkThreads / 32;
constexpr int kRowsPerWarp = kChunk / kChunkWarps;  // 128 = 4 steps of 32
constexpr int kSteps = kRowsPerWarp / 32;

__global__ void __launch_bounds__(kChunkThreads)
hist_kernel(const int32_t* __restrict__ ids, int R, int E, int NW, int32_t* __restrict__ hist,
            uint32_t* status) {
    extern __shared__ int32_t sh[];  // [E]
    const int c = blockIdx.x;
    pdl_trigger();
    pdl_wait();  // ids come from the routing kernel
    for (int e = threadIdx.x; e < E; e += kChunkThreads) sh[e] = 0;
    __syncthreads();
    const int beg = c * kChunk, end = min(R, beg + kChunk);
    bool bad = false;
    for (int src = beg + threadIdx.x; src < end; src += kChunkThreads) {
        const int id = __ldg(ids + src);
        if ((unsigned)id < (unsigned)E) atomicAdd(&sh[id], 1);
        else bad = true;
    }
    if (bad) set_status(status, MOE_DEVERR_BAD_EXPERT_ID);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += kChunkThreads) hist[(size_t)c * E + e] = sh[e];
}

// 256 threads, E <= 1024 (4 experts per thread in the scan); small enough to run beside a
// resident tensor-core GEMM CTA (the shared experts run concurrently on another stream).
__global__ void __launch_bounds__(kChunkThreads)
scatter_kernel(const int32_t* __restrict__ ids, int R, int E, int NW, const int32_t* __restrict__ hist,
               int32_t* __restrict__ counts, int32_t* __restrict__ offsets, int32_t* __restrict__ row_idx) {
    // [kChunkWarps][E]: per-warp counts, then per-warp first rows; [E] expert totals, then this
    // chunk's first rows; [E] the counts of the chunks before this one
    extern __shared__ int32_t sh[];
    __shared__ int warp_tot[kChunkWarps];
    int32_t* cfirst = sh + kChunkWarps * E;
    int32_t* before = cfirst + E;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int c = blockIdx.x;
    pdl_trigger();
    pdl_wait();  // the histograms (and, through the histogram kernel's own wait, the ids)
    for (int i = tid; i < kChunkWarps * E; i += kChunkThreads) sh[i] = 0;
    // every expert's total over the chunks, and its count in the chunks before this one
    for (int e = tid; e < E; e += kChunkThreads) {
        int tot = 0, pre = 0;
        for (int q = 0; q < NW; ++q) {
            const int v = hist[(size_t)q * E + e];
            tot += v;
            pre += q < c ? v : 0;
        }
        cfirst[e] = tot;
        before[e] = pre;
    }
    __syncthreads();
    // exclusive scan of the totals over experts: 4 consecutive experts per thread, then across threads
    {
        const int e0 = tid * 4;
        int loc[4], run = 0;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            loc[i] = run;
            run += e0 + i < E ? cfirst[e0 + i] : 0;
        }
        int incl = run;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            const int n = __shfl_up_sync(0xffffffffu, incl, off);
            if (lane >= off) incl += n;
        }
        if (lane == 31) warp_tot[warp] = incl;
        __syncthreads();
        int wbase = 0;
        for (int w = 0; w < warp; ++w) wbase += warp_tot[w];
        const int tbase = wbase + incl - run;
        if (c == 0) {
#pragma unroll
            for (int i = 0; i < 4; ++i)
                if (e0 + i < E) {
                    counts[e0 + i] = cfirst[e0 + i];
                    offsets[e0 + i] = tbase + loc[i];
                }
            if (tid == kChunkThreads - 1) offsets[E] = tbase + run;
        }
        __syncthreads();  // every total read before any is overwritten
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (e0 + i < E) cfirst[e0 + i] = tbase + loc[i] + before[e0 + i];
    }
    const int beg = c * kChunk + warp * kRowsPerWarp, end = min(R, c * kChunk + kChunk);
    int id[kSteps], rank[kSteps];
#pragma unroll
    for (int q = 0; q < kSteps; ++q) {  // all loads first
        const int src = beg + q * 32 + lane;
        id[q] = src < end ? __ldg(ids + src) : -1;
    }
    __syncthreads();
    int32_t* cnt = sh + warp * E;
    const unsigned lt_mask = (1u << lane) - 1u;
#pragma unroll
    for (int q = 0; q < kSteps; ++q) {
        const bool ok = (unsigned)id[q] < (unsigned)E;
        const unsigned group = __match_any_sync(0xffffffffu, ok ? (unsigned)id[q] : 0xffffffffu);
        const int r = __popc(group & lt_mask);
        const int first = ok ? cnt[id[q]] : 0;
        __syncwarp();
        if (ok && r == 0) cnt[id[q]] = first + __popc(group);
        __syncwarp();
        rank[q] = first + r;
        if (!ok) id[q] = -1;
    }
    __syncthreads();
    // per expert: the chunk's first row plus the counts of the earlier warps
    for (int e = threadIdx.x; e < E; e += kChunkThreads) {
        int run = cfirst[e];
        for (int w = 0; w < kChunkWarps; ++w) {
            const int v = sh[w * E + e];
            sh[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();
#pragma unroll
    for (int q = 0; q < kSteps; ++q) {
        const int src = beg + q * 32 + lane;
        if (src < end) row_idx[src] = id[q] >= 0 ? cnt[id[q]] + rank[q] : -1;
    }
}

constexpr int kCopyThreads = 128;
constexpr int kCopyUnroll = 4;

__global__ void __launch_bounds__(kCopyThreads)
permute_rows_kernel(const uint4* __restrict__ x, int nvec, const int32_t* __restrict__ row_idx, int T,
                    int k, int R, uint4* __restrict__ out) {
    __shared__ int dst[32];
    pdl_trigger();
    pdl_wait();  // row_idx comes from the scatter kernel
    for (int t = blockIdx.x; t < T; t += gridDim.x) {
        if (threadIdx.x < k) {
            const int d = row_idx[(size_t)t * k + threadIdx.x];
            dst[threadIdx.x] = (d >= 0 && d < R) ? d : -1;
        }
        __syncthreads();
        const uint4* xr = x + (size_t)t * nvec;
        for (int v0 = threadIdx.x; v0 < nvec; v0 += kCopyUnroll * kCopyThreads) {
            uint4 val[kCopyUnroll];
#pragma unroll
            for (int u = 0; u < kCopyUnroll; ++u) {
                const int v = v0 + u * kCopyThreads;
                if (v < nvec) val[u] = __ldcs(xr + v);  // read once: streaming
            }
            for (int j = 0; j < k; ++j) {
                const int d = dst[j];
                if (d < 0) continue;
                uint4* orow = out + (size_t)d * nvec;
#pragma unroll
                for (int u = 0; u < kCopyUnroll; ++u) {
                    const int v = v0 + u * kCopyThreads;
                    if (v < nvec) orow[v] = val[u];
                }
            }
        }
        __syncthreads();
    }
}

__global__ void pack_w13_kernel(const uint4* __restrict__ wg, const uint4* __restrict__ wu, int E, int I,
                                int Ip, int nvec, uint4* __restrict__ packed) {
    const int64_t rows = (int64_t)E * 2 * Ip;
    for (int64_t row = blockIdx.x; row < rows; row += gridDim.x) {
        const int e = (int)(row / (2 * Ip));
        const int r = (int)(row % (2 * Ip));
        const int q = r % 256;
        const int i = (r / 256) * 128 + (q & 127);
        const uint4* src = i < I ? ((q < 128 ? wg : wu) + ((size_t)e * I + i) * nvec) : nullptr;
        uint4* dst = packed + (size_t)row * nvec;
        for (int v = threadIdx.x; v < nvec; v += blockDim.x)
            dst[v] = src ? src[v] : make_uint4(0, 0, 0, 0);
    }
}

// Tiled weight layout: out[g][nt][kb][r][0..128 B) = w[g][256*nt + r][128*kb .. 128*kb + 128 B),
// zero past the matrix.  One 16-byte chunk per thread and step, writes in output order.
__global__ void tile_weights_kernel(const uint8_t* __restrict__ w, int G, int n_rows, int row_bytes, int NT, int KBt,
                                    uint4* __restrict__ out) {
    const int64_t total = (int64_t)G * NT * KBt * 256 * 8;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
        const int c = (int)(i & 7);
        int64_t t = i >> 3;
        const int r = (int)(t & 255);
        t >>= 8;
        const int kb = (int)(t % KBt);
        t /= KBt;
        const int nt = (int)(t % NT);
        const int64_t g = t / NT;
        const int row = nt * 256 + r;
        const int64_t byte = (int64_t)kb * 128 + c * 16;
        uint4 v = make_uint4(0, 0, 0, 0);
        if (row < n_rows && byte < row_bytes)
            v = __ldg(reinterpret_cast<const uint4*>(w + (g * n_rows + row) * (int64_t)row_bytes + byte));
        out[i] = v;
    }
}

}  // namespace

size_t tiled_weight_bytes(int G, int n_rows, int row_bytes) {
    return (size_t)G * (size_t)ceil_div(n_rows, 256) * (size_t)ceil_div(row_bytes, 128) * 256 * 128;
}

moe_status_t launch_tile_weights(const void* w, int G, int n_rows, int row_bytes, void* tiled, cudaStream_t s) {
    const int NT = (int)ceil_div(n_rows, 256), KBt = (int)ceil_div(row_bytes, 128);
    const int64_t total = (int64_t)G * NT * KBt * 256 * 8;
    if (total == 0) return MOE_OK;
    const int grid = (int)std::min<int64_t>(ceil_div(total, 256), (int64_t)sm_count() * 16);
    tile_weights_kernel<<<grid, 256, 0, s>>>(static_cast<const uint8_t*>(w), G, n_rows, row_bytes, NT, KBt,
                                             static_cast<uint4*>(tiled));
    note_launch();
    return last_launch_status();
}

size_t init_routing_scratch_bytes(int T, int E, int k) {
    const int64_t R = (int64_t)T * k;
    const int64_t NW = ceil_div(R, kChunk);
    return (size_t)(NW > 0 ? NW : 1) * (size_t)E * sizeof(int32_t);
}

moe_status_t launch_init_routing_index(const int32_t* ids, int R, int E, int32_t* counts, int32_t* offsets,
                                       int32_t* row_idx, int32_t* scratch, uint32_t* status, cudaStream_t s) {
    const int NW = (int)ceil_div(R, kChunk);
    if (NW == 0) {  // no rows: every expert empty
        MOE_CUDA_TRY(cudaMemsetAsync(counts, 0, (size_t)E * sizeof(int32_t), s));
        MOE_CUDA_TRY(cudaMemsetAsync(offsets, 0, (size_t)(E + 1) * sizeof(int32_t), s));
        return MOE_OK;
    }
    MOE_CUDA_TRY(launch_pdl(hist_kernel, dim3(NW), dim3(kChunkThreads), (size_t)E * sizeof(int32_t), s, ids, R, E,
                            NW, scratch, status));
    note_launch();
    MOE_CUDA_TRY(launch_pdl(scatter_kernel, dim3(NW), dim3(kChunkThreads),
                            (size_t)(kChunkWarps + 2) * E * sizeof(int32_t), s, ids, R, E, NW,
                            static_cast<const int32_t*>(scratch), counts, offsets, row_idx));
    note_launch();
    return MOE_OK;
}

moe_status_t launch_permute_rows(const void* x, size_t row_bytes, const int32_t* row_idx, int T, int k,
                                 void* expanded_x, cudaStream_t s, int blocks_per_sm) {
    if (T == 0) return MOE_OK;
    const int nvec = (int)(row_bytes / 16);
    const int grid = (int)std::min<int64_t>(T, (int64_t)sm_count() * std::max(1, blocks_per_sm));
    MOE_CUDA_TRY(launch_pdl(permute_rows_kernel, dim3(grid), dim3(kCopyThreads), 0, s,
                            static_cast<const uint4*>(x), nvec, row_idx, T, k, T * k,
                            static_cast<uint4*>(expanded_x)));
    note_launch();
    return MOE_OK;
}

moe_status_t launch_pack_w13(const void* w_gate, const void* w_up, size_t esize, int E, int H, int I,
                             void* packed, cudaStream_t s) {
    const int Ip = (int)round_up((size_t)I, 128);
    const int nvec = (int)((size_t)H * esize / 16);
    const int64_t rows = (int64_t)E * 2 * Ip;
    const int grid = (int)std::min<int64_t>(rows, (int64_t)sm_count() * 32);
    pack_w13_kernel<<<grid, 128, 0, s>>>(static_cast<const uint4*>(w_gate), static_cast<const uint4*>(w_up),
                                         E, I, Ip, nvec, static_cast<uint4*>(packed));
    note_launch();
    return last_launch_status();
}

}  // namespace moe
