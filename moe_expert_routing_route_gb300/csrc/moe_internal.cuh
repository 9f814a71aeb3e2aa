// Internal declarations of libmoe: launchers each .cu file provides, and the
// small helpers they share.  Not part of the public ABI (that is include/moe.h).
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cstdint>
#include <cstddef>
#include <algorithm>
#include <utility>

#include "moe.h"

namespace moe {

// ---- launch bookkeeping ------------------------------------------------------
void note_launch();                    // counts one kernel launch
moe_status_t last_launch_status();     // MOE_ERR_CUDA if the last launch failed
int sm_count();                        // SMs of the current device (cached per device)

#define MOE_TRY(expr)                           \
    do {                                        \
        moe_status_t _st = (expr);              \
        if (_st != MOE_OK) return _st;          \
    } while (0)

#define MOE_CUDA_TRY(expr)                      \
    do {                                        \
        if ((expr) != cudaSuccess) return MOE_ERR_CUDA; \
    } while (0)

// Programmatic dependent launch: the kernel may be scheduled while the previous kernel on the
// stream is still running; it must call pdl_wait() before reading anything that work earlier on
// the stream wrote (that wait covers the previous grid's completion and, through its own wait,
// everything before it).  With no running predecessor kernel this is an ordinary launch.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
inline int64_t ceil_div(int64_t a, int64_t b) { return (a + b - 1) / b; }
inline size_t round_up(size_t a, size_t b) { return (a + b - 1) / b * b; }
inline size_t dt_size(moe_dtype_t dt) { return dt == MOE_BF16 ? 2 : 4; }

// ---- device helpers -------------------------------------------------------------
__device__ __forceinline__ void set_status(uint32_t* status, uint32_t bit) {
    if (status) atomicOr(status, bit);
}
// The dependent grid (launched with launch_pdl) may be scheduled once every CTA of this grid has
// called this or exited; it still waits in pdl_wait() for this grid to complete.
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// Waits until the preceding grid on the stream has completed and its writes are visible.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- launchers (stream-ordered, no host sync) ------------------------------------
// route.cu
// n_group <= 1: flat top-k; otherwise group-limited (topk_group groups kept,
// rule 0 = group max, rule 1 = sum of the group's two largest scores).
// nsplit > 1: the logits arrive as nsplit partial sums, slice i at logits + i*slice_stride
// (0: T*E); they are added in slice order and the sums written back to slice 0.
moe_status_t launch_route_topk(const float* logits, const float* bias, int T, int E, int k, int renorm,
                               int32_t* ids, float* w, cudaStream_t s, int n_group = 1, int topk_group = 1,
                               int rule = 0, int nsplit = 1, int64_t slice_stride = 0);

// permute.cu
size_t init_routing_scratch_bytes(int T, int E, int k);
moe_status_t launch_init_routing_index(const int32_t* ids, int R, int E, int32_t* counts,
                                       int32_t* offsets, int32_t* row_idx, int32_t* scratch,
                                       uint32_t* status, cudaStream_t s);
// blocks_per_sm: grid = SMs x this (16 saturates HBM alone; the layer takes 2 when the
// shared experts' GEMM runs beside the copy, so fewer copy warps compete for its issue slots)
moe_status_t launch_permute_rows(const void* x, size_t row_bytes, const int32_t* row_idx, int T, int k,
                                 void* expanded_x, cudaStream_t s, int blocks_per_sm = 16);
// The tiled weight layout of the tensor-core GEMMs' B operand: [G][ceil(n/256)][ceil(row_bytes/128)][256][128 B]
// (each 256-row x 128-byte box one contiguous 32 KB block), zero-padded.
size_t tiled_weight_bytes(int G, int n_rows, int row_bytes);
moe_status_t launch_tile_weights(const void* w, int G, int n_rows, int row_bytes, void* tiled, cudaStream_t s);
moe_status_t launch_pack_w13(const void* w_gate, const void* w_up, size_t esize, int E, int H, int I,
                             void* packed, cudaStream_t s);

// ep.cu: Double-Routing pieces (re-routing, unsort, the virtual-rank exchange).
size_t re_routing_plan_ints(int W, int El);
moe_status_t launch_re_routing(const void* x_recv, size_t row_bytes, const int32_t* counts, int W, int El, int N,
                               void* x_sorted, int32_t* gidx, int32_t* tpl, int32_t* local_off, int32_t* plan,
                               uint32_t* status, cudaStream_t s);
moe_status_t launch_unsort_rows(const void* y_sorted, size_t row_bytes, const int32_t* gidx, int N, void* out,
                                uint32_t* status, cudaStream_t s);
struct EpBuffers {
    int W, T, E, k;
    size_t row_bytes;
    const void* x;          // [T,H]
    const int32_t* ids;     // [T,k]
    int32_t* row_idx;       // [T*k]: per source rank, rows local to the rank
    void* expanded;         // [T*k,H]: the source ranks' expanded rows, rank after rank
    void* recv;             // [T*k,H]: rows as received, receiving rank after rank
    void* sorted;           // [T*k,H]: received rows sorted by local expert
    int32_t* gidx;          // [T*k]: sorted row -> received row
    int32_t* scratch;       // ep_scratch_ints(W, E)
    int32_t* hist_scratch;  // init-routing histogram scratch for T/W tokens
    uint32_t* status;
};
size_t ep_scratch_ints(int W, int E);
moe_status_t ep_route_and_dispatch(const EpBuffers& b, cudaStream_t s);
size_t ep_recv_start_int(int W, int E);      // int offsets of recv_start and of the global
size_t ep_expert_offsets_int(int W, int E);  // expert offsets inside the EP scratch
const int32_t* ep_rank_offsets(const EpBuffers& b, int q);  // [E/W + 1] rows of rank q's experts in `sorted`
const int32_t* ep_expert_offsets(const EpBuffers& b);       // [E + 1] rows of every expert in `sorted`
moe_status_t ep_combine(const EpBuffers& b, const void* y_sorted, void* y_recv, void* y_expanded, cudaStream_t s);

// quant.cu: FP8 (e4m3) block quantisation.
// pow2: power-of-two block scales (the format the block-scaled tensor-core GEMM takes).
// pdl: programmatic dependent launch (false on the second stream, as the other launchers)
moe_status_t launch_quantize_rows_fp8(const void* a, moe_dtype_t dt, int64_t rows, int cols, uint8_t* codes,
                                      float* scales, int ld_scales, cudaStream_t s, bool pow2 = false,
                                      bool pdl = true);
moe_status_t launch_quantize_tiles_fp8(const void* w, moe_dtype_t dt, int G, int rows, int cols, uint8_t* codes,
                                       float* scales, cudaStream_t s, bool pow2 = false);

// finalize.cu
moe_status_t launch_finalize(const void* y, int64_t y_rows, const void* skip, const float* w,
                             const int32_t* row_idx, moe_dtype_t dt, int T, int H, int k, void* out,
                             uint32_t* status, cudaStream_t s);

// gemm_tc.cu: bf16 tcgen05 grouped GEMM, C = A B^T per group.
// TC_EPI_FFN: one pair-tile launch runs an up projection (SwiGLU) and then the down projection of
// its output (launch_tc_pair_ffn)
enum TcEpilogue { TC_EPI_SWIGLU = 0, TC_EPI_BF16 = 1, TC_EPI_F32 = 2, TC_EPI_FFN = 3 };
struct TcGroupedGemm {
    const void* A;            // [M, K] bf16, row stride K
    int M;                    // rows of A
    int K;
    const int32_t* offsets;   // [G+1] device, or nullptr for one group [0, M)
    int G;
    const void* B;            // [G * Nb, K] bf16
    int Nb;                   // B rows per group
    int N;                    // valid output columns per group
    void* C;                  // output base (row r of A -> row r of C)
    int64_t ldc;              // elements
    TcEpilogue epi;
    uint32_t* status;
    int ksplit = 1;               // fp32 output only: at most this many K slices, slice s written at
    int64_t c_split_stride = 0;   // C + s * c_split_stride (elements); the caller sums the slices
    bool smem_headroom = false;   // pair tiles: take the 6-stage ring, leaving ~24 KB of shared memory per SM
                                  // for kernels of other streams (the 7-stage ring leaves under 1 KB)
    bool b_tiled = false;         // B in the tiled layout (tiled_weight_bytes(G, Nb, 2K)); bf16/SwiGLU epilogues only
    int max_ctas = 0;             // persistent grid cap (0: one CTA per SM), leaving SMs to other streams' kernels
    bool pdl = true;              // programmatic dependent launch (false for kernels on the second stream, whose
                                  // followers placed early hold SMs the first stream's kernels need)
    bool exact_split = false;     // fp32 output: exactly ksplit K slices (the slices of another launch over more
                                  // rows, so that the partial sums agree bit for bit)
    int part = 0;                 // rows of each group to cover: all (0), the pair-tile part (1) or the tail (2)
};
moe_status_t launch_tc_grouped_gemm(const TcGroupedGemm& g, cudaStream_t s);
// One dense FFN (one group, no offsets: the shared experts) in one persistent pair-tile launch:
// the up projection's tiles (SwiGLU epilogue into up.C), then the down projection's (down.A ==
// up.C), whose tiles of 256 rows start as soon as every up tile of those rows is stored.  sync:
// ceil(M / 256) zeroed ints of device memory.  UNSUPPORTED unless both would take pair tiles.
moe_status_t launch_tc_pair_ffn(const TcGroupedGemm& up, const TcGroupedGemm& down, int* sync, cudaStream_t s);
int tc_gate_splits(int M, int N, int K, int max_split);  // K slices the fp32 launch will use

// gemm_fp8.cu: e4m3 block-scaled grouped GEMM (bf16 out), C = A B^T per group.
struct TcFp8GroupedGemm {
    const void* A;            // [M, K] e4m3 codes
    int M;
    int K;
    const int32_t* offsets;   // [G+1] device, or nullptr for one group [0, M)
    int G;
    const void* B;            // [G * Nb, K] e4m3 codes
    int Nb;                   // B rows per group (a multiple of 256)
    int N;                    // valid output columns per group
    void* C;                  // bf16 output
    int64_t ldc;
    TcEpilogue epi;           // TC_EPI_SWIGLU or TC_EPI_BF16
    const float* a_scales;    // [M][lda_scales]: one per 1x128 block of A
    int lda_scales;
    const float* b_scales;    // [G][Nb/128][ceil(K/128)]: one per 128x128 tile of B
    uint32_t* status;
    uint8_t* q = nullptr;     // SwiGLU: also quantise h in 1x128 blocks into codes [M, N] (C may then be null)
    float* q_scales = nullptr;  // [M][ldq]
    int ldq = 0;
    // Power-of-two scales: the tensor cores apply them (kind::mxf8f6f4 block
    // scaling, one accumulator per tile, no promotion on CUDA cores) and the
    // SwiGLU epilogue quantises h with power-of-two scales too.  Every scale of A
    // and B must then be a power of two (its exponent is what is used).
    bool pow2 = false;
    bool b_tiled = false;     // B codes in the tiled layout (tiled_weight_bytes(G, Nb, K))
    bool pdl = true;          // programmatic dependent launch (as TcGroupedGemm::pdl)
};
moe_status_t launch_tc_fp8_grouped_gemm(const TcFp8GroupedGemm& g, cudaStream_t s);
int tc_packed_block();        // rows of gate (and of up) per packed block: 128

// gemm_simt.cu: fp32 (FFMA) GEMMs of the same shapes.
moe_status_t launch_simt_gate(const float* x, const float* wr, int T, int H, int E, float* logits,
                              cudaStream_t s);
// pdl: programmatic dependent launch (as TcGroupedGemm::pdl)
moe_status_t launch_simt_grouped_ffn_up(const float* a, int M, int H, const int32_t* offsets, int G,
                                        const float* w13_packed, int Ip, int I, float* h,
                                        uint32_t* status, cudaStream_t s, bool pdl = true);
moe_status_t launch_simt_grouped_down(const float* h, int M, int I, const int32_t* offsets, int G,
                                      const float* w2, int H, float* y, uint32_t* status,
                                      cudaStream_t s, bool pdl = true);

}  // namespace moe
