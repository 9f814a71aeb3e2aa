/*
 * moe.h -- C ABI of libmoe, the single-GPU MoE layer hot path for GB300 (sm_103a).
 *
 *   logits = x Wr^T                     (gate GEMM)
 *   top-k routing                       (moe_route_topk)
 *   init-routing permutation            (moe_init_routing)
 *   per-expert SwiGLU FFN, grouped GEMM (moe_grouped_ffn)
 *   finalize-routing + shared expert    (moe_finalize_routing)
 *   all of the above on one stream      (moe_layer_forward)
 *
 * Sources for the operations (cited per entry point below):
 *   [BLOG] "Lower latency and higher throughput with multi-node DeepSeek
 *          deployment" (Perplexity blog): §Expert Parallelism, §Roofline /
 *          GroupGEMM, §Roofline / GEMM, §Quantization, §CUDA Graph, §MoE Router.
 *   [CANN] "DeepSeek-R1 prefill inference optimisation on Atlas A3"
 *          (cann-recipes-infer): §MoE deployment strategy, Double-Routing
 *          steps 1 (init-routing), 6 (argsort inverse) and 8 (finalize-routing).
 *
 * Conventions shared by every entry point:
 *   - Every pointer argument is a DEVICE pointer unless its name ends in _host.
 *     The caller allocates and owns all memory, including workspaces; the
 *     library never allocates, frees or synchronises (except
 *     moe_check_device_status and moe_layer_forward_host, which say so).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *     stream).  The entry points other than moe_layer_forward_host,
 *     moe_check_device_status and moe_init_routing_noalloc issue no host
 *     synchronisation, so a sequence of them can be captured into a CUDA graph.
 *   - Device pointers must be 16-byte aligned.  Matrices are row-major and
 *     contiguous; weights are stored like Linear weights, [out, in] with the
 *     reduction dimension contiguous.
 *   - dtype: MOE_F32 (float) or MOE_BF16 (bfloat16).  Accumulation is fp32.
 *   - Argument errors are returned synchronously (MOE_ERR_INVALID_ARG,
 *     MOE_ERR_UNSUPPORTED) before anything is enqueued.  A failed launch returns
 *     MOE_ERR_CUDA.  Data errors found on the device (an expert id outside
 *     [0,E), a row index outside its buffer, inconsistent offsets, a bounded
 *     wait that ran out) never trap: the kernel skips the offending row, sets a
 *     bit in the status word at the start of the workspace and carries on.
 *     Every entry point that takes a workspace clears that word first;
 *     moe_check_device_status reads it.  After a data error the outputs are
 *     unspecified.
 *   - Sizes: 0 <= T, 1 <= k <= min(E, 32), E <= 1024, H % 8 == 0, I % 8 == 0,
 *     T*k < 2^31.  T == 0 is a no-op.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1, /* null pointer, size out of range, workspace too small */
    MOE_ERR_UNSUPPORTED = 2, /* valid request outside what the kernels handle (alignment, dtype, shape) */
    MOE_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
    MOE_ERR_DEVICE = 4       /* moe_check_device_status: the device status word is non-zero */
} moe_status_t;

typedef enum moe_dtype { MOE_F32 = 0, MOE_BF16 = 1 } moe_dtype_t;

/* Bits of the device status word (first 4 bytes of a workspace). */
#define MOE_DEVERR_BAD_EXPERT_ID 0x1u /* init-routing met an id outside [0,E) */
#define MOE_DEVERR_BAD_ROW_INDEX 0x2u /* finalize met an expanded_row_idx outside [0,rows) */
#define MOE_DEVERR_BAD_OFFSETS 0x4u   /* grouped FFN got decreasing or out-of-range offsets */
#define MOE_DEVERR_TIMEOUT 0x8u       /* a bounded on-chip wait gave up (about one second) */

/* Every workspace starts with this many bytes of header (the status word). */
#define MOE_WS_HEADER_BYTES 256

/* Version of this ABI; bumped on any incompatible change.  2: moe_layer_desc
 * ends with a weight_layout field; weight_format takes MOE_WEIGHTS_FP8_POW2. */
int moe_abi_version(void);

/* Human-readable name of a status code (static storage). */
const char* moe_status_string(moe_status_t status);

/* Number of kernels this library has launched in this process (all devices). */
uint64_t moe_kernel_launch_count(void);

/* Diagnostic of the bounded on-chip waits (no counterpart on the pages): one
 * CTA waits on an mbarrier that nothing arrives on.  Its first warp gives up
 * after limit_ns (1 ns .. 10 s) and sets MOE_DEVERR_TIMEOUT in the status word
 * of `ws` (cleared first); its second warp, which has no limit of its own,
 * leaves through the shared abort flag the first one raises.  *outcome
 * (device, uint32) receives bit 0 when the first warp timed out and bit 1 when
 * the second left through the flag.  No trap, no hang; asynchronous. */
moe_status_t moe_diag_bounded_wait(uint64_t limit_ns, void* ws, uint32_t* outcome, moe_stream_t stream);

/* Synchronises `stream`, then reads and returns the status word of `ws` in
 * *word (may be NULL).  Returns MOE_OK if the word is zero, MOE_ERR_DEVICE if
 * not, MOE_ERR_CUDA if the synchronisation failed.  This call blocks. */
moe_status_t moe_check_device_status(const void* ws, moe_stream_t stream, uint32_t* word);

/* ---------------------------------------------------------------------------
 * Gate GEMM.  [BLOG §Roofline / GEMM]: a Linear projection is [m,k]x[k,n].
 *   logits[t,e] = sum_h x[t,h] * w_router[e,h]        (fp32 accumulate and out)
 * x [T,H], w_router [E,H] in dt; logits [T,E] fp32.
 * bf16 runs on tcgen05 tensor cores; fp32 runs on the FFMA pipes. */
moe_status_t moe_gate_logits(const void* x, const void* w_router, moe_dtype_t dt, int T, int H,
                             int E, float* logits, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Top-k routing.  [BLOG §MoE Router]: top-k of the router scores, keeping
 * the indices of the selected experts; [BLOG §Expert Parallelism]: each token
 * goes to k distinct routed experts whose outputs are summed with weights.
 *   s_e        = logits[t,e] + expert_bias[e]   (one fp32 add; bias may be NULL)
 *   topk_ids   = the k experts with the largest s, in descending order of s;
 *                equal scores go to the lower expert id (ids are distinct)
 *   topk_w     = softmax over all E scores, taken at the selected experts;
 *                with renormalize != 0 divided by their sum (so they sum to 1)
 * logits [T,E] fp32, finite; expert_bias [E] fp32 or NULL;
 * topk_ids [T,k] int32, topk_w [T,k] fp32 (outputs, row-major). */
moe_status_t moe_route_topk(const float* logits, const float* expert_bias, int T, int E, int k,
                            int renormalize, int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/* Group-limited top-k.  [BLOG §MoE Router]: flat routing is the special case
 * of DeepSeek routing in which the selected group is all experts.  The E
 * experts form n_group contiguous groups of E/n_group; a group's score is the
 * largest s_e in it (group_rule 0) or the sum of its two largest s_e as one
 * fp32 add (group_rule 1); the topk_group best groups are kept (ties to the
 * lower group index); topk_ids are the k best experts of the kept groups
 * (descending s, ties to the lower id).  Weights as in moe_route_topk (softmax
 * over all E scores at the selected experts, renormalised when asked).
 * 1 <= n_group <= 32, E % n_group == 0, 1 <= topk_group <= n_group,
 * k <= topk_group * E/n_group; group_rule 1 needs E/n_group >= 2.
 * n_group == 1 is exactly moe_route_topk. */
#define MOE_GROUP_SCORE_MAX 0
#define MOE_GROUP_SCORE_TOP2_SUM 1
moe_status_t moe_route_topk_grouped(const float* logits, const float* expert_bias, int T, int E, int k,
                                    int n_group, int topk_group, int group_rule, int renormalize,
                                    int32_t* topk_ids, float* topk_w, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Init-routing.  [CANN §MoE deployment, Double-Routing step 1]: expand every
 * token k times and sort the copies by expert, returning expanded_x,
 * expanded_row_idx (which restores the original order) and tokens_per_expert.
 * With source row src = t*k + j (token-major):
 *   tokens_per_expert[e] = #{src : topk_ids[src] == e}
 *   expert_offsets[e]    = sum_{e' < e} tokens_per_expert[e'],  expert_offsets[E] = T*k
 *   expanded_row_idx[src] = expert_offsets[id] + #{src' < src : topk_ids[src'] == id}
 *   expanded_x[expanded_row_idx[src], :] = x[src / k, :]
 * i.e. a stable sort by expert id; no token is dropped or padded.
 * x [T,H] dt; topk_ids [T,k] int32 (ids need not be distinct);
 * outputs expanded_x [T*k,H] dt, expanded_row_idx [T*k] int32,
 * tokens_per_expert [E] int32, expert_offsets [E+1] int32.
 * ws: at least moe_init_routing_workspace_bytes(T,E,k) bytes (scratch +
 * status word).  An id outside [0,E) is not counted, its expanded_row_idx is
 * -1 and MOE_DEVERR_BAD_EXPERT_ID is set. */
size_t moe_init_routing_workspace_bytes(int T, int E, int k);
moe_status_t moe_init_routing(const void* x, moe_dtype_t dt, const int32_t* topk_ids, int T, int H,
                              int E, int k, void* expanded_x, int32_t* expanded_row_idx,
                              int32_t* tokens_per_expert, int32_t* expert_offsets, void* ws,
                              size_t ws_bytes, moe_stream_t stream);

/* Init-routing without a workspace, for callers that cannot allocate device
 * memory: for example a serving engine that gives all device memory to its own
 * pool at start-up and permits no further cudaMalloc, a latency-critical loop
 * that must not pay cudaMalloc's implicit synchronisation, or a C program with
 * no device allocator.  The pages have no counterpart to this entry point.
 * Outputs and argument meanings are those of moe_init_routing; the caller still
 * passes every input and output buffer.
 * Scratch: a fixed 1 MiB array in this library's device memory (262144 int32),
 * held on every GPU that loads the library until the process exits.  A call
 * needs ceil(T*k/1024)*E of those ints (E=256: up to 1,048,576 expanded rows);
 * a larger call returns MOE_ERR_UNSUPPORTED.  No allocation of any kind is made.
 * The first call on a device looks up the array's device address (with that
 * device current) and keeps it; make that first call before any stream
 * capture.  The address is tied to the device's context: the first call after
 * a cudaDeviceReset of that device (a new context) looks it up again, so make
 * that call outside stream capture too.  All calls share the array and it
 * keeps the last call's contents (every entry a call reads is rewritten by
 * that call, so nothing needs clearing), but calls whose kernels overlap on
 * the GPU race on it.  There is
 * no status word: an id outside [0,E) shows as expanded_row_idx = -1 and is not
 * counted in tokens_per_expert. */
moe_status_t moe_init_routing_noalloc(const void* x, moe_dtype_t dt, const int32_t* topk_ids, int T, int H,
                                      int E, int k, void* expanded_x, int32_t* expanded_row_idx,
                                      int32_t* tokens_per_expert, int32_t* expert_offsets,
                                      moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Expert weight packing for the grouped FFN.  Interleaves each expert's gate
 * and up projections in blocks of 128 output rows so that one GEMM tile holds
 * matching gate and up columns (the SwiGLU epilogue needs both):
 *   Ip = I rounded up to a multiple of 128
 *   packed[e, 256*b + r,       :] = w_gate[e, 128*b + r, :]   (0 <= r < 128)
 *   packed[e, 256*b + 128 + r, :] = w_up  [e, 128*b + r, :]
 * rows past I are zero.  w_gate, w_up [E,I,H] dt; packed [E, 2*Ip, H] dt,
 * moe_w13_packed_bytes(dt,E,H,I) bytes.  Shared experts are packed the same
 * way with E = 1 and I = S*I (their gate/up rows stacked). */
size_t moe_w13_packed_bytes(moe_dtype_t dt, int E, int H, int I);
moe_status_t moe_pack_w13(const void* w_gate, const void* w_up, moe_dtype_t dt, int E, int H, int I,
                          void* w13_packed, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Tiled weight layout.  [BLOG §Roofline / GroupGEMM]: at about 128 rows per
 * expert the grouped GEMM streams its weights from HBM.  The tensor-core GEMM
 * reads a weight as boxes of 256 rows x 128 bytes of K; in the row-major layout
 * such a box is 256 pieces 2*K bytes apart, in this layout it is one contiguous
 * 32 KB block, which HBM serves faster (fewer DRAM rows opened per byte):
 *   tiled[g][t][b][r][0..128 B) = w[g][256*t + r][128*b .. 128*b + 128 B)
 * for t < ceil(n_rows/256), b < ceil(row_bytes/128), zero past the matrix.
 * w: [G][n_rows][row_bytes] (any element type; row_bytes % 16 == 0); tiled:
 * moe_tiled_weight_bytes(G, n_rows, row_bytes) bytes.  For a layer, tile the
 * moe_pack_w13 output ([E][2*Ip][H], row_bytes = 2*H for bf16), w2 ([E][H][I]),
 * and the shared w13 ([1][2*Ips][H]) and w2 ([1][H][S*I]). */
size_t moe_tiled_weight_bytes(int G, int n_rows, int row_bytes);
moe_status_t moe_tile_weights(const void* w, int G, int n_rows, int row_bytes, void* tiled, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Grouped SwiGLU expert FFN.  [BLOG §Roofline / GroupGEMM]: g groups, group i
 * multiplies [m_i,k]x[k,n]; here group e is expert e's segment of rows
 * [expert_offsets[e], expert_offsets[e+1]) of `a`.  [BLOG §Expert Parallelism]
 * and [BLOG §Quantization] (SiLU):
 *   h[r,:] = silu(a[r,:] Wgate_e^T) * (a[r,:] Wup_e^T),  silu(z) = z/(1+exp(-z))
 *   y[r,:] = h[r,:] W2_e^T
 * h is stored in dt (fp32 accumulate, one rounding), y likewise.  Group sizes
 * are read on the device (no host round trip), so expert_offsets can be the
 * output of moe_init_routing on the same stream.
 * a [rows,H] dt; expert_offsets [E+1] int32 (device), or NULL for one group of
 * all `rows` rows (E must then be 1); w13_packed from moe_pack_w13; w2 [E,H,I];
 * y [rows,H] dt (rows outside every segment are left untouched).
 * ws: at least moe_grouped_ffn_workspace_bytes(dt,rows,I) bytes (h + status).
 * bf16 runs on tcgen05 tensor cores (TMA-fed, persistent, device-side tile
 * scheduler); fp32 runs on the FFMA pipes.  bf16 tiles are 128 rows on one SM,
 * or 256 rows on a two-CTA cluster (tcgen05.mma.cta_group::2) once the groups
 * average 256 rows or more; the environment variable MOE_GEMM_TILE=single or
 * MOE_GEMM_TILE=pair, read at every launch, forces one shape.  Both give the
 * same result up to fp32 summation order.  With pair tiles over 128 groups or
 * more that average 512 rows or more, each group's tail of at most 128 rows goes
 * to a second, single-CTA launch instead of a half-empty pair tile (the same
 * bits); MOE_GEMM_MIXED=1 or 0 forces that split on or off. */
/* moe_grouped_ffn with both weights in the tiled layout (moe_tile_weights of the
 * moe_pack_w13 output and of w2); bf16 only.  Same arguments and results. */
moe_status_t moe_grouped_ffn_tiled(const void* a, moe_dtype_t dt, const int32_t* expert_offsets, int E, int rows,
                                   int H, int I, const void* w13_tiled, const void* w2_tiled, void* y, void* ws,
                                   size_t ws_bytes, moe_stream_t stream);
size_t moe_grouped_ffn_workspace_bytes(moe_dtype_t dt, int rows, int I);
moe_status_t moe_grouped_ffn(const void* a, moe_dtype_t dt, const int32_t* expert_offsets, int E,
                             int rows, int H, int I, const void* w13_packed, const void* w2, void* y,
                             void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * FP8 block quantisation.  [BLOG §Quantization]: DeepSeek-V3/R1 quantises per
 * block -- weights statically with one scale per 128x128 tile, activations on
 * the fly with one scale per 128-element vector.  Format e4m3 (largest finite
 * 448); a block's scale is amax/448 in fp32 (1 for an all-zero block); a value's
 * code is round-to-nearest-even of fl32(v/scale), saturated at +-448.
 *
 * moe_quantize_rows_fp8: a [rows, cols] dt -> codes [rows, cols] uint8, scales
 * [rows, ld_scales] fp32 (ld_scales >= ceil(cols/128); 1x128 blocks).
 * moe_quantize_weights_fp8: w [G, n_out, k_in] dt -> codes [G, n_out, k_in],
 * scales [G][ceil(n_out/128)][ceil(k_in/128)] (128x128 tiles).  For w13 pass the
 * moe_pack_w13 output (n_out = 2*Ip); for the shared experts G = 1. */
moe_status_t moe_quantize_rows_fp8(const void* a, moe_dtype_t dt, int64_t rows, int cols, uint8_t* codes,
                                   float* scales, int ld_scales, moe_stream_t stream);
moe_status_t moe_quantize_weights_fp8(const void* w, moe_dtype_t dt, int G, int n_out, int k_in, uint8_t* codes,
                                      float* scales, moe_stream_t stream);

/* The same two quantisers with power-of-two block scales (the second scale
 * format).  [BLOG §Quantization] fixes the blocks but not the scales' number
 * format; here each scale is the smallest power of two 2^e with amax/2^e <= 448
 * (1 for an all-zero block, e >= -127), so a block's largest magnitude lands in
 * (224, 448] and a code is the nearest e4m3 value of an exact division.  The
 * scales are still written as fp32 values.  Arguments as above. */
moe_status_t moe_quantize_rows_fp8_pow2(const void* a, moe_dtype_t dt, int64_t rows, int cols, uint8_t* codes,
                                        float* scales, int ld_scales, moe_stream_t stream);
moe_status_t moe_quantize_weights_fp8_pow2(const void* w, moe_dtype_t dt, int G, int n_out, int k_in,
                                           uint8_t* codes, float* scales, moe_stream_t stream);

/* Grouped SwiGLU expert FFN with FP8 weights and activations ([BLOG
 * §Quantization], [BLOG §Roofline / GroupGEMM]): products are block-scaled,
 *   C[m,n] = sum_b sa[m,b] * sb[n/128,b] * sum_{k in block b} qa[m,k] qb[n,k],
 * h = silu(gate) * up is rounded to bf16 and quantised in 1x128 blocks for the
 * down projection by the up GEMM's own epilogue (the workspace keeps the bf16
 * h, its codes and its scales); y [rows, H] bf16.  aq [rows, H] codes with a_scales
 * [rows, lda_scales]; w13q/w13s and w2q/w2s from moe_quantize_weights_fp8;
 * expert_offsets as in moe_grouped_ffn.  H % 256 == 0, I % 16 == 0.
 * ws: moe_grouped_ffn_fp8_workspace_bytes(rows, I) bytes. */
size_t moe_grouped_ffn_fp8_workspace_bytes(int rows, int I);
moe_status_t moe_grouped_ffn_fp8(const uint8_t* aq, const float* a_scales, int lda_scales,
                                 const int32_t* expert_offsets, int E, int rows, int H, int I, const uint8_t* w13q,
                                 const float* w13s, const uint8_t* w2q, const float* w2s, void* y, void* ws,
                                 size_t ws_bytes, moe_stream_t stream);

/* moe_grouped_ffn_fp8 with power-of-two scales on every operand (from the _pow2
 * quantisers): the same product, but the tensor cores apply the scales
 * (block-scaled MMA taking one 8-bit exponent per 32 K elements of every row of
 * A and column of B), so each tile accumulates in one TMEM accumulator with no
 * per-block promotion on CUDA cores; h is quantised with power-of-two scales.
 * A scale that is not a power of two acts as its exponent (rounded down to a
 * power of two).  Arguments, workspace and sizes as moe_grouped_ffn_fp8. */
moe_status_t moe_grouped_ffn_fp8_pow2(const uint8_t* aq, const float* a_scales, int lda_scales,
                                      const int32_t* expert_offsets, int E, int rows, int H, int I,
                                      const uint8_t* w13q, const float* w13s, const uint8_t* w2q, const float* w2s,
                                      void* y, void* ws, size_t ws_bytes, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Finalize-routing.  [CANN §MoE deployment, Double-Routing step 8]: restore
 * the token order through expanded_src_to_dst_row, weight by scales=topk_weight
 * and add the shared expert output (skip1):
 *   out[t,:] = skip[t,:] + sum_j topk_w[t,j] * y[expanded_row_idx[t*k+j], :]
 * summed in fp32 and rounded once to dt.  y [y_rows,H] dt; skip [T,H] dt or
 * NULL; topk_w [T,k] fp32; expanded_row_idx [T*k] int32; out [T,H] dt.
 * ws: NULL, or a workspace of at least MOE_WS_HEADER_BYTES whose status word
 * receives MOE_DEVERR_BAD_ROW_INDEX for an index outside [0,y_rows) (that
 * term is skipped either way). */
moe_status_t moe_finalize_routing(const void* y, int64_t y_rows, const void* skip, const float* topk_w,
                                  const int32_t* expanded_row_idx, moe_dtype_t dt, int T, int H, int k,
                                  void* out, void* ws, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * Re-routing.  [CANN §MoE deployment, Double-Routing step 4]: after the
 * token AlltoAll a rank holds, from each of W source ranks in rank order, that
 * source's rows for the rank's E_local experts, grouped by local expert in
 * expert order (the layout init-routing gives a contiguous expert range).
 * Re-routing sorts them by local expert, stable (source order, then arrival):
 *   x_sorted[i, :] = x_recv[gathered_ids_unsort[i], :]
 *   tokens_per_local_expert[e] = sum_p counts[p, e];  local_offsets = exclusive scan [E_local+1]
 * counts [W, E_local] int32 (device); x_recv, x_sorted [N, H] dt with N the
 * sum of counts (checked on the device: a mismatch moves no rows and sets
 * MOE_DEVERR_BAD_OFFSETS); gathered_ids_unsort [N] int32.
 * ws: moe_re_routing_workspace_bytes(W, E_local) bytes. */
size_t moe_re_routing_workspace_bytes(int W, int E_local);
moe_status_t moe_re_routing(const void* x_recv, moe_dtype_t dt, const int32_t* counts, int W, int E_local, int N,
                            int H, void* x_sorted, int32_t* gathered_ids_unsort, int32_t* tokens_per_local_expert,
                            int32_t* local_offsets, void* ws, size_t ws_bytes, moe_stream_t stream);

/* [CANN §MoE deployment, Double-Routing step 6]: the rows back in received
 * order, the page's index_select with the argsort of gathered_ids_unsort:
 *   out[gathered_ids_unsort[i], :] = y_sorted[i, :]
 * y_sorted, out [N, H] dt; ws NULL or a workspace whose status word receives
 * MOE_DEVERR_BAD_ROW_INDEX for an index outside [0, N). */
moe_status_t moe_unsort_rows(const void* y_sorted, moe_dtype_t dt, const int32_t* gathered_ids_unsort, int N, int H,
                             void* out, void* ws, moe_stream_t stream);

/* ---------------------------------------------------------------------------
 * The whole layer.  [BLOG §Expert Parallelism]: out[t] = shared(x_t) +
 * sum_j w_j FFN_{e_j}(x_t) with 8-of-256 style top-k routing; the steps above
 * run back to back on one stream with fixed grids and no host synchronisation
 * ([BLOG §Quantization]: persistent kernels read the routing counts on the
 * device; [BLOG §CUDA Graph]: the call can be captured in a CUDA graph). */
typedef struct moe_layer_desc {
    int T;  /* tokens */
    int H;  /* hidden size */
    int E;  /* routed experts */
    int k;  /* experts per token */
    int I;  /* intermediate size of one expert */
    int S;  /* shared experts (each of intermediate size I); 0 = none */
    moe_dtype_t dtype;
    int renormalize;           /* top-k weights renormalised to sum 1 */
    const void* w_router;      /* [E,H] */
    const float* expert_bias;  /* [E] fp32 added to the logits, or NULL */
    const void* w13;           /* moe_pack_w13(w_gate [E,I,H], w_up [E,I,H]) */
    const void* w2;            /* [E,H,I] */
    const void* w13_shared;    /* moe_pack_w13 with E=1, I=S*I of the stacked shared gate/up [S*I,H]; NULL iff S == 0 */
    const void* w2_shared;     /* [H, S*I]: the shared down projections side by side; NULL iff S == 0 */
    int n_group;               /* 0 or 1: flat top-k; > 1: group-limited (moe_route_topk_grouped) */
    int topk_group;            /* groups kept when n_group > 1 */
    int group_rule;            /* MOE_GROUP_SCORE_MAX or MOE_GROUP_SCORE_TOP2_SUM */
    int weight_format;         /* MOE_WEIGHTS_NATIVE, MOE_WEIGHTS_FP8 or MOE_WEIGHTS_FP8_POW2 (bf16 layers only) */
    const float* w13_scales;   /* FP8: tile scales of w13 [E][2*Ip/128][ceil(H/128)] (moe_quantize_weights_fp8) */
    const float* w2_scales;    /* FP8: tile scales of w2 [E][H/128][ceil(I/128)] */
    const float* w13_shared_scales; /* FP8: [1][2*Ips/128][ceil(H/128)], Ips = S*I rounded up to 128 */
    const float* w2_shared_scales;  /* FP8: [1][H/128][ceil(S*I/128)] */
    int weight_layout;         /* MOE_LAYOUT_ROWS (0) or MOE_LAYOUT_TILED (bf16 layers): the four expert
                                  weights above (w13, w2 and the shared ones; for FP8 their codes) passed
                                  through moe_tile_weights; w_router and the FP8 scales stay as they are */
} moe_layer_desc;

/* Expert-weight layouts of moe_layer_desc (and of moe_grouped_ffn_tiled). */
#define MOE_LAYOUT_ROWS 0
#define MOE_LAYOUT_TILED 1

/* Weight formats of moe_layer_desc.  With MOE_WEIGHTS_FP8 the w13/w2 pointers
 * (routed and shared) hold e4m3 codes in the same layouts (one byte per
 * element) with 128x128 tile scales beside them; the activations are quantised
 * on the fly in 1x128 blocks ([BLOG §Quantization]); the gate GEMM, routing and
 * all outputs stay bf16.  Requires dtype MOE_BF16, H % 256 == 0, I % 16 == 0. */
#define MOE_WEIGHTS_NATIVE 0
#define MOE_WEIGHTS_FP8 1
/* As MOE_WEIGHTS_FP8 with power-of-two scales everywhere (weights quantised
 * with moe_quantize_weights_fp8_pow2; x and h quantised on the fly the same
 * way), so the expert GEMMs run as block-scaled tensor-core MMAs. */
#define MOE_WEIGHTS_FP8_POW2 2

/* Layer steps timed by moe_layer_forward_timed.  "shared" (both projections of
 * the shared experts) runs on a second stream of the library's, forked when
 * the gate starts and joined before "up", concurrently with gate, route,
 * init_routing and permute_rows; "up" and "down" are the routed experts.  In
 * FP8 layers with shared experts, "shared" also holds the quantisation of x
 * (its codes are waited for before permute_rows); without them, "gate" does. */
#define MOE_NUM_STAGES 8
const char* moe_stage_name(int stage); /* "gate", "route", "init_routing", "permute_rows",
                                          "shared", "up", "down", "finalize" */

/* Workspace fields of the layer (intermediates a caller may inspect). */
typedef enum moe_ws_field {
    MOE_WS_LOGITS = 0,            /* [T,E] fp32 (bf16 layers: room for 8 K slices, the sums in the first) */
    MOE_WS_TOPK_IDS = 1,          /* [T,k] int32 */
    MOE_WS_TOPK_W = 2,            /* [T,k] fp32 */
    MOE_WS_TOKENS_PER_EXPERT = 3, /* [E] int32 */
    MOE_WS_EXPERT_OFFSETS = 4,    /* [E+1] int32 */
    MOE_WS_EXPANDED_ROW_IDX = 5,  /* [T*k] int32 */
    MOE_WS_EXPANDED_X = 6,        /* [T*k,H] dt */
    MOE_WS_H_ROUTED = 7,          /* [T*k,I] dt */
    MOE_WS_H_SHARED = 8,          /* [T,S*I] dt */
    MOE_WS_Y_ROUTED = 9,          /* [T*k,H] dt */
    MOE_WS_Y_SHARED = 10,         /* [T,H] dt */
    MOE_WS_X_IN = 11,             /* [T,H] dt: staging for moe_layer_forward_host */
    MOE_WS_OUT = 12,              /* [T,H] dt: staging for moe_layer_forward_host */
    MOE_WS_XQ = 13,               /* FP8 only: [T,H] e4m3 codes of x */
    MOE_WS_XQ_SCALES = 14,        /* FP8 only: [T, ceil(H/128) rounded up to 4] fp32 */
    MOE_WS_EXPANDED_XQ = 15,      /* FP8 only: [T*k,H] codes, expert-sorted */
    MOE_WS_EXPANDED_XQ_SCALES = 16, /* FP8 only: [T*k, ...] fp32 */
    MOE_WS_HQ = 17,               /* FP8 only: [T*k,I] codes of h */
    MOE_WS_HQ_SCALES = 18,        /* FP8 only: [T*k, ceil(I/128) rounded up to 4] fp32 */
    MOE_WS_HQ_SHARED = 19,        /* FP8 only: [T,S*I] codes of the shared h */
    MOE_WS_HQ_SHARED_SCALES = 20, /* FP8 only: [T, ceil(S*I/128) rounded up to 4] fp32 */
    MOE_WS_NUM_FIELDS = 21
} moe_ws_field;

size_t moe_layer_workspace_bytes(const moe_layer_desc* desc);
moe_status_t moe_layer_workspace_field(const moe_layer_desc* desc, moe_ws_field field, size_t* offset,
                                       size_t* bytes);

/* x [T,H] dt, out [T,H] dt, ws of moe_layer_workspace_bytes(desc) bytes.
 * T == 0 is a no-op that returns MOE_OK (x, out and ws may then be NULL).
 * With S > 0 the first call on a device creates the library's second stream
 * and three events for that device (no device memory is allocated); make that
 * first call outside stream capture.  The call's work forks onto that stream
 * and joins back into `stream`.  bf16 layers with T >= 256 run the shared
 * experts' two projections as one launch; the environment variable
 * MOE_SHARED_FUSED=0 keeps two launches (the same bits). */
moe_status_t moe_layer_forward(const moe_layer_desc* desc, const void* x, void* out, void* ws,
                               size_t ws_bytes, moe_stream_t stream);

/* As moe_layer_forward, also recording stage_events[2*i] (cudaEvent_t) when
 * stage i starts and stage_events[2*i+1] when it ends (2*MOE_NUM_STAGES events;
 * NULL entries are skipped).  The "shared" stage's events are recorded on the
 * library's second stream. */
moe_status_t moe_layer_forward_timed(const moe_layer_desc* desc, const void* x, void* out, void* ws,
                                     size_t ws_bytes, moe_stream_t stream, void* const* stage_events);

/* SMs that moe_layer_forward gives the shared experts' GEMMs (persistent CTAs,
 * in pairs) for the whole of the routed up projection, which takes the other
 * SMs, so that the shared experts run beside it and only the routed down
 * projection waits for them.  0 (the default) when the shared experts instead
 * take every SM beside the routing steps and both routed GEMMs wait for them.
 * The environment variable MOE_SHARED_SMS = n asks for the split (n rounded up
 * to a pair; granted for bf16 layers with native weights and S > 0 when n is at
 * most a quarter of the SMs).  The results are the same bits either way.
 * Reads the current device's SM count; -1 for a NULL desc. */
int moe_layer_shared_expert_sms(const moe_layer_desc* desc);

/* The layer through expert-parallel Double-Routing with W virtual ranks on
 * one GPU ([CANN §MoE deployment], steps 1-8): rank p owns tokens
 * [p*T/W, (p+1)*T/W) and experts [p*E/W, (p+1)*E/W); init-routing runs per
 * rank, the token AlltoAll and its reverse are device-side copies of row
 * blocks sized from the per-rank counts on the device, each rank re-routes,
 * runs its experts, un-sorts and returns the rows, and finalize runs per rank.
 * The output equals moe_layer_forward's bit for bit.  1 <= W <= 32,
 * T % W == 0, E % W == 0; ws of moe_layer_workspace_bytes_ep(desc, W) bytes. */
size_t moe_layer_workspace_bytes_ep(const moe_layer_desc* desc, int W);
moe_status_t moe_layer_forward_ep(const moe_layer_desc* desc, int W, const void* x, void* out, void* ws,
                                  size_t ws_bytes, moe_stream_t stream);

/* Intermediates of moe_layer_forward_ep that stay in its workspace after the
 * call (for inspection; the routing fields MOE_WS_LOGITS, MOE_WS_TOPK_IDS and
 * MOE_WS_TOPK_W sit at the offsets moe_layer_workspace_field gives).
 * [CANN §MoE deployment], steps 3-4: rank q's received rows arrive grouped by
 * source rank, each source's rows in global-expert order; re-routing sorts them
 * by local expert (stable), remembering where each sorted row came from. */
typedef enum moe_ws_field_ep {
    MOE_WS_EP_X_SORTED = 0,              /* [T*k,H] dt: every rank's re-routed rows, rank after rank */
    MOE_WS_EP_GATHERED_IDS_UNSORT = 1,   /* [T*k] int32: the receive-buffer row (all ranks, rank after
                                            rank) each sorted row was taken from */
    MOE_WS_EP_RECV_START = 2,            /* [W+1] int32: first received row of each rank */
    MOE_WS_EP_EXPERT_OFFSETS = 3,        /* [E+1] int32: rows of each global expert in X_SORTED */
    MOE_WS_EP_NUM_FIELDS = 4
} moe_ws_field_ep;
moe_status_t moe_layer_workspace_field_ep(const moe_layer_desc* desc, int W, moe_ws_field_ep field,
                                          size_t* offset, size_t* bytes);

/* End to end from HOST memory: copies x_host [T,H] into the workspace, runs
 * the layer, copies the result to out_host [T,H] and synchronises `stream`
 * (this call blocks).  Pinned host buffers give asynchronous copies.  The
 * copies run on two library-owned copy streams in row chunks of 1024 tokens,
 * overlapping the shared experts (input side) and finalize (output side); the
 * result equals moe_layer_forward's bit for bit.  The first call on a device
 * creates those streams and their events (make it outside stream capture).
 * T == 0 returns MOE_OK without touching any buffer. */
moe_status_t moe_layer_forward_host(const moe_layer_desc* desc, const void* x_host, void* out_host,
                                    void* ws, size_t ws_bytes, moe_stream_t stream);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
