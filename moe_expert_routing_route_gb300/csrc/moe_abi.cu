// C ABI of libmoe (declared in include/moe.h): argument checks, workspace
// layout and the stream-ordered composition of the layer.
//
// "Lower latency and higher throughput with multi-node DeepSeek deployment"
// (Perplexity blog), §Expert Parallelism (the layer: routed experts summed with
// weights plus the shared expert), §Quantization (kernels read the routing
// counts on the device; fixed grids), §CUDA Graph (no host synchronisation so
// the whole forward can be captured).  "DeepSeek-R1 prefill inference
// optimisation on Atlas A3" (cann-recipes-infer), §MoE deployment strategy
// (init-routing / expert compute / finalize-routing split of the layer).
#include "moe_internal.cuh"

#include <atomic>
#include <climits>
#include <cstdlib>
#include <mutex>

namespace moe {

namespace {
std::atomic<uint64_t> g_launches{0};
int g_sm_count[64] = {0};

constexpr size_t kAlign = 256;

bool bad_dtype(moe_dtype_t dt) { return dt != MOE_F32 && dt != MOE_BF16; }

moe_status_t check_sizes(int T, int H, int E, int k) {
    if (T < 0 || H <= 0 || E <= 0 || k <= 0) return MOE_ERR_INVALID_ARG;
    if (E > 1024 || k > 32 || k > E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * k >= INT_MAX) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

uint32_t* status_word(void* ws) { return static_cast<uint32_t*>(ws); }

moe_status_t clear_status(void* ws, cudaStream_t s) {
    if (!ws) return MOE_OK;
    MOE_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(uint32_t), s));
    return MOE_OK;
}

int packed_rows(int I) { return 2 * (int)round_up((size_t)I, (size_t)tc_packed_block()); }

// Grouped FFN halves: up (SwiGLU into h) and down (h into y); bf16 on tcgen05,
// fp32 on the FFMA pipes.  offsets == nullptr means one dense group of `rows`.
// headroom: leave shared memory on every SM for kernels running beside this one
// tiled: the weight is in the tiled layout (bf16 only)
// max_ctas: persistent grid cap (bf16; 0 = every SM)
// pdl: programmatic dependent launch; false on the second stream, where a follower placed early
// holds SMs that the first stream's routing kernels need (measured: mid_bf16 0.566 -> 0.542 ms,
// dsv3_prefill 3.986 -> 3.965 ms without it there)
moe_status_t ffn_up(const void* a, moe_dtype_t dt, const int32_t* offsets, int G, int rows, int H, int I,
                    const void* w13p, void* h, uint32_t* status, cudaStream_t s, bool headroom = false,
                    bool tiled = false, int max_ctas = 0, bool pdl = true) {
    if (rows == 0) return MOE_OK;
    if (dt == MOE_BF16) {
        TcGroupedGemm up{a, rows, H, offsets, G, w13p, packed_rows(I), I, h, I, TC_EPI_SWIGLU, status};
        up.smem_headroom = headroom;
        up.b_tiled = tiled;
        up.max_ctas = max_ctas;
        up.pdl = pdl;
        return launch_tc_grouped_gemm(up, s);
    }
    if (tiled) return MOE_ERR_UNSUPPORTED;
    return launch_simt_grouped_ffn_up(static_cast<const float*>(a), rows, H, offsets, G,
                                      static_cast<const float*>(w13p), packed_rows(I) / 2, I, static_cast<float*>(h),
                                      status, s, pdl);
}

moe_status_t ffn_down(const void* h, moe_dtype_t dt, const int32_t* offsets, int G, int rows, int H, int I,
                      const void* w2, void* y, uint32_t* status, cudaStream_t s, bool headroom = false,
                      bool tiled = false, int max_ctas = 0, bool pdl = true) {
    if (rows == 0) return MOE_OK;
    if (dt == MOE_BF16) {
        TcGroupedGemm down{h, rows, I, offsets, G, w2, H, H, y, H, TC_EPI_BF16, status};
        down.smem_headroom = headroom;
        down.b_tiled = tiled;
        down.max_ctas = max_ctas;
        down.pdl = pdl;
        return launch_tc_grouped_gemm(down, s);
    }
    if (tiled) return MOE_ERR_UNSUPPORTED;
    return launch_simt_grouped_down(static_cast<const float*>(h), rows, I, offsets, G, static_cast<const float*>(w2),
                                    H, static_cast<float*>(y), status, s, pdl);
}

// The shared experts (one dense FFN over all T rows, bf16) in one pair-tile launch when both of
// its GEMMs take pair tiles: the down projection's tiles of 256 rows start as soon as the up
// projection has stored those rows, instead of after the up projection's last tile (measured on
// the DeepSeek-V3 prefill layer: see the design notes).  MOE_SHARED_FUSED=0 keeps two launches.
// Returns MOE_ERR_UNSUPPORTED when the shapes take the two-launch path.
moe_status_t shared_ffn_fused(const void* x, int T, int H, int SI, const void* w13s, const void* w2s, void* hs,
                              void* ys, int* sync, uint32_t* status, cudaStream_t s, bool headroom, bool tiled) {
    if (const char* e = std::getenv("MOE_SHARED_FUSED"))
        if (e[0] == '0') return MOE_ERR_UNSUPPORTED;
    TcGroupedGemm up{x, T, H, nullptr, 1, w13s, packed_rows(SI), SI, hs, SI, TC_EPI_SWIGLU, status};
    TcGroupedGemm down{hs, T, SI, nullptr, 1, w2s, H, H, ys, H, TC_EPI_BF16, status};
    up.smem_headroom = down.smem_headroom = headroom;
    up.b_tiled = down.b_tiled = tiled;
    up.pdl = down.pdl = false;
    MOE_CUDA_TRY(cudaMemsetAsync(sync, 0, (size_t)ceil_div(T, 256) * sizeof(int), s));
    return launch_tc_pair_ffn(up, down, sync, s);
}

// FP8 halves: the up projection (SwiGLU into bf16 h) followed by the 1x128
// quantisation of h, and the down projection.  Scale rows are padded to a
// multiple of 4 floats so they can be permuted as 16-byte vectors.
int scale_ld(int cols) { return (int)round_up((size_t)ceil_div(cols, 128), 4); }

// pow2: power-of-two scales throughout (block-scaled tensor-core MMAs).
moe_status_t ffn_up_fp8(const uint8_t* aq, const float* as, int lda_s, const int32_t* offsets, int G, int rows, int H,
                        int I, const void* w13q, const float* w13s, void* h, uint8_t* hq, float* hs,
                        uint32_t* status, cudaStream_t s, bool pow2, bool tiled = false, bool pdl = true) {
    if (rows == 0) return MOE_OK;
    // the SwiGLU epilogue writes the down projection's FP8 input directly; bf16 h
    // is stored too only when the caller gives a buffer for it (h may be null)
    TcFp8GroupedGemm up{aq, rows, H, offsets, G, w13q, packed_rows(I), I, h, I, TC_EPI_SWIGLU, as, lda_s,
                        w13s, status, hq, hs, scale_ld(I), pow2, tiled, pdl};
    return launch_tc_fp8_grouped_gemm(up, s);
}

moe_status_t ffn_down_fp8(const uint8_t* hq, const float* hs, const int32_t* offsets, int G, int rows, int H, int I,
                          const void* w2q, const float* w2s, void* y, uint32_t* status, cudaStream_t s, bool pow2,
                          bool tiled = false, bool pdl = true) {
    if (rows == 0) return MOE_OK;
    TcFp8GroupedGemm down{hq, rows, I, offsets, G, w2q, H, H, y, H, TC_EPI_BF16, hs, scale_ld(I), w2s, status,
                          nullptr, nullptr, 0, pow2, tiled, pdl};
    return launch_tc_fp8_grouped_gemm(down, s);
}

moe_status_t gate(const void* x, const void* wr, moe_dtype_t dt, int T, int H, int E, float* logits,
                  cudaStream_t s) {
    if (T == 0) return MOE_OK;
    if (dt == MOE_BF16) {
        TcGroupedGemm g{x, T, H, nullptr, 1, wr, E, E, logits, E, TC_EPI_F32, nullptr};
        return launch_tc_grouped_gemm(g, s);
    }
    return launch_simt_gate(static_cast<const float*>(x), static_cast<const float*>(wr), T, H, E, logits, s);
}

// K slices of the layer's gate GEMM (bf16 on tensor cores only); the route
// kernel adds them.  The workspace holds kMaxGateSplits slices so that its size
// does not depend on the device; the launch picks at most that many.
constexpr int kMaxGateSplits = 8;
int gate_splits(const moe_layer_desc& d) {
    if (d.dtype != MOE_BF16 || d.T <= 0) return 1;
    return tc_gate_splits(d.T, d.E, d.H, kMaxGateSplits);
}

// The layer's gate GEMM: bf16 splits K (the route kernel adds the slices), fp32
// runs unsplit.  Every layer path uses this so that their logits agree bit for bit.
// The launch plans from the same maximum as gate_splits, so both arrive at the
// same slice count.
moe_status_t layer_gate(const moe_layer_desc& d, const void* x, float* logits, int* nsplit, cudaStream_t s) {
    *nsplit = gate_splits(d);
    if (d.dtype == MOE_BF16) {
        TcGroupedGemm g{x, d.T, d.H, nullptr, 1, d.w_router, d.E, d.E, logits, d.E, TC_EPI_F32, nullptr,
                        kMaxGateSplits, (int64_t)d.T * d.E};
        return launch_tc_grouped_gemm(g, s);
    }
    return gate(x, d.w_router, d.dtype, d.T, d.H, d.E, logits, s);
}

// The gate for rows [r0, r1) only, with the K slices of the whole batch's gate (nsplit from
// gate_splits), writing rows r0.. of every slice: the same logits, bit for bit, as layer_gate.
moe_status_t layer_gate_rows(const moe_layer_desc& d, const void* x, float* logits, int r0, int r1, int nsplit,
                             cudaStream_t s) {
    const void* xr = static_cast<const char*>(x) + (size_t)r0 * d.H * dt_size(d.dtype);
    float* lr = logits + (size_t)r0 * d.E;
    if (d.dtype == MOE_BF16) {
        TcGroupedGemm g{xr, r1 - r0, d.H, nullptr, 1, d.w_router, d.E, d.E, lr, d.E, TC_EPI_F32, nullptr,
                        nsplit, (int64_t)d.T * d.E};
        g.exact_split = true;
        return launch_tc_grouped_gemm(g, s);
    }
    return gate(xr, d.w_router, d.dtype, r1 - r0, d.H, d.E, lr, s);
}

// ---- layer workspace layout ----
struct Layout {
    size_t off[MOE_WS_NUM_FIELDS];
    size_t bytes[MOE_WS_NUM_FIELDS];
    size_t scratch_off, scratch_bytes, sync_off, total;
};

Layout layout(const moe_layer_desc& d) {
    Layout L{};
    const size_t b = dt_size(d.dtype);
    const size_t T = (size_t)d.T, H = (size_t)d.H, E = (size_t)d.E, R = (size_t)d.T * d.k, I = (size_t)d.I,
                 S = (size_t)d.S;
    L.bytes[MOE_WS_LOGITS] = T * E * 4 * (d.dtype == MOE_BF16 ? kMaxGateSplits : 1);
    L.bytes[MOE_WS_TOPK_IDS] = R * 4;
    L.bytes[MOE_WS_TOPK_W] = R * 4;
    L.bytes[MOE_WS_TOKENS_PER_EXPERT] = E * 4;
    L.bytes[MOE_WS_EXPERT_OFFSETS] = (E + 1) * 4;
    L.bytes[MOE_WS_EXPANDED_ROW_IDX] = R * 4;
    L.bytes[MOE_WS_EXPANDED_X] = R * H * b;
    L.bytes[MOE_WS_H_ROUTED] = R * I * b;
    L.bytes[MOE_WS_H_SHARED] = T * S * I * b;
    L.bytes[MOE_WS_Y_ROUTED] = R * H * b;
    L.bytes[MOE_WS_Y_SHARED] = T * H * b;
    L.bytes[MOE_WS_X_IN] = T * H * b;
    L.bytes[MOE_WS_OUT] = T * H * b;
    if (d.weight_format == MOE_WEIGHTS_FP8 || d.weight_format == MOE_WEIGHTS_FP8_POW2) {
        const size_t SI = S * I;
        L.bytes[MOE_WS_XQ] = T * H;
        L.bytes[MOE_WS_XQ_SCALES] = T * scale_ld(d.H) * 4;
        L.bytes[MOE_WS_EXPANDED_XQ] = R * H;
        L.bytes[MOE_WS_EXPANDED_XQ_SCALES] = R * scale_ld(d.H) * 4;
        L.bytes[MOE_WS_HQ] = R * I;
        L.bytes[MOE_WS_HQ_SCALES] = R * scale_ld(d.I) * 4;
        L.bytes[MOE_WS_HQ_SHARED] = T * SI;
        L.bytes[MOE_WS_HQ_SHARED_SCALES] = SI ? T * scale_ld((int)SI) * 4 : 0;
        L.bytes[MOE_WS_EXPANDED_X] = 0;  // the bf16 expanded rows are not used
    }
    size_t cur = MOE_WS_HEADER_BYTES;
    for (int f = 0; f < MOE_WS_NUM_FIELDS; ++f) {
        L.off[f] = cur;
        cur += round_up(L.bytes[f], kAlign);
    }
    L.scratch_off = cur;
    L.scratch_bytes = init_routing_scratch_bytes(d.T, d.E, d.k);
    cur += round_up(L.scratch_bytes, kAlign);
    L.sync_off = cur;  // the fused shared-expert FFN's counter per 256 rows
    cur += round_up((size_t)ceil_div(std::max(d.T, 1), 256) * 4, kAlign);
    L.total = cur;
    return L;
}

moe_status_t check_grouping(int E, int k, int n_group, int topk_group, int rule) {
    if (n_group <= 1) return MOE_OK;
    if (n_group > 32 || E % n_group != 0) return MOE_ERR_INVALID_ARG;
    if (topk_group < 1 || topk_group > n_group) return MOE_ERR_INVALID_ARG;
    if ((int64_t)k > (int64_t)topk_group * (E / n_group)) return MOE_ERR_INVALID_ARG;
    if (rule != MOE_GROUP_SCORE_MAX && rule != MOE_GROUP_SCORE_TOP2_SUM) return MOE_ERR_INVALID_ARG;
    if (rule == MOE_GROUP_SCORE_TOP2_SUM && E / n_group < 2) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status_t check_desc(const moe_layer_desc* d) {
    if (!d) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_sizes(d->T, d->H, d->E, d->k));
    MOE_TRY(check_grouping(d->E, d->k, d->n_group, d->topk_group, d->group_rule));
    if (bad_dtype(d->dtype) || d->I <= 0 || d->S < 0) return MOE_ERR_INVALID_ARG;
    if (d->I % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (!d->w_router || !d->w13 || !d->w2) return MOE_ERR_INVALID_ARG;
    if (d->S > 0 && (!d->w13_shared || !d->w2_shared)) return MOE_ERR_INVALID_ARG;
    if ((int64_t)d->S * d->I >= INT_MAX / 2) return MOE_ERR_INVALID_ARG;
    if (d->weight_format != MOE_WEIGHTS_NATIVE && d->weight_format != MOE_WEIGHTS_FP8 &&
        d->weight_format != MOE_WEIGHTS_FP8_POW2)
        return MOE_ERR_INVALID_ARG;
    if (d->weight_format != MOE_WEIGHTS_NATIVE) {
        if (d->dtype != MOE_BF16 || d->H % 256 != 0 || d->I % 16 != 0) return MOE_ERR_UNSUPPORTED;
        if (!d->w13_scales || !d->w2_scales) return MOE_ERR_INVALID_ARG;
        if (d->S > 0 && (!d->w13_shared_scales || !d->w2_shared_scales)) return MOE_ERR_INVALID_ARG;
    }
    if (d->weight_layout != MOE_LAYOUT_ROWS && d->weight_layout != MOE_LAYOUT_TILED) return MOE_ERR_INVALID_ARG;
    if (d->weight_layout == MOE_LAYOUT_TILED && d->dtype != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    if (!aligned16(d->w_router) || !aligned16(d->w13) || !aligned16(d->w2) || !aligned16(d->expert_bias) ||
        !aligned16(d->w13_shared) || !aligned16(d->w2_shared))
        return MOE_ERR_UNSUPPORTED;
    return MOE_OK;
}

// Shared experts on a fixed share of the SMs beside the routed up projection: with
// MOE_SHARED_SMS = n (rounded up to whole CTA pairs, at most a quarter of the SMs) their GEMMs take n
// persistent CTAs, the routed up projection the other SMs, and only the routed down projection waits
// for them.  By default (0) they take every SM beside the routing steps and both routed GEMMs wait.
// Measured on the DeepSeek-V3 prefill layer (4096 tokens, 128 rows per expert) the split loses: the
// routed up projection slows in proportion to the SMs it gives up (2344 us on 148 SMs, 2635 on 132,
// 2659 on 126; each SM's TMA pipeline, not HBM alone, sets its rate), more than the ~125 us the
// shared experts add beside the routing steps.
int shared_expert_ctas(const moe_layer_desc& d) {
    if (d.S <= 0 || d.dtype != MOE_BF16 || d.weight_format != MOE_WEIGHTS_NATIVE || d.T <= 0) return 0;
    const char* e = std::getenv("MOE_SHARED_SMS");
    const int n = ((e ? std::atoi(e) : 0) + 1) & ~1;  // whole CTA pairs
    return n > 0 && n <= sm_count() / 4 ? n : 0;
}

template <typename T>
T* at(void* ws, size_t off) {
    return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

// Stage timing: ev[2*i] before stage i, ev[2*i+1] after it (caller's events).
enum Stage { ST_GATE = 0, ST_ROUTE, ST_INIT, ST_PERMUTE, ST_SHARED, ST_UP, ST_DOWN, ST_FINALIZE };
moe_status_t mark(void* const* ev, int stage, int end, cudaStream_t s) {
    void* e = ev ? ev[2 * stage + end] : nullptr;
    if (e) MOE_CUDA_TRY(cudaEventRecord(static_cast<cudaEvent_t>(e), s));
    return MOE_OK;
}

// Per-device side stream for the shared experts, with the fork/join events.
// The shared experts depend only on x, so they run on the side stream while
// the main stream computes the gate logits, routes and permutes the tokens -- kernels that leave most of
// the SMs idle ("Lower latency and higher throughput with multi-node DeepSeek
// deployment", §Dispatch Overlap: the shared expert is computed while the
// tokens are being dispatched).  The mutex keeps each call's record/wait pairs
// together when several host threads use one device.
struct SideStream {
    cudaStream_t stream = nullptr;
    cudaEvent_t fork = nullptr, join = nullptr, xq = nullptr;  // xq: FP8 layers' x codes are ready
    std::mutex mu;
};
SideStream g_side[64];
std::mutex g_side_init;

moe_status_t side_stream(SideStream** out) {
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    SideStream& ss = g_side[dev];
    std::lock_guard<std::mutex> lock(g_side_init);
    if (!ss.stream) {
        int lo = 0, hi = 0;
        MOE_CUDA_TRY(cudaDeviceGetStreamPriorityRange(&lo, &hi));
        MOE_CUDA_TRY(cudaStreamCreateWithPriority(&ss.stream, cudaStreamNonBlocking, lo));
        MOE_CUDA_TRY(cudaEventCreateWithFlags(&ss.fork, cudaEventDisableTiming));
        MOE_CUDA_TRY(cudaEventCreateWithFlags(&ss.join, cudaEventDisableTiming));
        MOE_CUDA_TRY(cudaEventCreateWithFlags(&ss.xq, cudaEventDisableTiming));
    }
    *out = &ss;
    return MOE_OK;
}

// Host-buffer path: x arrives and out leaves in row chunks on two library-owned
// copy streams, so the copies overlap the shared experts (x side) and the
// finalize kernel (out side) instead of bracketing the whole layer.
constexpr int kMaxIoChunks = 8;
struct HostPipe {
    cudaStream_t h2d = nullptr, d2h = nullptr;
    cudaEvent_t entry = nullptr, done = nullptr, in[kMaxIoChunks] = {}, out[kMaxIoChunks] = {};
    std::mutex mu;
};
HostPipe g_pipe[64];
std::mutex g_pipe_init;

moe_status_t host_pipe(HostPipe** out) {
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= 64) return MOE_ERR_UNSUPPORTED;
    HostPipe& hp = g_pipe[dev];
    std::lock_guard<std::mutex> lock(g_pipe_init);
    if (!hp.h2d) {
        MOE_CUDA_TRY(cudaStreamCreateWithFlags(&hp.h2d, cudaStreamNonBlocking));
        MOE_CUDA_TRY(cudaStreamCreateWithFlags(&hp.d2h, cudaStreamNonBlocking));
        MOE_CUDA_TRY(cudaEventCreateWithFlags(&hp.entry, cudaEventDisableTiming));
        MOE_CUDA_TRY(cudaEventCreateWithFlags(&hp.done, cudaEventDisableTiming));
        for (int c = 0; c < kMaxIoChunks; ++c) {
            MOE_CUDA_TRY(cudaEventCreateWithFlags(&hp.in[c], cudaEventDisableTiming));
            MOE_CUDA_TRY(cudaEventCreateWithFlags(&hp.out[c], cudaEventDisableTiming));
        }
    }
    *out = &hp;
    return MOE_OK;
}

struct HostIO {
    const void* x_host;  // [T,H] dt, copied into the x buffer the layer reads
    void* out_host;      // [T,H] dt, receives the layer's output
    HostPipe* pipe;
};

// Rows [c0, c1) of chunk c when T rows are cut into n nearly equal chunks.
inline void chunk_rows(int T, int n, int c, int& c0, int& c1) {
    c0 = (int)((int64_t)T * c / n);
    c1 = (int)((int64_t)T * (c + 1) / n);
}

moe_status_t layer_forward(const moe_layer_desc* d, const void* x, void* out, void* ws, size_t ws_bytes,
                           cudaStream_t s, void* const* ev, const HostIO* io = nullptr) {
    MOE_TRY(check_desc(d));
    if (d->T == 0) {  // an empty batch: nothing to read or write (pointers may be null)
        for (int i = 0; i < MOE_NUM_STAGES; ++i) {
            MOE_TRY(mark(ev, i, 0, s));
            MOE_TRY(mark(ev, i, 1, s));
        }
        return MOE_OK;
    }
    if (!x || !out || !ws) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_UNSUPPORTED;
    const Layout L = layout(*d);
    if (ws_bytes < L.total) return MOE_ERR_INVALID_ARG;
    const int T = d->T, H = d->H, E = d->E, k = d->k, I = d->I, R = T * k;
    const int SI = d->S * d->I;
    const moe_dtype_t dt = d->dtype;
    uint32_t* status = status_word(ws);
    float* logits = at<float>(ws, L.off[MOE_WS_LOGITS]);
    int32_t* ids = at<int32_t>(ws, L.off[MOE_WS_TOPK_IDS]);
    float* w = at<float>(ws, L.off[MOE_WS_TOPK_W]);
    int32_t* counts = at<int32_t>(ws, L.off[MOE_WS_TOKENS_PER_EXPERT]);
    int32_t* offsets = at<int32_t>(ws, L.off[MOE_WS_EXPERT_OFFSETS]);
    int32_t* row_idx = at<int32_t>(ws, L.off[MOE_WS_EXPANDED_ROW_IDX]);
    void* ex = at<void>(ws, L.off[MOE_WS_EXPANDED_X]);
    void* h = at<void>(ws, L.off[MOE_WS_H_ROUTED]);
    void* hs = at<void>(ws, L.off[MOE_WS_H_SHARED]);
    void* y = at<void>(ws, L.off[MOE_WS_Y_ROUTED]);
    void* ys = at<void>(ws, L.off[MOE_WS_Y_SHARED]);
    int32_t* scratch = at<int32_t>(ws, L.scratch_off);

    const bool fp8 = d->weight_format == MOE_WEIGHTS_FP8 || d->weight_format == MOE_WEIGHTS_FP8_POW2;
    const bool pow2 = d->weight_format == MOE_WEIGHTS_FP8_POW2;
    const bool tiled = d->weight_layout == MOE_LAYOUT_TILED;
    uint8_t* xq = at<uint8_t>(ws, L.off[MOE_WS_XQ]);
    float* xs = at<float>(ws, L.off[MOE_WS_XQ_SCALES]);
    uint8_t* exq = at<uint8_t>(ws, L.off[MOE_WS_EXPANDED_XQ]);
    float* exs = at<float>(ws, L.off[MOE_WS_EXPANDED_XQ_SCALES]);
    uint8_t* hq = at<uint8_t>(ws, L.off[MOE_WS_HQ]);
    float* hqs = at<float>(ws, L.off[MOE_WS_HQ_SCALES]);
    uint8_t* hsq = at<uint8_t>(ws, L.off[MOE_WS_HQ_SHARED]);
    float* hss = at<float>(ws, L.off[MOE_WS_HQ_SHARED_SCALES]);
    const int ldx = scale_ld(H);

    SideStream* side = nullptr;
    if (SI > 0) MOE_TRY(side_stream(&side));
    std::unique_lock<std::mutex> side_lock;
    if (side) side_lock = std::unique_lock<std::mutex>(side->mu);

    MOE_TRY(clear_status(ws, s));
    const size_t row_bytes = (size_t)H * dt_size(dt);
    // host path: chunks of T/1024 rows (at most kMaxIoChunks), one when T is small
    const int io_chunks = io ? std::max(1, std::min(kMaxIoChunks, (T + 1023) / 1024)) : 0;
    const bool chunked_shared = io && side && !fp8;  // FP8 shared experts read x quantised on the main stream
    // gate and top-k chunk by chunk as x arrives too (per-token work; the sort needs the whole batch)
    const bool chunked_gate = io && !fp8 && io_chunks > 1;
    if (io) {
        HostPipe* hp = io->pipe;
        MOE_CUDA_TRY(cudaEventRecord(hp->entry, s));  // after the status reset and all earlier work on s
        MOE_CUDA_TRY(cudaStreamWaitEvent(hp->h2d, hp->entry, 0));
        for (int c = 0; c < io_chunks; ++c) {
            int c0, c1;
            chunk_rows(T, io_chunks, c, c0, c1);
            MOE_CUDA_TRY(cudaMemcpyAsync(static_cast<char*>(const_cast<void*>(x)) + (size_t)c0 * row_bytes,
                                         static_cast<const char*>(io->x_host) + (size_t)c0 * row_bytes,
                                         (size_t)(c1 - c0) * row_bytes, cudaMemcpyHostToDevice, hp->h2d));
            MOE_CUDA_TRY(cudaEventRecord(hp->in[c], hp->h2d));
        }
        if (chunked_shared) {
            // shared experts chunk by chunk as x arrives (they depend on x alone)
            cudaStream_t ss = side->stream;
            MOE_CUDA_TRY(cudaStreamWaitEvent(ss, hp->entry, 0));
            MOE_TRY(mark(ev, ST_SHARED, 0, ss));
            for (int c = 0; c < io_chunks; ++c) {
                int c0, c1;
                chunk_rows(T, io_chunks, c, c0, c1);
                MOE_CUDA_TRY(cudaStreamWaitEvent(ss, hp->in[c], 0));
                const char* xc = static_cast<const char*>(x) + (size_t)c0 * row_bytes;
                char* hsc = static_cast<char*>(hs) + (size_t)c0 * SI * dt_size(dt);
                char* ysc = static_cast<char*>(ys) + (size_t)c0 * row_bytes;
                // both projections in one launch, leaving shared memory for the gate and routing kernels
                // that run beside it chunk by chunk (the device-buffer forward's choice too)
                moe_status_t st = MOE_ERR_UNSUPPORTED;
                if (dt == MOE_BF16)
                    st = shared_ffn_fused(xc, c1 - c0, H, SI, d->w13_shared, d->w2_shared, hsc, ysc,
                                          at<int>(ws, L.sync_off), status, ss, true, tiled);
                if (st == MOE_ERR_UNSUPPORTED) {
                    MOE_TRY(ffn_up(xc, dt, nullptr, 1, c1 - c0, H, SI, d->w13_shared, hsc, status, ss, false, tiled, 0,
                                   false));
                    MOE_TRY(ffn_down(hsc, dt, nullptr, 1, c1 - c0, H, SI, d->w2_shared, ysc, status, ss, false, tiled,
                                     0, false));
                } else {
                    MOE_TRY(st);
                }
            }
            MOE_TRY(mark(ev, ST_SHARED, 1, ss));
            MOE_CUDA_TRY(cudaEventRecord(side->join, ss));
        }
        if (!chunked_gate) MOE_CUDA_TRY(cudaStreamWaitEvent(s, hp->in[io_chunks - 1], 0));  // the gate reads all of x
    }
    MOE_TRY(mark(ev, ST_GATE, 0, s));
    // fork: the shared experts need x alone (FP8: its codes), so they branch off
    // before the gate; the gate is enqueued first and starts first
    const bool fork = side && !chunked_shared;
    // FP8: x is quantised (1x128 blocks) on the second stream ahead of the shared experts that read
    // its codes, and the main stream waits for the codes only at the permute (the gate reads x);
    // without a second stream, here
    const bool xq_side = fp8 && fork;
    if (fp8 && !xq_side) MOE_TRY(launch_quantize_rows_fp8(x, dt, T, H, xq, xs, ldx, s, pow2));
    const int shared_ctas = fork && !fp8 ? shared_expert_ctas(*d) : 0;  // > 0: beside the routed up projection
    if (fork) MOE_CUDA_TRY(cudaEventRecord(side->fork, s));
    int nsplit = 1;
    if (chunked_gate) {
        // each chunk's logits and top-k as soon as its rows of x have arrived
        nsplit = gate_splits(*d);
        for (int c = 0; c < io_chunks; ++c) {
            int c0, c1;
            chunk_rows(T, io_chunks, c, c0, c1);
            MOE_CUDA_TRY(cudaStreamWaitEvent(s, io->pipe->in[c], 0));
            MOE_TRY(layer_gate_rows(*d, x, logits, c0, c1, nsplit, s));
            MOE_TRY(launch_route_topk(logits + (size_t)c0 * E, d->expert_bias, c1 - c0, E, k, d->renormalize,
                                      ids + (size_t)c0 * k, w + (size_t)c0 * k, s, d->n_group, d->topk_group,
                                      d->group_rule, nsplit, (int64_t)T * E));
        }
    } else {
        MOE_TRY(layer_gate(*d, x, logits, &nsplit, s));
    }
    MOE_TRY(mark(ev, ST_GATE, 1, s));
    if (chunked_shared) {
        // launched above
    } else if (fork) {
        // shared experts on the side stream, beside the gate and the routing steps
        MOE_CUDA_TRY(cudaStreamWaitEvent(side->stream, side->fork, 0));
        cudaStream_t ss = side->stream;
        MOE_TRY(mark(ev, ST_SHARED, 0, ss));
        if (fp8) {
            MOE_TRY(launch_quantize_rows_fp8(x, dt, T, H, xq, xs, ldx, ss, pow2, false));
            MOE_CUDA_TRY(cudaEventRecord(side->xq, ss));
            MOE_TRY(ffn_up_fp8(xq, xs, ldx, nullptr, 1, T, H, SI, d->w13_shared, d->w13_shared_scales, nullptr, hsq, hss,
                               status, ss, pow2, tiled, false));
            MOE_TRY(ffn_down_fp8(hsq, hss, nullptr, 1, T, H, SI, d->w2_shared, d->w2_shared_scales, ys, status, ss,
                                 pow2, tiled, false));
        } else {
            // the routing kernels (histogram and scatter use shared memory) run beside them
            moe_status_t st = MOE_ERR_UNSUPPORTED;
            if (dt == MOE_BF16 && shared_ctas == 0)
                st = shared_ffn_fused(x, T, H, SI, d->w13_shared, d->w2_shared, hs, ys, at<int>(ws, L.sync_off), status,
                                      ss, true, tiled);
            if (st == MOE_ERR_UNSUPPORTED) {
                MOE_TRY(ffn_up(x, dt, nullptr, 1, T, H, SI, d->w13_shared, hs, status, ss, true, tiled, shared_ctas,
                               false));
                MOE_TRY(ffn_down(hs, dt, nullptr, 1, T, H, SI, d->w2_shared, ys, status, ss, true, tiled,
                                 shared_ctas, false));
            } else {
                MOE_TRY(st);
            }
        }
        MOE_TRY(mark(ev, ST_SHARED, 1, ss));
        MOE_CUDA_TRY(cudaEventRecord(side->join, ss));
    } else {
        MOE_TRY(mark(ev, ST_SHARED, 0, s));
        MOE_TRY(mark(ev, ST_SHARED, 1, s));
    }
    MOE_TRY(mark(ev, ST_ROUTE, 0, s));
    if (!chunked_gate)
        MOE_TRY(launch_route_topk(logits, d->expert_bias, T, E, k, d->renormalize, ids, w, s, d->n_group,
                                  d->topk_group, d->group_rule, nsplit));
    MOE_TRY(mark(ev, ST_ROUTE, 1, s));
    MOE_TRY(mark(ev, ST_INIT, 0, s));
    MOE_TRY(launch_init_routing_index(ids, R, E, counts, offsets, row_idx, scratch, status, s));
    MOE_TRY(mark(ev, ST_INIT, 1, s));
    MOE_TRY(mark(ev, ST_PERMUTE, 0, s));
    if (fp8) {
        if (xq_side) MOE_CUDA_TRY(cudaStreamWaitEvent(s, side->xq, 0));
        MOE_TRY(launch_permute_rows(xq, (size_t)H, row_idx, T, k, exq, s));
        MOE_TRY(launch_permute_rows(xs, (size_t)ldx * 4, row_idx, T, k, exs, s));
    } else {
        // beside the shared experts' GEMM on every SM: two copy blocks per SM (measured on dsv3_prefill:
        // the shared branch 329 -> 312 us; the copy itself unchanged at ~112 us, still off the critical
        // path); beside it on a share of the SMs, eight.  In the host path the shared experts ran chunk
        // by chunk while x arrived and only the last chunk's remain, so the copy is the longer branch
        // and takes sixteen (dsv3_prefill from host buffers: 4.55-4.57 -> 4.51-4.52 ms)
        const int copy_blocks = !side || chunked_shared ? 16 : (shared_ctas ? 8 : 2);
        MOE_TRY(launch_permute_rows(x, (size_t)H * dt_size(dt), row_idx, T, k, ex, s, copy_blocks));
    }
    MOE_TRY(mark(ev, ST_PERMUTE, 1, s));
    // join: GEMMs on every SM start after the shared experts; with the SMs split, only the down projection
    if (side && !shared_ctas) MOE_CUDA_TRY(cudaStreamWaitEvent(s, side->join, 0));
    MOE_TRY(mark(ev, ST_UP, 0, s));
    if (fp8)
        MOE_TRY(ffn_up_fp8(exq, exs, ldx, offsets, E, R, H, I, d->w13, d->w13_scales, nullptr, hq, hqs, status, s, pow2,
                           tiled));
    else MOE_TRY(ffn_up(ex, dt, offsets, E, R, H, I, d->w13, h, status, s, false, tiled,
                        shared_ctas ? sm_count() - shared_ctas : 0));
    MOE_TRY(mark(ev, ST_UP, 1, s));
    if (side && shared_ctas) MOE_CUDA_TRY(cudaStreamWaitEvent(s, side->join, 0));
    MOE_TRY(mark(ev, ST_DOWN, 0, s));
    if (fp8) MOE_TRY(ffn_down_fp8(hq, hqs, offsets, E, R, H, I, d->w2, d->w2_scales, y, status, s, pow2, tiled));
    else MOE_TRY(ffn_down(h, dt, offsets, E, R, H, I, d->w2, y, status, s, false, tiled));
    MOE_TRY(mark(ev, ST_DOWN, 1, s));
    MOE_TRY(mark(ev, ST_FINALIZE, 0, s));
    if (!io) {
        MOE_TRY(launch_finalize(y, R, SI > 0 ? ys : nullptr, w, row_idx, dt, T, H, k, out, status, s));
    } else {
        // finalize chunk c, then its rows leave on the copy stream while chunk c+1 runs
        HostPipe* hp = io->pipe;
        for (int c = 0; c < io_chunks; ++c) {
            int c0, c1;
            chunk_rows(T, io_chunks, c, c0, c1);
            const size_t o = (size_t)c0 * row_bytes;
            MOE_TRY(launch_finalize(y, R, SI > 0 ? static_cast<const char*>(ys) + o : nullptr, w + (size_t)c0 * k,
                                    row_idx + (size_t)c0 * k, dt, c1 - c0, H, k, static_cast<char*>(out) + o,
                                    status, s));
            MOE_CUDA_TRY(cudaEventRecord(hp->out[c], s));
            MOE_CUDA_TRY(cudaStreamWaitEvent(hp->d2h, hp->out[c], 0));
            MOE_CUDA_TRY(cudaMemcpyAsync(static_cast<char*>(io->out_host) + o, static_cast<const char*>(out) + o,
                                         (size_t)(c1 - c0) * row_bytes, cudaMemcpyDeviceToHost, hp->d2h));
        }
        MOE_CUDA_TRY(cudaEventRecord(hp->done, hp->d2h));
        MOE_CUDA_TRY(cudaStreamWaitEvent(s, hp->done, 0));  // the caller's stream covers the copies
    }
    MOE_TRY(mark(ev, ST_FINALIZE, 1, s));
    return MOE_OK;
}

// ---- expert-parallel Double-Routing on one GPU ----
struct EpLayout {
    size_t recv_off, sorted_off, gidx_off, scratch_off, total;
};

EpLayout ep_layout(const moe_layer_desc& d, int W, const Layout& L) {
    EpLayout e{};
    const size_t R = (size_t)d.T * d.k, rb = (size_t)d.H * dt_size(d.dtype);
    size_t cur = L.total;
    e.recv_off = cur;
    cur += round_up(R * rb, kAlign);
    e.sorted_off = cur;
    cur += round_up(R * rb, kAlign);
    e.gidx_off = cur;
    cur += round_up(R * 4, kAlign);
    e.scratch_off = cur;
    cur += round_up(ep_scratch_ints(W, d.E) * 4, kAlign);
    e.total = cur;
    return e;
}

moe_status_t check_ep(const moe_layer_desc* d, int W) {
    MOE_TRY(check_desc(d));
    if (d->weight_format != MOE_WEIGHTS_NATIVE) return MOE_ERR_UNSUPPORTED;
    if (W < 1 || W > 32 || d->T % W != 0 || d->E % W != 0) return MOE_ERR_INVALID_ARG;
    return MOE_OK;
}

moe_status_t layer_forward_ep(const moe_layer_desc* d, int W, const void* x, void* out, void* ws, size_t ws_bytes,
                              cudaStream_t s) {
    MOE_TRY(check_ep(d, W));
    if (!x || !out || !ws) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_UNSUPPORTED;
    const Layout L = layout(*d);
    const EpLayout EL = ep_layout(*d, W, L);
    if (ws_bytes < EL.total) return MOE_ERR_INVALID_ARG;
    if (d->T == 0) return MOE_OK;
    const int T = d->T, H = d->H, E = d->E, k = d->k, I = d->I, R = T * k, SI = d->S * d->I;
    const int El = E / W, Tp = T / W, Rp = Tp * k;
    const moe_dtype_t dt = d->dtype;
    const bool tiled = d->weight_layout == MOE_LAYOUT_TILED;
    const size_t rb = (size_t)H * dt_size(dt), eb = dt_size(dt);
    uint32_t* status = status_word(ws);
    float* logits = at<float>(ws, L.off[MOE_WS_LOGITS]);
    int32_t* ids = at<int32_t>(ws, L.off[MOE_WS_TOPK_IDS]);
    float* w = at<float>(ws, L.off[MOE_WS_TOPK_W]);
    void* h = at<void>(ws, L.off[MOE_WS_H_ROUTED]);
    void* hs = at<void>(ws, L.off[MOE_WS_H_SHARED]);
    void* y = at<void>(ws, L.off[MOE_WS_Y_ROUTED]);
    void* ys = at<void>(ws, L.off[MOE_WS_Y_SHARED]);
    EpBuffers b{W, T, E, k, rb, x, ids, at<int32_t>(ws, L.off[MOE_WS_EXPANDED_ROW_IDX]),
                at<void>(ws, L.off[MOE_WS_EXPANDED_X]), at<void>(ws, EL.recv_off), at<void>(ws, EL.sorted_off),
                at<int32_t>(ws, EL.gidx_off), at<int32_t>(ws, EL.scratch_off), at<int32_t>(ws, L.scratch_off), status};

    SideStream* side = nullptr;
    if (SI > 0) MOE_TRY(side_stream(&side));
    std::unique_lock<std::mutex> side_lock;
    if (side) side_lock = std::unique_lock<std::mutex>(side->mu);

    MOE_TRY(clear_status(ws, s));
    if (side) MOE_CUDA_TRY(cudaEventRecord(side->fork, s));  // the shared experts need x alone
    int nsplit = 1;
    MOE_TRY(layer_gate(*d, x, logits, &nsplit, s));
    if (side) {
        MOE_CUDA_TRY(cudaStreamWaitEvent(side->stream, side->fork, 0));
        MOE_TRY(ffn_up(x, dt, nullptr, 1, T, H, SI, d->w13_shared, hs, status, side->stream, false, tiled, 0, false));
        MOE_TRY(ffn_down(hs, dt, nullptr, 1, T, H, SI, d->w2_shared, ys, status, side->stream, false, tiled, 0,
                         false));
        MOE_CUDA_TRY(cudaEventRecord(side->join, side->stream));
    }
    MOE_TRY(launch_route_topk(logits, d->expert_bias, T, E, k, d->renormalize, ids, w, s, d->n_group, d->topk_group,
                              d->group_rule, nsplit));
    MOE_TRY(ep_route_and_dispatch(b, s));  // steps 1-4
    if (side) MOE_CUDA_TRY(cudaStreamWaitEvent(s, side->join, 0));
    // step 5: each rank's experts on its sorted rows.  The ranks' sorted rows lie
    // rank after rank in one buffer and rank q owns experts [q*El, (q+1)*El), so
    // the ranks' local segments together segment the buffer by global expert: on
    // one GPU all ranks' expert GEMMs run as one persistent launch per projection
    // (the same tiles as W launches of El experts, without W tails).
    MOE_TRY(ffn_up(b.sorted, dt, ep_expert_offsets(b), E, R, H, I, d->w13, h, status, s, false, tiled));
    MOE_TRY(ffn_down(h, dt, ep_expert_offsets(b), E, R, H, I, d->w2, y, status, s, false, tiled));
    // steps 6-7: back to received order, back to the source ranks (into the free buffers)
    MOE_TRY(ep_combine(b, y, b.recv, b.expanded, s));
    // step 8: finalize on each source rank
    for (int p = 0; p < W; ++p)
        MOE_TRY(launch_finalize(static_cast<const char*>(b.expanded) + (size_t)p * Rp * rb, Rp,
                                SI > 0 ? static_cast<const char*>(ys) + (size_t)p * Tp * rb : nullptr,
                                w + (size_t)p * Tp * k, b.row_idx + (size_t)p * Rp, dt, Tp, H, k,
                                static_cast<char*>(out) + (size_t)p * Tp * rb, status, s));
    return MOE_OK;
}

}  // namespace

void note_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

moe_status_t last_launch_status() { return cudaGetLastError() == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

int sm_count() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 1;
    int& c = g_sm_count[dev & 63];
    if (c == 0) {
        int v = 0;
        cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
        c = v > 0 ? v : 1;
    }
    return c;
}

}  // namespace moe

namespace moe {
namespace {

moe_status_t quantize_rows(const void* a, moe_dtype_t dt, int64_t rows, int cols, uint8_t* codes, float* scales,
                           int ld_scales, moe_stream_t stream, bool pow2) {
    if (bad_dtype(dt) || rows < 0 || cols <= 0 || ld_scales < (cols + 127) / 128) return MOE_ERR_INVALID_ARG;
    if (rows == 0) return MOE_OK;
    if (!a || !codes || !scales) return MOE_ERR_INVALID_ARG;
    return launch_quantize_rows_fp8(a, dt, rows, cols, codes, scales, ld_scales, reinterpret_cast<cudaStream_t>(stream),
                                    pow2);
}

moe_status_t quantize_weights(const void* w, moe_dtype_t dt, int G, int n_out, int k_in, uint8_t* codes,
                              float* scales, moe_stream_t stream, bool pow2) {
    if (bad_dtype(dt) || G <= 0 || n_out <= 0 || k_in <= 0) return MOE_ERR_INVALID_ARG;
    if (!w || !codes || !scales) return MOE_ERR_INVALID_ARG;
    return launch_quantize_tiles_fp8(w, dt, G, n_out, k_in, codes, scales, reinterpret_cast<cudaStream_t>(stream),
                                     pow2);
}

moe_status_t grouped_ffn(const void* a, moe_dtype_t dt, const int32_t* expert_offsets, int E, int rows, int H, int I,
                         const void* w13_packed, const void* w2, void* y, void* ws, size_t ws_bytes,
                         moe_stream_t stream, bool tiled) {
    if (bad_dtype(dt) || rows < 0 || H <= 0 || I <= 0 || E <= 0 || E > 1024) return MOE_ERR_INVALID_ARG;
    if (!expert_offsets && E != 1) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0 || I % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < moe_grouped_ffn_workspace_bytes(dt, rows, I)) return MOE_ERR_INVALID_ARG;
    if (rows > 0 && (!a || !w13_packed || !w2 || !y)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(w13_packed) || !aligned16(w2) || !aligned16(y) || !aligned16(ws))
        return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MOE_TRY(clear_status(ws, s));
    void* h = at<void>(ws, MOE_WS_HEADER_BYTES);
    MOE_TRY(ffn_up(a, dt, expert_offsets, E, rows, H, I, w13_packed, h, status_word(ws), s, false, tiled));
    return ffn_down(h, dt, expert_offsets, E, rows, H, I, w2, y, status_word(ws), s, false, tiled);
}

moe_status_t grouped_ffn_fp8(const uint8_t* aq, const float* a_scales, int lda_scales, const int32_t* expert_offsets,
                             int E, int rows, int H, int I, const uint8_t* w13q, const float* w13s, const uint8_t* w2q,
                             const float* w2s, void* y, void* ws, size_t ws_bytes, moe_stream_t stream, bool pow2) {
    if (rows < 0 || H <= 0 || I <= 0 || E <= 0 || E > 1024 || lda_scales < (H + 127) / 128) return MOE_ERR_INVALID_ARG;
    if (!expert_offsets && E != 1) return MOE_ERR_INVALID_ARG;
    if (H % 256 != 0 || I % 16 != 0) return MOE_ERR_UNSUPPORTED;
    if (!ws || ws_bytes < moe_grouped_ffn_fp8_workspace_bytes(rows, I)) return MOE_ERR_INVALID_ARG;
    if (rows > 0 && (!aq || !a_scales || !w13q || !w13s || !w2q || !w2s || !y)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(aq) || !aligned16(w13q) || !aligned16(w2q) || !aligned16(y) || !aligned16(ws))
        return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MOE_TRY(clear_status(ws, s));
    void* h = at<void>(ws, MOE_WS_HEADER_BYTES);
    uint8_t* hq = at<uint8_t>(ws, MOE_WS_HEADER_BYTES + round_up((size_t)rows * I * 2, kAlign));
    float* hs = at<float>(ws, MOE_WS_HEADER_BYTES + round_up((size_t)rows * I * 2, kAlign) +
                                  round_up((size_t)rows * I, kAlign));
    MOE_TRY(ffn_up_fp8(aq, a_scales, lda_scales, expert_offsets, E, rows, H, I, w13q, w13s, h, hq, hs, status_word(ws),
                       s, pow2));
    return ffn_down_fp8(hq, hs, expert_offsets, E, rows, H, I, w2q, w2s, y, status_word(ws), s, pow2);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_abi_version(void) { return 2; }

const char* moe_status_string(moe_status_t st) {
    switch (st) {
        case MOE_OK: return "MOE_OK";
        case MOE_ERR_INVALID_ARG: return "MOE_ERR_INVALID_ARG";
        case MOE_ERR_UNSUPPORTED: return "MOE_ERR_UNSUPPORTED";
        case MOE_ERR_CUDA: return "MOE_ERR_CUDA";
        case MOE_ERR_DEVICE: return "MOE_ERR_DEVICE";
    }
    return "MOE_ERR_UNKNOWN";
}

uint64_t moe_kernel_launch_count(void) { return g_launches.load(std::memory_order_relaxed); }

moe_status_t moe_check_device_status(const void* ws, moe_stream_t stream, uint32_t* word) {
    if (!ws) return MOE_ERR_INVALID_ARG;
    uint32_t v = 0;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    MOE_CUDA_TRY(cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, s));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    if (word) *word = v;
    return v ? MOE_ERR_DEVICE : MOE_OK;
}

moe_status_t moe_gate_logits(const void* x, const void* w_router, moe_dtype_t dt, int T, int H, int E,
                             float* logits, moe_stream_t stream) {
    MOE_TRY(check_sizes(T, H, E, 1));
    if (bad_dtype(dt)) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!x || !w_router || !logits) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(w_router) || !aligned16(logits)) return MOE_ERR_UNSUPPORTED;
    return gate(x, w_router, dt, T, H, E, logits, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_route_topk(const float* logits, const float* expert_bias, int T, int E, int k, int renormalize,
                            int32_t* topk_ids, float* topk_w, moe_stream_t stream) {
    MOE_TRY(check_sizes(T, 8, E, k));
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    return launch_route_topk(logits, expert_bias, T, E, k, renormalize ? 1 : 0, topk_ids, topk_w,
                             reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_route_topk_grouped(const float* logits, const float* expert_bias, int T, int E, int k, int n_group,
                                    int topk_group, int group_rule, int renormalize, int32_t* topk_ids, float* topk_w,
                                    moe_stream_t stream) {
    MOE_TRY(check_sizes(T, 8, E, k));
    if (n_group < 1) return MOE_ERR_INVALID_ARG;
    MOE_TRY(check_grouping(E, k, n_group, topk_group, group_rule));
    if (T == 0) return MOE_OK;
    if (!logits || !topk_ids || !topk_w) return MOE_ERR_INVALID_ARG;
    return launch_route_topk(logits, expert_bias, T, E, k, renormalize ? 1 : 0, topk_ids, topk_w,
                             reinterpret_cast<cudaStream_t>(stream), n_group, topk_group, group_rule);
}

size_t moe_re_routing_workspace_bytes(int W, int E_local) {
    if (W <= 0 || E_local <= 0) return 0;
    return MOE_WS_HEADER_BYTES + round_up(re_routing_plan_ints(W, E_local) * 4, kAlign);
}

moe_status_t moe_re_routing(const void* x_recv, moe_dtype_t dt, const int32_t* counts, int W, int E_local, int N, int H,
                            void* x_sorted, int32_t* gathered_ids_unsort, int32_t* tokens_per_local_expert,
                            int32_t* local_offsets, void* ws, size_t ws_bytes, moe_stream_t stream) {
    if (bad_dtype(dt) || W < 1 || W > 4096 || E_local < 1 || E_local > 1024 || N < 0 || H <= 0)
        return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (!counts || !tokens_per_local_expert || !local_offsets || !ws) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < moe_re_routing_workspace_bytes(W, E_local)) return MOE_ERR_INVALID_ARG;
    if (N > 0 && (!x_recv || !x_sorted || !gathered_ids_unsort)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x_recv) || !aligned16(x_sorted) || !aligned16(ws)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MOE_TRY(clear_status(ws, s));
    return launch_re_routing(x_recv, (size_t)H * dt_size(dt), counts, W, E_local, N, x_sorted, gathered_ids_unsort,
                             tokens_per_local_expert, local_offsets, at<int32_t>(ws, MOE_WS_HEADER_BYTES),
                             status_word(ws), s);
}

moe_status_t moe_unsort_rows(const void* y_sorted, moe_dtype_t dt, const int32_t* gathered_ids_unsort, int N, int H,
                             void* out, void* ws, moe_stream_t stream) {
    if (bad_dtype(dt) || N < 0 || H <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (N == 0) return MOE_OK;
    if (!y_sorted || !gathered_ids_unsort || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y_sorted) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MOE_TRY(clear_status(ws, s));
    return launch_unsort_rows(y_sorted, (size_t)H * dt_size(dt), gathered_ids_unsort, N, out,
                              ws ? status_word(ws) : nullptr, s);
}


moe_status_t moe_quantize_rows_fp8(const void* a, moe_dtype_t dt, int64_t rows, int cols, uint8_t* codes,
                                   float* scales, int ld_scales, moe_stream_t stream) {
    return quantize_rows(a, dt, rows, cols, codes, scales, ld_scales, stream, false);
}

moe_status_t moe_quantize_rows_fp8_pow2(const void* a, moe_dtype_t dt, int64_t rows, int cols, uint8_t* codes,
                                        float* scales, int ld_scales, moe_stream_t stream) {
    return quantize_rows(a, dt, rows, cols, codes, scales, ld_scales, stream, true);
}

moe_status_t moe_quantize_weights_fp8(const void* w, moe_dtype_t dt, int G, int n_out, int k_in, uint8_t* codes,
                                      float* scales, moe_stream_t stream) {
    return quantize_weights(w, dt, G, n_out, k_in, codes, scales, stream, false);
}

moe_status_t moe_quantize_weights_fp8_pow2(const void* w, moe_dtype_t dt, int G, int n_out, int k_in,
                                           uint8_t* codes, float* scales, moe_stream_t stream) {
    return quantize_weights(w, dt, G, n_out, k_in, codes, scales, stream, true);
}

size_t moe_grouped_ffn_fp8_workspace_bytes(int rows, int I) {
    if (rows < 0 || I <= 0) return 0;
    return MOE_WS_HEADER_BYTES + round_up((size_t)rows * I * 2, kAlign) + round_up((size_t)rows * I, kAlign) +
           round_up((size_t)rows * scale_ld(I) * 4, kAlign);
}


moe_status_t moe_grouped_ffn_fp8(const uint8_t* aq, const float* a_scales, int lda_scales,
                                 const int32_t* expert_offsets, int E, int rows, int H, int I, const uint8_t* w13q,
                                 const float* w13s, const uint8_t* w2q, const float* w2s, void* y, void* ws,
                                 size_t ws_bytes, moe_stream_t stream) {
    return grouped_ffn_fp8(aq, a_scales, lda_scales, expert_offsets, E, rows, H, I, w13q, w13s, w2q, w2s, y, ws,
                           ws_bytes, stream, false);
}

moe_status_t moe_grouped_ffn_fp8_pow2(const uint8_t* aq, const float* a_scales, int lda_scales,
                                      const int32_t* expert_offsets, int E, int rows, int H, int I,
                                      const uint8_t* w13q, const float* w13s, const uint8_t* w2q, const float* w2s,
                                      void* y, void* ws, size_t ws_bytes, moe_stream_t stream) {
    return grouped_ffn_fp8(aq, a_scales, lda_scales, expert_offsets, E, rows, H, I, w13q, w13s, w2q, w2s, y, ws,
                           ws_bytes, stream, true);
}

size_t moe_init_routing_workspace_bytes(int T, int E, int k) {
    if (T < 0 || E <= 0 || k <= 0) return 0;
    return MOE_WS_HEADER_BYTES + round_up(init_routing_scratch_bytes(T, E, k), kAlign);
}

moe_status_t moe_init_routing(const void* x, moe_dtype_t dt, const int32_t* topk_ids, int T, int H, int E, int k,
                              void* expanded_x, int32_t* expanded_row_idx, int32_t* tokens_per_expert,
                              int32_t* expert_offsets, void* ws, size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_sizes(T, H, E, k));
    if (bad_dtype(dt)) return MOE_ERR_INVALID_ARG;
    if (!ws || ws_bytes < moe_init_routing_workspace_bytes(T, E, k)) return MOE_ERR_INVALID_ARG;
    if (!tokens_per_expert || !expert_offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !topk_ids || !expanded_x || !expanded_row_idx)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(expanded_x) || !aligned16(ws)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MOE_TRY(clear_status(ws, s));
    const int R = T * k;
    MOE_TRY(launch_init_routing_index(topk_ids, R, E, tokens_per_expert, expert_offsets, expanded_row_idx,
                                      at<int32_t>(ws, MOE_WS_HEADER_BYTES), status_word(ws), s));
    return launch_permute_rows(x, (size_t)H * dt_size(dt), expanded_row_idx, T, k, expanded_x, s);
}

size_t moe_w13_packed_bytes(moe_dtype_t dt, int E, int H, int I) {
    if (bad_dtype(dt) || E <= 0 || H <= 0 || I <= 0) return 0;
    return (size_t)E * packed_rows(I) * (size_t)H * dt_size(dt);
}

moe_status_t moe_pack_w13(const void* w_gate, const void* w_up, moe_dtype_t dt, int E, int H, int I,
                          void* w13_packed, moe_stream_t stream) {
    if (bad_dtype(dt) || E <= 0 || H <= 0 || I <= 0) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (!w_gate || !w_up || !w13_packed) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w_gate) || !aligned16(w_up) || !aligned16(w13_packed)) return MOE_ERR_UNSUPPORTED;
    return launch_pack_w13(w_gate, w_up, dt_size(dt), E, H, I, w13_packed, reinterpret_cast<cudaStream_t>(stream));
}

size_t moe_grouped_ffn_workspace_bytes(moe_dtype_t dt, int rows, int I) {
    if (bad_dtype(dt) || rows < 0 || I <= 0) return 0;
    return MOE_WS_HEADER_BYTES + round_up((size_t)rows * I * dt_size(dt), kAlign);
}

moe_status_t moe_grouped_ffn(const void* a, moe_dtype_t dt, const int32_t* expert_offsets, int E, int rows, int H,
                             int I, const void* w13_packed, const void* w2, void* y, void* ws, size_t ws_bytes,
                             moe_stream_t stream) {
    return grouped_ffn(a, dt, expert_offsets, E, rows, H, I, w13_packed, w2, y, ws, ws_bytes, stream, false);
}

moe_status_t moe_grouped_ffn_tiled(const void* a, moe_dtype_t dt, const int32_t* expert_offsets, int E, int rows,
                                   int H, int I, const void* w13_tiled, const void* w2_tiled, void* y, void* ws,
                                   size_t ws_bytes, moe_stream_t stream) {
    if (dt != MOE_BF16) return MOE_ERR_UNSUPPORTED;
    return grouped_ffn(a, dt, expert_offsets, E, rows, H, I, w13_tiled, w2_tiled, y, ws, ws_bytes, stream, true);
}

size_t moe_tiled_weight_bytes(int G, int n_rows, int row_bytes) {
    if (G <= 0 || n_rows <= 0 || row_bytes <= 0 || row_bytes % 16 != 0) return 0;
    return tiled_weight_bytes(G, n_rows, row_bytes);
}

moe_status_t moe_tile_weights(const void* w, int G, int n_rows, int row_bytes, void* tiled, moe_stream_t stream) {
    if (G <= 0 || n_rows <= 0 || row_bytes <= 0) return MOE_ERR_INVALID_ARG;
    if (row_bytes % 16 != 0) return MOE_ERR_UNSUPPORTED;
    if (!w || !tiled) return MOE_ERR_INVALID_ARG;
    if (!aligned16(w) || !aligned16(tiled)) return MOE_ERR_UNSUPPORTED;
    return launch_tile_weights(w, G, n_rows, row_bytes, tiled, reinterpret_cast<cudaStream_t>(stream));
}



moe_status_t moe_finalize_routing(const void* y, int64_t y_rows, const void* skip, const float* topk_w,
                                  const int32_t* expanded_row_idx, moe_dtype_t dt, int T, int H, int k, void* out,
                                  void* ws, moe_stream_t stream) {
    MOE_TRY(check_sizes(T, H, 32, k));
    if (bad_dtype(dt) || y_rows < 0) return MOE_ERR_INVALID_ARG;
    if (T == 0) return MOE_OK;
    if (!y || !topk_w || !expanded_row_idx || !out) return MOE_ERR_INVALID_ARG;
    if (!aligned16(y) || !aligned16(skip) || !aligned16(out) || !aligned16(ws)) return MOE_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MOE_TRY(clear_status(ws, s));
    return launch_finalize(y, y_rows, skip, topk_w, expanded_row_idx, dt, T, H, k, out,
                           ws ? status_word(ws) : nullptr, s);
}

const char* moe_stage_name(int stage) {
    static const char* names[MOE_NUM_STAGES] = {"gate",   "route", "init_routing", "permute_rows",
                                                "shared", "up",    "down",         "finalize"};
    return (stage >= 0 && stage < MOE_NUM_STAGES) ? names[stage] : "";
}

int moe_layer_shared_expert_sms(const moe_layer_desc* desc) {
    if (!desc) return -1;
    return shared_expert_ctas(*desc);
}

size_t moe_layer_workspace_bytes(const moe_layer_desc* desc) {
    if (!desc || check_sizes(desc->T, desc->H, desc->E, desc->k) != MOE_OK || desc->I <= 0 || desc->S < 0 ||
        bad_dtype(desc->dtype))
        return 0;
    return layout(*desc).total;
}

moe_status_t moe_layer_workspace_field(const moe_layer_desc* desc, moe_ws_field field, size_t* offset,
                                       size_t* bytes) {
    if (!desc || field < 0 || field >= MOE_WS_NUM_FIELDS) return MOE_ERR_INVALID_ARG;
    if (check_sizes(desc->T, desc->H, desc->E, desc->k) != MOE_OK || desc->I <= 0 || desc->S < 0 ||
        bad_dtype(desc->dtype))
        return MOE_ERR_INVALID_ARG;
    const Layout L = layout(*desc);
    if (offset) *offset = L.off[field];
    if (bytes) *bytes = L.bytes[field];
    return MOE_OK;
}

moe_status_t moe_layer_forward(const moe_layer_desc* desc, const void* x, void* out, void* ws, size_t ws_bytes,
                               moe_stream_t stream) {
    return layer_forward(desc, x, out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

moe_status_t moe_layer_forward_timed(const moe_layer_desc* desc, const void* x, void* out, void* ws, size_t ws_bytes,
                                     moe_stream_t stream, void* const* stage_events) {
    return layer_forward(desc, x, out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream), stage_events);
}

size_t moe_layer_workspace_bytes_ep(const moe_layer_desc* desc, int W) {
    if (check_ep(desc, W) != MOE_OK) return 0;
    return ep_layout(*desc, W, layout(*desc)).total;
}

moe_status_t moe_layer_workspace_field_ep(const moe_layer_desc* desc, int W, moe_ws_field_ep field, size_t* offset,
                                          size_t* bytes) {
    MOE_TRY(check_ep(desc, W));
    const EpLayout EL = ep_layout(*desc, W, layout(*desc));
    const size_t R = (size_t)desc->T * desc->k;
    size_t off = 0, nb = 0;
    switch (field) {
        case MOE_WS_EP_X_SORTED: off = EL.sorted_off; nb = R * desc->H * dt_size(desc->dtype); break;
        case MOE_WS_EP_GATHERED_IDS_UNSORT: off = EL.gidx_off; nb = R * 4; break;
        case MOE_WS_EP_RECV_START: off = EL.scratch_off + 4 * ep_recv_start_int(W, desc->E); nb = (W + 1) * 4; break;
        case MOE_WS_EP_EXPERT_OFFSETS:
            off = EL.scratch_off + 4 * ep_expert_offsets_int(W, desc->E);
            nb = ((size_t)desc->E + 1) * 4;
            break;
        default: return MOE_ERR_INVALID_ARG;
    }
    if (offset) *offset = off;
    if (bytes) *bytes = nb;
    return MOE_OK;
}

moe_status_t moe_layer_forward_ep(const moe_layer_desc* desc, int W, const void* x, void* out, void* ws,
                                  size_t ws_bytes, moe_stream_t stream) {
    return layer_forward_ep(desc, W, x, out, ws, ws_bytes, reinterpret_cast<cudaStream_t>(stream));
}

moe_status_t moe_layer_forward_host(const moe_layer_desc* desc, const void* x_host, void* out_host, void* ws,
                                    size_t ws_bytes, moe_stream_t stream) {
    MOE_TRY(check_desc(desc));
    if (desc->T == 0) return MOE_OK;  // an empty batch (pointers may be null)
    if (!x_host || !out_host || !ws) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < layout(*desc).total) return MOE_ERR_INVALID_ARG;
    const Layout L = layout(*desc);
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    void* xin = at<void>(ws, L.off[MOE_WS_X_IN]);
    void* xout = at<void>(ws, L.off[MOE_WS_OUT]);
    HostPipe* hp = nullptr;
    MOE_TRY(host_pipe(&hp));
    std::lock_guard<std::mutex> lock(hp->mu);
    const HostIO io{x_host, out_host, hp};
    MOE_TRY(layer_forward(desc, xin, xout, ws, ws_bytes, s, nullptr, &io));
    MOE_CUDA_TRY(cudaStreamSynchronize(s));
    return MOE_OK;
}

}  // extern "C"
