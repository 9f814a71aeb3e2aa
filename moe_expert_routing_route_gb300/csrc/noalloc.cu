// Init-routing for callers that cannot allocate device memory.
//
// moe_init_routing needs a caller-provided workspace for the per-chunk expert
// histogram.  Some callers cannot provide one: a serving engine that hands all
// device memory to its own pool at start-up and allows no further cudaMalloc,
// a latency-critical loop that must not pay cudaMalloc's implicit device-wide
// synchronisation, or a plain C host program with no device allocator at
// hand.  moe_init_routing_noalloc computes the same outputs with its scratch in
// a fixed array in this library's device memory instead.
//
// The array is a file-scope __device__ variable: every GPU that loads the
// library holds it (1 MiB) until the process exits.  Host code cannot use the
// array's name as a device address, so the first call on each device looks the
// address up with cudaGetSymbolAddress while that device is current and keeps
// it; later calls on that device reuse it.  The address belongs to the device's
// context: after a cudaDeviceReset the module is loaded again into a new
// context, possibly elsewhere, so the kept address is tagged with the context's
// process-unique id and looked up again when the current context's id differs.
// All calls share the one array and it keeps whatever the last call left
// there.  The histogram kernel rewrites every entry a call reads, so nothing
// has to be cleared between calls, but two calls whose kernels overlap on the
// GPU (different streams, or different host threads on one device) race on the
// array and corrupt each other's results.
#include "moe_internal.cuh"

#include <cuda.h>

#include <mutex>

namespace moe {
namespace {

constexpr size_t kNoAllocScratchInts = 262144;  // 1 MiB of int32
static __device__ __align__(256) int32_t g_noalloc_scratch[kNoAllocScratchInts];

constexpr int kMaxDevices = 64;
std::mutex g_setup_mutex;
struct ScratchAddr {
    int32_t* ptr = nullptr;
    unsigned long long ctx_id = 0;  // id of the context the address belongs to (0: unknown)
};
ScratchAddr g_scratch[kMaxDevices];

typedef CUresult (*CtxGetCurrentFn)(CUcontext*);
typedef CUresult (*CtxGetIdFn)(CUcontext, unsigned long long*);

// Id of the calling thread's current context, 0 when there is none or the
// driver cannot say (then a kept address is trusted as it is).
unsigned long long current_context_id() {
    static CtxGetCurrentFn get_current = nullptr;
    static CtxGetIdFn get_id = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_current = reinterpret_cast<CtxGetCurrentFn>(p);
        p = nullptr;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetId", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            get_id = reinterpret_cast<CtxGetIdFn>(p);
    });
    if (!get_current || !get_id) return 0;
    CUcontext ctx = nullptr;
    unsigned long long id = 0;
    if (get_current(&ctx) != CUDA_SUCCESS || !ctx || get_id(ctx, &id) != CUDA_SUCCESS) return 0;
    return id;
}

// Device address of the array for the current device (set up on first use in
// each context of that device).
moe_status_t scratch_for_current_device(int32_t** out) {
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    if (dev < 0 || dev >= kMaxDevices) return MOE_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_setup_mutex);
    ScratchAddr& a = g_scratch[dev];
    const unsigned long long id = current_context_id();
    if (!a.ptr || (id != 0 && id != a.ctx_id)) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return MOE_ERR_CUDA;
        a.ptr = static_cast<int32_t*>(p);
        a.ctx_id = current_context_id();  // the lookup made the device's context current
    }
    *out = a.ptr;
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_init_routing_noalloc(const void* x, moe_dtype_t dt, const int32_t* topk_ids, int T,
                                                 int H, int E, int k, void* expanded_x, int32_t* expanded_row_idx,
                                                 int32_t* tokens_per_expert, int32_t* expert_offsets,
                                                 moe_stream_t stream) {
    if (T < 0 || H <= 0 || E <= 0 || k <= 0 || E > 1024 || k > 32 || k > E) return MOE_ERR_INVALID_ARG;
    if ((int64_t)T * k >= INT32_MAX) return MOE_ERR_INVALID_ARG;
    if (dt != MOE_F32 && dt != MOE_BF16) return MOE_ERR_INVALID_ARG;
    if (H % 8 != 0) return MOE_ERR_UNSUPPORTED;
    if (!tokens_per_expert || !expert_offsets) return MOE_ERR_INVALID_ARG;
    if (T > 0 && (!x || !topk_ids || !expanded_x || !expanded_row_idx)) return MOE_ERR_INVALID_ARG;
    if (!aligned16(x) || !aligned16(expanded_x)) return MOE_ERR_UNSUPPORTED;
    // the histogram holds ceil(T*k / 1024) * E ints; larger requests do not fit
    if (init_routing_scratch_bytes(T, E, k) > kNoAllocScratchInts * sizeof(int32_t)) return MOE_ERR_UNSUPPORTED;
    int32_t* scratch = nullptr;
    MOE_TRY(scratch_for_current_device(&scratch));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const int R = T * k;
    MOE_TRY(launch_init_routing_index(topk_ids, R, E, tokens_per_expert, expert_offsets, expanded_row_idx, scratch,
                                      nullptr, s));
    return launch_permute_rows(x, (size_t)H * dt_size(dt), expanded_row_idx, T, k, expanded_x, s);
}
