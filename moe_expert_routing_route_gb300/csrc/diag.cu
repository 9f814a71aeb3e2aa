// Diagnostic: exercises the bounded on-chip wait the tensor-core kernels use.
//
// One CTA of two warps initialises an mbarrier that nothing ever arrives on.
// Warp 0 waits on it with the given limit: the wait runs out, raises the
// shared abort flag and sets MOE_DEVERR_TIMEOUT in the status word.  Warp 1
// waits on the same barrier with no limit of its own and must leave because of
// the abort flag -- the path every role of the GEMM kernels takes when another
// role gives up.  Both warps then return normally: no trap, no hang, and the
// CUDA context stays usable.
#include "tc_ptx.cuh"

namespace moe {
namespace {

using namespace tc;

__global__ void __launch_bounds__(64) bounded_wait_kernel(uint64_t limit_ns, uint32_t* status, uint32_t* outcome) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    const int warp = threadIdx.x >> 5;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    bool ok;
    if (warp == 0) ok = wait_phase(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
    else ok = wait_phase(smem_u32(&bar), 0, &abort_flag, status, ~0ull);
    // outcome bit 0: warp 0 timed out; bit 1: warp 1 left through the abort flag
    if ((threadIdx.x & 31) == 0 && !ok) atomicOr(outcome, 1u << warp);
    __syncthreads();
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" moe_status_t moe_diag_bounded_wait(uint64_t limit_ns, void* ws, uint32_t* outcome, moe_stream_t stream) {
    if (!ws || !outcome || limit_ns == 0 || limit_ns > 10000000000ull) return MOE_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    MOE_CUDA_TRY(cudaMemsetAsync(ws, 0, sizeof(uint32_t), s));
    MOE_CUDA_TRY(cudaMemsetAsync(outcome, 0, sizeof(uint32_t), s));
    bounded_wait_kernel<<<1, 64, 0, s>>>(limit_ns, static_cast<uint32_t*>(ws), outcome);
    note_launch();
    return last_launch_status();
}
