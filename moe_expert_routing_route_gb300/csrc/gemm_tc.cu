// Grouped GEMM on the 5th-generation tensor cores (tcgen05 + TMEM), fed by TMA.
//
// "Lower latency and higher throughput with multi-node DeepSeek deployment"
// (Perplexity blog):
//   §Roofline / GroupGEMM: g groups, group i computes [m_i,k]x[k,n]; FLOPs
//     2*g*m*k*n, I/O bytes g*(m*k + n*k + m*n) -- here group e is expert e's
//     segment of the expert-sorted rows.
//   §Quantization: a fixed number of persistent kernels read the routing
//     information on the device to find how many tokens each expert got and
//     split the work dynamically, instead of sizing work by buffer upper
//     bounds (which breaks under CUDA graphs).  The grid here is one CTA per
//     SM; every CTA rebuilds the tile table from the expert offsets in device
//     memory and walks the tiles blockIdx.x, blockIdx.x + gridDim.x, ...
//   §Quantization: SiLU is applied to the up-projection output; here it is
//     fused into the GEMM epilogue (SwiGLU: h = silu(gate) * up).
//
// Per CTA (192 threads):
//   warp 0, one lane   TMA producer: A tile [128 x 64] and B tile [BN x 64]
//                      per k-block into a ring of shared-memory stages
//   warp 1, one lane   MMA issuer: 4 x tcgen05.mma (M=128, N=BN, K=16) per
//                      stage into one of two TMEM accumulators; tcgen05.commit
//                      frees the stage / publishes the accumulator
//   warps 2..5         epilogue: tcgen05.ld of the accumulator (one row per
//                      thread), SwiGLU / bf16 / fp32 conversion, masked stores
// The two TMEM accumulators let the epilogue of tile i overlap the MMAs of
// tile i+1.  Tiles are ordered (expert, n-tile, m-tile) with m fastest, so the
// CTAs working on the m-tiles of one weight panel run side by side and share
// it through L2.  Rows of a tile past the expert's segment belong to the next
// expert (or are zero-filled past the buffer by TMA); they cost MMA work but
// are never stored.
//
// Every wait on an mbarrier is bounded (about one second): on timeout the
// waiting role raises an abort flag in shared memory and MOE_DEVERR_TIMEOUT in
// the status word, every role leaves its loop, the producer waits (bounded) for
// the copies it issued, the MMA thread waits (bounded) for its MMAs, and TMEM
// is freed before the CTA exits.  No trap, no unbounded spin.
#include "tc_ptx.cuh"

#include <algorithm>
#include <climits>
#include <cstdlib>
#include <cstring>

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;      // MMA M (rows of A per tile), cta_group::1
constexpr int BK = 64;       // k-block: one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;   // K of one tcgen05.mma kind::f16
constexpr int kThreads = 192;
constexpr int kMaxGroups = 1024;
constexpr int kPackBlock = 128;  // gate rows (and up rows) per packed block

constexpr int kOutBox = 32 * 128;  // bf16 epilogue: one warp's 32 rows x 64 columns, staged for a TMA store

template <int BN>
struct Cfg {
    static constexpr int A_BYTES = BM * BK * 2;
    static constexpr int B_BYTES = BN * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
    static constexpr int STAGES = BN == 256 ? 4 : (BN == 128 ? 6 : 8);
    static constexpr int TMEM_COLS = 2 * BN;  // two fp32 accumulators
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr int OUT_BYTES = 4 * kOutBox;  // one staging box per epilogue warp
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + OUT_BYTES + NUM_BARS * 8 + 16 +
                                   (size_t)(3 * kMaxGroups + 1) * 4;
};

struct Params {
    const int32_t* offsets;
    int G, M, K, Nb, N, NT;
    int b_tiled, b_nt;        // B in the tiled layout, with b_nt 256-row tiles per group
    int c_tma;                // bf16 epilogue: C written through mapC (TMA stores of staged 32 x 64 boxes)
    int ksplit;               // K split into this many slices (fp32 outputs only), each written at
    int64_t c_split_stride;   // C + slice * c_split_stride
    int part;                 // rows of each group this launch covers (split_rows)
    void* C;
    int64_t ldc;
    uint32_t* status;
    // TC_EPI_FFN, phase 2 (the down projection of phase 1's output C): its tiles follow phase 1's
    // total1; a tile of m-block m waits until sync[m] == sync_target (every phase-1 tile of the
    // m-block counted once per epilogue warp of both CTAs)
    int total1, NT2, KB2, Nb2, N2, b_nt2, sync_target;
    void* C2;
    int64_t ldc2;
    int* sync;
};

// tile -> (group, m-tile, n-tile, K slice).  prefix[g] = first tile of group g,
// prefix[G] = total; tiles of a group are n-major, then m, K slice fastest.
__device__ __forceinline__ void decode_tile(int tile, const int* prefix, int G, int NT, int S, int& g, int& m,
                                            int& n, int& ks) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    g = lo;
    const int local = tile - prefix[g];
    const int mts = (prefix[g + 1] - prefix[g]) / NT;  // m-tiles x slices
    n = local / mts;
    const int rem = local - n * mts;
    m = rem / S;
    ks = rem - m * S;
}

// Rows [a, b) of a group that a launch covers.  part 0: all of them.  Mixed tile shapes split a
// group between two launches: part 1, the pair-tile launch, takes its 256-row blocks, and the tail
// too when more than 128 rows are left (one more, partly filled pair tile); part 2, a single-CTA
// launch, takes a tail of at most 128 rows (one m-tile) -- instead of a pair tile that would be
// half or more the next group's rows.  Left alone when the offsets are bad (the caller flags them).
__device__ __forceinline__ void split_rows(int part, int& a, int& b) {
    if (part == 0 || b < a) return;
    const int blocks = (b - a) >> 8, tail = (b - a) & 255;
    const int cut = a + (blocks << 8) + (tail > 128 ? tail : 0);
    if (part == 1) b = cut;
    else a = cut;
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// Store 32 consecutive outputs of one row (columns col0..col0+31, valid below N).
template <int EPI>
__device__ __forceinline__ void store_row32(void* C, int64_t ldc, int64_t row, int col0, int N,
                                            const float (&v)[32]) {
    if (EPI == TC_EPI_F32) {
        float* dst = static_cast<float*>(C) + row * ldc + col0;
        if (col0 + 32 <= N && (ldc & 3) == 0) {
#pragma unroll
            for (int q = 0; q < 8; ++q)
                reinterpret_cast<float4*>(dst)[q] = make_float4(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3]);
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (col0 + c < N) dst[c] = v[c];
        }
    } else {
        __nv_bfloat16* dst = static_cast<__nv_bfloat16*>(C) + row * ldc + col0;
        if (col0 + 32 <= N) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                uint4 u;
                u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
                u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
                u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
                u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
                reinterpret_cast<uint4*>(dst)[q] = u;
            }
        } else {
#pragma unroll
            for (int c = 0; c < 32; ++c)
                if (col0 + c < N) dst[c] = __float2bfloat16_rn(v[c]);
        }
    }
}

// 64 values of one row into a staging box laid out as the 128-byte swizzled TMA
// box expects: 16-byte chunk c of row r at r*128 + ((c ^ (r % 8)) * 16).
__device__ __forceinline__ void stage_row64_sw128(uint8_t* box, int r, const float* v) {
#pragma unroll
    for (int c = 0; c < 8; ++c) {
        uint4 u;
        u.x = pack_bf16x2(v[8 * c + 0], v[8 * c + 1]);
        u.y = pack_bf16x2(v[8 * c + 2], v[8 * c + 3]);
        u.z = pack_bf16x2(v[8 * c + 4], v[8 * c + 5]);
        u.w = pack_bf16x2(v[8 * c + 6], v[8 * c + 7]);
        *reinterpret_cast<uint4*>(box + r * 128 + ((c ^ (r & 7)) << 4)) = u;
    }
}

template <int BN, int EPI>
__global__ void __launch_bounds__(kThreads, 1)
tc_grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                       const __grid_constant__ CUtensorMap mapC, const __grid_constant__ Params p) {
    using Cf = Cfg<BN>;
    constexpr int STAGES = Cf::STAGES;
    constexpr uint32_t IDESC = idesc_bf16(BM, BN);
    static_assert(EPI != TC_EPI_SWIGLU || BN == 2 * kPackBlock, "SwiGLU tiles hold one packed block");

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cf::A_BYTES;
    uint8_t* sOut = sB + STAGES * Cf::B_BYTES;  // 1024-aligned: stage sizes are multiples of 1 KB
    uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + Cf::OUT_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cf::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* prefix = reinterpret_cast<int*>(tmem_slot + 4);  // [G+1]
    int* gstart = prefix + kMaxGroups + 1;               // [G]
    int* gend = gstart + kMaxGroups;                     // [G]

    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
    auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + 2 + a); };
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, NT = p.NT;

    // Launched after another kernel.  Only the up projection lets its follower (the down projection,
    // which cannot share an SM with it anyway) be scheduled early: the gate's follower (top-k) placed
    // early competes for SMs with the shared experts' GEMM on the other stream, and the down
    // projection's (finalize) waits beside it and slows it (DeepSeek-V3 prefill layer: 4.006 ->
    // 3.978 ms with the down projection releasing nothing early; as a CUDA graph 4.061 -> 4.018).
    if constexpr (EPI == TC_EPI_SWIGLU) pdl_trigger();
    pdl_wait();  // before any read of what earlier work on the stream wrote
    // ---- group table from the device-side offsets ----
    for (int g = threadIdx.x; g < G; g += kThreads) {
        int a = 0, b = p.M;
        if (p.offsets) {
            a = p.offsets[g];
            b = p.offsets[g + 1];
        }
        if (a < 0 || b < a || b > p.M) {
            set_status(p.status, MOE_DEVERR_BAD_OFFSETS);
            a = b = 0;
        }
        split_rows(p.part, a, b);
        gstart[g] = a;
        gend[g] = b;
    }
    if (threadIdx.x == 0) *abort_flag = 0;
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        for (int g0 = 0; g0 < G; g0 += 32) {
            const int g = g0 + lane;
            const int v = g < G ? (gend[g] - gstart[g] + BM - 1) / BM * NT * p.ksplit : 0;
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int nb = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += nb;
            }
            if (g < G) prefix[g] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            prefix[G] = run;
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(full_bar(s), 1);
                mbar_init(empty_bar(s), 1);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(tfull_bar(a), 1);
                mbar_init(tempty_bar(a), 4);
            }
            mbar_init(drain_bar, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            prefetch_tensormap(&mapA);
            prefetch_tensormap(&mapB);
        }
    } else if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), Cf::TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = prefix[G];
    const int KB = (p.K + BK - 1) / BK;
    const int KBS = (KB + p.ksplit - 1) / p.ksplit;  // k-blocks per slice (the host keeps every slice non-empty)

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int s = 0;
            uint32_t ph = 0, issued = 0, issued_par = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                int g, m, n, ks;
                decode_tile(tile, prefix, G, NT, p.ksplit, g, m, n, ks);
                const int row0 = gstart[g] + m * BM;
                const int brow = g * p.Nb + n * BN;
                const int tbase = (g * p.b_nt + n) * KB;  // tiled B: this tile's first 256-row box
                const int kb1 = min(KB, (ks + 1) * KBS);
                for (int kb = ks * KBS; kb < kb1; ++kb) {
                    if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), Cf::STAGE_BYTES);
                    tma_load_2d(smem_u32(sA + s * Cf::A_BYTES), &mapA, full_bar(s), kb * BK, row0);
                    if (p.b_tiled)  // one contiguous 32 KB box
                        tma_load_2d(smem_u32(sB + s * Cf::B_BYTES), &mapB, full_bar(s), 0, (tbase + kb) * BN);
                    else
                        tma_load_2d(smem_u32(sB + s * Cf::B_BYTES), &mapB, full_bar(s), kb * BK, brow);
                    issued |= 1u << s;
                    issued_par = (issued_par & ~(1u << s)) | (ph << s);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            // every copy this thread started has landed before the CTA exits
            for (int q = 0; q < STAGES; ++q)
                if ((issued >> q) & 1u) wait_drain(full_bar(q), (issued_par >> q) & 1u, p.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer ----------------
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                int g, m, n, ks;
                decode_tile(tile, prefix, G, NT, p.ksplit, g, m, n, ks);
                const int kb0 = ks * KBS, kb1 = min(KB, kb0 + KBS);
                if (!wait_phase(tempty_bar(acc), aph ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN);
                for (int kb = kb0; kb < kb1; ++kb) {
                    if (!wait_phase(full_bar(s), ph, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = smem_desc_sw128(smem_u32(sA + s * Cf::A_BYTES));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + s * Cf::B_BYTES));
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)  // +32 bytes per K=16 slice
                        mma_bf16(d, adesc + 2u * kk, bdesc + 2u * kk, IDESC, (kb != kb0) | (kk != 0));
                    mma_commit(empty_bar(s));
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(tfull_bar(acc));
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1u;
                }
            }
            // all MMAs issued by this thread are complete before TMEM is freed
            mma_commit(drain_bar);
            wait_drain(drain_bar, 0, p.status);
        }
    } else {
        // ---------------- epilogue: warps 2..5 ----------------
        const int eg = warp & 3;  // TMEM lane group this warp may access
        const int r = eg * 32 + lane;
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = blockIdx.x; tile < total; tile += gridDim.x) {
            int g, m, n, ks;
            decode_tile(tile, prefix, G, NT, p.ksplit, g, m, n, ks);
            void* C = static_cast<char*>(p.C) + ks * p.c_split_stride * (EPI == TC_EPI_F32 ? 4 : 2);
            const int64_t row = (int64_t)gstart[g] + (int64_t)m * BM + r;
            const bool valid = row < gend[g];
            // warp-uniform decision: the TMEM loads below are .sync.aligned
            if (!__all_sync(0xffffffffu, wait_phase(tfull_bar(acc), aph, abort_flag, p.status))) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(eg * 32) << 16) + (uint32_t)(acc * BN);
            if (EPI == TC_EPI_SWIGLU) {
#pragma unroll 1
                for (int c = 0; c < kPackBlock; c += 32) {
                    uint32_t gr[32], ur[32];
                    tmem_ld32(taddr + c, gr);
                    tmem_ld32(taddr + kPackBlock + c, ur);
                    float h[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float gv = __uint_as_float(gr[i]);
                        h[i] = gv / (1.0f + __expf(-gv)) * __uint_as_float(ur[i]);
                    }
                    if (valid) store_row32<EPI>(C, p.ldc, row, n * kPackBlock + c, p.N, h);
                }
            } else if (EPI == TC_EPI_BF16 && p.c_tma && __all_sync(0xffffffffu, valid)) {
                // all 32 rows of this warp inside the expert's segment: 32 x 64 boxes through the
                // warp's staging box, each leaving as one TMA store (full lines instead of 16-byte
                // pieces of 32 rows per store instruction)
                uint8_t* box = sOut + (warp - 2) * kOutBox;
                const int row0 = gstart[g] + m * BM + eg * 32;
#pragma unroll 1
                for (int c = 0; c < BN; c += 64) {
                    uint32_t v0[32], v1[32];
                    tmem_ld32(taddr + c, v0);
                    tmem_ld32(taddr + c + 32, v1);
                    float v[64];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        v[i] = __uint_as_float(v0[i]);
                        v[32 + i] = __uint_as_float(v1[i]);
                    }
                    if (lane == 0) bulk_wait_read_all();  // the previous box has left
                    __syncwarp();
                    stage_row64_sw128(box, lane, v);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0 && n * BN + c < p.N) {
                        tma_store_2d(&mapC, smem_u32(box), n * BN + c, row0);
                        bulk_commit();
                    }
                }
            } else {
#pragma unroll 1
                for (int c = 0; c < BN; c += 32) {
                    uint32_t vr[32];
                    tmem_ld32(taddr + c, vr);
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(vr[i]);
                    if (valid) store_row32<EPI>(C, p.ldc, row, n * BN + c, p.N, v);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty_bar(acc));
            if (++acc == 2) {
                acc = 0;
                aph ^= 1u;
            }
        }
        if (EPI == TC_EPI_BF16 && lane == 0) bulk_wait_all();  // staged stores done before the CTA leaves
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cf::TMEM_COLS);
    }
}

// ---------------------------------------------------------------------------
// Pair tiles: a cluster of two CTAs on one tcgen05.mma.cta_group::2 (M = 256).
//
// A tile is 256 rows x 256 columns.  Each CTA of the pair loads its own 128
// rows of A and its own half of the 256 B rows (SwiGLU: rank 0 the 128 gate
// rows, rank 1 the 128 up rows of the packed block), i.e. 32 KB per k-block
// instead of the 48 KB a 128 x 256 tile on one SM needs.  The fill rate one SM
// sustains is bounded by the bytes it keeps in flight, so the same 192 KB of
// stages now cover 6 k-blocks and feed the tensor core for 3/2 as long.
//
// Protocol (rank = %cluster_ctarank; rank 0 is the leader):
//   both producers   wait their own empty[s]; the leader arms its full[s] with
//                    the bytes of both CTAs; both load into their own shared
//                    memory with completion counted on the leader's full[s]
//   leader MMA       waits full[s], issues 4 x mma.cta_group::2, commits with
//                    multicast to empty[s] of both CTAs; after a tile, commits
//                    to tfull[acc] of both CTAs; waits tempty[acc] (8 warps:
//                    4 local + 4 remote) before reusing an accumulator
//   both epilogues   wait their own tfull[acc], read their own TMEM lanes
//                    (their 128 rows), store, arrive on the leader's tempty
// Cluster barriers after setup (barriers initialised, TMEM allocated) and
// before TMEM is freed (every pair MMA drained).  Waits are bounded as in the
// single-CTA kernel; a CTA that aborts stops signalling and its peer's waits
// run out in turn.
constexpr int BM2 = 256;  // rows per pair tile
constexpr int BN2 = 256;  // columns per pair tile (each CTA holds BN2 / 2 B rows)

// Shared memory: the stage ring, the barriers and a tile prefix over the
// groups (segment bounds are read from the offsets themselves).  Up to 256
// groups leave room for 7 stages; more groups take 6.
template <int STAGES_, int MAXG_>
struct Cfg2 {
    static constexpr int A_BYTES = 128 * BK * 2;
    static constexpr int B_BYTES = (BN2 / 2) * BK * 2;
    static constexpr int STAGE_BYTES = A_BYTES + B_BYTES;  // per CTA
    static constexpr int STAGES = STAGES_;
    static constexpr int MAXG = MAXG_;
    static constexpr int TMEM_COLS = 2 * BN2;
    static constexpr int NUM_BARS = 2 * STAGES + 5;
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + NUM_BARS * 8 + 16 + (size_t)(MAXG + 1) * 4;
};
static_assert(Cfg2<7, 256>::SMEM <= 232448, "pair-tile stages exceed shared memory");
static_assert(Cfg2<6, 1024>::SMEM <= 232448, "pair-tile stages exceed shared memory");

template <int EPI, int STAGES_, int MAXG_>
__global__ void __launch_bounds__(kThreads, 1)
tc_pair_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                    const __grid_constant__ CUtensorMap mapA2, const __grid_constant__ CUtensorMap mapB2,
                    const __grid_constant__ Params p) {
    using Cf = Cfg2<STAGES_, MAXG_>;
    constexpr int STAGES = Cf::STAGES;
    constexpr uint32_t IDESC = idesc_bf16(BM2, BN2);
    static_assert(EPI != TC_EPI_F32, "fp32 outputs use the single-CTA kernel");
    constexpr bool FFN = EPI == TC_EPI_FFN;  // phase 1 SwiGLU into C, phase 2 bf16 into C2 (mapA2, mapB2)

    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * Cf::A_BYTES;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sB + STAGES * Cf::B_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Cf::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* prefix = reinterpret_cast<int*>(tmem_slot + 4);  // [G+1]

    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
    auto tfull_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + a); };
    auto tempty_bar = [&](int a) { return smem_u32(bars + 2 * STAGES + 2 + a); };
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;
    const int pair = blockIdx.x >> 1, npairs = gridDim.x >> 1;
    const int G = p.G, NT = p.NT;
    // rows [a, b) of group g; a group with bad offsets gets no tiles, so every
    // decoded tile's group has valid bounds
    auto seg = [&](int g, int& a, int& b) {
        a = p.offsets ? __ldg(p.offsets + g) : 0;
        b = p.offsets ? __ldg(p.offsets + g + 1) : p.M;
        if (a >= 0 && b <= p.M) split_rows(p.part, a, b);
    };
    // tile -> (phase, group, m-tile, n-tile).  Two-phase launches (one group) order each phase
    // m-tile by m-tile, n fastest, so that the rows of an m-tile are finished early in phase 1
    auto decode = [&](int tile, int& phs, int& g, int& m, int& n) {
        if constexpr (FFN) {
            g = 0;
            phs = tile >= p.total1 ? 1 : 0;
            const int t = phs ? tile - p.total1 : tile, nt = phs ? p.NT2 : p.NT;
            m = t / nt;
            n = t - m * nt;
        } else {
            int ks;
            phs = 0;
            decode_tile(tile, prefix, G, NT, 1, g, m, n, ks);
        }
    };

    if constexpr (EPI == TC_EPI_SWIGLU) pdl_trigger();  // as in the single-CTA kernel
    pdl_wait();  // before any read of what earlier work on the stream wrote
    if (threadIdx.x == 0) *abort_flag = 0;
    if (warp == 0) {
        int run = 0;
        for (int g0 = 0; g0 < G; g0 += 32) {
            const int g = g0 + lane;
            int v = 0;
            if (g < G) {
                int a, b;
                seg(g, a, b);
                if (a < 0 || b < a || b > p.M) set_status(p.status, MOE_DEVERR_BAD_OFFSETS);
                else v = (b - a + BM2 - 1) / BM2 * NT;
            }
            int incl = v;
#pragma unroll
            for (int off = 1; off < 32; off <<= 1) {
                const int nb = __shfl_up_sync(0xffffffffu, incl, off);
                if (lane >= off) incl += nb;
            }
            if (g < G) prefix[g] = run + incl - v;
            run += __shfl_sync(0xffffffffu, incl, 31);
        }
        if (lane == 0) {
            prefix[G] = run;
            for (int s = 0; s < STAGES; ++s) {
                mbar_init(full_bar(s), 1);
                mbar_init(empty_bar(s), 1);
            }
            for (int a = 0; a < 2; ++a) {
                mbar_init(tfull_bar(a), 1);
                mbar_init(tempty_bar(a), 8);
            }
            mbar_init(drain_bar, 1);
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            prefetch_tensormap(&mapA);
            prefetch_tensormap(&mapB);
        }
    } else if (warp == 1) {
        tmem_alloc_pair(smem_u32(tmem_slot), Cf::TMEM_COLS);
    }
    tc_fence_before();
    cluster_sync_all();  // the peer's barriers exist before anything signals them
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = FFN ? p.total1 + p.total1 / NT * p.NT2 : prefix[G];
    const int KB = (p.K + BK - 1) / BK;

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer (both CTAs) ----------------
            int s = 0;
            uint32_t ph = 0, issued = 0, issued_par = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < total; tile += npairs) {
                int phs, g, m, n;
                decode(tile, phs, g, m, n);
                int ga, gb;
                seg(g, ga, gb);
                const CUtensorMap* mA = phs ? &mapA2 : &mapA;
                const CUtensorMap* mB = phs ? &mapB2 : &mapB;
                const int kbn = phs ? p.KB2 : KB;
                const int row0 = ga + m * BM2 + (int)rank * 128;
                const int brow = g * (phs ? p.Nb2 : p.Nb) + n * BN2 + (int)rank * (BN2 / 2);
                const int tbase = (g * (phs ? p.b_nt2 : p.b_nt) + n) * kbn;  // tiled B: the tile's first box
                if (FFN && phs) {
                    // phase 2 reads the rows phase 1 wrote: wait until every phase-1 tile of this
                    // m-tile is stored (bounded), then order that view before the TMA reads
                    const uint64_t t0 = globaltimer();
                    while (ld_acquire_gpu(p.sync + m) < p.sync_target) {
                        if (*abort_flag) {
                            ok = false;
                            break;
                        }
                        if (globaltimer() - t0 > kWaitLimitNs) {
                            *abort_flag = 1;
                            set_status(p.status, MOE_DEVERR_TIMEOUT);
                            ok = false;
                            break;
                        }
                    }
                    if (!ok) break;
                    fence_proxy_async_global();
                }
                for (int kb = 0; kb < kbn; ++kb) {
                    if (!wait_phase(empty_bar(s), ph ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    if (leader) mbar_arrive_expect_tx(full_bar(s), 2 * Cf::STAGE_BYTES);
                    const uint32_t fb = mapa_shared(full_bar(s), 0);  // the leader's full[s]
                    tma_load_2d_pair(smem_u32(sA + s * Cf::A_BYTES), mA, fb, kb * BK, row0);
                    if (p.b_tiled)  // this CTA's half of a contiguous 256-row box
                        tma_load_2d_pair(smem_u32(sB + s * Cf::B_BYTES), mB, fb, 0,
                                         (tbase + kb) * BN2 + (int)rank * (BN2 / 2));
                    else
                        tma_load_2d_pair(smem_u32(sB + s * Cf::B_BYTES), mB, fb, kb * BK, brow);
                    issued |= 1u << s;
                    issued_par = (issued_par & ~(1u << s)) | (ph << s);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            if (leader) {
                // the leader's full barriers count both CTAs' bytes of every stage it armed
                for (int q = 0; q < STAGES; ++q)
                    if ((issued >> q) & 1u) wait_drain(full_bar(q), (issued_par >> q) & 1u, p.status);
            } else if (!ok) {
                // stopped early: give copies still in flight time to land before exit
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 200000ull) {
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ---------------- MMA issuer (leader only) ----------------
            int s = 0, acc = 0;
            uint32_t ph = 0, aph = 0;
            bool ok = true;
            for (int tile = pair; ok && tile < total; tile += npairs) {
                const int kbn = FFN && tile >= p.total1 ? p.KB2 : KB;
                if (!wait_phase(tempty_bar(acc), aph ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                const uint32_t d = tmem_base + (uint32_t)(acc * BN2);
                for (int kb = 0; kb < kbn; ++kb) {
                    if (!wait_phase(full_bar(s), ph, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint64_t adesc = smem_desc_sw128(smem_u32(sA + s * Cf::A_BYTES));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + s * Cf::B_BYTES));
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        mma_bf16_pair(d, adesc + 2u * kk, bdesc + 2u * kk, IDESC, (kb | kk) != 0);
                    mma_commit_pair_mc(empty_bar(s), 0x3);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit_pair_mc(tfull_bar(acc), 0x3);
                if (++acc == 2) {
                    acc = 0;
                    aph ^= 1u;
                }
            }
            mma_commit_pair(drain_bar);
            wait_drain(drain_bar, 0, p.status);
        }
    } else {
        // ---------------- epilogue: warps 2..5 of both CTAs ----------------
        const int eg = warp & 3;
        const int r = eg * 32 + lane;
        int acc = 0;
        uint32_t aph = 0;
        for (int tile = pair; tile < total; tile += npairs) {
            int phs, g, m, n;
            decode(tile, phs, g, m, n);
            int ga, gb;
            seg(g, ga, gb);
            const int64_t row = (int64_t)ga + (int64_t)m * BM2 + (int64_t)rank * 128 + r;
            const bool valid = row < gb;
            if (!__all_sync(0xffffffffu, wait_phase(tfull_bar(acc), aph, abort_flag, p.status))) break;
            tc_fence_after();
            const uint32_t taddr = tmem_base + ((uint32_t)(eg * 32) << 16) + (uint32_t)(acc * BN2);
            if (EPI == TC_EPI_SWIGLU || (FFN && !phs)) {
#pragma unroll 1
                for (int c = 0; c < kPackBlock; c += 32) {
                    uint32_t gr[32], ur[32];
                    tmem_ld32(taddr + c, gr);
                    tmem_ld32(taddr + kPackBlock + c, ur);
                    float h[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const float gv = __uint_as_float(gr[i]);
                        h[i] = gv / (1.0f + __expf(-gv)) * __uint_as_float(ur[i]);
                    }
                    if (valid) store_row32<TC_EPI_SWIGLU>(p.C, p.ldc, row, n * kPackBlock + c, p.N, h);
                }
                if (FFN) {
                    // count this warp's rows of the m-tile as stored (every lane's stores are
                    // visible GPU-wide before the count; phase 2 acquires it)
                    __threadfence();
                    __syncwarp();
                    if (lane == 0) atomicAdd(p.sync + m, 1);
                }
            } else {
                void* C = FFN ? p.C2 : p.C;
                const int64_t ldc = FFN ? p.ldc2 : p.ldc;
                const int N = FFN ? p.N2 : p.N;
#pragma unroll 1
                for (int c = 0; c < BN2; c += 32) {
                    uint32_t vr[32];
                    tmem_ld32(taddr + c, vr);
                    float v[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(vr[i]);
                    if (valid) store_row32<TC_EPI_BF16>(C, ldc, row, n * BN2 + c, N, v);
                }
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) {
                if (leader) mbar_arrive(tempty_bar(acc));
                else mbar_arrive_cluster(mapa_shared(tempty_bar(acc), 0));
            }
            if (++acc == 2) {
                acc = 0;
                aph ^= 1u;
            }
        }
    }

    __syncwarp();
    tc_fence_before();
    cluster_sync_all();  // every pair MMA has completed and no CTA signals the other any more
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cf::TMEM_COLS);
    }
}

// K slices actually launched for a requested count: each slice takes
// ceil(KB / requested) k-blocks, so none is left empty.
int effective_splits(int K, int requested) {
    const int KB = (int)ceil_div(K, BK);
    const int S = std::max(1, std::min(requested, KB));
    return (int)ceil_div(KB, ceil_div(KB, S));
}

template <int BN, int EPI>
moe_status_t launch_impl(const TcGroupedGemm& g, cudaStream_t s) {
    using Cf = Cfg<BN>;
    static std::once_flag attr_once[64];
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        attr_err = cudaFuncSetAttribute(tc_grouped_gemm_kernel<BN, EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        (int)Cf::SMEM);
    });
    MOE_CUDA_TRY(attr_err);

    CUtensorMap ma, mb;
    const int b_nt = (int)ceil_div(g.Nb, 256), KBt = (int)ceil_div(g.K, BK);
    if (!make_map(&ma, g.A, (uint64_t)g.K, (uint64_t)g.M, BM)) return MOE_ERR_CUDA;
    if (g.b_tiled) {
        // box rows are addressed with int coordinates
        if (BN != 256 || (int64_t)g.G * b_nt * KBt * 256 >= INT_MAX) return MOE_ERR_UNSUPPORTED;
        if (!make_map(&mb, g.B, (uint64_t)BK, (uint64_t)g.G * b_nt * KBt * 256, BN)) return MOE_ERR_CUDA;
    } else if (!make_map(&mb, g.B, (uint64_t)g.K, (uint64_t)g.G * g.Nb, BN)) {
        return MOE_ERR_CUDA;
    }

    // bf16 output through TMA stores when the map can describe it (else direct stores)
    CUtensorMap mc;
    const bool c_tma = EPI == TC_EPI_BF16 && g.C && g.ksplit <= 1 &&
                       make_store_map_bf16(&mc, g.C, (uint64_t)g.N, (uint64_t)g.M, (uint64_t)g.ldc, 32);
    if (!c_tma) mc = ma;  // never read

    Params p{};
    p.offsets = g.offsets;
    p.G = g.G;
    p.M = g.M;
    p.K = g.K;
    p.Nb = g.Nb;
    p.N = g.N;
    p.b_tiled = g.b_tiled ? 1 : 0;
    p.b_nt = b_nt;
    p.c_tma = c_tma ? 1 : 0;
    p.NT = EPI == TC_EPI_SWIGLU ? g.Nb / BN : (int)ceil_div(g.N, BN);
    p.ksplit = EPI == TC_EPI_F32 ? (g.exact_split ? g.ksplit : effective_splits(g.K, g.ksplit)) : 1;
    p.c_split_stride = g.c_split_stride;
    p.C = g.C;
    p.ldc = g.ldc;
    p.status = g.status;
    p.part = g.part;

    const int64_t max_tiles = (int64_t)p.NT * p.ksplit * (ceil_div(g.M, BM) + (g.offsets ? g.G : 0));
    const int ctas = g.max_ctas > 0 ? std::min(g.max_ctas, sm_count()) : sm_count();
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(ctas, max_tiles));
    if (g.pdl) {
        MOE_CUDA_TRY(launch_pdl(tc_grouped_gemm_kernel<BN, EPI>, dim3(grid), dim3(kThreads), Cf::SMEM, s, ma, mb, mc,
                                p));
    } else {
        tc_grouped_gemm_kernel<BN, EPI><<<grid, kThreads, Cf::SMEM, s>>>(ma, mb, mc, p);
        MOE_CUDA_TRY(cudaGetLastError());
    }
    note_launch();
    return MOE_OK;
}

// g2, sync: TC_EPI_FFN only (g the up projection, g2 the down projection of its output)
template <int EPI, int STAGES, int MAXG>
moe_status_t launch_pair_impl(const TcGroupedGemm& g, cudaStream_t s, const TcGroupedGemm* g2 = nullptr,
                              int* sync = nullptr) {
    using Cf = Cfg2<STAGES, MAXG>;
    constexpr bool FFN = EPI == TC_EPI_FFN;
    if (FFN != (g2 != nullptr) || (FFN && (!sync || g.G != 1 || g.offsets || g2->G != 1 || g2->offsets ||
                                           g2->b_tiled != g.b_tiled || g2->M != g.M)))
        return MOE_ERR_INVALID_ARG;
    static std::once_flag attr_once[64];
    static int max_clusters[64];
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    cudaError_t attr_err = cudaSuccess;

    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // as launch_pdl, when g.pdl
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = Cf::SMEM;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;

    std::call_once(attr_once[dev & 63], [&] {
        attr_err = cudaFuncSetAttribute(tc_pair_gemm_kernel<EPI, STAGES, MAXG>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Cf::SMEM);
        if (attr_err != cudaSuccess) return;
        // pairs that fit on the device at once (clusters live within one GPC)
        cudaLaunchConfig_t q = cfg;
        q.gridDim = dim3(2 * (sm_count() / 2));
        int n = 0;
        attr_err = cudaOccupancyMaxActiveClusters(&n, tc_pair_gemm_kernel<EPI, STAGES, MAXG>, &q);
        max_clusters[dev & 63] = n;
    });
    MOE_CUDA_TRY(attr_err);
    const int pairs_max = max_clusters[dev & 63];
    if (pairs_max < 1) return MOE_ERR_UNSUPPORTED;

    // A: 128-row boxes of [M, K]; B: this CTA's 128 rows of a 256-row block (row-major or tiled)
    auto maps = [](const TcGroupedGemm& q, CUtensorMap& ma, CUtensorMap& mb) -> moe_status_t {
        const int b_nt = (int)ceil_div(q.Nb, 256), KBt = (int)ceil_div(q.K, BK);
        if (!make_map(&ma, q.A, (uint64_t)q.K, (uint64_t)q.M, 128)) return MOE_ERR_CUDA;
        if (q.b_tiled) {
            if ((int64_t)q.G * b_nt * KBt * 256 >= INT_MAX) return MOE_ERR_UNSUPPORTED;
            if (!make_map(&mb, q.B, (uint64_t)BK, (uint64_t)q.G * b_nt * KBt * 256, BN2 / 2)) return MOE_ERR_CUDA;
        } else if (!make_map(&mb, q.B, (uint64_t)q.K, (uint64_t)q.G * q.Nb, BN2 / 2)) {
            return MOE_ERR_CUDA;
        }
        return MOE_OK;
    };
    CUtensorMap ma, mb, ma2, mb2;
    const int b_nt = (int)ceil_div(g.Nb, 256);
    MOE_TRY(maps(g, ma, mb));
    if (FFN) {
        MOE_TRY(maps(*g2, ma2, mb2));
    } else {
        ma2 = ma;  // never read
        mb2 = mb;
    }

    Params p{};
    p.offsets = g.offsets;
    p.G = g.G;
    p.M = g.M;
    p.K = g.K;
    p.Nb = g.Nb;
    p.N = g.N;
    p.b_tiled = g.b_tiled ? 1 : 0;
    p.b_nt = b_nt;
    p.c_tma = 0;
    p.NT = EPI != TC_EPI_BF16 ? g.Nb / BN2 : (int)ceil_div(g.N, BN2);
    p.ksplit = 1;
    p.c_split_stride = 0;
    p.C = g.C;
    p.ldc = g.ldc;
    p.status = g.status;
    p.part = g.part;

    int64_t max_tiles = (int64_t)p.NT * (ceil_div(g.M, BM2) + (g.offsets ? g.G : 0));
    if (FFN) {
        const int mt = (int)ceil_div(g.M, BM2);
        p.total1 = p.NT * mt;
        p.NT2 = (int)ceil_div(g2->N, BN2);
        p.KB2 = (int)ceil_div(g2->K, BK);
        p.Nb2 = g2->Nb;
        p.N2 = g2->N;
        p.b_nt2 = (int)ceil_div(g2->Nb, 256);
        p.C2 = g2->C;
        p.ldc2 = g2->ldc;
        p.sync = sync;
        p.sync_target = 8 * p.NT;  // every phase-1 tile of an m-tile, once per epilogue warp of both CTAs
        max_tiles = p.total1 + (int64_t)mt * p.NT2;
    }
    const int pair_cap = g.max_ctas > 0 ? std::min(pairs_max, std::max(1, g.max_ctas / 2)) : pairs_max;
    const int pairs = (int)std::max<int64_t>(1, std::min<int64_t>(pair_cap, max_tiles));
    cfg.gridDim = dim3(2 * pairs);
    cfg.numAttrs = g.pdl ? 2 : 1;  // the occupancy query above takes the cluster shape alone
    MOE_CUDA_TRY(cudaLaunchKernelEx(&cfg, tc_pair_gemm_kernel<EPI, STAGES, MAXG>, ma, mb, ma2, mb2, p));
    note_launch();
    return last_launch_status();
}

template <int EPI>
moe_status_t launch_pair(const TcGroupedGemm& g, cudaStream_t s) {
    return g.G <= 256 && !g.smem_headroom ? launch_pair_impl<EPI, 7, 256>(g, s) : launch_pair_impl<EPI, 6, 1024>(g, s);
}

// Pair tiles for each group's 256-row blocks and a single-CTA launch for the tails of at most 128
// rows (split_rows), for grouped launches that take pair tiles.  A tail on a single-CTA tile costs
// one SM where a pair tile costs two, but the second launch waits for the first and ends in a
// partial wave of its own, a cost that only many groups' tails outweigh.  Measured: the Zipf-skewed
// DeepSeek-V3 prefill batch (256 experts, 512 rows each on average) 10.79-10.92 -> 10.29-10.33 ms;
// its 32-expert slice (512 rows each) 1.276 -> 1.334 ms; mid_bf16 (64 experts, 384 rows each)
// 0.526-0.530 -> 0.582-0.584 ms.  So: 128 groups or more, averaging two 256-row blocks or more.
// MOE_GEMM_MIXED=1 or 0 forces the choice; a forced MOE_GEMM_TILE=pair keeps pair tiles throughout.
bool mixed_tiles(const TcGroupedGemm& g) {
    if (!g.offsets || g.G < 2) return false;
    if (const char* e = std::getenv("MOE_GEMM_TILE"))
        if (std::strcmp(e, "pair") == 0) return false;
    if (const char* e = std::getenv("MOE_GEMM_MIXED")) return e[0] == '1';
    return g.G >= 128 && (int64_t)g.M >= (int64_t)2 * BM2 * g.G;
}

template <int EPI>
moe_status_t launch_mixed(const TcGroupedGemm& g, cudaStream_t s) {
    TcGroupedGemm pairs = g, tails = g;
    pairs.part = 1;
    tails.part = 2;
    MOE_TRY(launch_pair<EPI>(pairs, s));
    // programmatic: its blocks wait (griddepcontrol.wait) for the pair launch, which waited for
    // everything before it
    return launch_impl<256, EPI>(tails, s);
}

// Tile shape for the bf16 / SwiGLU outputs.  MOE_GEMM_TILE = "single" or "pair"
// forces one; otherwise pair tiles (256 rows) are used once the groups average
// 256 rows or more, where the halved operand fill per SM pays, and single-CTA
// tiles (128 rows) below that, where a pair tile would mostly hold the next
// group's rows and double the A traffic.
bool use_pair_tiles(const TcGroupedGemm& g) {
    if (const char* e = std::getenv("MOE_GEMM_TILE")) {
        if (std::strcmp(e, "single") == 0) return false;
        if (std::strcmp(e, "pair") == 0) return true;
    }
    return (int64_t)g.M >= (int64_t)BM2 * g.G;
}

// Gate-style launches (one dense problem, fp32 out): pick the n-tile width and
// the number of K slices.  A CTA's k-blocks run at roughly the larger of their
// MMA time (2*BN cycles), their operand fill ((16 KB + BN*128 B) at ~128 B per
// cycle) and a floor of ~700 cycles set by the load latency one pipeline
// covers; cost = waves x k-blocks per tile x that.  Ties go to fewer slices,
// then to the wider tile.
void plan_f32(int M, int N, int K, int max_split, int& bn_out, int& split_out) {
    const int sms = sm_count();
    const int64_t KB = ceil_div(K, BK);
    int64_t best_cost = INT64_MAX;
    bn_out = 256;
    split_out = 1;
    for (int S = 1; S <= max_split; S *= 2) {
        for (int bn : {256, 128, 64}) {
            const int64_t tiles = ceil_div(M, BM) * ceil_div(N, bn) * S;
            const int64_t waves = ceil_div(tiles, sms);
            const int64_t per_kb = std::max<int64_t>({2 * bn, (16384 + (int64_t)bn * 128) / 128, 700});
            const int64_t cost = waves * ceil_div(KB, S) * per_kb;
            if (cost < best_cost) {
                best_cost = cost;
                bn_out = bn;
                split_out = S;
            }
        }
    }
}

}  // namespace

int tc_packed_block() { return kPackBlock; }

int tc_gate_splits(int M, int N, int K, int max_split) {
    int bn, split;
    plan_f32(M, N, K, std::max(1, max_split), bn, split);
    return effective_splits(K, split);
}

moe_status_t launch_tc_pair_ffn(const TcGroupedGemm& up, const TcGroupedGemm& down, int* sync, cudaStream_t s) {
    if (up.M == 0) return MOE_OK;
    if (up.epi != TC_EPI_SWIGLU || down.epi != TC_EPI_BF16 || down.A != up.C || up.Nb % (2 * kPackBlock) != 0)
        return MOE_ERR_INVALID_ARG;
    if (!use_pair_tiles(up) || !use_pair_tiles(down)) return MOE_ERR_UNSUPPORTED;
    return up.smem_headroom ? launch_pair_impl<TC_EPI_FFN, 6, 1024>(up, s, &down, sync)
                            : launch_pair_impl<TC_EPI_FFN, 7, 256>(up, s, &down, sync);
}

moe_status_t launch_tc_grouped_gemm(const TcGroupedGemm& g, cudaStream_t s) {
    if (g.M == 0 || g.G == 0) return MOE_OK;
    if (g.G > kMaxGroups) return MOE_ERR_UNSUPPORTED;
    switch (g.epi) {
        case TC_EPI_SWIGLU:
            if (g.Nb % (2 * kPackBlock) != 0) return MOE_ERR_INVALID_ARG;
            if (!use_pair_tiles(g)) return launch_impl<256, TC_EPI_SWIGLU>(g, s);
            if (!mixed_tiles(g)) return launch_pair<TC_EPI_SWIGLU>(g, s);
            return launch_mixed<TC_EPI_SWIGLU>(g, s);
        case TC_EPI_BF16:
            if (!use_pair_tiles(g)) return launch_impl<256, TC_EPI_BF16>(g, s);
            if (!mixed_tiles(g)) return launch_pair<TC_EPI_BF16>(g, s);
            return launch_mixed<TC_EPI_BF16>(g, s);
        case TC_EPI_F32: {
            if (g.b_tiled) return MOE_ERR_UNSUPPORTED;
            int bn, split;
            plan_f32(g.M, g.N, g.K, std::max(1, g.ksplit), bn, split);
            TcGroupedGemm gs = g;
            if (g.exact_split) {
                if (g.ksplit < 1 || effective_splits(g.K, g.ksplit) != g.ksplit) return MOE_ERR_INVALID_ARG;
            } else {
                gs.ksplit = split;
            }
            switch (bn) {
                case 64: return launch_impl<64, TC_EPI_F32>(gs, s);
                case 128: return launch_impl<128, TC_EPI_F32>(gs, s);
                default: return launch_impl<256, TC_EPI_F32>(gs, s);
            }
        }
    }
    return MOE_ERR_INVALID_ARG;
}

}  // namespace moe
