// Grouped GEMM with FP8 (e4m3) block-scaled operands on tcgen05 tensor cores.
//
// "Lower latency and higher throughput with multi-node DeepSeek deployment"
// (Perplexity blog), §Quantization: activations carry one fp32 scale per
// 128-element vector along K (computed on the fly), weights one per 128x128
// tile, so a product is
//   C[m,n] = sum_b sa[m,b] * sb[n/128,b] * (sum_{k in block b} qa[m,k] * qb[n,k]).
// §Roofline / GroupGEMM: the grouped product over expert segments, as in the
// bf16 kernel (gemm_tc.cu), with the same persistent grid and device-side
// tile scheduler reading the expert offsets.
//
// One 128-wide K block is one pipeline stage and one scale block.  The MMA
// warp multiplies each K block into a fresh fp32 partial in TMEM (four
// kind::f8f6f4 instructions, K = 32 each), alternating between two partial
// buffers.  Eight epilogue warps -- two per TMEM lane group, each owning half of
// the tile's columns -- fold every partial into register accumulators with
// sa * sb (the promotion the block scales need), then apply SwiGLU or convert
// and store once per tile.  With a code buffer, the SwiGLU epilogue also
// quantises h for the down projection in place (the 1x128 activation blocks of
// §Quantization, computed on the fly): h is rounded to bf16, the two warps that
// hold the two 64-column halves of a 128-column block swap their partial amax
// through shared memory (an mbarrier per TMEM lane group, bounded wait), and
// each writes its 64 e4m3 codes; the first warp writes the block's scale.
// Rows of a tile past the expert's segment are
// computed and never stored, as in the bf16 kernel.  Waits are bounded as in
// the bf16 kernel (about one second, then abort without trapping).
//
// With power-of-two scales (the MX instantiation) the tensor cores apply the
// scales themselves: kind::mxf8f6f4 block-scaled MMAs take one UE8M0 exponent
// per 32 K elements for every row of A and every column of B, read from TMEM,
// and accumulate the whole tile in one TMEM accumulator, so nothing is promoted
// on CUDA cores.  A 128-element scale block covers four MMAs, so each 32-bit
// TMEM word holds the exponents of four consecutive K blocks and the
// instruction's scale-factor ids pick the byte.  Layout (the tensor cores read
// the A exponent of row m at lane m, column sfa + m/32, and the B exponent of
// column n at lane n%32 of the reading row's lane group, column sfb + n/32):
// per group of 16 K blocks there are four slots (one per four K blocks), each
// starting on an 8-column boundary: the A exponents of slot s at columns
// [8s, 8s+8) (a row's word repeated over them, so lane group w finds it at
// column 8s + w) and the B exponents at [32+8s, 40+8s) (the same eight words in
// all four lane groups).  Two such groups alternate; the first epilogue warp of
// each lane group writes them from the scale arrays while the MMAs run, and
// hands each over through an mbarrier.  The tile's accumulator is drained into
// registers once, at the end of the tile, after which the MMAs of the next tile
// start while the epilogue finishes this one.
#include "fp8_codec.cuh"
#include "tc_ptx.cuh"

#include <climits>

namespace moe {
namespace {

using namespace tc;

constexpr int BM = 128;
constexpr int BK = 128;  // bytes (= e4m3 elements) of K per stage: one swizzle row, one scale block
constexpr int UMMA_K = 32;
constexpr int BN = 256;
constexpr int kEpiWarps = 8;              // epilogue warps: kSplit per TMEM lane group
constexpr int kSplit = kEpiWarps / 4;     // warps sharing a lane group, each on 128/kSplit columns of a chunk
constexpr int kCols = 128 / kSplit;       // columns of each of a thread's two chunks
constexpr int kThreads = 64 + 32 * kEpiWarps;
static_assert(kSplit >= 2 && kCols % 16 == 0, "epilogue split");
constexpr int kMaxGroups = 1024;
constexpr int A_BYTES = BM * BK;
constexpr int B_BYTES = BN * BK;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int TMEM_COLS = 2 * BN;  // two partial buffers (MX: the accumulator and the scale factors)
constexpr int kSfGroup = 16;       // MX: K blocks per scale-factor group (4 per 32-bit TMEM word)
constexpr int kSfCols = 64;        // MX: TMEM columns of one group: A slots at +8s, B slots at +32+8s (s < 4)
constexpr int kSfBase = BN;        // MX: the two groups at columns 256 and 320
constexpr int XAMAX_FLOATS = 2 * kSplit * BM;  // [tile parity][column part][row]
constexpr int kOutBox = 32 * kCols * 2;        // one warp's 32 rows x kCols bf16 columns (128-byte rows)
static_assert(kCols * 2 == 128, "a staged output row is one 128-byte swizzle row");

// Shared-memory plan per epilogue.  The bf16 epilogue with fp32 scales (the down
// projection) stages each finished tile in shared memory and writes it with TMA
// stores, so its warps go straight back to folding the next tile's partials
// instead of waiting on 16-byte row-by-row global stores; the 64 KB staging area
// takes the place of one pipeline stage.
// With power-of-two scales the tile's accumulator is read out once and the next tile's MMAs start
// while the epilogue stores it, so direct stores cost nothing there and the four-stage ring is kept
// (dsv3_prefill_fp8_pow2 down 699 -> 681 us against staging).
template <int EPI, bool MX>
struct Plan {
    static constexpr int STAGES = EPI == TC_EPI_BF16 && !MX ? 3 : 4;
    static constexpr int OUT_BYTES = EPI == TC_EPI_BF16 && !MX ? kEpiWarps * 2 * kOutBox : 0;
    // full, empty, partial (MX: accumulator) full/empty, drain, 4 amax exchanges, MX scale groups full/empty
    static constexpr int NUM_BARS = 2 * STAGES + 13;
    static constexpr size_t SMEM = 1024 + (size_t)STAGES * STAGE_BYTES + OUT_BYTES + NUM_BARS * 8 + 16 +
                                   (size_t)(3 * kMaxGroups + 1) * 4 + (size_t)XAMAX_FLOATS * 4;
};

struct Params {
    const int32_t* offsets;  // [G+1] or nullptr: one group of M rows
    int G, M, K, Nb, N, NT, KB;
    int b_tiled, b_nt;       // B in the tiled layout, with b_nt 256-row tiles per group
    void* C;
    int64_t ldc;
    const float* a_scales;  // [M][lda_s]
    int lda_s;
    const float* b_scales;  // [G][Nb/128][KB]
    int c_tma;              // bf16 epilogue: C is written through mapC (TMA stores of staged tiles)
    uint8_t* q;             // SwiGLU only, nullable: e4m3 codes of h [M][N]
    float* q_scales;        // [M][ldq]: one per 1x128 block of h
    int ldq;
    uint32_t* status;
};

__device__ __forceinline__ void decode_tile(int tile, const int* prefix, int G, int NT, int& g, int& m, int& n) {
    int lo = 0, hi = G - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (prefix[mid] <= tile) lo = mid;
        else hi = mid - 1;
    }
    g = lo;
    const int local = tile - prefix[g];
    const int mt = (prefix[g + 1] - prefix[g]) / NT;
    n = local / mt;
    m = local - n * mt;
}

// (d0, d1) += (a0, a1) * f on the packed two-lane fp32 FMA; each lane rounds
// like fmaf, so the promotion costs half the issue slots of scalar FMAs.
__device__ __forceinline__ void ffma2(float& d0, float& d1, uint32_t a0, uint32_t a1, float f) {
    asm("{\n\t.reg .b64 ra, rf, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rf, {%4, %4};\n\t"
        "mov.b64 rd, {%0, %1};\n\t"
        "fma.rn.f32x2 rd, ra, rf, rd;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "+f"(d0), "+f"(d1)
        : "r"(a0), "r"(a1), "f"(f));
}

// Parity of the index of `tile` among this CTA's tiles (blockIdx.x, +gridDim.x, ...).
__device__ __forceinline__ int tile_parity(int tile, int first, int stride) { return ((tile - first) / stride) & 1; }

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
    __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<uint32_t*>(&v);
}

// NV consecutive bf16 outputs of one row (columns col0.., valid below N).
template <int NV>
__device__ __forceinline__ void store_row(__nv_bfloat16* C, int64_t ldc, int64_t row, int col0, int N,
                                          const float* v) {
    __nv_bfloat16* dst = C + row * ldc + col0;
    if (col0 + NV <= N) {
#pragma unroll
        for (int q = 0; q < NV / 8; ++q) {
            uint4 u;
            u.x = pack_bf16x2(v[8 * q + 0], v[8 * q + 1]);
            u.y = pack_bf16x2(v[8 * q + 2], v[8 * q + 3]);
            u.z = pack_bf16x2(v[8 * q + 4], v[8 * q + 5]);
            u.w = pack_bf16x2(v[8 * q + 6], v[8 * q + 7]);
            reinterpret_cast<uint4*>(dst)[q] = u;
        }
    } else {
#pragma unroll
        for (int c = 0; c < NV; ++c)
            if (col0 + c < N) dst[c] = __float2bfloat16_rn(v[c]);
    }
}

// One warp's 32 x 64 bf16 block into a staging box laid out as the 128-byte
// swizzled TMA box expects: 16-byte chunk c of row r at r*128 + ((c ^ (r % 8)) * 16).
// Lane r writes its row; eight consecutive rows cover all banks.
__device__ __forceinline__ void stage_row_sw128(uint8_t* box, int r, const float* v) {
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

// Four exponent bytes (UE8M0) of the power-of-two scales v[kb0 .. kb0+3] (127 past kb_end).
__device__ __forceinline__ uint32_t pack_exponents(const float* v, int kb0, int kb_end) {
    uint32_t w = 0;
#pragma unroll
    for (int b = 0; b < 4; ++b) w |= (kb0 + b < kb_end ? fp8::ue8m0(__ldg(v + kb0 + b)) : 127u) << (8 * b);
    return w;
}

template <int EPI, bool MX>
__global__ void __launch_bounds__(kThreads, 1)
tc_fp8_grouped_gemm_kernel(const __grid_constant__ CUtensorMap mapA, const __grid_constant__ CUtensorMap mapB,
                           const __grid_constant__ CUtensorMap mapC, const __grid_constant__ Params p) {
    constexpr uint32_t IDESC = MX ? idesc_mx_e4m3(BM, BN) : idesc_e4m3(BM, BN);
    constexpr int STAGES = Plan<EPI, MX>::STAGES;
    extern __shared__ uint8_t smem_raw[];
    const uint32_t raw_addr = smem_u32(smem_raw);
    uint8_t* smem = smem_raw + (((raw_addr + 1023u) & ~1023u) - raw_addr);
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * A_BYTES;
    uint8_t* sOut = sB + STAGES * B_BYTES;  // bf16 epilogue: kEpiWarps x 2 staging boxes (1024-aligned)
    uint64_t* bars = reinterpret_cast<uint64_t*>(sOut + Plan<EPI, MX>::OUT_BYTES);
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + Plan<EPI, MX>::NUM_BARS);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* prefix = reinterpret_cast<int*>(tmem_slot + 4);
    int* gstart = prefix + kMaxGroups + 1;
    int* gend = gstart + kMaxGroups;
    float* xamax = reinterpret_cast<float*>(gend + kMaxGroups);  // [2][2][BM]

    auto full_bar = [&](int s) { return smem_u32(bars + s); };
    auto empty_bar = [&](int s) { return smem_u32(bars + STAGES + s); };
    auto pfull_bar = [&](int j) { return smem_u32(bars + 2 * STAGES + j); };
    auto pempty_bar = [&](int j) { return smem_u32(bars + 2 * STAGES + 2 + j); };
    const uint32_t drain_bar = smem_u32(bars + 2 * STAGES + 4);
    auto xchg_bar = [&](int eg) { return smem_u32(bars + 2 * STAGES + 5 + eg); };
    auto sffull_bar = [&](int q) { return smem_u32(bars + 2 * STAGES + 9 + q); };    // MX
    auto sfempty_bar = [&](int q) { return smem_u32(bars + 2 * STAGES + 11 + q); };  // MX

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int G = p.G, NT = p.NT, KB = p.KB;

    // launched after another kernel; only the up projection lets its follower be scheduled early
    // (as in the bf16 kernels: the down projection's follower would wait beside it and slow it)
    if constexpr (EPI == TC_EPI_SWIGLU) pdl_trigger();
    pdl_wait();  // before any read of what earlier work on the stream wrote
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
        gstart[g] = a;
        gend[g] = b;
    }
    if (threadIdx.x == 0) *abort_flag = 0;
    __syncthreads();
    if (warp == 0) {
        int run = 0;
        for (int g0 = 0; g0 < G; g0 += 32) {
            const int g = g0 + lane;
            const int v = g < G ? (gend[g] - gstart[g] + BM - 1) / BM * NT : 0;
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
            for (int j = 0; j < 2; ++j) {
                mbar_init(pfull_bar(j), 1);
                mbar_init(pempty_bar(j), kEpiWarps);
            }
            mbar_init(drain_bar, 1);
            for (int eg = 0; eg < 4; ++eg) mbar_init(xchg_bar(eg), kSplit);  // the warps of a lane group
            for (int q = 0; q < 2; ++q) {
                mbar_init(sffull_bar(q), 4);  // the scale writer of each lane group
                mbar_init(sfempty_bar(q), 1);
            }
            asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            prefetch_tensormap(&mapA);
            prefetch_tensormap(&mapB);
        }
    } else if (warp == 1) {
        tmem_alloc(smem_u32(tmem_slot), TMEM_COLS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int total = prefix[G];

    if (warp == 0) {
        if (lane == 0) {
            // ---------------- TMA producer ----------------
            int s = 0;
            uint32_t ph = 0, issued = 0, issued_par = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                int g, m, n;
                decode_tile(tile, prefix, G, NT, g, m, n);
                const int row0 = gstart[g] + m * BM;
                const int brow = g * p.Nb + n * BN;
                const int tbase = (g * p.b_nt + n) * KB;  // tiled B: this tile's first 256-row box
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_phase_fast(empty_bar(s), ph ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    mbar_arrive_expect_tx(full_bar(s), STAGE_BYTES);
                    tma_load_2d(smem_u32(sA + s * A_BYTES), &mapA, full_bar(s), kb * BK, row0);
                    if (p.b_tiled)  // one contiguous 32 KB box
                        tma_load_2d(smem_u32(sB + s * B_BYTES), &mapB, full_bar(s), 0, (tbase + kb) * BN);
                    else
                        tma_load_2d(smem_u32(sB + s * B_BYTES), &mapB, full_bar(s), kb * BK, brow);
                    issued |= 1u << s;
                    issued_par = (issued_par & ~(1u << s)) | (ph << s);
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
            }
            for (int q = 0; q < STAGES; ++q)
                if ((issued >> q) & 1u) wait_drain(full_bar(q), (issued_par >> q) & 1u, p.status);
        }
    } else if (warp == 1 && MX) {
        if (lane == 0) {
            // ---------------- MMA issuer, block-scaled: one accumulator per tile ----------------
            int s = 0, sq = 0;
            uint32_t ph = 0, dph = 0, sph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                // the epilogue has drained the previous tile's accumulator
                if (!wait_phase_fast(pempty_bar(0), dph ^ 1u, abort_flag, p.status)) break;
                tc_fence_after();
                for (int kb = 0; kb < KB; ++kb) {
                    if ((kb % kSfGroup) == 0) {
                        if (!wait_phase_fast(sffull_bar(sq), sph, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                    }
                    if (!wait_phase_fast(full_bar(s), ph, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t sf = tmem_base + (uint32_t)(kSfBase + sq * kSfCols);
                    const uint32_t slot = (uint32_t)((kb % kSfGroup) >> 2), id = (uint32_t)(kb & 3);
                    const uint32_t idesc = IDESC | idesc_sf_ids(id, id);
                    const uint64_t adesc = smem_desc_sw128(smem_u32(sA + s * A_BYTES));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + s * B_BYTES));
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)
                        mma_mx_e4m3(tmem_base, adesc + 2u * kk, bdesc + 2u * kk, idesc, sf + 8u * slot,
                                    sf + 32u + 8u * slot, (kb | kk) != 0);
                    mma_commit(empty_bar(s));
                    if ((kb % kSfGroup) == kSfGroup - 1 || kb == KB - 1) {
                        mma_commit(sfempty_bar(sq));
                        if (++sq == 2) {
                            sq = 0;
                            sph ^= 1u;
                        }
                    }
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                }
                if (!ok) break;
                mma_commit(pfull_bar(0));  // the tile's accumulator is complete
                dph ^= 1u;
            }
            mma_commit(drain_bar);
            wait_drain(drain_bar, 0, p.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ---------------- MMA issuer: one partial per K block ----------------
            int s = 0, j = 0;
            uint32_t ph = 0, pph = 0;
            bool ok = true;
            for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
                for (int kb = 0; kb < KB; ++kb) {
                    if (!wait_phase_fast(full_bar(s), ph, abort_flag, p.status) ||
                        !wait_phase_fast(pempty_bar(j), pph ^ 1u, abort_flag, p.status)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t d = tmem_base + (uint32_t)(j * BN);
                    const uint64_t adesc = smem_desc_sw128(smem_u32(sA + s * A_BYTES));
                    const uint64_t bdesc = smem_desc_sw128(smem_u32(sB + s * B_BYTES));
#pragma unroll
                    for (int kk = 0; kk < BK / UMMA_K; ++kk)  // +32 bytes per K=32 slice
                        mma_e4m3(d, adesc + 2u * kk, bdesc + 2u * kk, IDESC, kk != 0);
                    mma_commit(empty_bar(s));
                    mma_commit(pfull_bar(j));
                    if (++s == STAGES) {
                        s = 0;
                        ph ^= 1u;
                    }
                    if (++j == 2) {
                        j = 0;
                        pph ^= 1u;
                    }
                }
            }
            mma_commit(drain_bar);
            wait_drain(drain_bar, 0, p.status);
        }
    } else {
        // ---------------- epilogue: kEpiWarps warps, each (lane group, column part) ----------------
        const int eg = warp & 3;
        const int part = (warp - 2) >> 2;  // 0 .. kSplit-1
        const int r = eg * 32 + lane;
        // the thread's two kCols-column chunks: gate and up slices of a packed block (SwiGLU), or two
        // adjacent slices of one 128-column block
        const int colA = EPI == TC_EPI_SWIGLU ? part * kCols : part * 2 * kCols;
        const int colB = EPI == TC_EPI_SWIGLU ? 128 + part * kCols : part * 2 * kCols + kCols;
        const int nbA = EPI == TC_EPI_SWIGLU ? 0 : colA / 128;  // scale block of each chunk inside the tile
        const int nbB = EPI == TC_EPI_SWIGLU ? 1 : colB / 128;
        const int nblocks = p.Nb / 128;
        int j = 0;
        uint32_t pph = 0, xph = 0;
        float acc[2 * kCols];
        bool ok = true;
        // MX: the first warp of each lane group writes the scale-factor groups, in
        // the order the MMAs consume them (two buffers)
        int wq = 0;
        uint32_t wph = 0, dph = 0;
        const int n_sf_groups = (KB + kSfGroup - 1) / kSfGroup;
        auto write_sf_group = [&](int tile, int grp) -> bool {
            if (!__all_sync(0xffffffffu, wait_phase_fast(sfempty_bar(wq), wph ^ 1u, abort_flag, p.status)))
                return false;
            int g, m, n;
            decode_tile(tile, prefix, G, NT, g, m, n);
            const int64_t row = (int64_t)gstart[g] + (int64_t)m * BM + r;
            const int64_t srow = row < p.M ? row : p.M - 1;
            const float* sa_row = p.a_scales + srow * p.lda_s;
            const float* sb0 = p.b_scales + ((int64_t)g * nblocks + n * 2) * KB;  // columns 0..127 of the tile
            const float* sb1 = sb0 + KB;                                          // columns 128..255
            const int kb0 = grp * kSfGroup;
            uint32_t aw[32], bw[32];
#pragma unroll
            for (int sl = 0; sl < 4; ++sl) {
                const uint32_t a = pack_exponents(sa_row, kb0 + 4 * sl, KB);
                const uint32_t w0 = pack_exponents(sb0, kb0 + 4 * sl, KB), w1 = pack_exponents(sb1, kb0 + 4 * sl, KB);
#pragma unroll
                for (int c = 0; c < 8; ++c) {
                    aw[8 * sl + c] = a;  // lane group eg reads column 8*slot + eg
                    bw[8 * sl + c] = c < 4 ? w0 : w1;
                }
            }
            const uint32_t t = tmem_base + ((uint32_t)(eg * 32) << 16) + (uint32_t)(kSfBase + wq * kSfCols);
            tmem_st32(t, aw);        // A slots: columns [0, 32) of the group
            tmem_st32(t + 32u, bw);  // B slots: columns [32, 64), in every lane group
            tmem_wait_st();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(sffull_bar(wq));
            if (++wq == 2) {
                wq = 0;
                wph ^= 1u;
            }
            return true;
        };
        if (MX && part == 0 && (int)blockIdx.x < total) ok = write_sf_group(blockIdx.x, 0);
        for (int tile = blockIdx.x; ok && tile < total; tile += gridDim.x) {
            int g, m, n;
            decode_tile(tile, prefix, G, NT, g, m, n);
            const int64_t row = (int64_t)gstart[g] + (int64_t)m * BM + r;
            const bool valid = row < gend[g];
            const int64_t srow = row < p.M ? row : p.M - 1;  // scale row (rows past M are never stored)
            const float* sa_row = p.a_scales + srow * p.lda_s;
            const float* sbA = p.b_scales + ((int64_t)g * nblocks + n * 2 + nbA) * KB;
            const float* sbB = p.b_scales + ((int64_t)g * nblocks + n * 2 + nbB) * KB;
            if constexpr (MX) {
                // the rest of this tile's scale groups and the next tile's first, then the accumulator
                if (part == 0) {
                    for (int grp = 1; ok && grp < n_sf_groups; ++grp) ok = write_sf_group(tile, grp);
                    if (ok && tile + (int)gridDim.x < total) ok = write_sf_group(tile + gridDim.x, 0);
                }
                if (!ok) break;
                if (!__all_sync(0xffffffffu, wait_phase_fast(pfull_bar(0), dph, abort_flag, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(eg * 32) << 16);
#pragma unroll
                for (int q = 0; q < kCols / 16; ++q) {
                    uint32_t va[16], vb[16];
                    tmem_ld16x2(taddr + colA + 16 * q, taddr + colB + 16 * q, va, vb);
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        acc[16 * q + i] = __uint_as_float(va[i]);
                        acc[kCols + 16 * q + i] = __uint_as_float(vb[i]);
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pempty_bar(0));  // the next tile's MMAs may overwrite it
                dph ^= 1u;
            } else {
#pragma unroll
            for (int i = 0; i < 2 * kCols; ++i) acc[i] = 0.0f;
            float sa_next = __ldg(sa_row), sbA_next = __ldg(sbA), sbB_next = __ldg(sbB);
            for (int kb = 0; kb < KB; ++kb) {
                // bf16 epilogue: both chunks lie in one 128-column scale block, so one factor serves
                // (one scale load and one fewer register: dsv3_prefill_fp8 down 751 -> 738 us)
                const float fA = sa_next * sbA_next, fB = EPI == TC_EPI_BF16 ? fA : sa_next * sbB_next;
                if (kb + 1 < KB) {
                    sa_next = __ldg(sa_row + kb + 1);
                    sbA_next = __ldg(sbA + kb + 1);
                    sbB_next = __ldg(sbB + kb + 1);
                }
                if (!__all_sync(0xffffffffu, wait_phase_fast(pfull_bar(j), pph, abort_flag, p.status))) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(eg * 32) << 16) + (uint32_t)(j * BN);
                if constexpr (EPI == TC_EPI_BF16) {
                    // 16 columns of chunk A and of chunk B at a time; the next pair's loads are in
                    // flight while this pair is scaled and added (measured on the DeepSeek-V3 down
                    // projection: 765 -> 751 us; the SwiGLU instantiation, short of registers, slows)
                    uint32_t va[2][16], vb[2][16];
                    tmem_ld16x2_nowait(taddr + colA, taddr + colB, va[0], vb[0]);
                    tmem_wait_ld32(va[0], vb[0]);
#pragma unroll
                    for (int q = 0; q < kCols / 16; ++q) {
                        if (q + 1 < kCols / 16)
                            tmem_ld16x2_nowait(taddr + colA + 16 * (q + 1), taddr + colB + 16 * (q + 1),
                                               va[(q + 1) & 1], vb[(q + 1) & 1]);
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {  // two columns per packed FMA
                            ffma2(acc[16 * q + i], acc[16 * q + i + 1], va[q & 1][i], va[q & 1][i + 1], fA);
                            ffma2(acc[kCols + 16 * q + i], acc[kCols + 16 * q + i + 1], vb[q & 1][i],
                                  vb[q & 1][i + 1], fB);
                        }
                        if (q + 1 < kCols / 16) tmem_wait_ld32(va[(q + 1) & 1], vb[(q + 1) & 1]);
                    }
                } else {
#pragma unroll
                    for (int q = 0; q < kCols / 16; ++q) {  // 16 columns of chunk A and of chunk B
                        uint32_t va[16], vb[16];
                        tmem_ld16x2(taddr + colA + 16 * q, taddr + colB + 16 * q, va, vb);
#pragma unroll
                        for (int i = 0; i < 16; i += 2) {  // two columns per packed FMA
                            ffma2(acc[16 * q + i], acc[16 * q + i + 1], va[i], va[i + 1], fA);
                            ffma2(acc[kCols + 16 * q + i], acc[kCols + 16 * q + i + 1], vb[i], vb[i + 1], fB);
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(pempty_bar(j));
                if (++j == 2) {
                    j = 0;
                    pph ^= 1u;
                }
            }
            if (!ok) break;
            }
            __nv_bfloat16* C = static_cast<__nv_bfloat16*>(p.C);
            if (EPI == TC_EPI_SWIGLU) {
                // h in bf16 (the precision it is stored and quantised in)
                float h[kCols];
                float am = 0.0f;
                // silu(g) = g / (1 + e^-g) with the fast reciprocal (2 ulp; h is then rounded to bf16):
                // the IEEE division's 64 per thread sat on the tile's tail, which the next tile's
                // MMAs wait behind
#pragma unroll
                for (int i = 0; i < kCols; i += 2) {  // two roundings to bf16 per conversion
                    const __nv_bfloat162 hb = __floats2bfloat162_rn(
                        __fdividef(acc[i], 1.0f + __expf(-acc[i])) * acc[kCols + i],
                        __fdividef(acc[i + 1], 1.0f + __expf(-acc[i + 1])) * acc[kCols + i + 1]);
                    h[i] = __low2float(hb);
                    h[i + 1] = __high2float(hb);
                    am = fmaxf(am, fmaxf(fabsf(h[i]), fabsf(h[i + 1])));
                }
                const int col0 = n * 128 + part * kCols;
                if (valid && C) store_row<kCols>(C, p.ldc, row, col0, p.N, h);
                if (p.q) {
                    // amax of the 128-column block: the maximum over the kSplit warps' parts
                    float* slot = xamax + tile_parity(tile, blockIdx.x, gridDim.x) * kSplit * BM;
                    slot[part * BM + r] = am;
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xchg_bar(eg));
                    if (!__all_sync(0xffffffffu, wait_phase_fast(xchg_bar(eg), xph, abort_flag, p.status))) break;
                    xph ^= 1u;
#pragma unroll
                    for (int o = 0; o < kSplit; ++o) am = fmaxf(am, slot[o * BM + r]);
                    const float sc = fp8::scale_for(am, MX);
                    if (valid) {
                        // fl32(h / sc) with one division per block, as the row quantiser takes it
                        const float rsc = 1.0f / sc;
                        if (MX) {
#pragma unroll
                            for (int i = 0; i < kCols; ++i) h[i] = __fmul_rn(h[i], rsc);
                        } else if (fp8::quotient_ok(sc)) {
#pragma unroll
                            for (int i = 0; i < kCols; ++i) h[i] = fp8::quotient(h[i], sc, rsc);
                        } else {
#pragma unroll
                            for (int i = 0; i < kCols; ++i) h[i] = h[i] / sc;
                        }
                        uint8_t* qrow = p.q + row * (int64_t)p.N + col0;
#pragma unroll
                        for (int c = 0; c < kCols / 16; ++c) {  // 16 codes per store; N % 16 == 0
                            if (col0 + 16 * c < p.N) {
                                uint32_t w4[4];
#pragma unroll
                                for (int t = 0; t < 4; ++t)
                                    w4[t] = fp8::e4m3x4(h[16 * c + 4 * t], h[16 * c + 4 * t + 1],
                                                        h[16 * c + 4 * t + 2], h[16 * c + 4 * t + 3]);
                                reinterpret_cast<uint4*>(qrow)[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
                            }
                        }
                        if (part == 0) p.q_scales[row * (int64_t)p.ldq + n] = sc;
                    }
                }
            } else {
                // all 32 rows of this warp inside the expert's segment: stage and TMA-store
                // the two 32 x 64 blocks; a warp holding rows past the segment (they belong
                // to the next expert) stores its valid rows directly
                if (p.c_tma && __all_sync(0xffffffffu, valid)) {
                    uint8_t* box = sOut + (warp - 2) * 2 * kOutBox;
                    if (lane == 0) bulk_wait_read_all();  // the previous tile's boxes have left
                    __syncwarp();
                    stage_row_sw128(box, lane, acc);
                    stage_row_sw128(box + kOutBox, lane, acc + kCols);
                    fence_proxy_async_smem();
                    __syncwarp();
                    if (lane == 0) {
                        const int row0 = gstart[g] + m * BM + eg * 32;
                        if (n * BN + colA < p.N) tma_store_2d(&mapC, smem_u32(box), n * BN + colA, row0);
                        if (n * BN + colB < p.N) tma_store_2d(&mapC, smem_u32(box + kOutBox), n * BN + colB, row0);
                        bulk_commit();
                    }
                } else if (valid) {
                    store_row<kCols>(C, p.ldc, row, n * BN + colA, p.N, acc);
                    store_row<kCols>(C, p.ldc, row, n * BN + colB, p.N, acc + kCols);
                }
            }
        }
        if (EPI == TC_EPI_BF16 && lane == 0) bulk_wait_all();  // staged stores done before the CTA leaves
    }

    __syncwarp();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem_base, TMEM_COLS);
    }
}

template <int EPI, bool MX>
moe_status_t launch_impl(const TcFp8GroupedGemm& g, cudaStream_t s) {
    static std::once_flag attr_once[64];
    int dev = 0;
    MOE_CUDA_TRY(cudaGetDevice(&dev));
    cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once[dev & 63], [&] {
        attr_err = cudaFuncSetAttribute(tc_fp8_grouped_gemm_kernel<EPI, MX>,
                                        cudaFuncAttributeMaxDynamicSharedMemorySize, (int)Plan<EPI, MX>::SMEM);
    });
    MOE_CUDA_TRY(attr_err);
    CUtensorMap ma, mb, mc;
    const int b_nt = (int)ceil_div(g.Nb, 256), KBt = (int)ceil_div(g.K, BK);
    if (!make_map(&ma, g.A, (uint64_t)g.K, (uint64_t)g.M, BM, 1)) return MOE_ERR_CUDA;
    if (g.b_tiled) {
        // box rows are addressed with int coordinates
        if ((int64_t)g.G * b_nt * KBt * 256 >= INT_MAX) return MOE_ERR_UNSUPPORTED;
        if (!make_map(&mb, g.B, (uint64_t)BK, (uint64_t)g.G * b_nt * KBt * 256, BN, 1)) return MOE_ERR_CUDA;
    } else if (!make_map(&mb, g.B, (uint64_t)g.K, (uint64_t)g.G * g.Nb, BN, 1)) {
        return MOE_ERR_CUDA;
    }
    // bf16 output through TMA stores when the map can describe it (else direct stores)
    const bool c_tma = EPI == TC_EPI_BF16 && !MX && g.C &&  // staged tiles (fp32 scales)
                       make_store_map_bf16(&mc, g.C, (uint64_t)g.N, (uint64_t)g.M, (uint64_t)g.ldc, 32);
    if (!c_tma) mc = ma;  // never read
    Params p;
    p.offsets = g.offsets;
    p.G = g.G;
    p.M = g.M;
    p.K = g.K;
    p.Nb = g.Nb;
    p.N = g.N;
    p.NT = (int)ceil_div(g.Nb, BN);
    p.KB = (int)ceil_div(g.K, BK);
    p.C = g.C;
    p.ldc = g.ldc;
    p.a_scales = g.a_scales;
    p.lda_s = g.lda_scales;
    p.b_scales = g.b_scales;
    p.c_tma = c_tma ? 1 : 0;
    p.b_tiled = g.b_tiled ? 1 : 0;
    p.b_nt = b_nt;
    p.q = g.q;
    p.q_scales = g.q_scales;
    p.ldq = g.ldq;
    p.status = g.status;
    const int64_t max_tiles = (int64_t)p.NT * (ceil_div(g.M, BM) + (g.offsets ? g.G : 0));
    const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(sm_count(), max_tiles));
    if (g.pdl) {
        MOE_CUDA_TRY(launch_pdl(tc_fp8_grouped_gemm_kernel<EPI, MX>, dim3(grid), dim3(kThreads), Plan<EPI, MX>::SMEM, s,
                                ma, mb, mc, p));
    } else {
        tc_fp8_grouped_gemm_kernel<EPI, MX><<<grid, kThreads, Plan<EPI, MX>::SMEM, s>>>(ma, mb, mc, p);
        MOE_CUDA_TRY(cudaGetLastError());
    }
    note_launch();
    return MOE_OK;
}

}  // namespace

moe_status_t launch_tc_fp8_grouped_gemm(const TcFp8GroupedGemm& g, cudaStream_t s) {
    if (g.M == 0 || g.G == 0) return MOE_OK;
    if (g.G > kMaxGroups) return MOE_ERR_UNSUPPORTED;
    if (g.Nb % BN != 0 || g.K % 16 != 0) return MOE_ERR_INVALID_ARG;
    if (g.q && (g.epi != TC_EPI_SWIGLU || g.N % 16 != 0 || !g.q_scales || g.ldq < (int)ceil_div(g.N, 128)))
        return MOE_ERR_INVALID_ARG;
    if (!g.q && !g.C) return MOE_ERR_INVALID_ARG;
    switch (g.epi) {
        case TC_EPI_SWIGLU:
            return g.pow2 ? launch_impl<TC_EPI_SWIGLU, true>(g, s) : launch_impl<TC_EPI_SWIGLU, false>(g, s);
        case TC_EPI_BF16: return g.pow2 ? launch_impl<TC_EPI_BF16, true>(g, s) : launch_impl<TC_EPI_BF16, false>(g, s);
        default: return MOE_ERR_INVALID_ARG;
    }
}

}  // namespace moe
