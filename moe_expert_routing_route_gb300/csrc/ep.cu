// Expert-parallel Double-Routing on one GPU.
//
// "DeepSeek-R1 prefill inference optimisation on Atlas A3" (cann-recipes-infer),
// §MoE deployment strategy, Double-Routing:
//   step 1  init-routing on each rank's own tokens (sorted by global expert)
//   step 2  AlltoAll of tokens_per_expert -> send/receive splits
//   step 3  AlltoAll of the tokens to the ranks that own their experts
//   step 4  re-routing: the received tokens, grouped by source rank, are
//           sorted again by local expert; gathered_ids_unsort remembers where
//           each sorted row came from
//   step 5  routed experts on the sorted rows
//   step 6  rows back in received order by index_select with the argsort of
//           gathered_ids_unsort
//   step 7  AlltoAll back to the source ranks
//   step 8  finalize-routing on each source rank
// Here W virtual ranks share one GPU: rank p owns tokens [p*T/W, (p+1)*T/W)
// and experts [p*E/W, (p+1)*E/W).  The two AlltoAlls become one device-side
// copy of row blocks whose sizes and offsets are computed on the device from
// the per-source expert counts (no host round trip, as for the single-routing
// path).  Every row's expert FFN and the finalize sums are the same arithmetic
// as in moe_layer_forward, so both paths give the same output bit for bit.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr int kPlanThreads = 1024;

// Dispatch plan.  counts_all [W][E]: rows of source p for expert e (its
// init-routing counts).  Outputs:
//   xfer [W*W][3]: (src row in the sources' expanded rows, dst row in the
//                  receive buffer, rows) of block p -> q, indexed p*W + q
//   recv_start [W+1]: first row of rank q's received rows
//   counts_recv [W(q)][W(p)][El]: rows rank q receives from p for local expert e
__global__ void __launch_bounds__(kPlanThreads)
ep_dispatch_plan_kernel(const int32_t* __restrict__ counts_all, int W, int E, int El, int Rp,
                        int32_t* __restrict__ xfer, int32_t* __restrict__ recv_start,
                        int32_t* __restrict__ counts_recv) {
    __shared__ int size_pq[32 * 32];
    __shared__ int start_q[33];
    const int tid = threadIdx.x;
    if (tid < W * W) {
        const int p = tid / W, q = tid % W;
        int sum = 0;
        for (int e = 0; e < El; ++e) sum += counts_all[p * E + q * El + e];
        size_pq[p * W + q] = sum;
    }
    __syncthreads();
    if (tid == 0) {
        start_q[0] = 0;
        for (int q = 0; q < W; ++q) {
            int tot = 0;
            for (int p = 0; p < W; ++p) tot += size_pq[p * W + q];
            start_q[q + 1] = start_q[q] + tot;
        }
        for (int q = 0; q <= W; ++q) recv_start[q] = start_q[q];
    }
    __syncthreads();
    if (tid < W * W) {
        const int p = tid / W, q = tid % W;
        int src = p * Rp, dst = start_q[q];
        for (int q2 = 0; q2 < q; ++q2) src += size_pq[p * W + q2];
        for (int p2 = 0; p2 < p; ++p2) dst += size_pq[p2 * W + q];
        xfer[3 * tid + 0] = src;
        xfer[3 * tid + 1] = dst;
        xfer[3 * tid + 2] = size_pq[p * W + q];
    }
    for (int i = tid; i < W * W * El; i += kPlanThreads) {
        const int q = i / (W * El), p = (i / El) % W, e = i % El;
        counts_recv[i] = counts_all[p * E + q * El + e];
    }
}

// Re-routing plan for Q receiving ranks, one block per rank q.  Rank q's
// received rows start at base = recv_start[q] (0 when recv_start is null) and
// arrive in (source p, local expert e) order with counts c[q][p][e]; sorted,
// they go in (e, p) order.  Outputs:
//   rr [Q][P][El][3]: (src row, dst row, rows) of block (p, e) of rank q
//   tokens_per_local_expert [Q][El], local_offsets [Q][El+1] (from 0),
//   goff [Q][El+1] (= base + local_offsets: rows in the whole sorted buffer)
//   eoff [Q*El+1] (nullable): the same offsets as one array over all ranks' experts
//     in rank order; with ranks laid out contiguously (base[q+1] = base[q] + rows
//     of rank q) it segments the whole sorted buffer by global expert
// expect_rows >= 0: the rank's rows must add up to it, else every block is
// emptied and the status bit is set.
__global__ void __launch_bounds__(kPlanThreads)
re_routing_plan_kernel(const int32_t* __restrict__ counts_recv, const int32_t* __restrict__ recv_start, int P,
                       int El, int expect_rows, int32_t* __restrict__ rr, int32_t* __restrict__ tpl,
                       int32_t* __restrict__ local_off, int32_t* __restrict__ goff, int32_t* __restrict__ eoff,
                       uint32_t* status) {
    __shared__ int scan_buf[1025];
    __shared__ int arrive_base;  // rows of earlier sources
    __shared__ int total_rows;
    const int q = blockIdx.x, tid = threadIdx.x;
    const int base = recv_start ? recv_start[q] : 0;
    const int32_t* c = counts_recv + (size_t)q * P * El;
    // tokens per local expert and their exclusive scan (serial over El <= 1024 in thread 0 is
    // avoided: each thread sums its expert, then a shared-memory scan by thread 0 of El values)
    int t_e = 0;
    if (tid < El)
        for (int p = 0; p < P; ++p) t_e += c[p * El + tid];
    if (tid < El) scan_buf[tid] = t_e;
    __syncthreads();
    if (tid == 0) {
        int run = 0;
        for (int e = 0; e < El; ++e) {
            const int v = scan_buf[e];
            scan_buf[e] = run;
            run += v;
        }
        scan_buf[El] = run;
        total_rows = run;
        arrive_base = 0;
    }
    __syncthreads();
    const bool ok = expect_rows < 0 || total_rows == expect_rows;
    if (!ok && tid == 0) set_status(status, MOE_DEVERR_BAD_OFFSETS);
    if (tid <= El) {
        local_off[(size_t)q * (El + 1) + tid] = ok ? scan_buf[tid] : 0;
        goff[(size_t)q * (El + 1) + tid] = base + (ok ? scan_buf[tid] : 0);
        // rank q writes its El starts; the last rank also writes the end
        if (eoff && (tid < El || q == gridDim.x - 1)) eoff[(size_t)q * El + tid] = base + (ok ? scan_buf[tid] : 0);
    }
    if (tid < El) tpl[(size_t)q * El + tid] = ok ? t_e : 0;
    int dst_run = tid < El ? scan_buf[tid] : 0;  // next sorted row of expert tid
    __syncthreads();
    for (int p = 0; p < P; ++p) {
        // exclusive scan of c[p][*] over e gives the arrival offsets inside source p
        const int v = tid < El ? c[p * El + tid] : 0;
        __syncthreads();
        if (tid < El) scan_buf[tid] = v;
        __syncthreads();
        if (tid == 0) {
            int run = 0;
            for (int e = 0; e < El; ++e) {
                const int x = scan_buf[e];
                scan_buf[e] = run;
                run += x;
            }
            scan_buf[El] = run;
        }
        __syncthreads();
        if (tid < El) {
            int32_t* ent = rr + ((size_t)(q * P + p) * El + tid) * 3;
            ent[0] = base + arrive_base + scan_buf[tid];
            ent[1] = base + dst_run;
            ent[2] = ok ? v : 0;
            dst_run += v;
        }
        __syncthreads();
        if (tid == 0) arrive_base += scan_buf[El];
        __syncthreads();
    }
}

// Copy row blocks: entry i moves table[i].n rows from row table[i].src of
// `src` to row table[i].dst of `dst` (swapped when reverse != 0).  gidx, when
// not null, receives gidx[dst row] = src row.  blockIdx.y splits an entry's rows.
__global__ void __launch_bounds__(256)
copy_row_blocks_kernel(const uint4* __restrict__ src, uint4* __restrict__ dst, int nvec,
                       const int32_t* __restrict__ table, int n_entries, int reverse, int32_t* __restrict__ gidx) {
    const int ent = blockIdx.x;
    if (ent >= n_entries) return;
    int s0 = table[3 * ent], d0 = table[3 * ent + 1];
    const int n = table[3 * ent + 2];
    if (reverse) {
        const int t = s0;
        s0 = d0;
        d0 = t;
    }
    const int per = (n + gridDim.y - 1) / gridDim.y;
    const int r0 = blockIdx.y * per, r1 = min(n, r0 + per);
    if (gidx)
        for (int r = r0 + threadIdx.x; r < r1; r += blockDim.x) gidx[d0 + r] = s0 + r;
    for (int r = r0; r < r1; ++r) {
        const uint4* srow = src + (size_t)(s0 + r) * nvec;
        uint4* drow = dst + (size_t)(d0 + r) * nvec;
        for (int v = threadIdx.x; v < nvec; v += blockDim.x) drow[v] = __ldcs(srow + v);
    }
}

// out[gidx[i]] = y_sorted[i] for i < N (indices outside [0, N) are skipped and flagged).
__global__ void __launch_bounds__(256)
unsort_rows_kernel(const uint4* __restrict__ y, int nvec, const int32_t* __restrict__ gidx, int N,
                   uint4* __restrict__ out, uint32_t* status) {
    for (int i = blockIdx.x; i < N; i += gridDim.x) {
        const int d = gidx[i];
        if (d < 0 || d >= N) {
            if (threadIdx.x == 0) set_status(status, MOE_DEVERR_BAD_ROW_INDEX);
            continue;
        }
        const uint4* yr = y + (size_t)i * nvec;
        uint4* orow = out + (size_t)d * nvec;
        for (int v = threadIdx.x; v < nvec; v += blockDim.x) orow[v] = __ldcs(yr + v);
    }
}

moe_status_t launch_copy_blocks(const void* src, void* dst, size_t row_bytes, const int32_t* table, int n_entries,
                                int reverse, int32_t* gidx, int avg_rows, cudaStream_t s) {
    if (n_entries == 0) return MOE_OK;
    const int nvec = (int)(row_bytes / 16);
    // enough blocks to keep HBM busy: about 8 per SM over all entries
    const int want = (int)std::max<int64_t>(1, (int64_t)sm_count() * 8 / n_entries);
    const int split = std::max(1, std::min(want, std::max(1, avg_rows)));
    dim3 grid((unsigned)n_entries, (unsigned)std::min(split, 65535));
    copy_row_blocks_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(src), static_cast<uint4*>(dst), nvec, table,
                                                n_entries, reverse, gidx);
    note_launch();
    return last_launch_status();
}

}  // namespace

size_t re_routing_plan_ints(int W, int El) { return (size_t)W * El * 3 + 2 * (size_t)(El + 1) + El; }

moe_status_t launch_re_routing(const void* x_recv, size_t row_bytes, const int32_t* counts, int W, int El, int N,
                               void* x_sorted, int32_t* gidx, int32_t* tpl, int32_t* local_off, int32_t* plan,
                               uint32_t* status, cudaStream_t s) {
    int32_t* rr = plan;
    int32_t* goff = plan + (size_t)W * El * 3;
    re_routing_plan_kernel<<<1, kPlanThreads, 0, s>>>(counts, nullptr, W, El, N, rr, tpl, local_off, goff, nullptr,
                                                      status);
    note_launch();
    MOE_TRY(last_launch_status());
    if (N == 0) return MOE_OK;
    return launch_copy_blocks(x_recv, x_sorted, row_bytes, rr, W * El, 0, gidx, std::max(1, N / (W * El)), s);
}

moe_status_t launch_unsort_rows(const void* y_sorted, size_t row_bytes, const int32_t* gidx, int N, void* out,
                                uint32_t* status, cudaStream_t s) {
    if (N == 0) return MOE_OK;
    const int grid = (int)std::min<int64_t>(N, (int64_t)sm_count() * 16);
    unsort_rows_kernel<<<grid, 256, 0, s>>>(static_cast<const uint4*>(y_sorted), (int)(row_bytes / 16), gidx, N,
                                            static_cast<uint4*>(out), status);
    note_launch();
    return last_launch_status();
}

size_t ep_scratch_ints(int W, int E) {
    const int El = E / W;
    return (size_t)W * E                    // counts_all
           + (size_t)W * (E + 1)            // offsets_all
           + (size_t)W * W * 3 + W + 1      // xfer, recv_start
           + (size_t)W * W * El             // counts_recv
           + (size_t)W * W * El * 3         // re-routing blocks
           + (size_t)W * El                 // tokens per local expert
           + 2 * (size_t)W * (El + 1)       // local and global offsets
           + (size_t)E + 1;                 // global offsets by global expert
}

moe_status_t ep_route_and_dispatch(const EpBuffers& b, cudaStream_t s) {
    const int W = b.W, E = b.E, El = E / W, Tp = b.T / W, Rp = Tp * b.k;
    int32_t* counts_all = b.scratch;
    int32_t* offsets_all = counts_all + (size_t)W * E;
    int32_t* xfer = offsets_all + (size_t)W * (E + 1);
    int32_t* recv_start = xfer + (size_t)W * W * 3;
    int32_t* counts_recv = recv_start + W + 1;
    int32_t* rr = counts_recv + (size_t)W * W * El;
    int32_t* tpl = rr + (size_t)W * W * El * 3;
    int32_t* local_off = tpl + (size_t)W * El;
    int32_t* goff = local_off + (size_t)W * (El + 1);
    int32_t* eoff = goff + (size_t)W * (El + 1);
    // step 1: init-routing per source rank (row indices local to the rank)
    for (int p = 0; p < W; ++p) {
        MOE_TRY(launch_init_routing_index(b.ids + (size_t)p * Rp, Rp, E, counts_all + (size_t)p * E,
                                          offsets_all + (size_t)p * (E + 1), b.row_idx + (size_t)p * Rp,
                                          b.hist_scratch, b.status, s));
        MOE_TRY(launch_permute_rows(static_cast<const char*>(b.x) + (size_t)p * Tp * b.row_bytes, b.row_bytes,
                                    b.row_idx + (size_t)p * Rp, Tp, b.k,
                                    static_cast<char*>(b.expanded) + (size_t)p * Rp * b.row_bytes, s));
    }
    // steps 2-3: splits and the token exchange
    ep_dispatch_plan_kernel<<<1, kPlanThreads, 0, s>>>(counts_all, W, E, El, Rp, xfer, recv_start, counts_recv);
    note_launch();
    MOE_TRY(last_launch_status());
    MOE_TRY(launch_copy_blocks(b.expanded, b.recv, b.row_bytes, xfer, W * W, 0, nullptr, Rp / W, s));
    // step 4: re-routing on every receiving rank
    re_routing_plan_kernel<<<W, kPlanThreads, 0, s>>>(counts_recv, recv_start, W, El, -1, rr, tpl, local_off, goff,
                                                      eoff, b.status);
    note_launch();
    MOE_TRY(last_launch_status());
    MOE_TRY(launch_copy_blocks(b.recv, b.sorted, b.row_bytes, rr, W * W * El, 0, b.gidx,
                               std::max(1, Rp / (W * El)), s));
    return MOE_OK;
}

size_t ep_recv_start_int(int W, int E) { return (size_t)W * E + (size_t)W * (E + 1) + (size_t)W * W * 3; }

size_t ep_expert_offsets_int(int W, int E) {
    const int El = E / W;
    return ep_recv_start_int(W, E) + W + 1 + (size_t)W * W * El + (size_t)W * W * El * 3 + (size_t)W * El +
           2 * (size_t)W * (El + 1);
}

const int32_t* ep_rank_offsets(const EpBuffers& b, int q) {
    const int W = b.W, E = b.E, El = E / W;
    const int32_t* goff = b.scratch + (size_t)W * E + (size_t)W * (E + 1) + (size_t)W * W * 3 + W + 1 +
                          (size_t)W * W * El + (size_t)W * W * El * 3 + (size_t)W * El + (size_t)W * (El + 1);
    return goff + (size_t)q * (El + 1);
}

const int32_t* ep_expert_offsets(const EpBuffers& b) {
    const int W = b.W, E = b.E, El = E / W;
    return ep_rank_offsets(b, 0) + (size_t)W * (El + 1);
}

moe_status_t ep_combine(const EpBuffers& b, const void* y_sorted, void* y_recv, void* y_expanded, cudaStream_t s) {
    const int W = b.W, E = b.E, Rp = (b.T / W) * b.k;
    const int32_t* xfer = b.scratch + (size_t)W * E + (size_t)W * (E + 1);
    // step 6: back to received order; step 7: back to the source ranks
    MOE_TRY(launch_unsort_rows(y_sorted, b.row_bytes, b.gidx, b.T * b.k, y_recv, b.status, s));
    return launch_copy_blocks(y_recv, y_expanded, b.row_bytes, xfer, W * W, 1, nullptr, Rp / W, s);
}

}  // namespace moe
