// route.cu -- routing counts, prefix offsets and stable expert-major ranks.
//
// What is computed ("dispatch_combine_shmem.py", "1. Implement Dispatch
// Operator"; "PTO MegaMoE Dispatch + Combine Fusion Example", FrontReorder
// Stage):
//   counts[e]           rows per expert (expert_token_nums_out)
//   offsets[e]          exclusive prefix of counts (the begin index of each
//                       expert's block in "Local data copy")
//   recv_cum[e*P + p]   inclusive running sum over (expert, partition)
//                       (ep_receive_count)
//   route_row[t*K + k]  row of route (t, k) (expandedRowIdx); -1 if inactive,
//                       -2 / -3 for a zero / copy expert (no row)
//   assist[row]         (partition, token in partition, slot)
// Row order is expert, then partition, then token, then slot.  Within one
// expert this is the route order, so a route's row is offsets[e] plus the
// number of earlier active routes with the same expert: the "token_repeat_num"
// of the send loop, computed here as a stable counting sort.
//
// GB300 design (not the pages' O((BS*K)^2) per-route count).  Routes are cut
// into chunks of 32..256 tokens (route_chunk_tokens) that never cross a
// partition boundary.
//   k_route_local  one CTA per chunk.  Each warp loads a contiguous slice of
//                  the chunk (all its loads issued at once), then walks it in
//                  order with warp_match: one shared-memory add per
//                  distinct expert per 32 routes gives every route its rank
//                  among same-expert routes of the warp.  Warp counts are
//                  then scanned across warps, giving each route its rank
//                  inside the chunk (written to route_row) and the chunk's
//                  per-expert histogram.
//   k_route_scan   one CTA: per expert, the histograms of all chunks are
//                  summed by several threads in parallel (contiguous chunk
//                  ranges, independent loads), the totals are scanned over
//                  experts (offsets), and every histogram entry is replaced
//                  by its chunk base: offsets[e] + counts of earlier chunks.
//                  It also writes recv_cum, the GEMM m-block schedule and the
//                  call's status word.
// The final row, base[chunk][e] + rank in chunk, is resolved by the kernel
// that next touches each token (row copy, quantisation, or k_route_resolve
// when no rows are copied), which also writes the triplet of the row.
// Single-kernel forms, which write the final rows themselves (the triplets
// still come from that next kernel):
//   k_route_single   one CTA, at most 2048 routes
//   k_route_cluster  one thread-block cluster of up to 16 CTAs, at most 65536
//                    routes; a hardware cluster barrier and distributed
//                    shared memory replace the grid barrier
//   k_route_fused    one cooperative CTA per chunk with a grid barrier, while
//                    all chunks fit on the GPU at once
// No global atomics decide a position, so the result is deterministic.
#include "common.cuh"
#include "ptx.cuh"

#include <algorithm>
#include <mutex>
#include <cooperative_groups.h>

namespace moe {
namespace {

constexpr uint32_t kFull = 0xffffffffu;
constexpr int kMaxWindows = (kRouteChunkTokensMax * kMaxTopK / kRouteWarps + 31) / 32;   // 16

// Lanes of the warp holding the same value as this lane, for values in
// [-4, 2^nbits): one ballot for the sign and one per bit.  The same mask as
// __match_any_sync for the non-negative values (negative values may share a
// group; callers use the mask only for experts), but built from votes, which
// pipeline across warps, where the match instruction was measured at about
// a hundred cycles a call, one call at a time per SM.
__device__ __forceinline__ uint32_t warp_match(int v, int nbits) {
    const uint32_t neg = __ballot_sync(kFull, v < 0);
    uint32_t m = (v < 0) ? neg : ~neg;
    for (int b = 0; b < nbits; ++b) {
        const bool bit = (v >> b) & 1;
        const uint32_t bb = __ballot_sync(kFull, bit);
        m &= bit ? bb : ~bb;
    }
    return m;
}
__device__ __forceinline__ int expert_bits(int64_t E) { return 32 - __clz((int)E - 1); }

struct ChunkRange {
    int64_t r0, r1;   // route range [r0, r1) (flat index t*K + k)
    int64_t p;        // partition
};

__device__ __forceinline__ ChunkRange chunk_range(const RouteDev &a, int64_t c) {
    ChunkRange cr;
    cr.p = c / a.chunks_per_partition;
    int64_t j = c % a.chunks_per_partition;
    int64_t t0 = cr.p * a.M + j * a.chunk_tokens;
    int64_t t1 = cr.p * a.M + min((j + 1) * a.chunk_tokens, a.M);
    cr.r0 = t0 * a.K;
    cr.r1 = t1 * a.K;
    return cr;
}

__global__ void __launch_bounds__(kRouteThreads)
k_route_local(RouteDev a, int32_t *local_rank) {
    extern __shared__ int32_t hw[];   // [kRouteWarps][E] warp counts, then warp bases
    __shared__ int any_bad;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t c = blockIdx.x;
    for (int64_t i = tid; i < kRouteWarps * a.E; i += blockDim.x) hw[i] = 0;
    if (tid == 0) any_bad = 0;
    pdl_wait();

    const ChunkRange cr = chunk_range(a, c);
    const int64_t n = cr.r1 - cr.r0;
    const int64_t per = ((n + kRouteWarps - 1) / kRouteWarps + 31) / 32 * 32;
    const int64_t w0 = min(cr.r0 + warp * per, cr.r1);
    const int64_t w1 = min(w0 + per, cr.r1);

    // all loads of the slice first (independent, so they are in flight together)
    int e_reg[kMaxWindows];
    int m_reg[kMaxWindows];
    const int32_t K32 = (int32_t)a.K;
    const int nwin = (int)((w1 - w0 + 31) / 32);   // warp-uniform
#pragma unroll
    for (int j = 0; j < kMaxWindows; ++j) {
        if (j >= nwin) break;
        const int64_t i = w0 + 32 * j + lane;
        e_reg[j] = -1;
        m_reg[j] = 1;
        if (i < w1) {
            e_reg[j] = __ldg(a.ids + i);
            if (a.mask_kind == 1) m_reg[j] = __ldg(a.mask + (cr.r0 / K32 + (int32_t)(i - cr.r0) / K32));
            else if (a.mask_kind == 2) m_reg[j] = __ldg(a.mask + i);
        }
    }
    // e_reg: the expert (>= 0), -1 inactive, -2 zero expert, -3 copy expert
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kMaxWindows; ++j) {
        if (j >= nwin) break;
        int e = -1;
        if (w0 + 32 * j + lane < w1 && m_reg[j] != 0) {
            e = route_code(e_reg[j], a);
            if (e == -4) { bad = true; e = -1; }
        }
        e_reg[j] = e;
    }
    __syncthreads();   // hw cleared

    int32_t *mine = hw + warp * a.E;
    const int nbits = expert_bits(a.E);
    int rl[kMaxWindows];
#pragma unroll
    for (int j = 0; j < kMaxWindows; ++j) {
        if (j >= nwin) break;
        rl[j] = -1;
        const int e = e_reg[j];
        const uint32_t grp = warp_match(e, nbits);
        if (e >= 0) rl[j] = mine[e] + __popc(grp & lanemask_lt());
        __syncwarp();
        if (e >= 0 && lane == __ffs(grp) - 1) mine[e] += __popc(grp);
        __syncwarp();
    }
    if (__any_sync(kFull, bad) && lane == 0) any_bad = 1;
    __syncthreads();
    // warp counts -> exclusive warp bases; chunk totals -> hist
    for (int64_t e = tid; e < a.E; e += blockDim.x) {
        int32_t run = 0;
#pragma unroll
        for (int w = 0; w < kRouteWarps; ++w) {
            const int32_t v = hw[w * a.E + e];
            hw[w * a.E + e] = run;
            run += v;
        }
        a.hist[c * a.E + e] = run;
    }
    if (tid == 0) a.bad[c] = any_bad;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kMaxWindows; ++j) {
        if (j >= nwin) break;
        const int64_t i = w0 + 32 * j + lane;
        if (i < w1) local_rank[i] = (e_reg[j] >= 0) ? rl[j] + mine[e_reg[j]] : e_reg[j];
    }
}

// Exclusive scan over a block of exactly 1024 threads; returns the thread's
// exclusive prefix and writes the block total to *total.
__device__ int block_exclusive_scan_1024(int v, int *scratch /*[33]*/, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = scratch[lane];
        int wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(kFull, wi, o);
            if (lane >= o) wi += n;
        }
        scratch[lane] = wi - w;   // exclusive prefix of warp totals
        if (lane == 31) scratch[32] = wi;
    }
    __syncthreads();
    int res = scratch[warp] + incl - v;
    *total = scratch[32];
    __syncthreads();
    return res;
}

__device__ long long block_exclusive_scan64_1024(long long v, long long *scratch, long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        long long n = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) scratch[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        long long w = scratch[lane];
        long long wi = w;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            long long n = __shfl_up_sync(kFull, wi, o);
            if (lane >= o) wi += n;
        }
        scratch[lane] = wi - w;
        if (lane == 31) scratch[32] = wi;
    }
    __syncthreads();
    const long long res = scratch[warp] + incl - v;
    *total = scratch[32];
    return res;
}

constexpr int kScanRegs = 32;   // chunk counts a scan thread keeps in registers

__global__ void __launch_bounds__(1024)
k_route_scan(RouteDev a, int64_t chunks, int64_t *counts, int32_t *offsets, int32_t *recv_cum,
             int32_t *sched) {
    __shared__ long long scratch64[33];
    __shared__ int tot_s[kMaxExperts];
    __shared__ int off_s[kMaxExperts];
    __shared__ int part_s[1024];
    pdl_wait();
    // tpe threads per expert; thread (e, j) owns the contiguous chunk range j.
    // Experts vary fastest across threads, so every load and store of a
    // chunk's histogram row is coalesced.
    int tpe = 1;
    while (tpe * 2 * a.E <= 1024 && tpe < 32) tpe *= 2;
    const int tid = threadIdx.x;
    const bool on = tid < tpe * a.E;
    const int e = on ? tid % (int)a.E : 0, j = on ? tid / (int)a.E : 0;
    const int64_t per = (chunks + tpe - 1) / tpe;
    const int64_t c0 = min((int64_t)j * per, chunks), c1 = on ? min(c0 + per, chunks) : c0;
    int vals[kScanRegs];
    int part = 0;
#pragma unroll
    for (int u = 0; u < kScanRegs; ++u) {
        vals[u] = (c0 + u < c1) ? a.hist[(c0 + u) * a.E + e] : 0;
        part += vals[u];
    }
    for (int64_t c = c0 + kScanRegs; c < c1; ++c) part += a.hist[c * a.E + e];   // long ranges
    part_s[tid] = part;
    __syncthreads();
    int excl = 0, total_e = 0;
    if (on) {
        for (int jj = 0; jj < tpe; ++jj) {
            const int v = part_s[jj * a.E + e];
            if (jj < j) excl += v;
            total_e += v;
        }
        if (j == 0) tot_s[e] = total_e;
    }
    __syncthreads();
    const int tv = (tid < a.E) ? tot_s[tid] : 0;
    // offsets (low half) and m-block starts (high half) in one 64-bit scan;
    // both sums stay below 2^31, so the halves never carry into each other
    const long long packed = (long long)tv | ((long long)((tv + kGemmBM - 1) / kGemmBM) << 32);
    long long ptotal;
    const long long pscan = block_exclusive_scan64_1024(packed, scratch64, &ptotal);
    const int total = (int)(ptotal & 0xffffffffll), mtotal = (int)(ptotal >> 32);
    if (tid < a.E) {
        off_s[tid] = (int)(pscan & 0xffffffffll);
        counts[tid] = tv;
        offsets[tid] = (int)(pscan & 0xffffffffll);
        if (sched) sched[tid] = (int)(pscan >> 32);
    }
    __syncthreads();
    if (on) {
        int run = off_s[e] + excl;
        // partition of chunk c0 and position inside it, then advanced by one per chunk
        const int cpp = (int)a.chunks_per_partition;
        int p = (int)(c0 / cpp), q = (int)(c0 - (int64_t)p * cpp);
        int32_t *rc = recv_cum + (int64_t)e * a.P;
        int32_t *h = a.hist + e;
        const int n = (int)(c1 - c0);
#pragma unroll
        for (int u = 0; u < kScanRegs; ++u) {
            if (u < n) {
                h[(c0 + u) * a.E] = run;
                run += vals[u];
                if (++q == cpp) { rc[p] = run; ++p; q = 0; }
            }
        }
        for (int u = kScanRegs; u < n; ++u) {
            const int v = h[(c0 + u) * a.E];
            h[(c0 + u) * a.E] = run;
            run += v;
            if (++q == cpp) { rc[p] = run; ++p; q = 0; }
        }
    }
    // status word of this call: invalid ids seen by any chunk
    int bad = 0;
    for (int64_t c = tid; c < chunks; c += blockDim.x) bad |= a.bad[c];
    bad = __syncthreads_or(bad);
    if (tid == 0) {
        offsets[a.E] = total;
        if (sched) sched[a.E] = mtotal;
        *a.status = bad ? MOE_DEV_BAD_EXPERT_ID : 0;
    }
}

// ---------------------------------------------------------------- single-kernel routing
// One CTA per chunk, launched cooperatively (all CTAs resident).  Phase 1 is
// k_route_local's count and rank, keeping each route's rank in registers.
// After a grid-wide barrier every CTA reads all chunk histograms and computes
// the per-expert totals, their exclusive scan (offsets) and its own chunk's
// bases, then writes the final row and triplet of each of its routes.  CTA 0
// also writes counts, offsets, recv_cum, the GEMM schedule and the status.
constexpr int kFusedLoads = 32;   // chunk counts loaded at once per expert

__global__ void __launch_bounds__(kRouteThreads)
k_route_fused(RouteDev a, int64_t chunks, int64_t *counts, int32_t *offsets, int32_t *recv_cum,
              int32_t *sched, int32_t *route_row) {
    extern __shared__ int32_t hw[];   // [kRouteWarps][E]; reused after the barrier
    __shared__ int any_bad;
    __shared__ long long scratch64[kRouteWarps + 1];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t c = blockIdx.x;
    for (int64_t i = tid; i < kRouteWarps * a.E; i += blockDim.x) hw[i] = 0;
    if (tid == 0) any_bad = 0;
    pdl_wait();

    // ---------------- phase 1: count and rank inside the chunk
    const ChunkRange cr = chunk_range(a, c);
    const int64_t n = cr.r1 - cr.r0;
    const int64_t per = ((n + kRouteWarps - 1) / kRouteWarps + 31) / 32 * 32;
    const int64_t w0 = min(cr.r0 + warp * per, cr.r1);
    const int64_t w1 = min(w0 + per, cr.r1);
    const int nwin = (int)((w1 - w0 + 31) / 32);
    const int32_t K32 = (int32_t)a.K;
    int e_reg[kMaxWindows];
    int m_reg[kMaxWindows];
#pragma unroll
    for (int j = 0; j < kMaxWindows; ++j) {
        if (j >= nwin) break;
        const int64_t i = w0 + 32 * j + lane;
        e_reg[j] = -1;
        m_reg[j] = 1;
        if (i < w1) {
            e_reg[j] = __ldg(a.ids + i);
            if (a.mask_kind == 1) m_reg[j] = __ldg(a.mask + (cr.r0 / K32 + (int32_t)(i - cr.r0) / K32));
            else if (a.mask_kind == 2) m_reg[j] = __ldg(a.mask + i);
        }
    }
    // e_reg: the expert (>= 0), -1 inactive, -2 zero expert, -3 copy expert
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kMaxWindows; ++j) {
        if (j >= nwin) break;
        int e = -1;
        if (w0 + 32 * j + lane < w1 && m_reg[j] != 0) {
            e = route_code(e_reg[j], a);
            if (e == -4) { bad = true; e = -1; }
        }
        e_reg[j] = e;
    }
    __syncthreads();
    int32_t *mine = hw + warp * a.E;
    const int nbits = expert_bits(a.E);
    int rl[kMaxWindows];
#pragma unroll
    for (int j = 0; j < kMaxWindows; ++j) {
        if (j >= nwin) break;
        rl[j] = -1;
        const int e = e_reg[j];
        const uint32_t grp = warp_match(e, nbits);
        if (e >= 0) rl[j] = mine[e] + __popc(grp & lanemask_lt());
        __syncwarp();
        if (e >= 0 && lane == __ffs(grp) - 1) mine[e] += __popc(grp);
        __syncwarp();
    }
    if (__any_sync(kFull, bad) && lane == 0) any_bad = 1;
    __syncthreads();
    for (int64_t e = tid; e < a.E; e += blockDim.x) {
        int32_t run = 0;
#pragma unroll
        for (int w = 0; w < kRouteWarps; ++w) {
            const int32_t v = hw[w * a.E + e];
            hw[w * a.E + e] = run;
            run += v;
        }
        a.hist[c * a.E + e] = run;
    }
    if (tid == 0) a.bad[c] = any_bad;
    __syncthreads();
#pragma unroll
    for (int j = 0; j < kMaxWindows; ++j) {
        if (j >= nwin) break;
        if (e_reg[j] >= 0) rl[j] += mine[e_reg[j]];   // rank inside the chunk
    }
    __threadfence();
    cooperative_groups::this_grid().sync();

    // ---------------- phase 2: totals, offsets, this chunk's bases
    int32_t *tot_s = hw;                 // [E]
    int32_t *below_s = hw + a.E;         // [E], later the chunk bases
    const bool lead = blockIdx.x == 0;
    const int cpp = (int)a.chunks_per_partition;
    int32_t *own_s = hw + 2 * a.E;       // [E] this chunk's own counts
    for (int64_t e = tid; e < a.E; e += blockDim.x) {
        int tot = 0, below = 0, own = 0;
        for (int64_t cb = 0; cb < chunks; cb += kFusedLoads) {
            int v[kFusedLoads];
#pragma unroll
            for (int u = 0; u < kFusedLoads; ++u)
                v[u] = (cb + u < chunks) ? a.hist[(cb + u) * a.E + e] : 0;
#pragma unroll
            for (int u = 0; u < kFusedLoads; ++u) {
                tot += v[u];
                if (cb + u < c) below += v[u];
                if (cb + u == c) own = v[u];
            }
        }
        tot_s[e] = tot;
        below_s[e] = below;
        own_s[e] = own;
    }
    __syncthreads();
    // exclusive scan over experts of (total, m-blocks), packed in 64 bits
    const int per_t = (int)((a.E + blockDim.x - 1) / blockDim.x);
    const int64_t e0 = (int64_t)tid * per_t, e1 = min(e0 + per_t, a.E);
    long long local = 0;
    for (int64_t e = e0; e < e1; ++e)
        local += (long long)tot_s[e] | ((long long)((tot_s[e] + kGemmBM - 1) / kGemmBM) << 32);
    long long incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long v = __shfl_up_sync(kFull, incl, o);
        if (lane >= o) incl += v;
    }
    if (lane == 31) scratch64[warp] = incl;
    __syncthreads();
    if (tid == 0) {
        long long run = 0;
        for (int w = 0; w < kRouteWarps; ++w) {
            const long long v = scratch64[w];
            scratch64[w] = run;
            run += v;
        }
        scratch64[kRouteWarps] = run;
    }
    __syncthreads();
    long long ex = scratch64[warp] + incl - local;
    int bad_all = 0;
    if (lead)
        for (int64_t cc = tid; cc < chunks; cc += blockDim.x) bad_all |= a.bad[cc];
    // the last chunk of a partition writes that partition's receive counts:
    // its own base plus its own count is the running sum through the partition
    const bool part_end = (c + 1) % cpp == 0;
    const int64_t pc = c / cpp;
    for (int64_t e = e0; e < e1; ++e) {
        const int off = (int)(ex & 0xffffffffll);
        const int tv = tot_s[e];
        below_s[e] += off;   // this chunk's base of expert e
        if (part_end) recv_cum[e * a.P + pc] = below_s[e] + own_s[e];
        if (lead) {
            counts[e] = tv;
            offsets[e] = off;
            if (sched) sched[e] = (int)(ex >> 32);
        }
        ex += (long long)tv | ((long long)((tv + kGemmBM - 1) / kGemmBM) << 32);
    }
    bad_all = __syncthreads_or(bad_all);
    if (lead && tid == 0) {
        const long long tot_all = scratch64[kRouteWarps];
        offsets[a.E] = (int)(tot_all & 0xffffffffll);
        if (sched) sched[a.E] = (int)(tot_all >> 32);
        *a.status = bad_all ? MOE_DEV_BAD_EXPERT_ID : 0;
    }
    // ---------------- final rows of this chunk's routes
#pragma unroll
    for (int j = 0; j < kMaxWindows; ++j) {
        if (j >= nwin) break;
        const int64_t i = w0 + 32 * j + lane;
        if (i >= w1) continue;
        // -1 inactive, -2 / -3 special expert; triplets are written by the next kernel
        route_row[i] = (e_reg[j] >= 0) ? below_s[e_reg[j]] + rl[j] : e_reg[j];
    }
}

// ---------------------------------------------------------------- one-CTA routing
// Tiny batches (at most kSingleMaxRoutes routes): one CTA of 32 warps does
// everything, so no grid barrier and no global round trip between the count
// and the final rows.  Larger batches go to the per-chunk kernels: ranking
// is issue-bound (two warp matches per 32 routes), and one SM ranking 16384
// routes was measured 4x slower than 32 CTAs with a grid barrier.  Each warp takes a contiguous slice of the route array
// (route order is row order within an expert), ranks it with warp_match
// as in k_route_local, and also counts its routes per (partition, expert) for
// the receive counts.  Per-warp counts are scanned across warps (stable
// ranks), their totals across experts (offsets, m-block starts), and the
// partition counts across partitions (recv_cum).
constexpr int kSingleThreads = 1024;
constexpr int kSingleWarps = kSingleThreads / 32;
constexpr int kSingleWindows = 2;   // 32-route windows per warp
constexpr int64_t kSingleMaxRoutes = (int64_t)kSingleWarps * kSingleWindows * 32;   // 2048
constexpr size_t kSingleSmemMax = 200 * 1024;

size_t route_single_smem(int64_t E, int64_t P) {
    return (size_t)(kSingleWarps + P + 1) * (size_t)E * sizeof(int32_t);
}

__global__ void __launch_bounds__(kSingleThreads)
k_route_single(RouteDev a, int64_t *counts, int32_t *offsets, int32_t *recv_cum, int32_t *sched,
               int32_t *route_row) {
    extern __shared__ int32_t sm[];
    __shared__ long long scratch64[33];
    const int E = (int)a.E, P = (int)a.P;
    int32_t *hw = sm;                       // [32][E] warp counts, then warp bases
    int32_t *hp = sm + kSingleWarps * E;    // [P][E] routes per (partition, expert)
    int32_t *off_s = hp + P * E;            // [E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < (kSingleWarps + P) * E; i += kSingleThreads) sm[i] = 0;
    pdl_wait();

    // T * K <= kSingleMaxRoutes, so every index below fits in 32 bits
    const int n = (int)(a.T * a.K), K32 = (int)a.K, M32 = (int)a.M;
    const int per = ((n + kSingleWarps - 1) / kSingleWarps + 31) / 32 * 32;
    const int w0 = min(warp * per, n), w1 = min(w0 + per, n);
    const int nwin = (w1 - w0 + 31) / 32;   // warp-uniform, <= kSingleWindows
    int e_reg[kSingleWindows];
    int m_reg[kSingleWindows];
#pragma unroll
    for (int j = 0; j < kSingleWindows; ++j) {
        if (j >= nwin) break;
        const int i = w0 + 32 * j + lane;
        e_reg[j] = -1;
        m_reg[j] = 1;
        if (i < w1) {
            e_reg[j] = __ldg(a.ids + i);
            if (a.mask_kind == 1) m_reg[j] = __ldg(a.mask + i / K32);
            else if (a.mask_kind == 2) m_reg[j] = __ldg(a.mask + i);
        }
    }
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kSingleWindows; ++j) {
        if (j >= nwin) break;
        int e = -1;
        if (w0 + 32 * j + lane < w1 && m_reg[j] != 0) {
            e = route_code(e_reg[j], a);
            if (e == -4) { bad = true; e = -1; }
        }
        e_reg[j] = e;
    }
    __syncthreads();   // counters cleared

    int32_t *mine = hw + warp * E;
    const int nbits = expert_bits(a.E);
    int rl[kSingleWindows];
#pragma unroll
    for (int j = 0; j < kSingleWindows; ++j) {
        if (j >= nwin) break;
        const int i = w0 + 32 * j + lane;
        const int e = e_reg[j];
        const int p = (e >= 0) ? (i / K32) / M32 : 0;
        const uint32_t grp = warp_match(e, nbits);
        rl[j] = (e >= 0) ? mine[e] + __popc(grp & lanemask_lt()) : -1;
        __syncwarp();
        if (e >= 0 && lane == __ffs(grp) - 1) mine[e] += __popc(grp);
        // partition counts (shared by all warps, hence atomic): one add per
        // expert group when the window lies in one partition, else one per route
        const int i_last = min(w0 + 32 * j + 31, w1 - 1);
        if ((w0 + 32 * j) / K32 / M32 == i_last / K32 / M32) {
            if (e >= 0 && lane == __ffs(grp) - 1) atomicAdd(&hp[p * E + e], (int)__popc(grp));
        } else if (e >= 0) {
            atomicAdd(&hp[p * E + e], 1);
        }
        __syncwarp();
    }
    __syncthreads();

    // per expert: warp counts -> exclusive warp bases, partition counts ->
    // inclusive running sums, and the total
    int tv = 0;
    if (tid < E) {
        int run = 0;
#pragma unroll 8
        for (int w = 0; w < kSingleWarps; ++w) {
            const int v = hw[w * E + tid];
            hw[w * E + tid] = run;
            run += v;
        }
        tv = run;
        int pr = 0;
        for (int p = 0; p < P; ++p) {
            pr += hp[p * E + tid];
            hp[p * E + tid] = pr;
        }
    }
    // offsets (low half) and m-block starts (high half) in one 64-bit scan
    const long long packed = (long long)tv | ((long long)((tv + kGemmBM - 1) / kGemmBM) << 32);
    long long ptotal;
    const long long pscan = block_exclusive_scan64_1024(packed, scratch64, &ptotal);
    if (tid < E) {
        const int off = (int)(pscan & 0xffffffffll);
        off_s[tid] = off;
        counts[tid] = tv;
        offsets[tid] = off;
        if (sched) sched[tid] = (int)(pscan >> 32);
    }
    const int bad_all = __syncthreads_or(bad);   // also publishes off_s and hp
    if (tid == 0) {
        offsets[E] = (int)(ptotal & 0xffffffffll);
        if (sched) sched[E] = (int)(ptotal >> 32);
        *a.status = bad_all ? MOE_DEV_BAD_EXPERT_ID : 0;
    }
    // receive counts, coalesced: entry (e, p) at e * P + p
    for (int q = tid; q < E * P; q += kSingleThreads) {
        const int e = q / P, p = q - e * P;
        recv_cum[q] = off_s[e] + hp[p * E + e];
    }
    // final rows
#pragma unroll
    for (int j = 0; j < kSingleWindows; ++j) {
        if (j >= nwin) break;
        const int i = w0 + 32 * j + lane;
        if (i >= w1) continue;
        // -1 inactive, -2 / -3 special expert; triplets are written by the next kernel
        route_row[i] = (e_reg[j] >= 0) ? off_s[e_reg[j]] + mine[e_reg[j]] + rl[j] : e_reg[j];
    }
}

// ---------------------------------------------------------------- one-cluster routing
// Mid-size batches: one thread-block cluster of up to 16 CTAs.  CTA j of the
// cluster takes the j-th contiguous range of the route array and counts and
// ranks it as k_route_single does (per warp, warp_match), keeping its
// per-(partition, expert) counts in shared memory.  Each CTA stores its
// per-expert totals into every CTA's shared memory (distributed shared
// memory stores, which complete under the barrier's release), and one
// hardware cluster barrier replaces the grid barrier and the global round
// trip of the histograms.  Every CTA then scans the totals over experts
// itself and writes the final rows of its range and the receive counts of
// the partitions that end inside it.
constexpr int kClThreads = 1024;
constexpr int kClWarps = kClThreads / 32;
constexpr int kClWindows = 4;      // 32-route windows per warp
constexpr int kClMaxParts = 8;     // partitions one CTA's range may touch
constexpr int kClMaxCtas = 16;
constexpr int64_t kClMaxRoutesPerCta = (int64_t)kClWarps * kClWindows * 32;   // 4096

size_t route_cluster_smem(int64_t E, int64_t C) {
    return (size_t)(kClWarps + kClMaxParts + 1 + C) * (size_t)E * sizeof(int32_t);
}

// Store v at the address of `local` in the shared memory of CTA `rank`.
__device__ __forceinline__ void st_peer_s32(int32_t *local, uint32_t rank, int v) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_u32(local)), "r"(rank));
    asm volatile("st.shared::cluster.s32 [%0], %1;" ::"r"(remote), "r"(v) : "memory");
}

__global__ void __launch_bounds__(kClThreads)
k_route_cluster(RouteDev a, int64_t per_cta, int64_t *counts, int32_t *offsets, int32_t *recv_cum,
                int32_t *sched, int32_t *route_row) {
    extern __shared__ int32_t sm[];
    __shared__ long long scratch64[33];
    __shared__ int32_t bad_s[kClMaxCtas];   // each CTA's invalid-id flag
    const int E = (int)a.E, P = (int)a.P;
    const int C = (int)gridDim.x;           // the grid is one cluster
    int32_t *hw = sm;                       // [32][E] warp counts, then warp bases
    int32_t *hp = hw + kClWarps * E;        // [kClMaxParts][E] per (partition in range, expert)
    int32_t *base_s = hp + kClMaxParts * E; // [E] this CTA's base of each expert
    int32_t *all_tot = base_s + E;          // [C][E] every CTA's totals, stored by that CTA
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_ctarank();
    // this CTA has started: peers may store into its shared memory once every
    // CTA has arrived here (the wait comes just before the first such store)
    cluster_arrive();
    for (int i = tid; i < (kClWarps + kClMaxParts) * E; i += kClThreads) sm[i] = 0;

    // The ids and the mask are inputs, which no kernel of this library writes,
    // so they are loaded before waiting on the previous kernel of the stream;
    // everything this kernel writes is written after the wait.
    // T * K <= kClMaxCtas * kClMaxRoutesPerCta, so indices fit in 32 bits
    const int n = (int)(a.T * a.K), K32 = (int)a.K, M32 = (int)a.M, MK = M32 * K32;
    const int r0 = min((int)(rank * per_cta), n), r1 = min(r0 + (int)per_cta, n);
    const int pfirst = (r0 < r1) ? r0 / MK : 0;
    const int per = ((r1 - r0 + kClWarps - 1) / kClWarps + 31) / 32 * 32;
    const int w0 = min(r0 + warp * per, r1), w1 = min(w0 + per, r1);
    const int nwin = (w1 - w0 + 31) / 32;   // warp-uniform, <= kClWindows
    int e_reg[kClWindows];
    int m_reg[kClWindows];
#pragma unroll
    for (int j = 0; j < kClWindows; ++j) {
        if (j >= nwin) break;
        const int i = w0 + 32 * j + lane;
        e_reg[j] = -1;
        m_reg[j] = 1;
        if (i < w1) {
            e_reg[j] = __ldg(a.ids + i);
            if (a.mask_kind == 1) m_reg[j] = __ldg(a.mask + i / K32);
            else if (a.mask_kind == 2) m_reg[j] = __ldg(a.mask + i);
        }
    }
    pdl_wait();
    bool bad = false;
#pragma unroll
    for (int j = 0; j < kClWindows; ++j) {
        if (j >= nwin) break;
        int e = -1;
        if (w0 + 32 * j + lane < w1 && m_reg[j] != 0) {
            e = route_code(e_reg[j], a);
            if (e == -4) { bad = true; e = -1; }
        }
        e_reg[j] = e;
    }
    __syncthreads();   // counters cleared

    int32_t *mine = hw + warp * E;
    const int nbits = expert_bits(a.E);
    int rl[kClWindows];
#pragma unroll
    for (int j = 0; j < kClWindows; ++j) {
        if (j >= nwin) break;
        const int i = w0 + 32 * j + lane;
        const int e = e_reg[j];
        const uint32_t grp = warp_match(e, nbits);
        rl[j] = (e >= 0) ? mine[e] + __popc(grp & lanemask_lt()) : -1;
        __syncwarp();
        if (e >= 0 && lane == __ffs(grp) - 1) mine[e] += __popc(grp);
        // partition counts (shared by all warps, hence atomic): one add per
        // expert group when the window lies in one partition (the common
        // case), else one per route
        const int pw0 = (w0 + 32 * j) / MK, pw1 = min(w0 + 32 * j + 31, w1 - 1) / MK;
        if (pw0 == pw1) {
            if (e >= 0 && lane == __ffs(grp) - 1) atomicAdd(&hp[(pw0 - pfirst) * E + e], (int)__popc(grp));
        } else if (e >= 0) {
            atomicAdd(&hp[(i / MK - pfirst) * E + e], 1);
        }
        __syncwarp();
    }
    const int bad_cta = __syncthreads_or(bad);
    cluster_wait();   // every CTA of the cluster has started
    // per expert: warp counts -> exclusive warp bases, partition counts ->
    // inclusive running sums within the range, and the CTA total
    if (tid < E) {
        int run = 0;
#pragma unroll 8
        for (int w = 0; w < kClWarps; ++w) {
            const int v = hw[w * E + tid];
            hw[w * E + tid] = run;
            run += v;
        }
        for (int j = 0; j < C; ++j) st_peer_s32(all_tot + rank * E + tid, (uint32_t)j, run);
        int pr = 0;
        for (int q = 0; q < kClMaxParts; ++q) {
            pr += hp[q * E + tid];
            hp[q * E + tid] = pr;
        }
    }
    if (tid < C) st_peer_s32(bad_s + rank, (uint32_t)tid, bad_cta);
    cluster_sync();   // every CTA's stores into this CTA have completed and are visible

    // totals over the cluster and this CTA's share below it
    int tv = 0, below = 0;
    if (tid < E) {
        for (int j = 0; j < C; ++j) {
            const int v = all_tot[j * E + tid];
            tv += v;
            if (j < (int)rank) below += v;
        }
    }
    int bad_all = (rank == 0 && tid < C) ? bad_s[tid] : 0;
    const long long packed = (long long)tv | ((long long)((tv + kGemmBM - 1) / kGemmBM) << 32);
    long long ptotal;
    const long long pscan = block_exclusive_scan64_1024(packed, scratch64, &ptotal);
    if (tid < E) {
        const int off = (int)(pscan & 0xffffffffll);
        base_s[tid] = off + below;
        if (rank == 0) {
            counts[tid] = tv;
            offsets[tid] = off;
            if (sched) sched[tid] = (int)(pscan >> 32);
        }
    }
    bad_all = __syncthreads_or(bad_all);   // also publishes base_s
    if (rank == 0 && tid == 0) {
        offsets[E] = (int)(ptotal & 0xffffffffll);
        if (sched) sched[E] = (int)(ptotal >> 32);
        *a.status = bad_all ? MOE_DEV_BAD_EXPERT_ID : 0;
    }
    // receive counts of the partitions whose last route lies in this range
    if (r0 < r1) {
        const int plast = (r1 - 1) / MK;
        for (int q = 0; q <= plast - pfirst; ++q) {
            const int p = pfirst + q;
            const int pend = (p + 1) * MK - 1;
            if (pend < r0 || pend >= r1) continue;
            for (int e = tid; e < E; e += kClThreads)
                recv_cum[(int64_t)e * P + p] = base_s[e] + hp[q * E + e];
        }
    }
    // final rows
#pragma unroll
    for (int j = 0; j < kClWindows; ++j) {
        if (j >= nwin) break;
        const int i = w0 + 32 * j + lane;
        if (i >= w1) continue;
        // -1 inactive, -2 / -3 special expert; triplets are written by the next kernel
        route_row[i] = (e_reg[j] >= 0) ? base_s[e_reg[j]] + mine[e_reg[j]] + rl[j] : e_reg[j];
    }
}

__global__ void k_route_resolve(RouteDev a, int32_t *route_row, int32_t *assist) {
    pdl_wait();
    const int64_t n = a.T * a.K;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x)
        resolve_route_row(a, i / a.K, (int)(i % a.K), route_row, assist);
}

// m-block schedule from offsets alone (for moe_grouped_ffn, which gets only
// the offsets from its caller).  It also starts the call's status word at 0.
__global__ void __launch_bounds__(1024)
k_sched(const int32_t *offsets, int64_t E, int32_t *sched, int32_t *status) {
    __shared__ int scratch[33];
    pdl_wait();
    const int e = threadIdx.x;
    int mb = 0;
    if (e < E) mb = max(0, offsets[e + 1] - offsets[e] + kGemmBM - 1) / kGemmBM;
    int total;
    int start = block_exclusive_scan_1024(e < E ? mb : 0, scratch, &total);
    if (e < E) sched[e] = start;
    if (e == 0) {
        sched[E] = total;
        *status = 0;
    }
}

}  // namespace

moe_status launch_route(const RouteDev &r, int64_t chunks, int64_t *counts, int32_t *offsets,
                        int32_t *recv_cum, int32_t *sched, int32_t *route_row,
                        cudaStream_t stream) {
    const size_t smem = (size_t)kRouteWarps * r.E * sizeof(int32_t);
    if (chunks > 0) {
        MOE_LAUNCH("route_local", k_route_local, (unsigned)chunks, kRouteThreads, smem, stream, r,
                   route_row);
    }
    MOE_LAUNCH("route_scan", k_route_scan, 1, 1024, 0, stream, r, chunks, counts, offsets,
               recv_cum, sched);
    return MOE_OK;
}

// Whether a cluster of C CTAs of k_route_cluster with `smem` bytes each can be
// scheduled (16 CTAs need the non-portable cluster size).  The answers are
// cached per (C, smem): the occupancy query is a driver call.
bool cluster_fits_query(int64_t C, size_t smem);
bool cluster_fits(int64_t C, size_t smem) {
    struct Entry { int64_t C; size_t smem; bool ok; };
    static std::mutex mu;
    static Entry cache[8];
    static int used = 0, next = 0;
    std::lock_guard<std::mutex> lock(mu);
    for (int i = 0; i < used; ++i)
        if (cache[i].C == C && cache[i].smem == smem) return cache[i].ok;
    const bool ok = cluster_fits_query(C, smem);
    cache[next] = Entry{C, smem, ok};
    next = (next + 1) % 8;
    if (used < 8) ++used;
    return ok;
}
bool cluster_fits_query(int64_t C, size_t smem) {
    static size_t configured = 0;
    if (smem > configured) {
        if (cudaFuncSetAttribute(k_route_cluster, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)smem) != cudaSuccess ||
            cudaFuncSetAttribute(k_route_cluster, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                 1) != cudaSuccess) {
            cudaGetLastError();
            return false;
        }
        configured = smem;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)C);
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = smem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int clusters = 0;
    if (cudaOccupancyMaxActiveClusters(&clusters, k_route_cluster, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return clusters >= 1;
}

moe_status launch_route_fused(RouteDev &r, int64_t chunks, int64_t *counts, int32_t *offsets,
                              int32_t *recv_cum, int32_t *sched, int32_t *route_row,
                              cudaStream_t stream) {
    const size_t ssm = route_single_smem(r.E, r.P);
    if (r.T * r.K <= kSingleMaxRoutes && ssm <= kSingleSmemMax) {
        if (!set_smem_limit((const void *)k_route_single, ssm)) return MOE_ERR_CUDA;
        r.rows_final = 1;
        MOE_LAUNCH("route_single", k_route_single, 1, kSingleThreads, ssm, stream, r, counts,
                   offsets, recv_cum, sched, route_row);
        return MOE_OK;
    }
    // one cluster: ranges of at most 4096 routes, each touching at most
    // kClMaxParts partitions
    const int64_t n = r.T * r.K;
    if (n <= (int64_t)kClMaxCtas * kClMaxRoutesPerCta) {
        const int64_t C = std::min<int64_t>(kClMaxCtas, std::max<int64_t>(2, (n + 1023) / 1024));
        const int64_t per_cta = ((n + C - 1) / C + 31) / 32 * 32;
        const int64_t parts = per_cta / (r.M * r.K) + 2;
        const size_t csm = route_cluster_smem(r.E, C);
        if (per_cta <= kClMaxRoutesPerCta && parts <= kClMaxParts && csm <= kSingleSmemMax &&
            cluster_fits(C, csm)) {
            r.rows_final = 1;
            MOE_LAUNCH_CLUSTER("route_cluster", k_route_cluster, (unsigned)C, kClThreads, csm, stream,
                               (unsigned)C, r, per_cta, counts, offsets, recv_cum, sched, route_row);
            return MOE_OK;
        }
    }
    const size_t smem = (size_t)kRouteWarps * r.E * sizeof(int32_t);
    int per_sm = 0;
    if (chunks > 0 &&
        cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, k_route_fused, kRouteThreads, smem) ==
            cudaSuccess &&
        chunks <= (int64_t)per_sm * num_sms()) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)chunks);
        cfg.blockDim = dim3(kRouteThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = stream;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeCooperative;
        attr[0].val.cooperative = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        r.rows_final = 1;
        const int tok = launch_begin("route_fused", stream, (unsigned)chunks);
        cudaError_t err = cudaLaunchKernelEx(&cfg, k_route_fused, r, chunks, counts, offsets,
                                             recv_cum, sched, route_row);
        if (err == cudaSuccess) err = cudaGetLastError();
        launch_end(tok, stream);
        if (err == cudaSuccess) return MOE_OK;
        return MOE_ERR_CUDA;
    }
    cudaGetLastError();
    r.rows_final = 0;
    return launch_route(r, chunks, counts, offsets, recv_cum, sched, route_row, stream);
}

moe_status launch_route_resolve(const RouteDev &r, int32_t *route_row, int32_t *assist,
                                cudaStream_t stream) {
    const int64_t n = r.T * r.K;
    if (n == 0) return MOE_OK;
    int64_t blocks = (n + 255) / 256;
    const int64_t cap = (int64_t)num_sms() * 8;
    if (blocks > cap) blocks = cap;
    MOE_LAUNCH("route_resolve", k_route_resolve, (unsigned)blocks, 256, 0, stream, r, route_row,
               assist);
    return MOE_OK;
}

moe_status launch_sched(const int32_t *offsets, int64_t E, int32_t *sched, int32_t *status,
                        cudaStream_t stream) {
    MOE_LAUNCH("sched", k_sched, 1, 1024, 0, stream, offsets, E, sched, status);
    return MOE_OK;
}

}  // namespace moe
