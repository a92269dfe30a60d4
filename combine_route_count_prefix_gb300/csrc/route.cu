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
//   route_row[t*K + k]  row of route (t, k) (expandedRowIdx), -1 if inactive
//   assist[row]         (partition, token in partition, slot)
// Row order is expert, then partition, then token, then slot.  Within one
// expert this is the route order, so a route's row is offsets[e] plus the
// number of earlier active routes with the same expert: the "token_repeat_num"
// of the send loop, computed here as a stable counting sort.
//
// GB300 design (not the pages' O((BS*K)^2) per-route count): three small
// kernels.  Routes are cut into chunks of at most 256 tokens that never cross a
// partition boundary.
//   k_route_count  one CTA per chunk; each warp counts a contiguous slice of
//                  the chunk with __match_any_sync (one shared-memory add per
//                  distinct expert per 32 routes) -> hist[chunk][e]
//   k_route_scan   one CTA: totals, exclusive scan over experts, per-chunk
//                  bases (scan over chunks for each expert), recv_cum, and the
//                  GEMM m-block schedule
//   k_route_rank   one CTA per chunk; recounts per warp, turns the counts into
//                  per-warp bases and walks the slice again in order, giving
//                  each route base + (same-expert lanes below it) and bumping
//                  the base by the group size.
// No global atomics decide a position, so the result is deterministic.
#include "common.cuh"

namespace moe {
namespace {

constexpr uint32_t kFull = 0xffffffffu;

struct ChunkRange {
    int64_t r0, r1;   // route range [r0, r1) (flat index t*K + k)
    int64_t p;        // partition
};

__device__ __forceinline__ ChunkRange chunk_range(const RouteDev &a, int64_t c) {
    ChunkRange cr;
    cr.p = c / a.chunks_per_partition;
    int64_t j = c % a.chunks_per_partition;
    int64_t t0 = cr.p * a.M + j * kRouteChunkTokens;
    int64_t t1 = cr.p * a.M + min((j + 1) * (int64_t)kRouteChunkTokens, a.M);
    cr.r0 = t0 * a.K;
    cr.r1 = t1 * a.K;
    return cr;
}

// Expert of route i, -1 if masked off, -2 if active but the id is not an expert.
__device__ __forceinline__ int route_expert(const RouteDev &a, int64_t i) {
    if (a.mask_kind == 1 && a.mask[i / a.K] == 0) return -1;
    if (a.mask_kind == 2 && a.mask[i] == 0) return -1;
    int e = a.ids[i];
    if (e < 0 || e >= a.E) return -2;
    return e;
}

__device__ __forceinline__ void warp_slice(const ChunkRange &cr, int warp, int64_t &w0, int64_t &w1) {
    int64_t n = cr.r1 - cr.r0;
    int64_t per = ((n + kRouteWarps - 1) / kRouteWarps + 31) / 32 * 32;
    w0 = min(cr.r0 + warp * per, cr.r1);
    w1 = min(w0 + per, cr.r1);
}

// Per-warp histogram of the warp's slice into sh[warp*E + e].  Returns whether
// the warp saw an invalid expert id.
__device__ __forceinline__ bool warp_count(const RouteDev &a, int64_t w0, int64_t w1, int32_t *row,
                                           int lane) {
    bool bad = false;
    for (int64_t base = w0; base < w1; base += 32) {
        int64_t i = base + lane;
        int e = (i < w1) ? route_expert(a, i) : -1;
        if (e == -2) { bad = true; e = -1; }
        uint32_t grp = __match_any_sync(kFull, e);
        if (e >= 0 && lane == __ffs(grp) - 1) row[e] += __popc(grp);
        __syncwarp();
    }
    return bad;
}

__global__ void __launch_bounds__(kRouteThreads)
k_route_count(RouteDev a) {
    extern __shared__ int32_t sh[];   // [kRouteWarps][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t c = blockIdx.x;
    for (int64_t i = tid; i < kRouteWarps * a.E; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    ChunkRange cr = chunk_range(a, c);
    int64_t w0, w1;
    warp_slice(cr, warp, w0, w1);
    bool bad = warp_count(a, w0, w1, sh + warp * a.E, lane);
    __shared__ int any_bad;
    if (tid == 0) any_bad = 0;
    __syncthreads();
    if (__any_sync(kFull, bad) && lane == 0) any_bad = 1;
    __syncthreads();
    if (tid == 0) a.bad[c] = any_bad;
    for (int64_t e = tid; e < a.E; e += blockDim.x) {
        int32_t s = 0;
#pragma unroll
        for (int w = 0; w < kRouteWarps; ++w) s += sh[w * a.E + e];
        a.hist[c * a.E + e] = s;
    }
}

// Exclusive scan over a block of exactly 1024 threads; returns the thread's
// exclusive prefix and writes the block total to *total.
__device__ int block_exclusive_scan_1024(int v, int *scratch /*[32]*/, int *total) {
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

__global__ void __launch_bounds__(1024)
k_route_scan(RouteDev a, int64_t chunks, int64_t *counts, int32_t *offsets, int32_t *recv_cum,
             int32_t *sched) {
    __shared__ int scratch[33];
    const int e = threadIdx.x;   // E <= 1024 = blockDim.x
    int tot = 0;
    if (e < a.E)
        for (int64_t c = 0; c < chunks; ++c) tot += a.hist[c * a.E + e];
    int total;
    int off = block_exclusive_scan_1024(e < a.E ? tot : 0, scratch, &total);
    int mblocks = (tot + kGemmBM - 1) / kGemmBM;
    int mtotal;
    int mstart = block_exclusive_scan_1024(e < a.E ? mblocks : 0, scratch, &mtotal);
    if (e < a.E) {
        counts[e] = tot;
        offsets[e] = off;
        if (sched) sched[e] = mstart;
        int run = off;
        for (int64_t c = 0; c < chunks; ++c) {
            int v = a.hist[c * a.E + e];
            a.hist[c * a.E + e] = run;
            run += v;
            if ((c + 1) % a.chunks_per_partition == 0 && recv_cum)
                recv_cum[e * a.P + c / a.chunks_per_partition] = run;
        }
    }
    // status word of this call: invalid ids seen by any chunk
    int bad = 0;
    for (int64_t c = e; c < chunks; c += blockDim.x) bad |= a.bad[c];
    bad = __syncthreads_or(bad);
    if (e == 0) {
        offsets[a.E] = total;
        if (sched) sched[a.E] = mtotal;
        *a.status = bad ? MOE_DEV_BAD_EXPERT_ID : 0;
    }
}

__global__ void __launch_bounds__(kRouteThreads)
k_route_rank(RouteDev a, int32_t *route_row, int32_t *assist) {
    extern __shared__ int32_t sh[];   // [kRouteWarps][E]
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int64_t c = blockIdx.x;
    for (int64_t i = tid; i < kRouteWarps * a.E; i += blockDim.x) sh[i] = 0;
    __syncthreads();
    ChunkRange cr = chunk_range(a, c);
    int64_t w0, w1;
    warp_slice(cr, warp, w0, w1);
    warp_count(a, w0, w1, sh + warp * a.E, lane);
    __syncthreads();
    // per-warp bases: chunk base from the scan plus the counts of earlier warps
    for (int64_t e = tid; e < a.E; e += blockDim.x) {
        int32_t run = a.hist[c * a.E + e];
#pragma unroll
        for (int w = 0; w < kRouteWarps; ++w) {
            int32_t v = sh[w * a.E + e];
            sh[w * a.E + e] = run;
            run += v;
        }
    }
    __syncthreads();
    int32_t *base = sh + warp * a.E;
    const int32_t pl = (int32_t)cr.p;
    for (int64_t b = w0; b < w1; b += 32) {
        int64_t i = b + lane;
        int e = (i < w1) ? route_expert(a, i) : -1;
        if (e < 0) e = -1;
        uint32_t grp = __match_any_sync(kFull, e);
        int row = -1;
        if (e >= 0) row = base[e] + __popc(grp & lanemask_lt());
        __syncwarp();
        if (e >= 0 && lane == __ffs(grp) - 1) base[e] += __popc(grp);
        __syncwarp();
        if (i < w1) {
            route_row[i] = row;
            if (row >= 0 && assist) {
                int64_t t = i / a.K;
                assist[3 * (int64_t)row + 0] = pl;
                assist[3 * (int64_t)row + 1] = (int32_t)(t - cr.p * a.M);
                assist[3 * (int64_t)row + 2] = (int32_t)(i - t * a.K);
            }
        }
    }
}

// m-block schedule from offsets alone (for moe_grouped_ffn, which gets only
// the offsets from its caller).
// It also starts the call's status word at 0.
__global__ void __launch_bounds__(1024)
k_sched(const int32_t *offsets, int64_t E, int32_t *sched, int32_t *status) {
    __shared__ int scratch[33];
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
                        int32_t *recv_cum, int32_t *sched, int32_t *route_row, int32_t *assist,
                        cudaStream_t stream) {
    size_t smem = (size_t)kRouteWarps * r.E * sizeof(int32_t);
    if (chunks > 0) {
        MOE_LAUNCH("route_count", k_route_count, (unsigned)chunks, kRouteThreads, smem, stream, r);
    }
    MOE_LAUNCH("route_scan", k_route_scan, 1, 1024, 0, stream, r, chunks, counts, offsets,
               recv_cum, sched);
    if (chunks > 0) {
        MOE_LAUNCH("route_rank", k_route_rank, (unsigned)chunks, kRouteThreads, smem, stream, r,
                   route_row, assist);
    }
    return MOE_OK;
}

moe_status launch_sched(const int32_t *offsets, int64_t E, int32_t *sched, int32_t *status,
                        cudaStream_t stream) {
    MOE_LAUNCH("sched", k_sched, 1, 1024, 0, stream, offsets, E, sched, status);
    return MOE_OK;
}

}  // namespace moe
