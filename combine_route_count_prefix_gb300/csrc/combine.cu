// combine.cu -- weighted combine / unpermute.
//
// out[t] = bf16( sum_{k active, ascending} p[t,k] * float(y[row(t,k)]) + float(shared[t]) )
// with a separately rounded fp32 multiply and add per slot, in slot order,
// from an accumulator starting at +0, then round-to-nearest-even to bf16:
// the combine loop of "dispatch_combine_shmem.py" ("2. Implement the Combine
// operator": cast, mul by expert_scales, add, CAST_RINT), with the shared
// expert term of "aclnnMoeDistributeCombineV4" (Function/Formula) added once
// after the routed sum, back in token order ("PTO MegaMoE ...", Unpermute).
//
// GB300 design: a persistent kernel, one CTA per SM, that moves whole
// contiguous row segments through shared memory with bulk (TMA) copies.  A
// work item is one segment (about half of a 7168-wide row) of one token; each
// CTA owns a contiguous block of tokens.  Warp 0 produces: its lanes load the
// route rows, mask bits and probabilities of 32 tokens into registers (all
// loads issued together, and the next batch's loads in flight while the
// current batch is issued); per item, lane 0 waits for a free stage, writes
// the item header (active slot count and their probabilities) and arms the
// stage's mbarrier with the byte count, and the lanes issue the item's bulk
// copies in parallel, one active row segment each plus the shared-expert
// segment.  Warps 1..15 consume a stage: each thread owns up to two 16-byte
// vectors of the segment, loads the rows' vectors from shared memory, adds
// them in slot order and stores the bf16 result.  Three stages of ~64 KB are
// in flight per SM; the copies bypass the SM's load-tracking limits and keep
// DRAM reads long and contiguous.  Measured on the decode workload: smaller
// stages (more of them) and whole-row stages (one copy per row) are both
// slower, so the time is set by the bytes in flight per SM against DRAM
// latency under load.  CTA b takes tokens from the last one down in steps of
// G (G CTAs), so the tokens in flight at any time are close together and so
// are their rows inside each expert's block.
#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kConsumerWarps = 15;   // with the producer, 16 warps: four per scheduler
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr int kVecsPerThread = 2;
constexpr int kMaxSegVecs = kConsumerWarps * 32 * kVecsPerThread;   // 512 vectors = 8 KB
constexpr int kMaxStages = 8;
constexpr size_t kStageTarget = 64 * 1024;
constexpr size_t kSmemBudget = 196 * 1024;
constexpr uint32_t kFull = 0xffffffffu;

// One work item: n terms in slot order with their probabilities; with
// special experts, term j adds p[j] * (stage slot src[j], or 0 when
// src[j] < 0: a zero expert).
struct ItemHdr {
    int32_t n;
    int32_t pad[3];
    float p[kMaxTopK];
    int32_t src[kMaxTopK];
};

struct CombineArgs {
    const uint4 *y;
    const int32_t *route_row;
    const float *probs;
    const uint8_t *mask;
    const uint4 *shared;
    const uint4 *ori_x;
    uint4 *out;
    int64_t T, H8, cap_rows, tokens_per_cta;
    int K, mask_kind, stages, nseg, seg_vecs, slots;
    int32_t *status;
};

__device__ __forceinline__ uint4 lds128(const void *p) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(smem_u32(p)));
    return v;
}

__device__ __forceinline__ void unpack8(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    return (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
           ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
}

// Stage slots: up to K row segments, the shared-expert segment (slot K) and,
// when copy experts exist, the oriX segment (slot K + 1).
__host__ __device__ inline size_t stage_bytes(int slots, int seg_vecs) {
    return (size_t)slots * seg_vecs * 16;
}

size_t smem_bytes(int K, int slots, int stages, int seg_vecs) {
    return 128 + (size_t)stages * stage_bytes(slots, seg_vecs) + stages * sizeof(ItemHdr) +
           2 * stages * sizeof(uint64_t) + 16 + 2 * 32 * (size_t)K * (sizeof(int32_t) + sizeof(float));
}

// Adds the shared-expert vector (slot K) if present, rounds to bf16, stores.
__device__ __forceinline__ void store_result(const CombineArgs &a, const uint8_t *src, int v,
                                             int64_t out_idx, float (&acc)[8]) {
    if (a.shared) {
        float f[8];
        unpack8(lds128(src + ((size_t)a.K * a.seg_vecs + v) * 16), f);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc[i] = __fadd_rn(acc[i], f[i]);
    }
    uint4 o;
    o.x = pack_bf16x2(acc[0], acc[1]);
    o.y = pack_bf16x2(acc[2], acc[3]);
    o.z = pack_bf16x2(acc[4], acc[5]);
    o.w = pack_bf16x2(acc[6], acc[7]);
    a.out[out_idx] = o;
}

// kSpecial: the shape has zero or copy experts (route_row codes -2 / -3).
template <bool kSpecial>
__global__ void __launch_bounds__(kThreads, 1)
k_combine(CombineArgs a) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 127) &
                                                ~(uintptr_t)127);
    const size_t sbytes = stage_bytes(a.slots, a.seg_vecs);
    uint8_t *bufs = smem;
    ItemHdr *hdrs = reinterpret_cast<ItemHdr *>(bufs + a.stages * sbytes);
    uint64_t *full = reinterpret_cast<uint64_t *>(hdrs + a.stages);
    uint64_t *empty = full + a.stages;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(empty + a.stages);
    int32_t *meta_row = reinterpret_cast<int32_t *>(empty + a.stages) + 4;   // [2][32*K]
    float *meta_p = reinterpret_cast<float *>(meta_row + 2 * 32 * a.K);    // [2][32*K]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < a.stages; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kConsumerWarps);
        }
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    __syncthreads();
    pdl_wait();

    // this CTA's tokens: T - 1 - (blockIdx.x + G * i) for i in [0, ntok).  Tokens are
    // taken from the last one down: the row copy writes rows in token order, so when
    // combine follows it the last tokens' rows are the ones most likely still in L2.
    const int64_t G = gridDim.x;
    const int64_t ntok = (a.T - blockIdx.x + G - 1) / G;
    auto token_of = [&](int64_t i) -> int64_t { return a.T - 1 - (blockIdx.x + G * i); };

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        int stage = 0;
        uint32_t phase = 0;
        int issued_phase[kMaxStages];
#pragma unroll
        for (int s = 0; s < kMaxStages; ++s) issued_phase[s] = -1;
        bool ok = true;
        int32_t rr[kMaxTopK];
        float pp[kMaxTopK];
        const uint64_t read_once = l2_policy_evict_first();
        // metadata of the batch starting at tb, for token tb + lane, into registers
        auto load_meta = [&](int64_t ib) {
            const bool in = ib + lane < ntok;
            const int64_t t = token_of(ib + lane);
            const bool tok = in && (a.mask_kind != 1 || a.mask[t] != 0);
#pragma unroll
            for (int k = 0; k < kMaxTopK; ++k) {
                rr[k] = -1;
                pp[k] = 0.0f;
                if (k < a.K && in) {
                    rr[k] = a.route_row[t * a.K + k];
                    pp[k] = a.probs[t * a.K + k];
                }
            }
#pragma unroll
            for (int k = 0; k < kMaxTopK; ++k) {
                if (k >= a.K) break;
                // a row; with special experts also a zero (-2) or copy (-3) slot
                bool on = tok && ((rr[k] >= 0 && rr[k] < a.cap_rows) ||
                                  (kSpecial && (rr[k] == -2 || (rr[k] == -3 && a.ori_x))));
                if (a.mask_kind == 2 && in) on = on && a.mask[t * a.K + k] != 0;
                rr[k] = on ? rr[k] : -1;
            }
        };
        auto store_meta = [&](int buf) {
            int32_t *mr = meta_row + buf * 32 * a.K + lane * a.K;
            float *mp = meta_p + buf * 32 * a.K + lane * a.K;
#pragma unroll
            for (int k = 0; k < kMaxTopK; ++k) {
                if (k >= a.K) break;
                mr[k] = rr[k];
                mp[k] = pp[k];
            }
        };
        if (ntok > 0) {
            load_meta(0);
            store_meta(0);
        }
        __syncwarp();
        int buf = 0;
        for (int64_t ib = 0; ib < ntok; ib += 32) {
            const bool more = ib + 32 < ntok;
            if (more) load_meta(ib + 32);          // in flight while this batch is issued
            // Lane 0 waits for the stage and writes its header; the copies are
            // issued by the lanes in parallel (a bulk copy costs its issuing
            // thread a few hundred cycles): lane k < K the row of slot k if it
            // has one, lane K the shared-expert row, lane K + 1 the token's
            // own row when a copy expert needs it.
            const int64_t ie = min(ib + 32, ntok);
            for (int64_t ii = ib; ok && ii < ie; ++ii) {
                const int64_t tt = token_of(ii);
                const int32_t *rows = meta_row + buf * 32 * a.K + (ii - ib) * a.K;
                const float *ps = meta_p + buf * 32 * a.K + (ii - ib) * a.K;
                const int32_t my_code = lane < a.K ? rows[lane] : -1;
                const uint32_t row_mask = __ballot_sync(kFull, my_code >= 0);
                const int my_slot = __popc(row_mask & ((1u << lane) - 1u));
                const int nrow = __popc(row_mask);
                const bool need_ori = kSpecial && __any_sync(kFull, my_code == -3);
                for (int seg = 0; seg < a.nseg; ++seg) {
                    bool w = true;
                    if (lane == 0) w = wait_bounded(&empty[stage], phase ^ 1u, abort_flag, a.status);
                    if (!__shfl_sync(kFull, w, 0)) {
                        ok = false;
                        break;
                    }
                    const int64_t v0 = (int64_t)seg * a.seg_vecs;
                    const uint32_t bytes = (uint32_t)(min((int64_t)a.seg_vecs, a.H8 - v0) * 16);
                    ItemHdr *h = hdrs + stage;
                    uint8_t *dst = bufs + stage * sbytes;
                    if (lane == 0) {
                        int n = 0;
                        if (kSpecial) {
                            int nr = 0;
                            for (int k = 0; k < a.K; ++k) {
                                const int32_t code = rows[k];
                                if (code == -1) continue;
                                h->p[n] = ps[k];
                                if (code >= 0) h->src[n] = nr++;
                                else if (code == -2) h->src[n] = -1;
                                else h->src[n] = a.K + 1;
                                ++n;
                            }
                        } else {
                            for (int k = 0; k < a.K; ++k)
                                if (rows[k] >= 0) h->p[n++] = ps[k];
                        }
                        h->n = n;
                        const uint32_t loads =
                            (uint32_t)(nrow + (a.shared ? 1 : 0) + (need_ori ? 1 : 0));
                        mbar_arrive_expect_tx(&full[stage], loads * bytes);
                        issued_phase[stage] = (int)phase;
                    }
                    __syncwarp();
                    // every input is read once: evict-first keeps the rows still to
                    // come (the row copy leaves the last tokens' rows in L2) in place
                    if (my_code >= 0)
                        bulk_load_hint(dst + (size_t)my_slot * a.seg_vecs * 16,
                                       a.y + (int64_t)my_code * a.H8 + v0, bytes, &full[stage],
                                       read_once);
                    else if (lane == a.K && a.shared)
                        bulk_load_hint(dst + (size_t)a.K * a.seg_vecs * 16,
                                       a.shared + tt * a.H8 + v0, bytes, &full[stage], read_once);
                    else if (lane == a.K + 1 && need_ori)
                        bulk_load_hint(dst + (size_t)(a.K + 1) * a.seg_vecs * 16,
                                       a.ori_x + tt * a.H8 + v0, bytes, &full[stage], read_once);
                    if (++stage == a.stages) { stage = 0; phase ^= 1u; }
                }
            }
            ok = __shfl_sync(kFull, ok, 0);
            __syncwarp();
            if (more) store_meta(buf ^ 1);
            __syncwarp();
            buf ^= 1;
            if (!ok) break;
        }
        // every copy issued must have landed before the CTA exits
        if (lane == 0)
            for (int s = 0; s < a.stages; ++s)
                if (issued_phase[s] >= 0)
                    wait_bounded(&full[s], (uint32_t)issued_phase[s], abort_flag, a.status, false);
    } else {
        // ------------------------------------------------------------ consumers
        const int c = threadIdx.x - 32;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int64_t ii = 0; ok && ii < ntok; ++ii) {
            const int64_t tt = token_of(ii);
            for (int seg = 0; seg < a.nseg; ++seg) {
                const bool w = wait_bounded(&full[stage], phase, abort_flag, a.status);
                if (!__all_sync(kFull, w)) { ok = false; break; }
                const ItemHdr *h = hdrs + stage;
                const uint8_t *src = bufs + stage * sbytes;
                const int64_t v0 = (int64_t)seg * a.seg_vecs;
                const int len = (int)min((int64_t)a.seg_vecs, a.H8 - v0);
                const int n = h->n;
                if (kSpecial) {
                    // the item's terms in registers; a zero-expert term adds p * 0
                    int sl[kMaxTopK];
                    float pr[kMaxTopK];
#pragma unroll
                    for (int j = 0; j < kMaxTopK; ++j) {
                        sl[j] = (j < n) ? h->src[j] : 0;
                        pr[j] = (j < n) ? h->p[j] : 0.0f;
                    }
#pragma unroll
                    for (int u = 0; u < kVecsPerThread; ++u) {
                        const int v = c + u * kConsumerWarps * 32;
                        if (v >= len) continue;
                        float acc[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
                        // up to 8 terms' vectors are loaded before any is used, so the
                        // shared-memory latency is paid once per 8 terms
#pragma unroll
                        for (int j0 = 0; j0 < kMaxTopK; j0 += 8) {
                            if (j0 >= n) break;
                            uint4 raw[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j)
                                if (j0 + j < n)
                                    raw[j] = lds128(src + ((size_t)(sl[j0 + j] < 0 ? 0 : sl[j0 + j]) *
                                                               a.seg_vecs + v) * 16);
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                if (j0 + j >= n) break;
                                const bool zero = sl[j0 + j] < 0;
                                float f[8];
                                unpack8(raw[j], f);
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    acc[i] = __fadd_rn(acc[i], __fmul_rn(pr[j0 + j], zero ? 0.0f : f[i]));
                            }
                        }
                        store_result(a, src, v, tt * a.H8 + v0 + v, acc);
                    }
                } else {
#pragma unroll
                    for (int u = 0; u < kVecsPerThread; ++u) {
                        const int v = c + u * kConsumerWarps * 32;
                        if (v >= len) continue;
                        float acc[8];
#pragma unroll
                        for (int i = 0; i < 8; ++i) acc[i] = 0.0f;
                        for (int j0 = 0; j0 < n; j0 += 8) {
                            // up to 8 rows' vectors loaded before any is used
                            uint4 raw[8];
                            float pj[8];
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                if (j0 + j < n) {
                                    raw[j] = lds128(src + ((size_t)(j0 + j) * a.seg_vecs + v) * 16);
                                    pj[j] = h->p[j0 + j];
                                }
                            }
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                if (j0 + j >= n) break;
                                float f[8];
                                unpack8(raw[j], f);
#pragma unroll
                                for (int i = 0; i < 8; ++i)
                                    acc[i] = __fadd_rn(acc[i], __fmul_rn(pj[j], f[i]));
                            }
                        }
                        store_result(a, src, v, tt * a.H8 + v0 + v, acc);
                    }
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[stage]);
                if (++stage == a.stages) { stage = 0; phase ^= 1u; }
            }
        }
    }
}

}  // namespace

moe_status launch_combine(const void *y, const int32_t *route_row, const float *probs,
                          const uint8_t *mask, int mask_kind, const void *shared,
                          const void *ori_x, bool special, void *out, int64_t T, int64_t K,
                          int64_t H, int64_t cap_rows, int32_t *status, cudaStream_t stream) {
    if (T == 0) return MOE_OK;
    const int64_t grid = T < num_sms() ? T : (int64_t)num_sms();
    CombineArgs a;
    a.y = static_cast<const uint4 *>(y);
    a.route_row = route_row;
    a.probs = probs;
    a.mask = mask;
    a.shared = static_cast<const uint4 *>(shared);
    a.ori_x = static_cast<const uint4 *>(ori_x);
    a.out = static_cast<uint4 *>(out);
    a.T = T;
    a.H8 = H / 8;
    a.cap_rows = cap_rows;
    a.K = (int)K;
    a.mask_kind = mask_kind;
    // segment length: at most 512 vectors, a multiple of 8 (128-byte aligned
    // copies), about 64 KB per stage over all slots
    a.slots = a.K + 1 + (ori_x ? 1 : 0);
    int64_t maxv = (int64_t)(kStageTarget / ((size_t)a.slots * 16));
    if (maxv > kMaxSegVecs) maxv = kMaxSegVecs;
    maxv = maxv / 8 * 8;
    if (maxv < 8) maxv = 8;
    a.nseg = (int)((a.H8 + maxv - 1) / maxv);
    a.seg_vecs = (int)(((a.H8 + a.nseg - 1) / a.nseg + 7) / 8 * 8);
    a.stages = (int)(kSmemBudget / stage_bytes(a.slots, a.seg_vecs));
    if (a.stages > kMaxStages) a.stages = kMaxStages;
    if (a.stages < 2) a.stages = 2;
    a.tokens_per_cta = 0;
    a.status = status;
    const size_t smem = smem_bytes(a.K, a.slots, a.stages, a.seg_vecs);
    if (!set_smem_limit(special ? (const void *)k_combine<true> : (const void *)k_combine<false>, smem))
        return MOE_ERR_CUDA;
    if (special) {
        MOE_LAUNCH("combine", k_combine<true>, (unsigned)grid, kThreads, smem, stream, a);
    } else {
        MOE_LAUNCH("combine", k_combine<false>, (unsigned)grid, kThreads, smem, stream, a);
    }
    return MOE_OK;
}

}  // namespace moe
