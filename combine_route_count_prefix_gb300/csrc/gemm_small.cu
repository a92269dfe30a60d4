// gemm_small.cu -- grouped int8 GEMMs for batches with few rows per expert.
//
// "PTO MegaMoE Dispatch + Combine Fusion Example", GMM1 / GMM2, and its
// Supported Cases (the sweep from 16 to 2048 tokens per rank): with a few
// routed rows per expert the GEMMs do little arithmetic per weight byte and
// their time is the time to read the weights.  This kernel reads them as int8
// (stored biased by +128), half the bytes of the fp16 images of the large-tile
// kernel, and widens them on chip straight into tensor memory: the weights are
// the MMA's A operand (M = 128 output channels, taken from TMEM) and the
// expert's rows its B operand (N = the rows present rounded up to 16, at most
// 128, from shared memory).  So the widened weights never pass through shared
// memory, whose bandwidth bounds a design that stages them there.
//
// Exactness is that of the large-tile kernel: fp16 images of int8 values,
// fp32 sums of at most 1024 products per accumulator, int32 totals in
// registers.
//
// Kernel shape (one persistent CTA per SM, 16 warps):
//   warp 0       weight producer: one biased-int8 TMA tile (128 rows x 128,
//                128-byte swizzle) per k-block into a 4-stage ring
//   warps 1, 3   MMA issuers: one thread spends ~130 cycles issuing each
//                tcgen05.mma whatever its N, and two threads issue at twice
//                the rate, so the 8 MMAs (K = 16) of a 128-deep k-block are
//                split: issuer i takes K [64 i, 64 i + 64) into its own 128
//                accumulator columns (the sums are exact integers, so how they
//                are split and added does not matter); warp 1 also owns TMEM
//                (512 columns: the issuers' 256 accumulator columns and four
//                64-column A stages)
//   warp 2       row producer: the tile's rows (fp16 images, 128-byte swizzle),
//                one TB-row TMA box per 64-wide half of a k-block, into a
//                4-stage ring; rows past the tile's (the next expert's, or zero
//                fill past the row capacity) come along and are never read
//                out: two large copies per k-block cost far less than one per
//                16 rows present, whose count bounded the kernel
//   warps 4..7   converters: thread (q, l) widens weight row 32 q + l of the
//                tile (128 values) and writes it to its own TMEM lane (64
//                columns, two fp16 values each)
//   warps 8..15  epilogue: warp % 4 selects the TMEM lane quadrant (32 output
//                channels), (warp - 8) / 4 the half of the tile's rows; adds
//                the two issuers' accumulators
// Tiles are (expert, TB-row block of its rows, 128-channel block), channel
// block fastest; the row block schedule is computed here from the offsets.
// Two tile heights:
//   TB = 64   each issuer's 128 columns hold two 64-column accumulators, so
//             the MMAs of one 1024-deep chunk run while the epilogue drains
//             the previous one (rows average at most 32 per expert);
//   TB = 128  one 128-column accumulator per issuer: an expert of up to 128
//             rows reads its weights once, at the cost of the MMAs waiting
//             for each drain; chunks are 16 k-blocks (each issuer sums 1024
//             products per row, still exact) to halve the drains.
// Every wait is bounded (about two seconds) and sets MOE_DEV_TIMEOUT.
#include "common.cuh"
#include "tcgen05.cuh"

#include <cudaTypedefs.h>

namespace moe {
namespace {

using namespace tc;

constexpr int BW = 128;                  // weight rows (output channels) per tile = MMA M
constexpr int BK = 128;                  // k-block
constexpr int BKH = 64;                  // one 128-byte swizzle atom of fp16 rows
constexpr int S8 = 4;                    // int8 weight ring stages
constexpr int SA = 4;                    // operand stages: TMEM A + shared-memory rows
constexpr int W8_BYTES = BW * BK;        // 16 KB
constexpr int CONV_WARP0 = 4;            // warps 4..7: TMEM lane quadrants 0..3
constexpr int EPI_WARP0 = 8;
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 32 * (EPI_WARP0 + EPI_WARPS);
constexpr uint32_t TMEM_COLS = 512;
constexpr int ISSUERS = 2;
constexpr uint32_t ACC_COLS = 128;       // per issuer
constexpr uint32_t A_COL0 = ISSUERS * ACC_COLS;
constexpr uint32_t A_STAGE_COLS = BK / 2;
constexpr size_t kBarrierBytes = 512;
// rows averaging at most this many per expert take the 64-row tiles
constexpr int64_t kNarrowTileMaxRowsPerExpert = 32;
static_assert(A_COL0 + SA * A_STAGE_COLS <= TMEM_COLS, "TMEM budget");
static_assert(BK / 16 == 4 * ISSUERS, "k-steps split between the issuers");
static_assert((2 * S8 + 2 * SA + 5) * 8 + 16 <= (int)kBarrierBytes, "barrier area");

// Sizes that follow from the tile height TB (64 or 128 rows).
template <int TB_>
struct SmallCfg {
    static constexpr int TB = TB_;
    static constexpr int NBUF = (int)ACC_COLS / TB;    // accumulators per issuer
    static constexpr int CHUNK_KB = TB == 64 ? 8 : 16;  // k-blocks per exact chunk
    static constexpr int B_HALF_BYTES = TB * BKH * 2;   // one 64-wide half of the rows: one TMA box
    static constexpr int B_BYTES = 2 * B_HALF_BYTES;
    static constexpr int EPI_COLS = TB / 2;             // tile rows per epilogue warp
    static constexpr size_t RING_BYTES = (size_t)SA * B_BYTES + (size_t)S8 * W8_BYTES;
    static constexpr size_t SMEM_BYTES =
        RING_BYTES + 1024 + kBarrierBytes + 2 * (kMaxExperts + 1) * sizeof(int32_t);
    static_assert(TB == 64 || TB == 128, "tile heights");
    static_assert(NBUF * TB == (int)ACC_COLS && NBUF <= 2, "accumulators");
    // each issuer adds BK / ISSUERS products per k-block into its accumulator;
    // fp32 holds every integer sum of at most 1024 int8 products exactly
    static_assert(CHUNK_KB * (BK / ISSUERS) <= 1024, "exact chunk");
    static_assert(SMEM_BYTES <= 232448, "shared memory budget");
};

struct SmallDev {
    const int32_t *offsets;
    const int32_t *sched;
    int E;
    int n_wblocks;      // ceil(Nout / 128)
    int num_kb;
    int Nout;
    int64_t cap_rows;
    int32_t *c_s32;
    float *g;
    const float *scale1;
    const float *s1;
    __nv_bfloat16 *y;
    const float *scale2;
    const float *s2;
    int32_t *status;
};

struct Tile {
    int e, row0, rows, wb;
};

template <int TB>
__device__ __forceinline__ Tile decode_tile(int64_t tile, int n_wblocks, int E,
                                            const int32_t *s_sched, const int32_t *s_off) {
    Tile t;
    const int mblk = (int)(tile / n_wblocks);
    t.wb = (int)(tile % n_wblocks);
    int lo = 0, hi = E - 1;
    while (lo < hi) {   // last expert whose first row block is <= mblk
        const int mid = (lo + hi + 1) >> 1;
        if (s_sched[mid] <= mblk) lo = mid; else hi = mid - 1;
    }
    t.e = lo;
    t.row0 = s_off[lo] + (mblk - s_sched[lo]) * TB;
    t.rows = min(TB, s_off[lo + 1] - t.row0);
    return t;
}

// Two biased bytes u0, u1 (w + 128) -> the fp16 pair (w0, w1): each byte goes
// into the low mantissa bits of the fp16 number 1024 (exponent 10, unit
// spacing), giving 1024 + u exactly, and one f16x2 subtraction of 1152 leaves
// w exactly.
__device__ __forceinline__ uint32_t widen_pair(uint32_t word, uint32_t sel) {
    uint32_t d;
    asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(__byte_perm(word, 0x64646464u, sel)), "r"(0x64806480u));
    return d;
}

// ---------------------------------------------------------------- epilogues
// acc[i] is the exact int32 sum of output channel `ch` (a row of the weight
// tile, lane quadrant q) for row t.row0 + c0 + i of the tile.
template <int EPI, int EPI_COLS>
__device__ __forceinline__ void epilogue_small(const SmallDev &p, const Tile &t, int q, int lane,
                                               int c0, const int32_t (&acc)[EPI_COLS]) {
    const int ch = t.wb * BW + q * 32 + lane;
    if (EPI == (int)Epi::S32) {
#pragma unroll
        for (int i = 0; i < EPI_COLS; ++i) {
            if (c0 + i >= t.rows) break;
            const int64_t row = (int64_t)t.row0 + c0 + i;
            if (row >= p.cap_rows) break;
            if (ch < p.Nout) p.c_s32[row * p.Nout + ch] = acc[i];
        }
    } else if (EPI == (int)Epi::SwiGLU) {
        // weight block wb, quadrant q: lanes 0..15 are SiLU-half channels
        // j = 64 wb + 16 q + lane, lanes 16..31 the multiplier channels N/2 + j
        const int Nh = p.Nout / 2;
        const int j = t.wb * 64 + q * 16 + (lane & 15);
        const bool gate = lane < 16;
        const float sc = __ldg(p.scale1 + (int64_t)t.e * p.Nout + (gate ? j : Nh + j));
#pragma unroll
        for (int i = 0; i < EPI_COLS; ++i) {
            if (c0 + i >= t.rows) break;
            const int64_t row = (int64_t)t.row0 + c0 + i;
            if (row >= p.cap_rows) break;
            const float h = __fmul_rn(__fmul_rn(__int2float_rn(acc[i]), sc), __ldg(p.s1 + row));
            const float m = __shfl_down_sync(0xffffffffu, h, 16);
            if (gate) p.g[row * Nh + j] = __fmul_rn(silu_f32(h), m);
        }
    } else {
        const float sc = ch < p.Nout ? __ldg(p.scale2 + (int64_t)t.e * p.Nout + ch) : 0.0f;
#pragma unroll
        for (int i = 0; i < EPI_COLS; ++i) {
            if (c0 + i >= t.rows) break;
            const int64_t row = (int64_t)t.row0 + c0 + i;
            if (row >= p.cap_rows) break;
            const float v = __fmul_rn(__fmul_rn(__int2float_rn(acc[i]), sc), __ldg(p.s2 + row));
            if (ch < p.Nout) p.y[row * p.Nout + ch] = __float2bfloat16_rn(v);
        }
    }
}

// ---------------------------------------------------------------- the kernel
template <int EPI, int TB_>
__global__ void __launch_bounds__(THREADS, 1)
k_gemm_small(const __grid_constant__ CUtensorMap tmRows, const __grid_constant__ CUtensorMap tmW,
             SmallDev p) {
    using Cfg = SmallCfg<TB_>;
    constexpr int TB = Cfg::TB, NBUF = Cfg::NBUF, CHUNK_KB = Cfg::CHUNK_KB;
    constexpr int B_HALF_BYTES = Cfg::B_HALF_BYTES, B_BYTES = Cfg::B_BYTES;
    constexpr int EPI_COLS = Cfg::EPI_COLS;
    constexpr size_t RING_BYTES = Cfg::RING_BYTES;
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint8_t *ringB = smem;                                   // SA x B_BYTES fp16 rows
    uint8_t *ring8 = ringB + (size_t)SA * B_BYTES;           // S8 x 16 KB biased int8 weights
    uint64_t *w8_full = reinterpret_cast<uint64_t *>(smem + RING_BYTES);
    uint64_t *w8_empty = w8_full + S8;
    // ab_full[s]: operand stage s is complete -- the four converter warps have
    // written its A columns and the row producer's copies have landed (one
    // barrier, so the issuers test one phase per k-block)
    uint64_t *ab_full = w8_empty + S8;
    uint64_t *ab_empty = ab_full + SA;
    uint64_t *acc_full = ab_empty + SA;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int32_t *s_sched = reinterpret_cast<int32_t *>(smem + RING_BYTES + kBarrierBytes);
    int32_t *s_off = s_sched + (kMaxExperts + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < S8; ++s) {
            mbar_init(&w8_full[s], 1);
            mbar_init(&w8_empty[s], 4);
        }
        for (int s = 0; s < SA; ++s) {
            mbar_init(&ab_full[s], 4 + 1);
            mbar_init(&ab_empty[s], ISSUERS);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], ISSUERS);
            mbar_init(&acc_empty[b], EPI_WARPS);
        }
        mbar_init(drain, ISSUERS);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmRows) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmW) : "memory");
    }
    pdl_wait();   // everything below may read what earlier kernels wrote
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_off[i] = p.offsets[i];
    __syncthreads();
    if (warp == 0) {
        // s_sched[e] = TB-row blocks of the experts before e (warp scan)
        int carry = 0;
        for (int base = 0; base < p.E; base += 32) {
            const int e = base + lane;
            const int c = e < p.E ? (s_off[e + 1] - s_off[e] + TB - 1) / TB : 0;
            int x = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, d);
                if (lane >= d) x += y;
            }
            if (e < p.E) s_sched[e] = carry + x - c;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) s_sched[p.E] = carry;
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t total_tiles = (int64_t)s_sched[p.E] * p.n_wblocks;
    const int num_chunks = (p.num_kb + CHUNK_KB - 1) / CHUNK_KB;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ weight producer
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[S8];
#pragma unroll
            for (int s = 0; s < S8; ++s) issued_phase[s] = -1;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const Tile t = decode_tile<TB>(tile, p.n_wblocks, p.E, s_sched, s_off);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bounded(&w8_empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&w8_full[stage], W8_BYTES);
                    tma_load_3d(ring8 + (size_t)stage * W8_BYTES, &tmW, &w8_full[stage], kb * BK,
                                t.wb * BW, t.e);
                    issued_phase[stage] = (int)phase;
                    if (++stage == S8) { stage = 0; phase ^= 1u; }
                }
            }
            for (int s = 0; s < S8; ++s)
                if (issued_phase[s] >= 0)
                    wait_bounded(&w8_full[s], (uint32_t)issued_phase[s], abort_flag, p.status, false);
        }
    } else if (warp == 2) {
        if (lane == 0) {
            // ------------------------------------------------ row producer
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[SA];
#pragma unroll
            for (int s = 0; s < SA; ++s) issued_phase[s] = -1;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const Tile t = decode_tile<TB>(tile, p.n_wblocks, p.E, s_sched, s_off);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bounded(&ab_empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    mbar_arrive_expect_tx(&ab_full[stage], (uint32_t)B_BYTES);
                    uint8_t *dst = ringB + (size_t)stage * B_BYTES;
                    for (int h = 0; h < 2; ++h)
                        tma_load_2d(dst + h * B_HALF_BYTES, &tmRows, &ab_full[stage], kb * BK + h * BKH,
                                    t.row0);
                    issued_phase[stage] = (int)phase;
                    if (++stage == SA) { stage = 0; phase ^= 1u; }
                }
            }
            for (int s = 0; s < SA; ++s)
                if (issued_phase[s] >= 0)
                    wait_bounded(&ab_full[s], (uint32_t)issued_phase[s], abort_flag, p.status, false);
        }
    } else if (warp >= CONV_WARP0 && warp < CONV_WARP0 + 4) {
        // ---------------------------------------------------- converters
        const int q = warp & 3;                 // TMEM lane quadrant of this warp
        const int row = q * 32 + lane;          // weight row of the tile = TMEM lane
        const uint32_t lane_addr = (uint32_t)(q * 32) << 16;
        int s8 = 0, sa = 0;
        uint32_t ph8 = 0, pha = 0;
        bool ok = true;
        for (int64_t tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
            for (int kb = 0; kb < p.num_kb; ++kb) {
                const bool w = wait_bounded(&w8_full[s8], ph8, abort_flag, p.status) &&
                               wait_bounded(&ab_empty[sa], pha ^ 1u, abort_flag, p.status);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                // row `row` of the tile: 128 bytes, 16-byte unit u at u ^ (row % 8)
                const uint8_t *src = ring8 + (size_t)s8 * W8_BYTES + row * 128;
                uint4 v[8];
#pragma unroll
                for (int i = 0; i < 8; ++i)
                    v[i] = *reinterpret_cast<const uint4 *>(src + ((i ^ (row & 7)) << 4));
#pragma unroll
                for (int h = 0; h < 2; ++h) {
                    uint32_t words[32];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const uint4 &x = v[4 * h + i];
                        const uint32_t b4[4] = {x.x, x.y, x.z, x.w};
#pragma unroll
                        for (int j = 0; j < 4; ++j) {
                            words[8 * i + 2 * j] = widen_pair(b4[j], 0x4140);       // bytes 0, 1
                            words[8 * i + 2 * j + 1] = widen_pair(b4[j], 0x4342);   // bytes 2, 3
                        }
                    }
                    tmem_st32(tmem_base + lane_addr + A_COL0 + (uint32_t)sa * A_STAGE_COLS + 32 * h,
                              words);
                }
                tmem_st_wait();
                tc_fence_before();
                __syncwarp();
                if (lane == 0) {
                    mbar_arrive(&w8_empty[s8]);
                    mbar_arrive(&ab_full[sa]);
                }
                if (++s8 == S8) { s8 = 0; ph8 ^= 1u; }
                if (++sa == SA) { sa = 0; pha ^= 1u; }
            }
        }
    } else if (warp == 1 || warp == 3) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuers
            const int is = warp >> 1;   // 0 or 1: K [64 is, 64 is + 64) of every k-block
            int stage = 0;
            uint32_t phase = 0;
            int accb = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                const Tile t = decode_tile<TB>(tile, p.n_wblocks, p.E, s_sched, s_off);
                const int n16 = ((t.rows + 15) / 16) * 16;
                const uint32_t idesc = idesc_f16(BW, n16);
                for (int kb0 = 0; ok && kb0 < p.num_kb; kb0 += CHUNK_KB) {
                    if (!wait_bounded(&acc_empty[accb], acc_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(is * ACC_COLS + accb * TB);
                    const int kb1 = min(kb0 + CHUNK_KB, p.num_kb);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!wait_bounded(&ab_full[stage], phase, abort_flag, p.status)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        const uint32_t a_tmem = tmem_base + A_COL0 + (uint32_t)stage * A_STAGE_COLS;
                        const uint32_t b_addr = smem_u32(ringB + (size_t)stage * B_BYTES);
#pragma unroll
                        for (int k = 0; k < 4; ++k)   // K = 16: 8 TMEM columns, 32 bytes of a row
                            mma_f16_ta(d_tmem, a_tmem + 32 * is + 8 * k,
                                       desc_sw128(b_addr + is * B_HALF_BYTES + 32 * k), idesc,
                                       (kb > kb0 || k > 0) ? 1u : 0u);
                        mma_commit(&ab_empty[stage]);
                        if (++stage == SA) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    mma_commit(&acc_full[accb]);
                    if (++accb == NBUF) { accb = 0; acc_phase ^= 1u; }
                }
            }
            mma_commit(drain);
            wait_bounded(drain, 0, abort_flag, p.status, false);
        }
    } else if (warp >= EPI_WARP0) {
        // ---------------------------------------------------- epilogue warps
        const int q = warp & 3;
        const int c0 = ((warp - EPI_WARP0) >> 2) * EPI_COLS;   // first tile row of this warp
        int accb = 0;
        uint32_t acc_phase = 0;
        // columns per TMEM load: 16 when a warp holds 64 rows' sums, so the load
        // buffer and the sums fit the registers together
        constexpr int LDW = EPI_COLS > 32 ? 16 : 32;
        for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            const Tile t = decode_tile<TB>(tile, p.n_wblocks, p.E, s_sched, s_off);
            const int nj = (t.rows - c0 + LDW - 1) / LDW;   // column groups holding rows (may be <= 0)
            int32_t acc[EPI_COLS];
#pragma unroll
            for (int i = 0; i < EPI_COLS; ++i) acc[i] = 0;
            bool ok = true;
            for (int c = 0; c < num_chunks; ++c) {
                const bool w = wait_bounded(&acc_full[accb], acc_phase, abort_flag, p.status);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr =
                    tmem_base + ((uint32_t)(q * 32) << 16) + (uint32_t)(accb * TB + c0);
#pragma unroll
                for (int j = 0; j < EPI_COLS / LDW; ++j) {
                    if (j < nj) {
#pragma unroll
                        for (int is = 0; is < ISSUERS; ++is) {
                            uint32_t r[LDW];
                            if constexpr (LDW == 32)
                                tmem_ld32(taddr + is * ACC_COLS + LDW * j, r);
                            else
                                tmem_ld16(taddr + is * ACC_COLS + LDW * j, r);
                            tmem_ld_wait();
#pragma unroll
                            for (int i = 0; i < LDW; ++i)
                                acc[LDW * j + i] += __float2int_rn(__uint_as_float(r[i]));
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[accb]);
                if (++accb == NBUF) { accb = 0; acc_phase ^= 1u; }
            }
            if (!ok) break;
            if (nj > 0) epilogue_small<EPI, EPI_COLS>(p, t, q, lane, c0, acc);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

template <int EPI, int TB>
moe_status launch_small_tb(const CUtensorMap &mr, const CUtensorMap &mw, const SmallDev &d,
                           cudaStream_t stream) {   // mr: boxes of TB rows
    constexpr size_t smem = SmallCfg<TB>::SMEM_BYTES;
    if (!set_smem_limit((const void *)k_gemm_small<EPI, TB>, smem)) return MOE_ERR_CUDA;
    const char *names[3] = {"gemm_s32_small", "gemm1_swiglu_small", "gemm2_dequant_small"};
    MOE_LAUNCH(names[EPI], (k_gemm_small<EPI, TB>), num_sms(), THREADS, smem, stream, mr, mw, d);
    return MOE_OK;
}

template <int EPI>
moe_status launch_small_epi(const CUtensorMap &mr, const CUtensorMap &mw, const SmallDev &d,
                            bool wide, cudaStream_t stream) {
    return wide ? launch_small_tb<EPI, 128>(mr, mw, d, stream)
                : launch_small_tb<EPI, 64>(mr, mw, d, stream);
}

}  // namespace

moe_status launch_grouped_gemm_small(Epi epi, const GemmArgs &a, cudaStream_t stream) {
    if (a.cap_rows <= 0 || a.E <= 0) return MOE_OK;
    if (a.Kd % 16 != 0) return MOE_ERR_SHAPE;   // byte rows must be 16-byte strided for TMA
    if (epi == Epi::SwiGLU && a.Nout % 128 != 0) return MOE_ERR_SHAPE;
    // the row capacity bounds the rows present: 64-row tiles while it averages
    // at most 32 rows per expert, else 128-row tiles
    const bool wide = a.cap_rows > kNarrowTileMaxRowsPerExpert * a.E;
    CUtensorMap mr, mw;
    const uint64_t rdims[2] = {(uint64_t)a.Kd, (uint64_t)a.cap_rows};
    const uint64_t rstr[1] = {(uint64_t)a.Kd * 2};
    const uint32_t rbox[2] = {BKH, wide ? 128u : 64u};
    const uint64_t wdims[3] = {(uint64_t)a.Kd, (uint64_t)a.Nout, (uint64_t)a.E};
    const uint64_t wstr[2] = {(uint64_t)a.Kd, (uint64_t)a.Kd * a.Nout};
    const uint32_t wbox[3] = {BK, BW, 1};
    if (!make_tensor_map(&mr, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, CU_TENSOR_MAP_SWIZZLE_128B, a.a_img, 2,
                         rdims, rstr, rbox))
        return MOE_ERR_CUDA;
    if (!make_tensor_map(&mw, CU_TENSOR_MAP_DATA_TYPE_UINT8, CU_TENSOR_MAP_SWIZZLE_128B, a.b_img, 3,
                         wdims, wstr, wbox))
        return MOE_ERR_CUDA;
    SmallDev d;
    d.offsets = a.offsets;
    d.sched = a.sched;
    d.E = (int)a.E;
    d.n_wblocks = (int)((a.Nout + BW - 1) / BW);
    d.num_kb = (int)((a.Kd + BK - 1) / BK);
    d.Nout = (int)a.Nout;
    d.cap_rows = a.cap_rows;
    d.c_s32 = a.c_s32;
    d.g = a.g;
    d.scale1 = a.scale1;
    d.s1 = a.s1;
    d.y = reinterpret_cast<__nv_bfloat16 *>(a.y);
    d.scale2 = a.scale2;
    d.s2 = a.s2;
    d.status = a.status;
    switch (epi) {
        case Epi::S32: return launch_small_epi<(int)Epi::S32>(mr, mw, d, wide, stream);
        case Epi::SwiGLU: return launch_small_epi<(int)Epi::SwiGLU>(mr, mw, d, wide, stream);
        case Epi::DequantBF16:
            return launch_small_epi<(int)Epi::DequantBF16>(mr, mw, d, wide, stream);
    }
    return MOE_ERR_PARAM_INVALID;
}

}  // namespace moe
