// gemm_tc.cu -- grouped int8 GEMMs on the 5th-generation tensor cores.
//
// "PTO MegaMoE Dispatch + Combine Fusion Example", GMM1 and GMM2: per local
// expert, int8 rows x int8 weights -> int32 accumulator -> per-channel fp32
// scale (fixpipe) -> epilogue.  Here every expert is local.
//
// Exact int8 products on tcgen05.  sm_103a has no tcgen05 int8 kind, so the
// int8 operands are stored as fp16 images (every integer in [-127, 127] is an
// fp16 number) and multiplied with tcgen05.mma kind::f16 into fp32 TMEM
// accumulators.  Each product is at most 127*127 = 16129 in magnitude and is
// exact in fp32, and a sum of at most 1024 of them stays below 2^24 =
// 16777216, where every integer is an fp32 number.  The K loop is therefore cut
// into chunks of 1024 (16 k-blocks of 64): each chunk's accumulator holds an
// exact integer, which the epilogue warps convert to int32 and add up in
// registers.  The int32 total is the exact int8 dot product.
//
// Kernel shape (one persistent CTA per SM, 320 threads):
//   warp 0      TMA producer: A tile 128 x 64 and B tile 256 x 64 (fp16,
//               128-byte swizzle) per k-block into a 4-stage shared-memory ring
//   warp 1      TMEM owner (allocates all 512 columns) and MMA issuer
//               (one thread): 4 x tcgen05.mma M=128 N=256 K=16 per k-block,
//               alternating between two 256-column TMEM accumulators, one
//               accumulator per 1024-deep K chunk
//   warps 2..9  epilogue: each (TMEM lane quadrant, column half) pair drains
//               its 32 rows x 128 columns per chunk with tcgen05.ld, keeps the
//               int32 sums in registers and, after the last chunk, applies the
//               epilogue and stores
// Tiles are (expert, 128-row block, 256-column block), enumerated from the
// per-expert m-block schedule computed on the device, column block fastest so
// that the CTAs in flight share the same rows of A and the same expert's
// weights in L2.  Rows past an expert's end are computed and never stored.
// Every wait is bounded: after about two seconds a wait gives up, sets
// MOE_DEV_TIMEOUT in the status word and the CTA drains and exits.
#include "common.cuh"
#include "tcgen05.cuh"

#include <cuda.h>
#include <cudaTypedefs.h>

namespace moe {
namespace {

using namespace tc;

constexpr int BM = kGemmBM;          // 128
constexpr int BN = kGemmBN;          // 256
#ifndef MOE_GEMM_BK
#define MOE_GEMM_BK 64
#endif
// k-block depth: 64 fp16 (128-byte rows, 128-byte swizzle, 4 stages of 48 KB)
// or 32 fp16 (64-byte rows, 64-byte swizzle, 9 stages of 24 KB)
constexpr int BK = MOE_GEMM_BK;
static_assert(BK == 64 || BK == 32, "k-block depth");
constexpr int STAGES = BK == 64 ? 4 : 9;
constexpr int A_BYTES = BM * BK * 2;
constexpr int B_BYTES = BN * BK * 2;
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int CHUNK_KB = 1024 / BK;  // 1024-deep exact chunk
constexpr int EPI_WARPS = 8;
constexpr int THREADS = 64 + 32 * EPI_WARPS;
constexpr uint32_t TMEM_COLS = 512;
constexpr size_t kBarrierBytes = 512;
constexpr size_t SMEM_BYTES = (size_t)STAGES * STAGE_BYTES + 1024 + kBarrierBytes +
                              2 * (kMaxExperts + 1) * sizeof(int32_t);
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// The CTA-pair variant: a 256 x 256 tile per cluster of two CTAs; each CTA
// stages its 128 rows of A and its 128 of the 256 weight rows (16 + 16 KB)
// per k-block, so six stages fit.
constexpr int P_STAGES = BK == 64 ? 6 : 12;
constexpr int P_B_BYTES = (BN / 2) * BK * 2;
constexpr int P_STAGE_BYTES = A_BYTES + P_B_BYTES;
constexpr size_t P_RING_BYTES = (size_t)P_STAGES * P_STAGE_BYTES;
constexpr size_t P_SMEM_BYTES = P_RING_BYTES + 1024 + kBarrierBytes +
                                2 * (kMaxExperts + 1) * sizeof(int32_t);
static_assert(P_SMEM_BYTES <= 232448, "shared memory budget");
static_assert((2 * P_STAGES + 5) * 8 + 16 <= (int)kBarrierBytes, "barriers");

// Shared-memory descriptor of a K-major tile with BK-element rows: 128-byte
// rows with the 128-byte swizzle, or 64-byte rows with the 64-byte swizzle
// (8-row groups 1024 or 512 bytes apart).
__device__ __forceinline__ uint64_t desc_k(uint32_t saddr) {
    if (BK == 64) return desc_sw128(saddr);
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);        // start address
    d |= (uint64_t)1 << 16;                          // leading byte offset (unused here)
    d |= (uint64_t)(512 >> 4) << 32;                 // stride byte offset: 8 rows x 64 B
    d |= (uint64_t)1 << 46;                          // descriptor version
    d |= (uint64_t)4 << 61;                          // swizzle: 64 B
    return d;
}
constexpr CUtensorMapSwizzle kTileSwizzle =
    BK == 64 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B;

struct GemmDev {
    const int32_t *offsets;
    const int32_t *sched;
    int E;
    int n_blocks;
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
    int y_vec32;        // y rows start on 32-byte boundaries: 32-byte stores
};

// One 32-byte store (eight 32-bit words) to a 32-byte aligned global address.
__device__ __forceinline__ void st_global_v8(void *p, uint32_t a, uint32_t b, uint32_t c,
                                             uint32_t d, uint32_t e, uint32_t f, uint32_t g,
                                             uint32_t h) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(a),
                 "r"(b), "r"(c), "r"(d), "r"(e), "r"(f), "r"(g), "r"(h)
                 : "memory");
}

struct Tile {
    int e, row0, rows, nb;
};

// Expert-major, then column-block-major order: expert e owns tiles
// [blk[e] * n_blocks, blk[e + 1] * n_blocks), where blk[e] counts the row
// blocks (of `rows_per_block` rows) of the experts before e, and walks every
// row block of one weight column block before the next column block.  The
// CTAs in flight then share few weight tiles, each read by all of the
// expert's row blocks while it is in L2, and the expert's rows stay in L2
// across its column blocks.  Returns the expert, the block's first row, its
// row count past row0 (may exceed the block; clipped by the caller) and the
// column block.
__device__ __forceinline__ Tile decode_tile_nmajor(int64_t tile, int n_blocks, int E,
                                                   const int32_t *s_blk, const int32_t *s_off,
                                                   int rows_per_block) {
    Tile t;
    int lo = 0, hi = E - 1;
    while (lo < hi) {   // last expert whose first tile is <= tile
        const int mid = (lo + hi + 1) >> 1;
        if ((int64_t)s_blk[mid] * n_blocks <= tile) lo = mid; else hi = mid - 1;
    }
    const int nm = s_blk[lo + 1] - s_blk[lo];   // >= 1: an expert with no rows owns no tile
    const int64_t local = tile - (int64_t)s_blk[lo] * n_blocks;
    t.e = lo;
    t.nb = (int)(local / nm);
    t.row0 = s_off[lo] + (int)(local % nm) * rows_per_block;
    t.rows = s_off[lo + 1] - t.row0;
    return t;
}

// ---------------------------------------------------------------- epilogues
// acc[i] is the exact int32 sum for row `row` and tile column hf*128 + i.
template <int EPI>
__device__ __forceinline__ void epilogue_store(const GemmDev &p, const Tile &t, int row, int hf,
                                               const int32_t (&acc)[128]) {
    if (EPI == (int)Epi::S32) {
        const int c0 = t.nb * BN + hf * 128;
        int4 *dst = reinterpret_cast<int4 *>(p.c_s32 + (int64_t)row * p.Nout + c0);
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (c0 + 4 * i < p.Nout)
                dst[i] = make_int4(acc[4 * i], acc[4 * i + 1], acc[4 * i + 2], acc[4 * i + 3]);
    } else if (EPI == (int)Epi::SwiGLU) {
        // packed columns hf*128 + [0, 64) are SiLU-half channels j0 + cc and
        // hf*128 + [64, 128) their multiplier channels Nh + j0 + cc.
        const int Nh = p.Nout / 2;
        const int j0 = t.nb * 128 + hf * 64;
        const float s1 = p.s1[row];
        const float *sc_a = p.scale1 + (int64_t)t.e * p.Nout + j0;
        const float *sc_b = sc_a + Nh;
        float4 *dst = reinterpret_cast<float4 *>(p.g + (int64_t)row * Nh + j0);
#pragma unroll
        for (int i = 0; i < 16; ++i) {
            const float4 sa = __ldg(reinterpret_cast<const float4 *>(sc_a) + i);
            const float4 sb = __ldg(reinterpret_cast<const float4 *>(sc_b) + i);
            const float sav[4] = {sa.x, sa.y, sa.z, sa.w};
            const float sbv[4] = {sb.x, sb.y, sb.z, sb.w};
            float o[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const int cc = 4 * i + u;
                float ha = __fmul_rn(__fmul_rn(__int2float_rn(acc[cc]), sav[u]), s1);
                float hb = __fmul_rn(__fmul_rn(__int2float_rn(acc[64 + cc]), sbv[u]), s1);
                o[u] = __fmul_rn(silu_f32(ha), hb);
            }
            dst[i] = make_float4(o[0], o[1], o[2], o[3]);
        }
    } else {
        const int c0 = t.nb * BN + hf * 128;
        const float s2 = p.s2[row];
        const float *sc = p.scale2 + (int64_t)t.e * p.Nout + c0;
        __nv_bfloat16 *dst = p.y + (int64_t)row * p.Nout + c0;
        // bf16 of (acc * scale2) * s2 for tile columns 8i .. 8i + 7, as four words
        auto dequant8 = [&](int i, uint32_t (&w)[4]) {
            const float4 sa = __ldg(reinterpret_cast<const float4 *>(sc) + 2 * i);
            const float4 sb = __ldg(reinterpret_cast<const float4 *>(sc) + 2 * i + 1);
            const float sv[8] = {sa.x, sa.y, sa.z, sa.w, sb.x, sb.y, sb.z, sb.w};
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                float lo = __fmul_rn(__fmul_rn(__int2float_rn(acc[8 * i + 2 * u]), sv[2 * u]), s2);
                float hi = __fmul_rn(__fmul_rn(__int2float_rn(acc[8 * i + 2 * u + 1]), sv[2 * u + 1]), s2);
                w[u] = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(lo)) |
                       ((uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(hi)) << 16);
            }
        };
        if (p.y_vec32 && c0 + 128 <= p.Nout) {
            // y rows start on 32-byte boundaries and c0 is a multiple of 128
#pragma unroll
            for (int i = 0; i < 16; i += 2) {
                uint32_t a[4], b[4];
                dequant8(i, a);
                dequant8(i + 1, b);
                st_global_v8(dst + 8 * i, a[0], a[1], a[2], a[3], b[0], b[1], b[2], b[3]);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 16; ++i) {
                if (c0 + 8 * i < p.Nout) {
                    uint32_t w[4];
                    dequant8(i, w);
                    reinterpret_cast<uint4 *>(dst)[i] = make_uint4(w[0], w[1], w[2], w[3]);
                }
            }
        }
    }
}

// ---------------------------------------------------------------- the kernel
template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
k_grouped_gemm(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
               GemmDev p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)STAGES * STAGE_BYTES);
    uint64_t *empty = full + STAGES;
    uint64_t *acc_full = empty + STAGES;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int32_t *s_sched = reinterpret_cast<int32_t *>(smem + (size_t)STAGES * STAGE_BYTES + kBarrierBytes);
    int32_t *s_off = s_sched + (kMaxExperts + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], 1);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], EPI_WARPS);
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    }
    pdl_wait();   // everything below may read what earlier kernels wrote
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) {
        s_sched[i] = p.sched[i];
        s_off[i] = p.offsets[i];
    }
    if (warp == 1) {
        tmem_alloc(tmem_slot, TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t total_tiles = (int64_t)s_sched[p.E] * p.n_blocks;
    const int num_chunks = (p.num_kb + CHUNK_KB - 1) / CHUNK_KB;

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer
            int stage = 0;
            uint32_t phase = 0;
            int issued_phase[STAGES];
#pragma unroll
            for (int s = 0; s < STAGES; ++s) issued_phase[s] = -1;
            for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
                Tile t = decode_tile_nmajor(tile, p.n_blocks, p.E, s_sched, s_off, BM);
                t.rows = min(t.rows, BM);
                bool ok = true;
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    uint8_t *sa = smem + (size_t)stage * STAGE_BYTES;
                    mbar_arrive_expect_tx(&full[stage], STAGE_BYTES);
                    tma_load_2d(sa, &tmA, &full[stage], kb * BK, t.row0);
                    tma_load_3d(sa + A_BYTES, &tmB, &full[stage], kb * BK, t.nb * BN, t.e);
                    issued_phase[stage] = (int)phase;
                    if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                }
                if (!ok) break;
            }
            // every issued load must have landed before the CTA may exit
            for (int s = 0; s < STAGES; ++s)
                if (issued_phase[s] >= 0)
                    wait_bounded(&full[s], (uint32_t)issued_phase[s], abort_flag, p.status, false);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            // ------------------------------------------------ MMA issuer
            constexpr uint32_t idesc = idesc_f16(BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int accb = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t tile = blockIdx.x; ok && tile < total_tiles; tile += gridDim.x) {
                for (int kb0 = 0; ok && kb0 < p.num_kb; kb0 += CHUNK_KB) {
                    if (!wait_bounded(&acc_empty[accb], acc_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(accb * BN);
                    const int kb1 = min(kb0 + CHUNK_KB, p.num_kb);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!wait_bounded(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + (size_t)stage * STAGE_BYTES);
                        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k) {
                            mma_f16(d_tmem, desc_k(a_addr + 32 * k), desc_k(b_addr + 32 * k),
                                    idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        }
                        mma_commit(&empty[stage]);
                        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    mma_commit(&acc_full[accb]);
                    if (++accb == 2) { accb = 0; acc_phase ^= 1u; }
                }
            }
            // no MMA may still be running when TMEM is released
            mma_commit(drain);
            wait_bounded(drain, 0, abort_flag, p.status, false);
        }
    } else {
        // ---------------------------------------------------- epilogue warps
        const int q = warp & 3;              // TMEM lane quadrant this warp may read
        const int hf = (warp - 2) >> 2;      // column half of the tile
        const int rloc = q * 32 + lane;
        int accb = 0;
        uint32_t acc_phase = 0;
        for (int64_t tile = blockIdx.x; tile < total_tiles; tile += gridDim.x) {
            Tile t = decode_tile_nmajor(tile, p.n_blocks, p.E, s_sched, s_off, BM);
            t.rows = min(t.rows, BM);
            int32_t acc[128];
            bool ok = true;
            for (int c = 0; c < num_chunks; ++c) {
                bool w = wait_bounded(&acc_full[accb], acc_phase, abort_flag, p.status);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                tc_fence_after();
                const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                                       (uint32_t)(accb * BN + hf * 128);
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    uint32_t r[32];
                    tmem_ld32(taddr + 32 * j, r);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int v = __float2int_rn(__uint_as_float(r[i]));
                        acc[32 * j + i] = (c == 0) ? v : acc[32 * j + i] + v;
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[accb]);
                if (++accb == 2) { accb = 0; acc_phase ^= 1u; }
            }
            if (!ok) break;
            if (rloc < t.rows && (int64_t)t.row0 + rloc < p.cap_rows)
                epilogue_store<EPI>(p, t, t.row0 + rloc, hf, acc);
        }
    }

    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------- CTA-pair variant
struct PairTile {
    int e, row0, rows, nb;   // row0/rows: this CTA's 128-row half (rows may be <= 0)
};

// This CTA's half of pair tile `tile` (decode_tile_nmajor's order over
// 256-row blocks).
__device__ __forceinline__ PairTile decode_pair_tile(int64_t tile, int n_blocks, int E,
                                                     const int32_t *s_psched, const int32_t *s_off,
                                                     uint32_t rank) {
    const Tile b = decode_tile_nmajor(tile, n_blocks, E, s_psched, s_off, 2 * BM);
    PairTile t;
    t.e = b.e;
    t.nb = b.nb;
    t.row0 = b.row0 + (int)rank * BM;
    t.rows = min(BM, b.rows - (int)rank * BM);
    return t;
}

// Clusters of two CTAs (ranks 0 and 1, on two SMs).  Per 256-row x 256-column
// tile, CTA r loads rows [128 r, 128 r + 128) of the tile's A and weight rows
// [128 r, 128 r + 128) of its B; one thread of CTA 0 issues M = 256, N = 256
// MMAs over both CTAs' halves, and each CTA's TMEM receives its own 128 rows of
// the accumulator, which its own epilogue warps drain as in k_grouped_gemm.
// Per SM, a k-block moves 32 KB of operands for the same arithmetic that
// costs the one-SM kernel 48 KB.
//   warp 0      TMA producer (each CTA, its own halves) into a 6-stage ring.
//               Both CTAs' loads complete on CTA 0's stage barrier (the
//               CTA-pair form of the tensor copy), which CTA 0's producer
//               arms with the bytes of both halves, so one wait covers the
//               whole stage and no thread relays the peer's landing.
//   warp 1      TMEM (pair allocation); CTA 0: MMA issuer
//   warps 2..9  epilogue; their accumulator-free signal goes to CTA 0
// Commits arrive on both CTAs' barriers (multicast).  Waits acquire at CTA
// scope and the epilogue's accumulator-free arrivals release at CTA scope:
// the barriers order tensor-memory and shared-memory use, which the tcgen05
// fences and the copies' transaction counts cover, and a cluster-scope release
// would stall each arrival behind the warp's outstanding output stores.  Every
// wait is bounded; both CTAs meet at a cluster barrier before either frees
// TMEM or exits.
template <int EPI>
__global__ void __launch_bounds__(THREADS, 1)
k_grouped_gemm_pair(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                    GemmDev p) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~(uintptr_t)1023);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + P_RING_BYTES);   // used in CTA 0
    uint64_t *empty = full + P_STAGES;
    uint64_t *acc_full = empty + P_STAGES;
    uint64_t *acc_empty = acc_full + 2;                                   // used in CTA 0
    uint64_t *drain = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(drain + 1);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    int32_t *s_off = reinterpret_cast<int32_t *>(smem + P_RING_BYTES + kBarrierBytes);
    int32_t *s_psched = s_off + (kMaxExperts + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < P_STAGES; ++s) {
            mbar_init(&full[s], 1);        // CTA 0's producer arms it with both halves' bytes
            mbar_init(&empty[s], 1);       // one commit per stage use
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(&acc_full[b], 1);
            mbar_init(&acc_empty[b], 2 * EPI_WARPS);   // both CTAs' epilogue warps
        }
        mbar_init(drain, 1);
        *abort_flag = 0;
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    if (warp == 0 && lane == 0) {
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmA) : "memory");
        asm volatile("prefetch.tensormap [%0];" ::"l"(&tmB) : "memory");
    }
    pdl_wait();   // everything below may read what earlier kernels wrote
    for (int i = threadIdx.x; i <= p.E; i += blockDim.x) s_off[i] = p.offsets[i];
    __syncthreads();
    if (warp == 0) {
        // s_psched[e] = 256-row blocks of the experts before e (warp scan)
        int carry = 0;
        for (int base = 0; base < p.E; base += 32) {
            const int e = base + lane;
            const int c = e < p.E ? (s_off[e + 1] - s_off[e] + 2 * BM - 1) / (2 * BM) : 0;
            int x = c;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, d);
                if (lane >= d) x += y;
            }
            if (e < p.E) s_psched[e] = carry + x - c;
            carry += __shfl_sync(0xffffffffu, x, 31);
        }
        if (lane == 0) s_psched[p.E] = carry;
    }
    if (warp == 1) {
        tmem_alloc_pair(tmem_slot, TMEM_COLS);
        tmem_relinquish_pair();
    }
    tc_fence_before();
    __syncthreads();
    cluster_sync();   // both CTAs' barriers and TMEM exist before any cross-CTA use
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    const int64_t total_tiles = (int64_t)s_psched[p.E] * p.n_blocks;
    const int num_chunks = (p.num_kb + CHUNK_KB - 1) / CHUNK_KB;
    const int64_t first = blockIdx.x >> 1, step = gridDim.x >> 1;   // cluster index and count

    if (warp == 0) {
        if (lane == 0) {
            // ------------------------------------------------ TMA producer (both CTAs)
            const uint32_t full0 = cluster_addr(full, 0);   // CTA 0's full[0]
            int stage = 0;
            uint32_t phase = 0;
            int armed_phase[P_STAGES];
#pragma unroll
            for (int s = 0; s < P_STAGES; ++s) armed_phase[s] = -1;
            bool ok = true;
            for (int64_t tile = first; ok && tile < total_tiles; tile += step) {
                const PairTile t = decode_pair_tile(tile, p.n_blocks, p.E, s_psched, s_off, rank);
                for (int kb = 0; kb < p.num_kb; ++kb) {
                    // freed by CTA 0's commit once the MMAs have read both halves
                    if (!wait_bounded(&empty[stage], phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    uint8_t *sa = smem + (size_t)stage * P_STAGE_BYTES;
                    if (leader) {
                        mbar_arrive_expect_tx(&full[stage], 2 * P_STAGE_BYTES);
                        armed_phase[stage] = (int)phase;
                    }
                    // rows past this CTA's half (or past the buffer) only reach
                    // accumulator rows that are never stored
                    const uint32_t fb = full0 + (uint32_t)(stage * sizeof(uint64_t));
                    tma_load_2d_pair(sa, &tmA, fb, kb * BK, t.row0);
                    tma_load_3d_pair(sa + A_BYTES, &tmB, fb, kb * BK,
                                     t.nb * BN + (int)rank * (BN / 2), t.e);
                    if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
                }
            }
            if (leader) {
                // every armed stage must have landed (both CTAs' halves) before exit
                for (int s = 0; s < P_STAGES; ++s)
                    if (armed_phase[s] >= 0)
                        wait_bounded(&full[s], (uint32_t)armed_phase[s], abort_flag, p.status, false);
            } else if (!ok) {
                // the peer's loads complete on CTA 0's barriers; after a give-up,
                // leave the copies still in flight time to land before exit
                const uint64_t t0 = globaltimer();
                while (globaltimer() - t0 < 100000ull) __nanosleep(2000);
            }
        }
    } else if (warp == 1) {
        if (lane == 0 && leader) {
            // ------------------------------------------------ MMA issuer (CTA 0)
            constexpr uint32_t idesc = idesc_f16(2 * BM, BN);
            int stage = 0;
            uint32_t phase = 0;
            int accb = 0;
            uint32_t acc_phase = 0;
            bool ok = true;
            for (int64_t tile = first; ok && tile < total_tiles; tile += step) {
                for (int kb0 = 0; ok && kb0 < p.num_kb; kb0 += CHUNK_KB) {
                    if (!wait_bounded(&acc_empty[accb], acc_phase ^ 1u, abort_flag, p.status)) { ok = false; break; }
                    tc_fence_after();
                    const uint32_t d_tmem = tmem_base + (uint32_t)(accb * BN);
                    const int kb1 = min(kb0 + CHUNK_KB, p.num_kb);
                    for (int kb = kb0; kb < kb1; ++kb) {
                        if (!wait_bounded(&full[stage], phase, abort_flag, p.status)) { ok = false; break; }
                        tc_fence_after();
                        const uint32_t a_addr = smem_u32(smem + (size_t)stage * P_STAGE_BYTES);
                        const uint32_t b_addr = a_addr + A_BYTES;
#pragma unroll
                        for (int k = 0; k < BK / 16; ++k)
                            mma_f16_pair(d_tmem, desc_k(a_addr + 32 * k), desc_k(b_addr + 32 * k),
                                         idesc, (kb > kb0 || k > 0) ? 1u : 0u);
                        mma_commit_pair(&empty[stage], 0x3);
                        if (++stage == P_STAGES) { stage = 0; phase ^= 1u; }
                    }
                    if (!ok) break;
                    mma_commit_pair(&acc_full[accb], 0x3);
                    if (++accb == 2) { accb = 0; acc_phase ^= 1u; }
                }
            }
            // no MMA may still be running when either CTA frees TMEM or exits
            mma_commit_pair(drain, 0x1);
            wait_bounded(drain, 0, abort_flag, p.status, false);
        }
    } else {
        // ---------------------------------------------------- epilogue warps (both CTAs)
        const int q = warp & 3;
        const int hf = (warp - 2) >> 2;
        const int rloc = q * 32 + lane;
        int accb = 0;
        uint32_t acc_phase = 0;
        for (int64_t tile = first; tile < total_tiles; tile += step) {
            const PairTile t = decode_pair_tile(tile, p.n_blocks, p.E, s_psched, s_off, rank);
            const bool rows_here = q * 32 < t.rows;   // warp-uniform
            int32_t acc[128];
            bool ok = true;
            for (int c = 0; c < num_chunks; ++c) {
                const bool w = wait_bounded(&acc_full[accb], acc_phase, abort_flag, p.status);
                if (!__all_sync(0xffffffffu, w)) { ok = false; break; }
                tc_fence_after();
                if (rows_here) {
                    const uint32_t taddr = tmem_base + ((uint32_t)(q * 32) << 16) +
                                           (uint32_t)(accb * BN + hf * 128);
#pragma unroll
                    for (int j = 0; j < 4; ++j) {
                        uint32_t r[32];
                        tmem_ld32(taddr + 32 * j, r);
                        tmem_ld_wait();
#pragma unroll
                        for (int i = 0; i < 32; ++i) {
                            const int v = __float2int_rn(__uint_as_float(r[i]));
                            acc[32 * j + i] = (c == 0) ? v : acc[32 * j + i] + v;
                        }
                    }
                }
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive_remote(&acc_empty[accb], 0);
                if (++accb == 2) { accb = 0; acc_phase ^= 1u; }
            }
            if (!ok) break;
            if (rows_here && rloc < t.rows && (int64_t)t.row0 + rloc < p.cap_rows) {
                Tile et;
                et.e = t.e;
                et.row0 = t.row0;
                et.rows = t.rows;
                et.nb = t.nb;
                epilogue_store<EPI>(p, et, t.row0 + rloc, hf, acc);
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    cluster_sync();
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem_base, TMEM_COLS);
}

// ---------------------------------------------------------------- host side
template <int EPI>
moe_status launch_epi(const CUtensorMap &ma, const CUtensorMap &mb, const GemmDev &d,
                      cudaStream_t stream) {
    if (!set_smem_limit((const void *)k_grouped_gemm<EPI>, SMEM_BYTES)) return MOE_ERR_CUDA;
    const char *names[3] = {"gemm_s32", "gemm1_swiglu", "gemm2_dequant"};
    MOE_LAUNCH(names[EPI], k_grouped_gemm<EPI>, num_sms(), THREADS, SMEM_BYTES, stream, ma, mb, d);
    return MOE_OK;
}

// Clusters of the pair kernel that fit on the GPU at once (0 if it cannot run);
// the persistent grid is twice that.
template <int EPI>
int pair_clusters() {
    static int cached = -1;
    if (cached < 0) {
        cached = 0;
        if (cudaFuncSetAttribute(k_grouped_gemm_pair<EPI>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 (int)P_SMEM_BYTES) != cudaSuccess) {
            cudaGetLastError();
            return cached;
        }
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3((unsigned)(num_sms() & ~1));
        cfg.blockDim = dim3(THREADS);
        cfg.dynamicSmemBytes = P_SMEM_BYTES;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = 2;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, (const void *)k_grouped_gemm_pair<EPI>, &cfg) !=
            cudaSuccess) {
            cudaGetLastError();
            n = 0;
        }
        cached = n;
    }
    return cached;
}

template <int EPI>
moe_status launch_epi_pair(const CUtensorMap &ma, const CUtensorMap &mb, const GemmDev &d,
                           int clusters, cudaStream_t stream) {
    const char *names[3] = {"gemm_s32_pair", "gemm1_swiglu_pair", "gemm2_dequant_pair"};
    MOE_LAUNCH_CLUSTER(names[EPI], k_grouped_gemm_pair<EPI>, 2 * clusters, THREADS, P_SMEM_BYTES,
                       stream, 2u, ma, mb, d);
    return MOE_OK;
}

GemmDev gemm_dev(const GemmArgs &a) {
    GemmDev d;
    d.offsets = a.offsets;
    d.sched = a.sched;
    d.E = (int)a.E;
    d.n_blocks = (int)((a.Nout + BN - 1) / BN);
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
    // 32-byte stores need every y row to start on a 32-byte boundary
    d.y_vec32 = a.y != nullptr && ((uintptr_t)a.y % 32) == 0 && ((a.Nout * 2) % 32) == 0;
    return d;
}

}  // namespace

bool make_tensor_map(CUtensorMap *m, CUtensorMapDataType dtype, CUtensorMapSwizzle swizzle,
                     const void *base, int rank, const uint64_t *dims,
                     const uint64_t *strides_bytes, const uint32_t *box) {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    }
    if (!fn) return false;
    cuuint64_t d[3], s[2];
    cuuint32_t b[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) { d[i] = dims[i]; b[i] = box[i]; }
    for (int i = 0; i < rank - 1; ++i) s[i] = strides_bytes[i];
    CUresult r = fn(m, dtype, (cuuint32_t)rank, const_cast<void *>(base), d, s, b, es,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

template <int EPI>
moe_status launch_pair_or_single(const GemmArgs &a, cudaStream_t stream, bool pair) {
    CUtensorMap ma, mb;
    const int clusters = pair ? pair_clusters<EPI>() : 0;
    const uint64_t adims[2] = {(uint64_t)a.Kd, (uint64_t)a.cap_rows};
    const uint64_t astr[1] = {(uint64_t)a.Kd * 2};
    const uint32_t abox[2] = {BK, BM};
    const uint64_t bdims[3] = {(uint64_t)a.Kd, (uint64_t)a.Nout, (uint64_t)a.E};
    const uint64_t bstr[2] = {(uint64_t)a.Kd * 2, (uint64_t)a.Kd * a.Nout * 2};
    const uint32_t bbox[3] = {BK, clusters > 0 ? (uint32_t)(BN / 2) : (uint32_t)BN, 1};
    if (!make_tensor_map(&ma, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kTileSwizzle, a.a_img, 2, adims,
                         astr, abox))
        return MOE_ERR_CUDA;
    if (!make_tensor_map(&mb, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, kTileSwizzle, a.b_img, 3, bdims,
                         bstr, bbox))
        return MOE_ERR_CUDA;
    const GemmDev d = gemm_dev(a);
    if (clusters > 0) return launch_epi_pair<EPI>(ma, mb, d, clusters, stream);
    return launch_epi<EPI>(ma, mb, d, stream);
}

moe_status launch_grouped_gemm(Epi epi, const GemmArgs &a, cudaStream_t stream, bool pair) {
    if (a.cap_rows <= 0 || a.E <= 0) return MOE_OK;
    switch (epi) {
        case Epi::S32: return launch_pair_or_single<(int)Epi::S32>(a, stream, pair);
        case Epi::SwiGLU: return launch_pair_or_single<(int)Epi::SwiGLU>(a, stream, pair);
        case Epi::DequantBF16: return launch_pair_or_single<(int)Epi::DequantBF16>(a, stream, pair);
    }
    return MOE_ERR_PARAM_INVALID;
}

}  // namespace moe
