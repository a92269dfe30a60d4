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
// GB300 design: the work item is one part (at most 512 16-byte vectors, i.e.
// half of a 7168-wide row) of one token, so a 2048-token batch has 4096 items
// and the last wave is short.  A CTA of 256 threads takes one item at a time:
// threads 0..K-1 fetch the token's route rows and probabilities into shared
// memory, then every thread issues the loads of its two vectors of ALL active
// rows (and of the shared-expert row) before it accumulates them in slot
// order, so 8 rows x 7 KB per CTA, two CTAs per SM, are in flight at once.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;
constexpr int kSlots = 2;                          // 16-byte vectors per thread per row
constexpr int kPartVecs = kThreads * kSlots;       // vectors per work item
constexpr int kRowsInFlight = 8;                   // rows loaded before accumulating

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
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

__global__ void __launch_bounds__(kThreads, 2)
k_combine(const uint4 *__restrict__ y, const int32_t *__restrict__ route_row,
          const float *__restrict__ probs, const uint8_t *__restrict__ mask, int mask_kind,
          const uint4 *__restrict__ shared, uint4 *__restrict__ out, int64_t T, int K, int64_t H8,
          int64_t cap_rows, int nparts) {
    __shared__ int32_t rows_s[kMaxTopK];
    __shared__ float ps_s[kMaxTopK];
    pdl_wait();
    const int64_t items = T * nparts;
    const int64_t per = (H8 + nparts - 1) / nparts;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t t = it / nparts;
        const int64_t v0 = (it % nparts) * per;
        const int64_t v1 = min(v0 + per, H8);
        __syncthreads();
        if (threadIdx.x < K) {
            const int k = threadIdx.x;
            const int32_t r = route_row[t * K + k];
            bool on = r >= 0 && r < cap_rows;
            if (mask_kind == 1) on = on && mask[t] != 0;
            if (mask_kind == 2) on = on && mask[t * K + k] != 0;
            rows_s[k] = on ? r : -1;
            ps_s[k] = probs[t * K + k];
        }
        __syncthreads();
        float acc[kSlots][8];
#pragma unroll
        for (int u = 0; u < kSlots; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
        // the shared-expert vectors are requested together with the rows
        uint4 sv[kSlots];
#pragma unroll
        for (int u = 0; u < kSlots; ++u) {
            const int64_t j = v0 + threadIdx.x + (int64_t)u * kThreads;
            sv[u] = make_uint4(0, 0, 0, 0);
            if (shared && j < v1) sv[u] = ld_stream(shared + t * H8 + j);
        }
        for (int kb = 0; kb < K; kb += kRowsInFlight) {
            uint4 v[kRowsInFlight][kSlots];
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q) {
                const int k = kb + q;
                const int32_t r = (k < K) ? rows_s[k] : -1;
#pragma unroll
                for (int u = 0; u < kSlots; ++u) {
                    const int64_t j = v0 + threadIdx.x + (int64_t)u * kThreads;
                    v[q][u] = make_uint4(0, 0, 0, 0);
                    if (r >= 0 && j < v1) v[q][u] = ld_stream(y + (int64_t)r * H8 + j);
                }
            }
#pragma unroll
            for (int q = 0; q < kRowsInFlight; ++q) {
                const int k = kb + q;
                if (k >= K || rows_s[k] < 0) continue;
                const float p = ps_s[k];
#pragma unroll
                for (int u = 0; u < kSlots; ++u) {
                    float f[8];
                    unpack8(v[q][u], f);
#pragma unroll
                    for (int i = 0; i < 8; ++i) acc[u][i] = __fadd_rn(acc[u][i], __fmul_rn(p, f[i]));
                }
            }
        }
#pragma unroll
        for (int u = 0; u < kSlots; ++u) {
            const int64_t j = v0 + threadIdx.x + (int64_t)u * kThreads;
            if (j >= v1) continue;
            if (shared) {
                float f[8];
                unpack8(sv[u], f);
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[u][i] = __fadd_rn(acc[u][i], f[i]);
            }
            uint4 o;
            o.x = pack_bf16x2(acc[u][0], acc[u][1]);
            o.y = pack_bf16x2(acc[u][2], acc[u][3]);
            o.z = pack_bf16x2(acc[u][4], acc[u][5]);
            o.w = pack_bf16x2(acc[u][6], acc[u][7]);
            out[t * H8 + j] = o;
        }
    }
}

}  // namespace

moe_status launch_combine(const void *y, const int32_t *route_row, const float *probs,
                          const uint8_t *mask, int mask_kind, const void *shared, void *out,
                          int64_t T, int64_t K, int64_t H, int64_t cap_rows, int32_t *status,
                          cudaStream_t stream) {
    (void)status;
    if (T == 0) return MOE_OK;
    const int64_t H8 = H / 8;
    const int nparts = (int)((H8 + kPartVecs - 1) / kPartVecs);
    int64_t grid = (int64_t)num_sms() * 2;
    if (grid > T * nparts) grid = T * nparts;
    MOE_LAUNCH("combine", k_combine, (unsigned)grid, kThreads, 0, stream, (const uint4 *)y,
               route_row, probs, mask, mask_kind, (const uint4 *)shared, (uint4 *)out, T, (int)K,
               H8, cap_rows, nparts);
    return MOE_OK;
}

}  // namespace moe
