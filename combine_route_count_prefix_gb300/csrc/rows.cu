// rows.cu -- the HBM-bound row kernels: dispatch copy, combine, the two
// dynamic quantisations and weight packing.
//
// All of them move whole rows as 16-byte vectors: a CTA takes one row (or one
// token) at a time, every thread loads its slice of the row into registers
// (up to 8 x 16 B), and then writes it once per destination.  H is a multiple
// of 8, so a 16-byte vector never straddles a row.
#include "common.cuh"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {
namespace {

constexpr int kRowThreads = 128;
constexpr int kVec = 8;                 // 16-byte vectors held per thread per pass
constexpr uint32_t kFull = 0xffffffffu;

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_hint(uint4 *p, const uint4 &v, uint64_t policy) {
    asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1,%2,%3,%4}, %5;" ::"l"(p), "r"(v.x),
                 "r"(v.y), "r"(v.z), "r"(v.w), "l"(policy)
                 : "memory");
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float (&f)[8]) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        f[2 * i] = __uint_as_float(w[i] << 16);
        f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
    }
}


__device__ __forceinline__ float block_max(float v, float *scratch /*[32]*/) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    if (lane == 0) scratch[warp] = v;
    __syncthreads();
    float r = scratch[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, scratch[w]);
    __syncthreads();
    return r;
}

// ---------------------------------------------------------------- dispatch copy
// expand_x[route_row[t*K+k]] = x[t] for every active route of token t.
// The rows of tokens t >= keep_from are stored with an L2 evict-last policy
// and the others evict-first: the combine reads tokens from the last one
// down, so the rows it reads first are still in L2 when it starts.
__global__ void __launch_bounds__(kRowThreads)
k_dispatch_rows(RouteDev ra, const uint4 *__restrict__ x, int32_t *__restrict__ route_row,
                int32_t *__restrict__ assist, uint4 *__restrict__ expand_x, int64_t H8,
                int64_t keep_from) {
    __shared__ int32_t rows[kMaxTopK];
    const int64_t T = ra.T;
    const int K = (int)ra.K;
    const uint64_t keep = l2_policy_evict_last(), pass = l2_policy_evict_first();
    uint4 v[kVec];
    auto load_row = [&](int64_t t, int64_t j0) {
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            int64_t j = j0 + (int64_t)u * kRowThreads;
            if (j < H8) v[u] = ld_stream(x + t * H8 + j);
        }
    };
    // The first token's row is loaded before waiting on the routing kernel, so that the
    // read of x overlaps it.  x is not written by anything this grid can overlap: the
    // routing kernel triggers its dependents only after its own wait has returned, i.e.
    // after every earlier kernel of the stream has finished.
    // The mask is an input too, so a token it switches off entirely is not loaded.
    bool preloaded = false;
    if ((int64_t)blockIdx.x < T && H8 <= (int64_t)kRowThreads * kVec) {
        const int64_t t = blockIdx.x;
        bool on = ra.mask_kind != 1 || ra.mask[t] != 0;
        if (ra.mask_kind == 2) {
            on = false;
            for (int k = 0; k < K; ++k) on = on || ra.mask[t * K + k] != 0;
        }
        if (on) {
            load_row(t, threadIdx.x);
            preloaded = true;
        }
    }
    pdl_wait();
    for (int64_t t = blockIdx.x; t < T; t += gridDim.x) {
        __syncthreads();
        if (threadIdx.x < K) rows[threadIdx.x] = resolve_route_row(ra, t, threadIdx.x, route_row, assist);
        __syncthreads();
        bool any = false;
        for (int k = 0; k < K; ++k) any = any || rows[k] >= 0;
        if (!any) {
            preloaded = false;
            continue;
        }
        for (int64_t j0 = threadIdx.x; j0 < H8; j0 += (int64_t)kRowThreads * kVec) {
            if (!preloaded) load_row(t, j0);
            preloaded = false;
            const uint64_t pol = t >= keep_from ? keep : pass;
            for (int k = 0; k < K; ++k) {
                int32_t r = rows[k];
                if (r < 0) continue;
                uint4 *dst = expand_x + (int64_t)r * H8;
#pragma unroll
                for (int u = 0; u < kVec; ++u) {
                    int64_t j = j0 + (int64_t)u * kRowThreads;
                    if (j < H8) st_hint(dst + j, v[u], pol);
                }
            }
        }
    }
}

// ---------------------------------------------------------------- quantisation of bf16 rows
// One source row (bf16, H8 vectors) -> int8 codes stored as fp16 images plus
// the fp32 scale, written to every destination row in rows[0..ndst).
// The whole row stays in registers: H8 <= kRowThreads * kVec (H <= 8192).
template <bool kFromRouteTable>
__global__ void __launch_bounds__(kRowThreads)
k_quant_bf16_rows(RouteDev ra, const uint4 *__restrict__ src, int32_t *__restrict__ route_row,
                  int32_t *__restrict__ assist, const int32_t *__restrict__ offsets, int64_t E,
                  int64_t T, int K, uint4 *__restrict__ q, float *__restrict__ s_out, int64_t H8) {
    __shared__ int32_t rows[kMaxTopK];
    __shared__ int32_t nrows;
    __shared__ float scratch[32];
    pdl_wait();
    // kFromRouteTable: one iteration per token t, destinations = its active routes.
    // otherwise:       one iteration per dispatched row r < offsets[E], destination = r.
    const int64_t n_items = kFromRouteTable ? T : min((int64_t)offsets[E], T);
    for (int64_t it = blockIdx.x; it < n_items; it += gridDim.x) {
        __syncthreads();
        if (kFromRouteTable) {
            // lane k resolves slot k; the active rows are packed in slot order
            if (threadIdx.x < 32) {
                const int k = threadIdx.x;
                const int32_t r = k < K ? resolve_route_row(ra, it, k, route_row, assist) : -1;
                const uint32_t act = __ballot_sync(kFull, r >= 0);
                if (r >= 0) rows[__popc(act & lanemask_lt())] = r;
                if (k == 0) nrows = __popc(act);
            }
        } else if (threadIdx.x == 0) {
            rows[0] = (int32_t)it;
            nrows = 1;
        }
        __syncthreads();
        const int n = nrows;
        if (n == 0) continue;
        uint4 v[kVec];
        float amax = 0.0f;
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            int64_t j = threadIdx.x + (int64_t)u * kRowThreads;
            v[u] = make_uint4(0, 0, 0, 0);
            if (j < H8) {
                v[u] = ld_stream(src + it * H8 + j);
                float f[8];
                unpack_bf16x8(v[u], f);
#pragma unroll
                for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(f[i]));
            }
        }
        amax = block_max(amax, scratch);
        const float s = __fdiv_rn(amax, 127.0f);
        const float rs = __frcp_rn(s);
        // 8 bf16 in -> 8 fp16 codes out: one 16-byte vector in, one out
        uint4 qv[kVec];
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            float f[8], c[8];
            unpack_bf16x8(v[u], f);
            quant_codes<8>(f, s, rs, c);
            qv[u] = make_uint4(pack_half2(c[0], c[1]), pack_half2(c[2], c[3]),
                               pack_half2(c[4], c[5]), pack_half2(c[6], c[7]));
        }
        for (int d = 0; d < n; ++d) {
            const int64_t r = rows[d];
            uint4 *dst = q + r * H8;
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                int64_t j = threadIdx.x + (int64_t)u * kRowThreads;
                if (j < H8) dst[j] = qv[u];
            }
            if (threadIdx.x == 0) s_out[r] = s;
        }
    }
}

// ---------------------------------------------------------------- quantised dispatch
// Row r of token t and expert e gets the dynamic int8 quantisation of
// float(x[t]) * smooth[e] (kSmooth) or of float(x[t]), as int8 bytes, and its
// scale.  Without smooth scales the token is quantised once and its codes are
// written to every one of its rows.
__device__ __forceinline__ uint2 pack_i8x8(const float (&c)[8]) {
    return make_uint2(pack_i8x4(c[0], c[1], c[2], c[3]), pack_i8x4(c[4], c[5], c[6], c[7]));
}

// The row stays in registers as its raw 16-byte vectors only: each pass
// (amax, then codes) unpacks them again, so a CTA needs about 60 registers a
// thread and eight or more CTAs (tokens) per SM keep their loads in flight.
template <bool kSmooth>
__global__ void __launch_bounds__(kRowThreads, 8)
k_dispatch_quant(RouteDev ra, const uint4 *__restrict__ x, const float4 *__restrict__ smooth,
                 int32_t *__restrict__ route_row, int32_t *__restrict__ assist,
                 uint2 *__restrict__ q, float *__restrict__ s_out, int64_t H8) {
    __shared__ int32_t rows[kMaxTopK];
    __shared__ int32_t experts[kMaxTopK];
    __shared__ int32_t nrows;
    __shared__ float scratch[32];
    const int K = (int)ra.K;
    // The token's row is read before its route rows are resolved, and the first
    // token's before the wait on the routing kernel (x and the mask are inputs
    // nothing in flight writes); a token the mask switches off entirely is not
    // read.  The route rows are resolved by one lane per slot, in parallel.
    uint4 raw[kVec];
    auto load_row = [&](int64_t t) {
        bool on = t < ra.T;
        if (on && ra.mask_kind == 1) on = ra.mask[t] != 0;
        if (on && ra.mask_kind == 2) {
            bool any = false;
            for (int k = 0; k < K; ++k) any = any || ra.mask[t * K + k] != 0;
            on = any;
        }
#pragma unroll
        for (int u = 0; u < kVec; ++u) {
            const int64_t j = threadIdx.x + (int64_t)u * kRowThreads;
            raw[u] = (on && j < H8) ? ld_stream(x + t * H8 + j) : make_uint4(0, 0, 0, 0);
        }
    };
    // v = float(x) (* smooth[e] for the destination expert, one rounded multiply)
    auto values = [&](int u, int64_t j, const float4 *sm, float (&v)[8]) {
        unpack_bf16x8(raw[u], v);
        if (kSmooth) {
            const float4 a = __ldg(sm + j * 2), b = __ldg(sm + j * 2 + 1);
            const float m[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = __fmul_rn(v[i], m[i]);
        }
    };
    // lane k resolves slot k of token t; the active rows are packed in slot order
    auto resolve_rows = [&](int64_t t) {
        if (threadIdx.x < 32) {
            const int k = threadIdx.x;
            const int32_t e = k < K ? ra.ids[t * K + k] : 0;
            const int32_t r = k < K ? resolve_route_row(ra, t, k, route_row, assist) : -1;
            const uint32_t act = __ballot_sync(kFull, r >= 0);
            if (r >= 0) {
                const int pos = __popc(act & lanemask_lt());
                rows[pos] = r;
                experts[pos] = e;
            }
            if (k == 0) nrows = __popc(act);
        }
    };
    if constexpr (!kSmooth) {
        // Every destination gets the token's own codes, which depend on x alone:
        // the first token's scale and codes are computed before the wait on the
        // routing kernel, so only its stores wait for the route rows.
        uint2 codes[kVec];
        float sc = 0.0f;
        auto quantise_token = [&]() {
            float amax = 0.0f;
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int64_t j = threadIdx.x + (int64_t)u * kRowThreads;
                if (j < H8) {
                    float v[8];
                    values(u, j, nullptr, v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
                }
            }
            amax = block_max(amax, scratch);
            sc = __fdiv_rn(amax, 127.0f);
            const float rs = __frcp_rn(sc);
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                float v[8], c[8];
                values(u, 0, nullptr, v);
                quant_codes<8>(v, sc, rs, c);
                codes[u] = pack_i8x8(c);
            }
        };
        load_row(blockIdx.x);
        quantise_token();
        pdl_wait();
        for (int64_t t = blockIdx.x; t < ra.T; t += gridDim.x) {
            if (t != blockIdx.x) {
                load_row(t);
                quantise_token();
            }
            __syncthreads();   // the previous token's rows are no longer read
            resolve_rows(t);
            __syncthreads();
            const int n = nrows;
            for (int d = 0; d < n; ++d) {
                const int64_t r = rows[d];
#pragma unroll
                for (int u = 0; u < kVec; ++u) {
                    const int64_t j = threadIdx.x + (int64_t)u * kRowThreads;
                    if (j < H8) q[r * H8 + j] = codes[u];
                }
                if (threadIdx.x == 0) s_out[r] = sc;
            }
        }
        return;
    }
    load_row(blockIdx.x);
    pdl_wait();
    for (int64_t t = blockIdx.x; t < ra.T; t += gridDim.x) {
        if (t != blockIdx.x) load_row(t);
        __syncthreads();   // the previous token's rows are no longer read
        resolve_rows(t);
        __syncthreads();
        const int n = nrows;
        if (n == 0) continue;
        // without smooth scales every destination gets the token's own codes
        for (int d = 0; d < (kSmooth ? n : 1); ++d) {
            const float4 *sm = kSmooth ? smooth + (int64_t)experts[d] * H8 * 2 : nullptr;
            float amax = 0.0f;
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int64_t j = threadIdx.x + (int64_t)u * kRowThreads;
                if (j < H8) {
                    float v[8];
                    values(u, j, sm, v);
#pragma unroll
                    for (int i = 0; i < 8; ++i) amax = fmaxf(amax, fabsf(v[i]));
                }
            }
            amax = block_max(amax, scratch);
            const float sc = __fdiv_rn(amax, 127.0f);
            const float rs = __frcp_rn(sc);
            const int d0 = kSmooth ? d : 0, d1 = kSmooth ? d + 1 : n;
#pragma unroll
            for (int u = 0; u < kVec; ++u) {
                const int64_t j = threadIdx.x + (int64_t)u * kRowThreads;
                if (j < H8) {
                    float v[8], c[8];
                    values(u, j, sm, v);
                    quant_codes<8>(v, sc, rs, c);
                    const uint2 packed = pack_i8x8(c);
                    for (int dd = d0; dd < d1; ++dd) q[(int64_t)rows[dd] * H8 + j] = packed;
                }
            }
            if (threadIdx.x == 0)
                for (int dd = d0; dd < d1; ++dd) s_out[rows[dd]] = sc;
        }
    }
}

// int8 rows (r < offsets[E]) -> fp16 images for the GEMM, scales copied.
__global__ void k_rows_i8_to_f16(const int4 *__restrict__ src, const float *__restrict__ sc_in,
                                 uint4 *__restrict__ dst, float *__restrict__ sc_out,
                                 const int32_t *__restrict__ offsets, int64_t E, int64_t H16,
                                 int64_t cap_rows) {
    pdl_wait();
    const int64_t R = min((int64_t)offsets[E], cap_rows);
    const int64_t n = R * H16;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int4 in = src[i];
        const int8_t *b = reinterpret_cast<const int8_t *>(&in);
        uint32_t w[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) w[k] = pack_half2((float)b[2 * k], (float)b[2 * k + 1]);
        dst[2 * i] = make_uint4(w[0], w[1], w[2], w[3]);
        dst[2 * i + 1] = make_uint4(w[4], w[5], w[6], w[7]);
        if (i % H16 == 0) sc_out[i / H16] = sc_in[i / H16];
    }
}

// ---------------------------------------------------------------- second quantisation
// g fp32 [rows, Nh] -> q2 fp16 images + s2, for rows r < offsets[E].
// One warp per row: the row's amax is a warp reduction, no block barrier, and
// a CTA keeps 8 rows in flight.  Rows up to 32 * 4 * kQ2Vec floats stay in
// registers; longer rows are read twice (the second read hits L2).
constexpr int kQ2Threads = 256;
constexpr int kQ2Vec = 16;
__global__ void __launch_bounds__(kQ2Threads)
k_quant2(const float4 *__restrict__ g, const int32_t *__restrict__ offsets, int64_t E,
         uint2 *__restrict__ q2, float *__restrict__ s2, int64_t Nh4, int64_t cap_rows) {
    pdl_wait();
    const int lane = threadIdx.x & 31;
    const int64_t R = min((int64_t)offsets[E], cap_rows);
    const int64_t warps = (int64_t)gridDim.x * (kQ2Threads / 32);
    for (int64_t r = blockIdx.x * (int64_t)(kQ2Threads / 32) + (threadIdx.x >> 5); r < R;
         r += warps) {
        const float4 *src = g + r * Nh4;
        uint2 *dst = q2 + r * Nh4;
        float amax = 0.0f;
        if (Nh4 <= 32 * kQ2Vec) {
            float4 v[kQ2Vec];
#pragma unroll
            for (int u = 0; u < kQ2Vec; ++u) {
                const int64_t j = lane + 32 * u;
                v[u] = (j < Nh4) ? __ldcs(src + j) : make_float4(0.f, 0.f, 0.f, 0.f);
            }
#pragma unroll
            for (int u = 0; u < kQ2Vec; ++u)
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v[u].x), fabsf(v[u].y)),
                                         fmaxf(fabsf(v[u].z), fabsf(v[u].w))));
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
            const float s = __fdiv_rn(amax, 127.0f);
            const float rs = __frcp_rn(s);
#pragma unroll
            for (int u = 0; u < kQ2Vec; ++u) {
                const int64_t j = lane + 32 * u;
                if (j < Nh4) {
                    const float a[4] = {v[u].x, v[u].y, v[u].z, v[u].w};
                    float c[4];
                    quant_codes<4>(a, s, rs, c);
                    dst[j] = make_uint2(pack_half2(c[0], c[1]), pack_half2(c[2], c[3]));
                }
            }
            if (lane == 0) s2[r] = s;
        } else {
            for (int64_t j = lane; j < Nh4; j += 32) {
                const float4 v = src[j];
                amax = fmaxf(amax, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
            }
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(kFull, amax, o));
            const float s = __fdiv_rn(amax, 127.0f);
            const float rs = __frcp_rn(s);
            for (int64_t j = lane; j < Nh4; j += 32) {
                const float4 v = src[j];
                const float a[4] = {v.x, v.y, v.z, v.w};
                float c[4];
                quant_codes<4>(a, s, rs, c);
                dst[j] = make_uint2(pack_half2(c[0], c[1]), pack_half2(c[2], c[3]));
            }
            if (lane == 0) s2[r] = s;
        }
    }
}

// ---------------------------------------------------------------- weight packing
// int8 -> fp16 image of the same integer (exact), 16 values per thread.
__device__ __forceinline__ void i8x16_to_f16(const int4 &in, uint4 &lo, uint4 &hi) {
    const int8_t *b = reinterpret_cast<const int8_t *>(&in);
    uint32_t w[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) w[i] = pack_half2((float)b[2 * i], (float)b[2 * i + 1]);
    lo = make_uint4(w[0], w[1], w[2], w[3]);
    hi = make_uint4(w[4], w[5], w[6], w[7]);
}

__global__ void k_i8_to_f16(const int4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n16) {
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x) {
        uint4 lo, hi;
        i8x16_to_f16(src[i], lo, hi);
        dst[2 * i] = lo;
        dst[2 * i + 1] = hi;
    }
}

__global__ void k_i8_to_f16_tail(const int8_t *__restrict__ src, __half *__restrict__ dst,
                                 int64_t start, int64_t n) {
    pdl_wait();
    int64_t i = start + blockIdx.x * (int64_t)blockDim.x + threadIdx.x;
    if (i < n) dst[i] = __float2half_rn((float)src[i]);
}

// W1 [E, N, H] -> packed fp16 [E, N, H] with rows reordered so that packed
// block b (rows 256b .. 256b+255) holds, for half h in {0, 1}:
//   rows 256b + 128h +  0..63 : SiLU-half channels 128b + 64h + (0..63)
//   rows 256b + 128h + 64..127: multiplier channels N/2 + 128b + 64h + (0..63)
// so one 256-column GEMM tile carries 128 complete SwiGLU pairs.
__global__ void k_pack_w1(const int8_t *__restrict__ w1, uint4 *__restrict__ out, int64_t E,
                          int64_t N, int64_t H) {
    pdl_wait();
    const int64_t H16 = H / 16;
    const int64_t total = E * N * H16;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        int64_t col16 = i % H16;
        int64_t prow = (i / H16) % N;
        int64_t e = i / (H16 * N);
        int64_t b = prow / 256, within = prow % 256, h = within / 128, ii = within % 128;
        int64_t src_row = (ii < 64) ? (128 * b + 64 * h + ii) : (N / 2 + 128 * b + 64 * h + (ii - 64));
        int4 in = *reinterpret_cast<const int4 *>(w1 + (e * N + src_row) * H + col16 * 16);
        uint4 lo, hi;
        i8x16_to_f16(in, lo, hi);
        out[2 * i] = lo;
        out[2 * i + 1] = hi;
    }
}

// W1 [E, N, H] -> biased bytes (w + 128) [E, N, H] with rows reordered for the
// small-batch GEMM: packed row 128b + 32q + l (b = 128-channel block, q = TMEM
// lane quadrant) holds
//   l <  16: SiLU-half channel         64b + 16q + l
//   l >= 16: multiplier channel  N/2 + 64b + 16q + (l - 16)
// so the two halves of a SwiGLU pair sit 16 TMEM lanes apart in one warp.
__global__ void k_pack_w1_i8(const int8_t *__restrict__ w1, uint4 *__restrict__ out, int64_t E,
                             int64_t N, int64_t H) {
    pdl_wait();
    const int64_t H16 = H / 16;
    const int64_t total = E * N * H16;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t col16 = i % H16;
        const int64_t prow = (i / H16) % N;
        const int64_t e = i / (H16 * N);
        const int64_t b = prow / 128, qq = (prow % 128) / 32, l = prow % 32;
        const int64_t j = 64 * b + 16 * qq + (l & 15);
        const int64_t src_row = l < 16 ? j : N / 2 + j;
        const uint4 v = *reinterpret_cast<const uint4 *>(w1 + (e * N + src_row) * H + col16 * 16);
        out[i] = make_uint4(v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u,
                            v.w ^ 0x80808080u);
    }
}

// int8 -> biased bytes (w + 128): flipping the sign bit of a two's-complement
// byte adds 128.  n16 = number of 16-byte vectors.
__global__ void k_bias_i8(const uint4 *__restrict__ src, uint4 *__restrict__ dst, int64_t n16) {
    pdl_wait();
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n16;
         i += (int64_t)gridDim.x * blockDim.x) {
        const uint4 v = src[i];
        dst[i] = make_uint4(v.x ^ 0x80808080u, v.y ^ 0x80808080u, v.z ^ 0x80808080u,
                            v.w ^ 0x80808080u);
    }
}

int grid_for(int64_t items, int per_sm) {
    int64_t g = (int64_t)num_sms() * per_sm;
    if (items < g) g = items;
    return (int)(g > 0 ? g : 1);
}

}  // namespace

#ifndef MOE_ROWS_L2_KEEP_MB
#define MOE_ROWS_L2_KEEP_MB 128
#endif
moe_status launch_dispatch_rows(const RouteDev &r, const void *x, int32_t *route_row,
                                int32_t *assist, void *expand_x, int64_t H, cudaStream_t stream) {
    if (r.T == 0) return MOE_OK;
    // the last tokens whose rows (K per token at most) fit the L2 budget
    const int64_t keep_tokens = ((int64_t)MOE_ROWS_L2_KEEP_MB << 20) / (r.K * H * 2);
    const int64_t keep_from = r.T > keep_tokens ? r.T - keep_tokens : 0;
    MOE_LAUNCH("dispatch_rows", k_dispatch_rows, grid_for(r.T, 16), kRowThreads, 0, stream, r,
               (const uint4 *)x, route_row, assist, (uint4 *)expand_x, H / 8, keep_from);
    return MOE_OK;
}

moe_status launch_quant_scatter(const RouteDev &r, const void *x, int32_t *route_row,
                                int32_t *assist, void *q1, float *s1, int64_t H,
                                cudaStream_t stream) {
    if (r.T == 0) return MOE_OK;
    MOE_LAUNCH("quant_scatter", k_quant_bf16_rows<true>, grid_for(r.T, 16), kRowThreads, 0, stream,
               r, (const uint4 *)x, route_row, assist, (const int32_t *)nullptr, (int64_t)0, r.T,
               (int)r.K, (uint4 *)q1, s1, H / 8);
    return MOE_OK;
}

moe_status launch_dispatch_quant(const RouteDev &r, const void *x, const float *smooth,
                                 int32_t *route_row, int32_t *assist, int8_t *q, float *scales,
                                 int64_t H, cudaStream_t stream) {
    if (r.T == 0) return MOE_OK;
    if (smooth) {
        MOE_LAUNCH("dispatch_quant", k_dispatch_quant<true>, grid_for(r.T, 16), kRowThreads, 0,
                   stream, r, (const uint4 *)x, (const float4 *)smooth, route_row, assist,
                   (uint2 *)q, scales, H / 8);
    } else {
        MOE_LAUNCH("dispatch_quant", k_dispatch_quant<false>, grid_for(r.T, 16), kRowThreads, 0,
                   stream, r, (const uint4 *)x, (const float4 *)nullptr, route_row, assist,
                   (uint2 *)q, scales, H / 8);
    }
    return MOE_OK;
}

moe_status launch_rows_i8_to_f16(const int8_t *rows, const float *scales, const int32_t *offsets,
                                 int64_t E, void *q1, float *s1, int64_t cap_rows, int64_t H,
                                 cudaStream_t stream) {
    if (cap_rows == 0) return MOE_OK;
    const int64_t n16 = cap_rows * (H / 16);
    MOE_LAUNCH("rows_i8_to_f16", k_rows_i8_to_f16, grid_for((n16 + 255) / 256, 8), 256, 0, stream,
               (const int4 *)rows, scales, (uint4 *)q1, s1, offsets, E, H / 16, cap_rows);
    return MOE_OK;
}

moe_status launch_quant_rows(const void *x_rows, const int32_t *offsets, int64_t E, void *q1,
                             float *s1, int64_t cap_rows, int64_t H, cudaStream_t stream) {
    if (cap_rows == 0) return MOE_OK;
    // T carries the row capacity here: rows >= cap_rows are never touched
    MOE_LAUNCH("quant_rows", k_quant_bf16_rows<false>, grid_for(cap_rows, 16), kRowThreads, 0,
               stream, RouteDev{}, (const uint4 *)x_rows, (int32_t *)nullptr, (int32_t *)nullptr,
               offsets, E, cap_rows, 1,
               (uint4 *)q1, s1, H / 8);
    return MOE_OK;
}

moe_status launch_quant2(const float *g, const int32_t *offsets, int64_t E, void *q2, float *s2,
                         int64_t cap_rows, int64_t Nh, cudaStream_t stream) {
    if (cap_rows == 0) return MOE_OK;
    MOE_LAUNCH("quant2", k_quant2, grid_for((cap_rows + 7) / 8, 8), kQ2Threads, 0, stream,
               (const float4 *)g, offsets, E, (uint2 *)q2, s2, Nh / 4, cap_rows);
    return MOE_OK;
}

moe_status launch_pack_w1(const int8_t *w1, void *w1p, int64_t E, int64_t N, int64_t H,
                          cudaStream_t stream) {
    int64_t total = E * N * (H / 16);
    if (total == 0) return MOE_OK;
    MOE_LAUNCH("pack_w1", k_pack_w1, grid_for((total + 255) / 256, 8), 256, 0, stream, w1,
               (uint4 *)w1p, E, N, H);
    return MOE_OK;
}

moe_status launch_pack_w1_i8(const int8_t *w1, void *w1p, int64_t E, int64_t N, int64_t H,
                             cudaStream_t stream) {
    int64_t total = E * N * (H / 16);
    if (total == 0) return MOE_OK;
    MOE_LAUNCH("pack_w1_i8", k_pack_w1_i8, grid_for((total + 255) / 256, 8), 256, 0, stream, w1,
               (uint4 *)w1p, E, N, H);
    return MOE_OK;
}

moe_status launch_bias_i8(const int8_t *src, void *dst, int64_t n, cudaStream_t stream) {
    const int64_t n16 = n / 16;   // callers pass multiples of 16
    if (n16 == 0) return MOE_OK;
    MOE_LAUNCH("bias_i8", k_bias_i8, grid_for((n16 + 255) / 256, 8), 256, 0, stream,
               (const uint4 *)src, (uint4 *)dst, n16);
    return MOE_OK;
}

moe_status launch_i8_to_f16(const int8_t *src, void *dst, int64_t n, cudaStream_t stream) {
    int64_t n16 = n / 16;
    if (n16 > 0) {
        MOE_LAUNCH("i8_to_f16", k_i8_to_f16, grid_for((n16 + 255) / 256, 8), 256, 0, stream,
                   (const int4 *)src, (uint4 *)dst, n16);
    }
    int64_t rem = n - n16 * 16;
    if (rem > 0) {
        MOE_LAUNCH("i8_to_f16_tail", k_i8_to_f16_tail, 1, 32, 0, stream, src, (__half *)dst,
                   n16 * 16, n);
    }
    return MOE_OK;
}

}  // namespace moe
