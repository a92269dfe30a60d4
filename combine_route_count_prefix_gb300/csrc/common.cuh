// common.cuh -- shared host/device definitions of the GB300 MoE library.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <stdint.h>
#include <stddef.h>

#include "moe_gb300.h"

namespace moe {

// ---------------------------------------------------------------- limits
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 16;
constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
constexpr int kRouteChunkTokensMax = 256;   // routing chunks never cross a partition
constexpr int kGemmBM = 128;             // GEMM tile rows (routed rows)
constexpr int kGemmBN = 256;             // GEMM tile columns (output channels)
constexpr size_t kAlign = 1024;

inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------- launch bookkeeping
// Every kernel launch goes through launch_begin/launch_end: they count launches
// and, when profiling is on, bracket the launch with a CUDA event pair recorded
// on the launching stream.
int launch_begin(const char *name, cudaStream_t stream, unsigned grid);
// Raises a kernel's dynamic shared-memory limit to at least `bytes`, once per
// kernel and size (thread-safe); false if the runtime refuses.
bool set_smem_limit(const void *kernel, size_t bytes);
void launch_end(int token, cudaStream_t stream);
int num_sms();

// Kernels are launched with programmatic stream serialization: a kernel may
// be scheduled while its predecessor on the stream drains, and waits in
// pdl_wait() (griddepcontrol.wait) before it reads anything the predecessor
// wrote.  Every kernel of this library calls pdl_wait() before its first
// dependent read.
#ifndef MOE_PDL_ATTRS
#define MOE_PDL_ATTRS 1
#endif
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = MOE_PDL_ATTRS;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// The same with a cluster of `cluster_x` CTAs along x (grid.x a multiple of it).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                               cudaStream_t stream, unsigned cluster_x, Args... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster_x;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1 + MOE_PDL_ATTRS;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

#define MOE_LAUNCH(name, kernel, grid, block, smem, stream, ...)                          \
    do {                                                                                  \
        int _tok = ::moe::launch_begin(name, stream, dim3(grid).x);                       \
        cudaError_t _err = ::moe::launch_pdl(kernel, dim3(grid), dim3(block), (smem),     \
                                             (stream), __VA_ARGS__);                      \
        if (_err == cudaSuccess) _err = cudaGetLastError();                               \
        ::moe::launch_end(_tok, stream);                                                  \
        if (_err != cudaSuccess) return MOE_ERR_CUDA;                                     \
    } while (0)

// Waits for the predecessor grid (its writes are visible afterwards), then
// lets the next kernel on the stream be launched: its CTAs are scheduled as
// resources free up and wait in their own pdl_wait, so its launch latency
// overlaps this kernel's execution.
__device__ __forceinline__ void pdl_wait() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

#define MOE_LAUNCH_CLUSTER(name, kernel, grid, block, smem, stream, cluster_x, ...)      \
    do {                                                                                  \
        int _tok = ::moe::launch_begin(name, stream, dim3(grid).x);                       \
        cudaError_t _err = ::moe::launch_pdl_cluster(kernel, dim3(grid), dim3(block),     \
                                                     (smem), (stream), (cluster_x),       \
                                                     __VA_ARGS__);                        \
        if (_err == cudaSuccess) _err = cudaGetLastError();                               \
        ::moe::launch_end(_tok, stream);                                                  \
        if (_err != cudaSuccess) return MOE_ERR_CUDA;                                     \
    } while (0)

// Optional log on stderr, set by the environment variable MOE_LOG (read
// once): 1 reports every error status on its way out of the library (where it
// arose: the function, or the failing call for MOE_TRY) and every non-zero
// device status word read back; 2 also every kernel launch.  0 (the default)
// prints nothing.
int log_level();
moe_status log_failure(const char *where, moe_status s);   // logs if enabled; returns s
#define MOE_FAIL(s) ::moe::log_failure(__func__, (s))
#define MOE_TRY(expr)                                                         \
    do {                                                                      \
        moe_status _s = (expr);                                               \
        if (_s != MOE_OK) return ::moe::log_failure(#expr, _s);               \
    } while (0)

// ---------------------------------------------------------------- workspace
// Regions of a workspace, byte offsets from its start (0 = region absent,
// except `status`, which is always at offset 0).  Each region is 1024-aligned.
struct Layout {
    size_t status = 0;        // int32 status word (+ padding to 1024)
    size_t hist = 0;          // int32 [chunks][E] routing histograms / bases
    size_t sched = 0;         // int32 [E+1] GEMM m-block starts per expert
    size_t route_row = 0;     // int32 [T*K]
    size_t assist = 0;        // int32 [T*K*3]
    size_t offsets = 0;       // int32 [E+1]
    size_t counts = 0;        // int64 [E]
    size_t recv_cum = 0;      // int32 [E*P]
    size_t q1 = 0;            // fp16 [T*K, H]  int8 values
    size_t s1 = 0;            // fp32 [T*K]
    size_t g = 0;             // fp32 [T*K, N/2]
    size_t q2 = 0;            // fp16 [T*K, N/2] int8 values
    size_t s2 = 0;            // fp32 [T*K]
    size_t y = 0;             // bf16 [T*K, H]
    size_t a_img = 0;         // fp16 images for the plain grouped GEMM
    size_t w_img = 0;
    size_t total = 0;
};

enum class Op { Dispatch, Combine, Ffn, Layer };

int64_t route_chunks(const moe_shape &s);
moe_status check_shape(const moe_shape *s, bool need_ffn);
Layout layout_for(const moe_shape &s, Op op);

// ---------------------------------------------------------------- device helpers
__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(((uint32_t)b) << 16);
}
__device__ __forceinline__ uint32_t lanemask_lt() {
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace moe

// ---------------------------------------------------------------- kernel-level entry points
// (host functions implemented in the .cu files, used by capi.cu)
namespace moe {

// Tokens per routing chunk: small batches use small chunks (more CTAs, a
// shorter serial walk per warp), large ones up to 256.  A function of T only.
inline int64_t route_chunk_tokens(int64_t T) {
    int64_t c = 64;
    while (c < kRouteChunkTokensMax && c * 128 < T) c *= 2;
    return c;
}

struct RouteDev {
    const int32_t *ids;
    const uint8_t *mask;
    int mask_kind;
    int64_t T, P, M, K, E;
    int64_t Z, C;          // zero and copy experts after the E MoE experts
    int64_t chunk_tokens;
    int64_t chunks_per_partition;
    int32_t *hist;     // [chunks][E]
    int32_t *bad;      // [chunks] 1 if the chunk saw an invalid expert id
    int32_t *status;
    int rows_final;    // 1: route_row already holds final rows (single-kernel routing)
};

// Route code of an active route's expert id: the id itself for a MoE expert,
// -2 for a zero expert, -3 for a copy expert, -4 for an id naming no expert.
__device__ __forceinline__ int route_code(int e, const RouteDev &a) {
    if (e >= 0 && e < a.E) return e;
    if (e >= a.E && e < a.E + a.Z) return -2;
    if (e >= a.E + a.Z && e < a.E + a.Z + a.C) return -3;
    return -4;
}

// Final row of route (t, k): route_row holds the route's rank inside its
// routing chunk (or -1) after launch_route; the chunk base of its expert is
// in r.hist after the scan.  Replaces route_row[t*K+k] by the row (unless
// the routing kernel already wrote final rows), writes the row's triplet
// (partition, token in partition, slot) and returns the row (-1 if
// inactive).  Called exactly once per route per call, by a kernel that
// spreads the routes over the whole GPU, so the triplets' scattered stores
// never sit on the routing kernel's few CTAs.
__device__ __forceinline__ int32_t resolve_route_row(const RouteDev &a, int64_t t, int k,
                                                     int32_t *route_row, int32_t *assist) {
    const int64_t i = t * a.K + k;
    const int32_t lr = route_row[i];
    if (lr < 0) return lr;   // inactive (-1) or a special expert (-2, -3): no row
    // T * K < 2^31, so token, partition and chunk indices fit in 32 bits
    const int32_t t32 = (int32_t)t, M32 = (int32_t)a.M;
    const int32_t p = t32 / M32;
    const int32_t tl = t32 - p * M32;
    int32_t row = lr;
    if (!a.rows_final) {
        const int e = a.ids[i];
        const int32_t c = p * (int32_t)a.chunks_per_partition + tl / (int32_t)a.chunk_tokens;
        row = a.hist[(int64_t)c * a.E + e] + lr;
        route_row[i] = row;
    }
    if (assist) {
        assist[3 * (int64_t)row + 0] = p;
        assist[3 * (int64_t)row + 1] = tl;
        assist[3 * (int64_t)row + 2] = k;
    }
    return row;
}

// Routing counts and scan: afterwards route_row holds ranks inside chunks
// (see resolve_route_row), r.hist the chunk bases.
moe_status launch_route(const RouteDev &r, int64_t chunks, int64_t *counts, int32_t *offsets,
                        int32_t *recv_cum, int32_t *sched, int32_t *route_row,
                        cudaStream_t stream);
// Single-kernel routing (count, rank, prefix and final rows in one launch: one
// CTA for tiny batches, one thread-block cluster for mid-size ones, one CTA
// per chunk with a grid barrier when all chunks fit on the GPU at once);
// otherwise launch_route.  Sets r.rows_final accordingly.  The triplets are
// written by the kernel that next reads route_row (resolve_route_row).
moe_status launch_route_fused(RouteDev &r, int64_t chunks, int64_t *counts, int32_t *offsets,
                              int32_t *recv_cum, int32_t *sched, int32_t *route_row,
                              cudaStream_t stream);
// Resolution alone, when no kernel copies or quantises the rows.
moe_status launch_route_resolve(const RouteDev &r, int32_t *route_row, int32_t *assist,
                                cudaStream_t stream);

// Resolves every route's row and copies x[t] to each of its rows.
moe_status launch_dispatch_rows(const RouteDev &r, const void *x, int32_t *route_row,
                                int32_t *assist, void *expand_x, int64_t H, cudaStream_t stream);

// status may be NULL (bounded waits that give up then only abort the kernel).
// special: the shape has zero or copy experts (route_row codes -2 / -3);
// ori_x is read by copy experts.
moe_status launch_combine(const void *y, const int32_t *route_row, const float *probs,
                          const uint8_t *mask, int mask_kind, const void *shared,
                          const void *ori_x, bool special, void *out, int64_t T, int64_t K,
                          int64_t H, int64_t cap_rows, int32_t *status, cudaStream_t stream);

// Resolves every route's row and writes the int8 codes (fp16 images) and
// scale of the quantised token x[t] to each of its rows.
moe_status launch_quant_scatter(const RouteDev &r, const void *x, int32_t *route_row,
                                int32_t *assist, void *q1, float *s1, int64_t H,
                                cudaStream_t stream);

// Quantised dispatch rows (int8 bytes) and their scales; resolves the rows.
moe_status launch_dispatch_quant(const RouteDev &r, const void *x, const float *smooth,
                                 int32_t *route_row, int32_t *assist, int8_t *q, float *scales,
                                 int64_t H, cudaStream_t stream);
moe_status launch_rows_i8_to_f16(const int8_t *rows, const float *scales, const int32_t *offsets,
                                 int64_t E, void *q1, float *s1, int64_t cap_rows, int64_t H,
                                 cudaStream_t stream);
moe_status launch_quant_rows(const void *x_rows, const int32_t *offsets, int64_t E, void *q1,
                             float *s1, int64_t cap_rows, int64_t H, cudaStream_t stream);


moe_status launch_quant2(const float *g, const int32_t *offsets, int64_t E, void *q2, float *s2,
                         int64_t cap_rows, int64_t Nh, cudaStream_t stream);

moe_status launch_sched(const int32_t *offsets, int64_t E, int32_t *sched, int32_t *status,
                        cudaStream_t stream);

moe_status launch_pack_w1(const int8_t *w1, void *w1p, int64_t E, int64_t N, int64_t H,
                          cudaStream_t stream);
moe_status launch_i8_to_f16(const int8_t *src, void *dst, int64_t n, cudaStream_t stream);
moe_status launch_pack_w1_i8(const int8_t *w1, void *w1p, int64_t E, int64_t N, int64_t H,
                             cudaStream_t stream);
moe_status launch_bias_i8(const int8_t *src, void *dst, int64_t n, cudaStream_t stream);

// Grouped GEMM on fp16 images of int8 operands (tcgen05, TMEM accumulators).
enum class Epi { S32 = 0, SwiGLU = 1, DequantBF16 = 2 };
struct GemmArgs {
    const void *a_img;        // fp16 [cap_rows, Kd]
    int64_t cap_rows;
    const void *b_img;        // fp16 [E, Nout, Kd]; biased bytes w + 128 for the int8-weight GEMM
    int64_t E, Nout, Kd;
    const int32_t *offsets;   // [E+1]; rows >= cap_rows are never stored
    const int32_t *sched;     // [E+1]
    // epilogue operands
    int32_t *c_s32;           // [cap_rows, Nout]
    float *g;                 // [cap_rows, Nout/2]
    const float *scale1;      // [E, Nout]
    const float *s1;          // [cap_rows]
    void *y;                  // bf16 [cap_rows, Nout]
    const float *scale2;      // [E, Nout]
    const float *s2;          // [cap_rows]
    int32_t *status;
};
// pair: 256-row tiles on clusters of two CTAs (falls back to one-SM tiles when
// no cluster of that kernel fits).
moe_status launch_grouped_gemm(Epi epi, const GemmArgs &a, cudaStream_t stream,
                               bool pair = false);
// The same GEMM for few rows per expert: the weights stream as biased bytes
// (b_img, w + 128; W1 in launch_pack_w1_i8's row order), are widened on chip
// into tensor memory and are the MMA's M side; the expert's rows are its N
// side, only as many as present.  Kd % 16 == 0 (and Nout % 128 == 0 for the
// SwiGLU epilogue).
moe_status launch_grouped_gemm_small(Epi epi, const GemmArgs &a, cudaStream_t stream);

}  // namespace moe
