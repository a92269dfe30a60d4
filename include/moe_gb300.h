/*
 * moe_gb300.h -- C ABI of the single-GPU MoE dispatch / grouped int8 FFN /
 * combine library for GB300 (sm_103a).  Library: libmoe_gb300.so.
 *
 * One GPU holds every expert.  The cross-rank exchange of the pages (shmem
 * puts, AllToAllV, HCCL windows) has no counterpart: routed rows are written
 * straight into an expert-major buffer in the same HBM.
 *
 * Pages the operations follow:
 *   "dispatch_combine_shmem.py"        TileLang-Ascend dispatch/combine example
 *   "aclnnMoeDistributeCombineV4"      CANN operator documentation
 *   "PTO MegaMoE Dispatch + Combine Fusion Example"
 *
 * Conventions for every entry point
 *   - Pointers named *_host are host memory; every other tensor pointer is a
 *     device pointer owned by the caller.  The library allocates and frees
 *     nothing, and synchronises nothing except in moe_read_device_status.
 *   - Work is enqueued on `stream` (0 = legacy default stream).  A call
 *     returns as soon as its kernels are enqueued.
 *   - Argument errors are reported synchronously, before any launch, through
 *     the return value; nothing is launched when a call fails.
 *   - Errors found by kernels (an expert id outside [0, E), a bounded wait
 *     that gave up) are recorded in a status word at the start of the
 *     workspace; the offending route is treated as inactive.  Each call that
 *     takes a workspace resets the word before its first kernel and later
 *     kernels of the call OR bits into it, so it describes the most recent
 *     call.  moe_read_device_status reads and clears it.
 *   - Every tensor pointer must be 16-byte aligned; workspace and packed
 *     weights must be 1024-byte aligned.
 *   - With T == 0 the per-token, per-route and per-row arrays are empty and
 *     may be NULL; the per-expert outputs of a dispatch are still written.
 *   - Results are deterministic: repeated calls give bitwise-identical
 *     outputs ("aclnnMoeDistributeCombineV4", Constraints: Deterministic
 *     Computation).
 *   - bf16 is IEEE binary32's upper half (stored as 2-byte words).
 *   - Concurrent calls that share a workspace race; give each stream its own.
 *   - Optional log on stderr, set by the environment variable MOE_LOG (read
 *     once per process): 1 reports every error status as it leaves the
 *     library (the function or failing internal call, and the status) and
 *     every non-zero device status word moe_read_device_status reads; 2 also
 *     every kernel launch (name and CTA count).  Unset or 0: nothing printed.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>
#include <cuda_runtime_api.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes.  The first three mirror the parameter-check codes in
 * "aclnnMoeDistributeCombineV4", Return Value. */
typedef enum moe_status {
    MOE_OK = 0,
    MOE_ERR_NULLPTR = 161001,        /* a required pointer is NULL */
    MOE_ERR_PARAM_INVALID = 161002,  /* an argument value is outside its range */
    MOE_ERR_SHAPE = 561002,          /* a shape is outside the supported range */
    MOE_ERR_WORKSPACE = 561003,      /* workspace too small */
    MOE_ERR_ALIGNMENT = 561004,      /* a pointer is not aligned as required */
    MOE_ERR_CUDA = 561005,           /* a CUDA launch or runtime call failed */
    MOE_ERR_UNSUPPORTED = 561006,    /* the device is not sm_103 / feature missing */
    MOE_ERR_TOO_LARGE = 561007       /* problem exceeds the fixed scratch of moe_dispatch_noalloc */
} moe_status;

/* Device status word bits (moe_read_device_status). */
#define MOE_DEV_BAD_EXPERT_ID  0x1   /* some active route had id outside [0, E) */
#define MOE_DEV_TIMEOUT        0x2   /* a bounded in-kernel wait gave up */

/*
 * Problem shape.  Notation of the pages: BS = T tokens on this GPU, split into
 * P source partitions of M = T / P consecutive tokens (a partition plays the
 * role of a source rank); H hidden size; E experts (moeExpertNum); K topK;
 * N the GMM1 output width (SwiGLU halves it).
 *   - T >= 0, P >= 1, T % P == 0
 *   - H >= 8, H % 8 == 0            (rows move as 16-byte vectors)
 *   - 1 <= E <= 1024; 1 <= K <= 16 ("aclnnMoeDistributeCombineV4",
 *     Constraints: 0 < K <= 16, moeExpertNum in (0, 1024])
 *   - N == 0 for dispatch/combine only; otherwise N % 256 == 0
 *   - mask_kind: 0 no xActiveMask, 1 per token uint8 [T], 2 per route uint8 [T, K]
 *   - has_shared: 1 if sharedExpertX is passed
 *   - zero_experts, copy_experts >= 0 ("aclnnMoeDistributeCombineV4",
 *     zeroExpertNum / copyExpertNum): a route to a zero expert contributes
 *     probs * 0 and one to a copy expert probs * oriX[t] to the combine; neither
 *     gets a row or a count.  Ids outside [0, E+Z+C) are invalid.
 *   - T * K * max(H, N) must stay below 2^31 elements per buffer row index space.
 */
typedef struct moe_shape {
    int64_t num_tokens;      /* T */
    int64_t num_partitions;  /* P */
    int64_t hidden;          /* H */
    int64_t num_experts;     /* E */
    int64_t topk;            /* K */
    int64_t ffn;             /* N, 0 = no expert FFN */
    int32_t mask_kind;
    int32_t has_shared;
    int64_t zero_experts;    /* Z: ids [E, E+Z) are zero experts (output 0) */
    int64_t copy_experts;    /* C: ids [E+Z, E+Z+C) are copy experts (output oriX) */
    int32_t ffn_path;        /* MOE_FFN_PATH_*: which grouped-GEMM kernels the FFN uses */
    int32_t reserved;        /* must be 0 */
} moe_shape;

/* Grouped-GEMM kernels of the expert FFN.  All give bit-identical results.
 *   LARGE: 128-row x 256-channel tiles on fp16 images of the weights, one
 *          SM each; for many rows per expert, where the tensor cores bound
 *          the time.
 *   LARGE_PAIR: 256-row x 256-channel tiles, each computed by a pair of SMs
 *          (a cluster of two CTAs sharing one 256-row MMA, each holding half
 *          of the rows and half of the weight channels, so a k-step moves a
 *          third less data per SM than LARGE).  Falls back to LARGE's kernel
 *          where no pair cluster fits.
 *   SMALL: the weights read as int8 (half the bytes), widened on chip into
 *          tensor memory as the MMA's 128-row side, against the expert's rows
 *          (the MMA's N); for few rows per expert, where reading the
 *          weights bounds the time ("PTO MegaMoE ...", Supported Cases: the M
 *          sweep from 16 tokens per rank).  Row tiles of 64 while the row
 *          capacity (T*K, or the rows of moe_grouped_gemm_s32's A) is at most
 *          32 per expert, else of 128, so that an expert of up to 128 rows
 *          reads its weights once.
 *   AUTO:  SMALL when T*K <= MOE_FFN_SMALL_ROWS_PER_EXPERT * E, else LARGE_PAIR.
 * moe_pack_weights writes the weight format(s) of the path in the shape it is
 * given, and the FFN calls read the format of theirs: pack with the same
 * ffn_path the FFN runs with (AUTO packs both formats). */
#define MOE_FFN_PATH_AUTO 0
#define MOE_FFN_PATH_LARGE 1
#define MOE_FFN_PATH_SMALL 2
#define MOE_FFN_PATH_LARGE_PAIR 3
/* Any other ffn_path value returns MOE_ERR_PARAM_INVALID. */
#define MOE_FFN_SMALL_ROWS_PER_EXPERT 128

/* ------------------------------------------------------------------------
 * Dispatch.
 * "dispatch_combine_shmem.py", "1. Implement Dispatch Operator": per-expert
 * route counts (SetStatus), prefix sums (GetCumSum, ep_receive_count), the
 * expert-major copy of token rows with (rank, token, k) triplets (send loop
 * and "Local data copy"), per-expert token counts (UpdateTokenNumsOut).
 * "PTO MegaMoE ...", FrontReorder Stage: expandedRowIdx, the route -> row index.
 *
 * x                  bf16 [T, H]
 * expert_ids         int32 [T, K]
 * x_active_mask      uint8 [T] or [T, K] per shape->mask_kind, else NULL
 * expand_x           bf16 [T*K, H] capacity; rows [0, R) are written, where
 *                    R = number of active routes; rows >= R are untouched
 * assist             int32 [T*K, 3]; row r gets (partition p, token t - p*M,
 *                    slot k); rows >= R untouched
 * expert_token_nums  int64 [E]; rows per expert
 * expert_offsets     int32 [E+1]; exclusive prefix of expert_token_nums,
 *                    expert_offsets[E] = R
 * ep_recv_counts     int32 [E*P]; inclusive running sum of the per-(expert,
 *                    partition) counts, expert-major
 * route_row          int32 [T*K]; row of route (t, k); -1 if inactive,
 *                    -2 for a zero expert, -3 for a copy expert
 * Row order: expert, then partition, then token, then slot.
 * expand_x may be NULL: only the bookkeeping is produced.
 * ------------------------------------------------------------------------ */
moe_status moe_dispatch_workspace_size(const moe_shape *shape, size_t *bytes);
moe_status moe_dispatch(const moe_shape *shape, const void *x, const int32_t *expert_ids,
                        const uint8_t *x_active_mask, void *expand_x, int32_t *assist,
                        int64_t *expert_token_nums, int32_t *expert_offsets,
                        int32_t *ep_recv_counts, int32_t *route_row,
                        void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Quantised dispatch: the dispatch above with int8 rows and one dynamic
 * scale per row ("aclnnMoeDistributeCombineV4", Example: the paired dispatch
 * call with a quantisation mode takes smooth scales [experts + 1, H] and returns
 * int8 expandX and dynamicScales [A]).  Row r of token t routed to expert e
 * holds q = clamp(rint(v / s), -127, 127) with v = float(x[t]) * smooth[e]
 * (or float(x[t]) when smooth_scales is NULL) and s = max|v| / 127, both in
 * fp32 with IEEE rounding; dynamic_scales[r] = s.
 * smooth_scales   fp32 [E, H] or NULL (rows past E, such as the shared
 *                 expert's row of an [E+1, H] array, are not read)
 * expand_x        int8 [T*K, H]; dynamic_scales fp32 [T*K]; rows >= R untouched
 * Other arguments and the workspace (moe_dispatch_workspace_size) as in
 * moe_dispatch.  H <= 8192.
 * ------------------------------------------------------------------------ */
moe_status moe_dispatch_quant(const moe_shape *shape, const void *x, const int32_t *expert_ids,
                              const uint8_t *x_active_mask, const float *smooth_scales,
                              int8_t *expand_x, float *dynamic_scales, int32_t *assist,
                              int64_t *expert_token_nums, int32_t *expert_offsets,
                              int32_t *ep_recv_counts, int32_t *route_row, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Combine.
 * "dispatch_combine_shmem.py", "2. Implement the Combine operator": per token,
 * the K returned rows are cast to fp32, multiplied by expert_scales[t, k] and
 * added in slot order into an fp32 accumulator, then rounded to bf16 to nearest
 * even.  "aclnnMoeDistributeCombineV4", Function/Formula: the shared-expert
 * term joins the sum; here it is added once, unscaled, after the routed sum.
 * "PTO MegaMoE ...", Unpermute: output in the original token order.
 *
 * No workspace is needed.
 * expand_x        bf16 [T*K, H] rows of the expert outputs (dispatch order)
 * route_row       int32 [T*K] from moe_dispatch (-1 inactive, -2 zero expert,
 *                 -3 copy expert)
 * expert_scales   fp32 [T, K]
 * x_active_mask   same mask as given to moe_dispatch, or NULL
 * shared_expert_x bf16 [T, H] or NULL (shape->has_shared must match)
 * ori_x           bf16 [T, H], the tokens before the FFN (oriXOptional);
 *                 required when shape->copy_experts > 0, else may be NULL
 * x_out           bf16 [T, H]; a token with no active route gets
 *                 bf16(shared) or +0
 * The multiply and add are separately rounded fp32 operations in slot order,
 * so the result is bitwise reproducible on any IEEE machine.
 * ------------------------------------------------------------------------ */
moe_status moe_combine(const moe_shape *shape, const void *expand_x, const int32_t *route_row,
                       const float *expert_scales, const uint8_t *x_active_mask,
                       const void *shared_expert_x, const void *ori_x, void *x_out,
                       cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Expert weights.  "PTO MegaMoE ...", Specification: "per-local-expert int8
 * packed weights" and fixpipe scales.  The caller's int8 weights are
 *   w1 int8 [E, N, H]   (row n = GMM1 output channel n, H contiguous)
 *   w2 int8 [E, H, N/2] (row c = GMM2 output channel c, N/2 contiguous)
 * Packing, done once per model, writes the operand format(s) of shape->ffn_path:
 *   LARGE, LARGE_PAIR: fp16 images of the int8 values (exact), 2 bytes
 *          per weight (E*N*H*2 and E*H*(N/2)*2 bytes);
 *   SMALL: the values as bytes biased by +128, 1 byte per weight;
 *   AUTO:  both, the bytes after the images, 3 bytes per weight.
 * W1's rows are reordered in each format (differently) so that every GEMM1
 * tile holds complete SwiGLU pairs.  The packed buffers are opaque; an FFN
 * call must use the ffn_path they were packed with.
 * ------------------------------------------------------------------------ */
moe_status moe_packed_weight_bytes(const moe_shape *shape, size_t *w1_bytes, size_t *w2_bytes);
moe_status moe_pack_weights(const moe_shape *shape, const int8_t *w1, const int8_t *w2,
                            void *w1_packed, void *w2_packed, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Grouped expert FFN on dispatched rows.
 * "PTO MegaMoE ...", GMM1 / SwiGLU / GMM2 Stages and the dequant of the
 * Combine stage.  For row r of expert e (rows [offsets[e], offsets[e+1])):
 *   q1, s1 = dynamic int8 quantisation of the row (s1 = max|x| / 127)
 *   acc1   = q1 . W1[e]^T                          exact int32
 *   h      = (float(acc1) * scale1[e]) * s1         fp32
 *   g      = silu(h[:N/2]) * h[N/2:]                fp32
 *   q2, s2 = dynamic int8 quantisation of g
 *   acc2   = q2 . W2[e]^T                          exact int32
 *   y      = bf16((float(acc2) * scale2[e]) * s2)
 * expand_x        bf16 [T*K, H] (rows [0, R) read)
 * expert_offsets  int32 [E+1] from moe_dispatch
 * w1_packed, w2_packed from moe_pack_weights; scale1 fp32 [E, N]; scale2 fp32 [E, H]
 * y               bf16 [T*K, H] (rows [0, R) written)
 * ------------------------------------------------------------------------ */
moe_status moe_grouped_ffn_workspace_size(const moe_shape *shape, size_t *bytes);
moe_status moe_grouped_ffn(const moe_shape *shape, const void *expand_x,
                           const int32_t *expert_offsets,
                           const void *w1_packed, const float *scale1,
                           const void *w2_packed, const float *scale2, void *y,
                           void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* The grouped FFN on rows that are already int8 (moe_dispatch_quant's
 * expand_x and dynamic_scales): the same stages as moe_grouped_ffn from the
 * GMM1 on; workspace from moe_grouped_ffn_workspace_size. */
moe_status moe_grouped_ffn_q(const moe_shape *shape, const int8_t *expand_x,
                             const float *dynamic_scales, const int32_t *expert_offsets,
                             const void *w1_packed, const float *scale1, const void *w2_packed,
                             const float *scale2, void *y, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * The whole layer in one call ("PTO MegaMoE ...", Functionality:
 *   out[token] = sum over its topK routes of probs * FFN_expert(x[token])):
 * dispatch bookkeeping, per-token quantisation scattered straight into
 * expert-major rows (FrontReorder quantises before the exchange; the result is
 * the same as quantising each dispatched copy), the grouped FFN, and combine.
 * Arguments as in the calls above; x_out bf16 [T, H].
 * ------------------------------------------------------------------------ */
moe_status moe_layer_workspace_size(const moe_shape *shape, size_t *bytes);
moe_status moe_layer(const moe_shape *shape, const void *x, const int32_t *expert_ids,
                     const float *expert_scales, const uint8_t *x_active_mask,
                     const void *shared_expert_x, const void *w1_packed, const float *scale1,
                     const void *w2_packed, const float *scale2, void *x_out,
                     void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* Device pointers into a workspace used by moe_layer or moe_grouped_ffn, for
 * inspection of the intermediate stages after the stream has finished.  Any
 * field a given call does not produce is NULL.  Layout of each:
 *   route_row int32 [T*K], assist int32 [T*K, 3], expert_offsets int32 [E+1],
 *   expert_token_nums int64 [E], ep_recv_counts int32 [E*P] (moe_layer only)
 *   q1 fp16 [T*K, H] (int8 values), s1 fp32 [T*K]
 *   g fp32 [T*K, N/2], q2 fp16 [T*K, N/2] (int8 values), s2 fp32 [T*K]
 *   y bf16 [T*K, H]                                                      */
typedef struct moe_stage_views {
    int32_t *route_row;
    int32_t *assist;
    int32_t *expert_offsets;
    int64_t *expert_token_nums;
    int32_t *ep_recv_counts;
    void *q1;
    float *s1;
    float *g;
    void *q2;
    float *s2;
    void *y;
} moe_stage_views;
moe_status moe_stage_views_get(const moe_shape *shape, int for_layer, void *workspace,
                               size_t workspace_bytes, moe_stage_views *views_host);

/* ------------------------------------------------------------------------
 * Grouped int8 GEMM with int32 output -- the GMM mainloop of the FFN with a
 * plain store epilogue ("PTO MegaMoE ...", GMM1: int8 x int8 -> int32
 * accumulator, per local expert).  C[r, n] = sum_i A[r, i] * W[e, n, i] for
 * rows r in [offsets[e], offsets[e+1]).
 *   A int8 [rows, Kd]; W int8 [E, N, Kd]; C int32 [rows, N]; rows >= offsets[E].
 *   N % 8 == 0, Kd % 8 == 0 (Kd % 16 == 0 for the SMALL kernel).
 * path: MOE_FFN_PATH_* (AUTO: SMALL when rows <= MOE_FFN_SMALL_ROWS_PER_EXPERT * E
 * and Kd % 16 == 0, else LARGE_PAIR).  A is first converted into fp16 images in
 * the workspace, and W into fp16 images (LARGE, LARGE_PAIR) or biased bytes
 * (SMALL).
 * ------------------------------------------------------------------------ */
moe_status moe_grouped_gemm_s32_workspace_size(int64_t rows, int64_t E, int64_t N, int64_t Kd,
                                               size_t *bytes);
moe_status moe_grouped_gemm_s32(int64_t rows, int64_t E, int64_t N, int64_t Kd,
                                const int32_t *expert_offsets, const int8_t *A,
                                const int8_t *W, int32_t *C, int path,
                                void *workspace, size_t workspace_bytes, cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Dispatch without any device allocation by the caller.
 * The pages have no counterpart: this entry point exists for callers that
 * cannot allocate device memory -- a runtime whose device memory is planned
 * once at load time, a plugin inside a framework that exposes no allocator,
 * or a latency-critical path on which an allocation is not allowed -- and so
 * cannot provide moe_dispatch's workspace.
 * Same arguments and results as moe_dispatch, minus the workspace: the
 * routing scratch lives in a fixed array in the library's own device memory
 * (moe_dispatch_noalloc_scratch_bytes() bytes, held on every GPU that loads
 * the library until the process exits).  Limit: chunks*E + chunks <= 262144,
 * where chunks = P * ceil(M / c) and the routing chunk c depends on T only:
 * c = 64, doubled while c < 256 and c * 128 < T (so c = 64 for T <= 8192,
 * 128 for T <= 16384, 256 above).  Larger problems return MOE_ERR_TOO_LARGE
 * before any launch.  The first call on a device looks up the array's device
 * address (cudaGetSymbolAddress) with that device current and caches it; make
 * that first call before any stream capture on the device.  The cached
 * address does not survive a cudaDeviceReset in the calling process.  All
 * calls share the array: calls whose kernels overlap on the GPU race.  Every
 * scratch entry a call reads is written earlier in the same call, so nothing
 * needs clearing between calls.  Invalid ids are treated as inactive, as in
 * moe_dispatch; the status word is kept in the scratch and is not reported.
 * Pointer alignment as in moe_dispatch.  No cudaMalloc, cudaFree or other
 * allocating call is made.
 * ------------------------------------------------------------------------ */
size_t moe_dispatch_noalloc_scratch_bytes(void);
moe_status moe_dispatch_noalloc(const moe_shape *shape, const void *x, const int32_t *expert_ids,
                                const uint8_t *x_active_mask, void *expand_x, int32_t *assist,
                                int64_t *expert_token_nums, int32_t *expert_offsets,
                                int32_t *ep_recv_counts, int32_t *route_row,
                                cudaStream_t stream);

/* Reads the device status word of `workspace` (synchronising `stream`),
 * stores it in *status_host (0 = no device-side error, else MOE_DEV_* bits)
 * and clears it. */
moe_status moe_read_device_status(void *workspace, cudaStream_t stream, int32_t *status_host);

/* ------------------------------------------------------------------------
 * Self-test of the bounded waits.  Every in-kernel wait of this library gives
 * up after a time limit (about 2 s), records MOE_DEV_TIMEOUT in the status
 * word and lets the kernel finish, so a lost completion surfaces as a status
 * instead of a hung stream (the pages bound waiting on the host side too:
 * "aclnnMoeDistributeCombineV4", the A2 sample synchronises its stream with a
 * 10 000 ms timeout).  This call runs that wait loop on a barrier nothing
 * arrives on, with no copy or MMA attached, for limit_ns nanoseconds
 * (0 < limit_ns <= 2e9): the status word of `workspace` must then read
 * MOE_DEV_TIMEOUT (moe_read_device_status), and the 8 bytes at offset 8 hold
 * the nanoseconds the wait took.  workspace: >= 16 bytes, 1024-aligned.
 * ------------------------------------------------------------------------ */
moe_status moe_wait_selftest(void *workspace, size_t workspace_bytes, uint64_t limit_ns,
                             cudaStream_t stream);

/* ------------------------------------------------------------------------
 * Instrumentation.
 * moe_launch_count: number of kernels this library has launched in the
 * process so far.
 * moe_profile_enable(1) makes every later launch record a CUDA event pair
 * on its own stream; moe_profile_report (after the streams are synchronised)
 * writes one line per kernel name: "name launches total_ms grid" (grid: the
 * CTAs of its last launch) into buf and clears the records.
 * moe_profile_enable(0) stops recording.
 * ------------------------------------------------------------------------ */
uint64_t moe_launch_count(void);
moe_status moe_profile_enable(int on);
moe_status moe_profile_report(char *buf_host, size_t buf_bytes);

/* Human-readable name of a status code (static storage). */
const char *moe_status_string(moe_status status);

#ifdef __cplusplus
}
#endif
#endif /* MOE_GB300_H */
