// capi.cu -- the C ABI (include/moe_gb300.h): argument checks, workspace
// layout, the order of kernels behind each entry point, launch counting and
// per-kernel event profiling.
#include "common.cuh"

#include <atomic>
#include <mutex>
#include <string>
#include <vector>
#include <map>
#include <cstdio>
#include <cstdlib>
#include <cstring>

namespace moe {

// ---------------------------------------------------------------- launch bookkeeping
namespace {
std::atomic<uint64_t> g_launches{0};
std::atomic<bool> g_profile{false};

struct ProfRecord {
    const char *name;
    cudaEvent_t start, stop;
    unsigned grid;   // CTAs launched
};
std::mutex g_prof_mu;
std::vector<ProfRecord> g_records;
std::vector<cudaEvent_t> g_event_pool;

cudaEvent_t take_event() {
    if (!g_event_pool.empty()) {
        cudaEvent_t e = g_event_pool.back();
        g_event_pool.pop_back();
        return e;
    }
    cudaEvent_t e = nullptr;
    cudaEventCreate(&e);
    return e;
}
}  // namespace

int log_level() {
    static const int level = [] {
        const char *e = getenv("MOE_LOG");
        return e ? atoi(e) : 0;
    }();
    return level;
}

moe_status log_failure(const char *where, moe_status s) {
    if (log_level() > 0) fprintf(stderr, "moe: %s: %s (%d)\n", where, moe_status_string(s), (int)s);
    return s;
}

int launch_begin(const char *name, cudaStream_t stream, unsigned grid) {
    g_launches.fetch_add(1, std::memory_order_relaxed);
    if (log_level() >= 2) fprintf(stderr, "moe: launch %s, %u CTAs\n", name, grid);
    if (!g_profile.load(std::memory_order_relaxed)) return -1;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    ProfRecord r{name, take_event(), take_event(), grid};
    cudaEventRecord(r.start, stream);
    g_records.push_back(r);
    return (int)g_records.size() - 1;
}

void launch_end(int token, cudaStream_t stream) {
    if (token < 0) return;
    std::lock_guard<std::mutex> lk(g_prof_mu);
    if (token < (int)g_records.size()) cudaEventRecord(g_records[token].stop, stream);
}

bool set_smem_limit(const void *kernel, size_t bytes) {
    static std::mutex mu;
    static std::vector<std::pair<const void *, size_t>> done;
    std::lock_guard<std::mutex> lk(mu);
    size_t *have = nullptr;
    for (auto &d : done)
        if (d.first == kernel) have = &d.second;
    if (have && *have >= bytes) return true;
    if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes) !=
        cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    if (have) *have = bytes;
    else done.emplace_back(kernel, bytes);
    return true;
}

int num_sms() {
    static int cached[64] = {0};
    int dev = 0;
    cudaGetDevice(&dev);
    if (dev < 0 || dev >= 64) dev = 0;
    if (cached[dev] == 0) {
        int n = 0;
        cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        cached[dev] = n > 0 ? n : 1;
    }
    return cached[dev];
}

// ---------------------------------------------------------------- shapes and layouts
int64_t route_chunks(const moe_shape &s) {
    if (s.num_tokens == 0) return 0;
    const int64_t M = s.num_tokens / s.num_partitions;
    const int64_t ct = route_chunk_tokens(s.num_tokens);
    return s.num_partitions * ((M + ct - 1) / ct);
}

moe_status check_shape(const moe_shape *s, bool need_ffn) {
    if (!s) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (s->num_tokens < 0 || s->num_partitions < 1 || s->num_tokens % s->num_partitions != 0)
        return MOE_FAIL(MOE_ERR_SHAPE);
    if (s->hidden < 8 || s->hidden % 8 != 0) return MOE_FAIL(MOE_ERR_SHAPE);
    if (s->num_experts < 1 || s->num_experts > kMaxExperts) return MOE_FAIL(MOE_ERR_SHAPE);
    if (s->topk < 1 || s->topk > kMaxTopK) return MOE_FAIL(MOE_ERR_SHAPE);
    if (s->mask_kind < 0 || s->mask_kind > 2) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    if (s->zero_experts < 0 || s->copy_experts < 0 ||
        s->num_experts + s->zero_experts + s->copy_experts > INT32_MAX)
        return MOE_FAIL(MOE_ERR_SHAPE);
    if (s->has_shared != 0 && s->has_shared != 1) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    if (s->ffn_path < MOE_FFN_PATH_AUTO || s->ffn_path > MOE_FFN_PATH_LARGE_PAIR || s->reserved != 0)
        return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    const int64_t cap = s->num_tokens * s->topk;
    if (cap > INT32_MAX) return MOE_FAIL(MOE_ERR_SHAPE);
    if (need_ffn) {
        if (s->ffn <= 0 || s->ffn % 256 != 0 || s->ffn > 8192) return MOE_FAIL(MOE_ERR_SHAPE);
        if (s->hidden % 16 != 0 || s->hidden > 8192) return MOE_FAIL(MOE_ERR_SHAPE);
    } else if (s->ffn < 0) {
        return MOE_FAIL(MOE_ERR_SHAPE);
    }
    return MOE_OK;
}

Layout layout_for(const moe_shape &s, Op op) {
    Layout L;
    const int64_t T = s.num_tokens, K = s.topk, E = s.num_experts, H = s.hidden, P = s.num_partitions;
    const int64_t cap = T * K, Nh = s.ffn / 2;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t at = off;
        off = align_up(off + (bytes ? bytes : 1), kAlign);
        return at;
    };
    L.status = take(4);
    if (op == Op::Dispatch || op == Op::Layer) {
        const int64_t C = route_chunks(s);
        L.hist = take((size_t)(C * E + C) * sizeof(int32_t));
    }
    if (op == Op::Ffn || op == Op::Layer) L.sched = take((size_t)(E + 1) * sizeof(int32_t));
    if (op == Op::Layer) {
        L.route_row = take((size_t)cap * sizeof(int32_t));
        L.assist = take((size_t)cap * 3 * sizeof(int32_t));
        L.offsets = take((size_t)(E + 1) * sizeof(int32_t));
        L.counts = take((size_t)E * sizeof(int64_t));
        L.recv_cum = take((size_t)(E * P) * sizeof(int32_t));
    }
    if (op == Op::Ffn || op == Op::Layer) {
        L.q1 = take((size_t)cap * H * 2);
        L.s1 = take((size_t)cap * sizeof(float));
        L.g = take((size_t)cap * Nh * sizeof(float));
        L.q2 = take((size_t)cap * Nh * 2);
        L.s2 = take((size_t)cap * sizeof(float));
    }
    if (op == Op::Layer) L.y = take((size_t)cap * H * 2);
    L.total = off;
    return L;
}

static bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

template <typename T>
static T *at(void *ws, size_t off) {
    return reinterpret_cast<T *>(reinterpret_cast<uint8_t *>(ws) + off);
}

static RouteDev route_dev(const moe_shape &s, const int32_t *ids, const uint8_t *mask, void *ws,
                          const Layout &L) {
    RouteDev r;
    r.ids = ids;
    r.mask = mask;
    r.mask_kind = s.mask_kind;
    r.T = s.num_tokens;
    r.P = s.num_partitions;
    r.M = s.num_tokens / s.num_partitions;
    r.K = s.topk;
    r.E = s.num_experts;
    r.Z = s.zero_experts;
    r.C = s.copy_experts;
    r.chunk_tokens = route_chunk_tokens(r.T);
    r.chunks_per_partition = (r.M + r.chunk_tokens - 1) / r.chunk_tokens;
    if (r.chunks_per_partition == 0) r.chunks_per_partition = 1;
    const int64_t C = route_chunks(s);
    r.hist = at<int32_t>(ws, L.hist);
    r.bad = r.hist + C * s.num_experts;
    r.status = at<int32_t>(ws, L.status);
    r.rows_final = 0;
    return r;
}

}  // namespace moe

using namespace moe;

// ====================================================================== C ABI
extern "C" {

const char *moe_status_string(moe_status st) {
    switch (st) {
        case MOE_OK: return "ok";
        case MOE_ERR_NULLPTR: return "required pointer is NULL";
        case MOE_ERR_PARAM_INVALID: return "argument value out of range";
        case MOE_ERR_SHAPE: return "shape not supported";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_ALIGNMENT: return "pointer misaligned";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_UNSUPPORTED: return "unsupported device";
        case MOE_ERR_TOO_LARGE: return "problem exceeds the fixed scratch of the allocation-free entry point";
    }
    return "unknown status";
}

uint64_t moe_launch_count(void) { return g_launches.load(); }

moe_status moe_profile_enable(int on) {
    g_profile.store(on != 0);
    return MOE_OK;
}

moe_status moe_profile_report(char *buf, size_t bytes) {
    if (!buf || bytes == 0) return MOE_FAIL(MOE_ERR_NULLPTR);
    std::lock_guard<std::mutex> lk(g_prof_mu);
    std::map<std::string, std::pair<int, double>> agg;
    std::map<std::string, unsigned> grid;
    std::vector<std::string> order;
    for (auto &r : g_records) {
        float ms = 0.0f;
        if (cudaEventElapsedTime(&ms, r.start, r.stop) != cudaSuccess) ms = -1.0f;
        auto it = agg.find(r.name);
        if (it == agg.end()) {
            order.push_back(r.name);
            agg[r.name] = {1, (double)ms};
        } else {
            it->second.first += 1;
            it->second.second += ms;
        }
        grid[r.name] = r.grid;
        g_event_pool.push_back(r.start);
        g_event_pool.push_back(r.stop);
    }
    g_records.clear();
    cudaGetLastError();
    std::string out;
    char line[256];
    for (auto &n : order) {
        snprintf(line, sizeof line, "%s %d %.6f %u\n", n.c_str(), agg[n].first, agg[n].second, grid[n]);
        out += line;
    }
    if (out.size() + 1 > bytes) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    memcpy(buf, out.c_str(), out.size() + 1);
    return MOE_OK;
}

moe_status moe_read_device_status(void *workspace, cudaStream_t stream, int32_t *status_host) {
    if (!workspace || !status_host) return MOE_FAIL(MOE_ERR_NULLPTR);
    int32_t v = 0;
    if (cudaMemcpyAsync(&v, workspace, sizeof v, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
        return MOE_FAIL(MOE_ERR_CUDA);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_FAIL(MOE_ERR_CUDA);
    if (cudaMemsetAsync(workspace, 0, sizeof v, stream) != cudaSuccess) return MOE_FAIL(MOE_ERR_CUDA);
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MOE_FAIL(MOE_ERR_CUDA);
    if (v != 0 && log_level() > 0) fprintf(stderr, "moe: device status word 0x%x\n", (unsigned)v);
    *status_host = v;
    return MOE_OK;
}

// ---------------------------------------------------------------- dispatch
moe_status moe_dispatch_workspace_size(const moe_shape *shape, size_t *bytes) {
    MOE_TRY(check_shape(shape, false));
    if (!bytes) return MOE_FAIL(MOE_ERR_NULLPTR);
    *bytes = layout_for(*shape, Op::Dispatch).total;
    return MOE_OK;
}

moe_status moe_dispatch(const moe_shape *shape, const void *x, const int32_t *expert_ids,
                        const uint8_t *x_active_mask, void *expand_x, int32_t *assist,
                        int64_t *expert_token_nums, int32_t *expert_offsets,
                        int32_t *ep_recv_counts, int32_t *route_row, void *workspace,
                        size_t workspace_bytes, cudaStream_t stream) {
    MOE_TRY(check_shape(shape, false));
    const moe_shape &s = *shape;
    // with T == 0 the per-token and per-route arrays are empty and may be NULL
    const bool empty = s.num_tokens == 0;
    if (!expert_token_nums || !expert_offsets || !ep_recv_counts || !workspace)
        return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && (!expert_ids || !assist || !route_row)) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && expand_x && !x) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && s.mask_kind != 0 && !x_active_mask) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (s.mask_kind == 0 && x_active_mask) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    if ((expand_x && (!aligned(x, 16) || !aligned(expand_x, 16))) || !aligned(workspace, kAlign))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    if (!aligned(expert_ids, 4) || !aligned(assist, 4) || !aligned(expert_token_nums, 8) ||
        !aligned(expert_offsets, 4) || !aligned(ep_recv_counts, 4) || !aligned(route_row, 4))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    const Layout L = layout_for(s, Op::Dispatch);
    if (workspace_bytes < L.total) return MOE_FAIL(MOE_ERR_WORKSPACE);
    RouteDev r = route_dev(s, expert_ids, x_active_mask, workspace, L);
    MOE_TRY(launch_route_fused(r, route_chunks(s), expert_token_nums, expert_offsets,
                               ep_recv_counts, nullptr, route_row, stream));
    if (expand_x) return launch_dispatch_rows(r, x, route_row, assist, expand_x, s.hidden, stream);
    return launch_route_resolve(r, route_row, assist, stream);
}

moe_status moe_dispatch_quant(const moe_shape *shape, const void *x, const int32_t *expert_ids,
                              const uint8_t *x_active_mask, const float *smooth_scales,
                              int8_t *expand_x, float *dynamic_scales, int32_t *assist,
                              int64_t *expert_token_nums, int32_t *expert_offsets,
                              int32_t *ep_recv_counts, int32_t *route_row, void *workspace,
                              size_t workspace_bytes, cudaStream_t stream) {
    MOE_TRY(check_shape(shape, false));
    const moe_shape &s = *shape;
    const bool empty = s.num_tokens == 0;
    if (s.hidden > 8192) return MOE_FAIL(MOE_ERR_SHAPE);
    if (!expert_token_nums || !expert_offsets || !ep_recv_counts || !workspace) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && (!x || !expert_ids || !assist || !route_row || !expand_x || !dynamic_scales))
        return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && s.mask_kind != 0 && !x_active_mask) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (s.mask_kind == 0 && x_active_mask) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    if (!aligned(x, 16) || !aligned(expand_x, 16) || !aligned(smooth_scales, 16) ||
        !aligned(workspace, kAlign) || !aligned(dynamic_scales, 4))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    const Layout L = layout_for(s, Op::Dispatch);
    if (workspace_bytes < L.total) return MOE_FAIL(MOE_ERR_WORKSPACE);
    RouteDev r = route_dev(s, expert_ids, x_active_mask, workspace, L);
    MOE_TRY(launch_route_fused(r, route_chunks(s), expert_token_nums, expert_offsets,
                               ep_recv_counts, nullptr, route_row, stream));
    return launch_dispatch_quant(r, x, smooth_scales, route_row, assist, expand_x, dynamic_scales,
                                 s.hidden, stream);
}

// ---------------------------------------------------------------- combine
moe_status moe_combine(const moe_shape *shape, const void *expand_x, const int32_t *route_row,
                       const float *expert_scales, const uint8_t *x_active_mask,
                       const void *shared_expert_x, const void *ori_x, void *x_out,
                       cudaStream_t stream) {
    MOE_TRY(check_shape(shape, false));
    const moe_shape &s = *shape;
    if (s.num_tokens == 0) return MOE_OK;
    if (!expand_x || !route_row || !expert_scales || !x_out) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (s.copy_experts > 0 && !ori_x) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (ori_x && !aligned(ori_x, 16)) return MOE_FAIL(MOE_ERR_ALIGNMENT);
    if (s.has_shared && !shared_expert_x) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!s.has_shared && shared_expert_x) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    if (s.mask_kind != 0 && !x_active_mask) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (s.mask_kind == 0 && x_active_mask) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    if (!aligned(expand_x, 16) || !aligned(x_out, 16) ||
        (shared_expert_x && !aligned(shared_expert_x, 16)) || !aligned(route_row, 4) ||
        !aligned(expert_scales, 4))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    return launch_combine(expand_x, route_row, expert_scales, x_active_mask, s.mask_kind,
                          shared_expert_x, s.copy_experts > 0 ? ori_x : nullptr,
                          s.zero_experts + s.copy_experts > 0, x_out, s.num_tokens, s.topk,
                          s.hidden, s.num_tokens * s.topk, nullptr, stream);
}

// ---------------------------------------------------------------- weights
// Formats a packed buffer holds, by the shape's ffn_path: fp16 images for the
// large-tile kernels, biased bytes for the small-batch kernel, both for AUTO
// (which picks by the row count of each call).  In a buffer holding both, the
// bytes follow the images.
static bool packs_f16(int32_t path) { return path != MOE_FFN_PATH_SMALL; }
static bool packs_i8(int32_t path) {
    return path == MOE_FFN_PATH_SMALL || path == MOE_FFN_PATH_AUTO;
}

moe_status moe_packed_weight_bytes(const moe_shape *shape, size_t *w1_bytes, size_t *w2_bytes) {
    MOE_TRY(check_shape(shape, true));
    if (!w1_bytes || !w2_bytes) return MOE_FAIL(MOE_ERR_NULLPTR);
    const moe_shape &s = *shape;
    const size_t per = (packs_f16(s.ffn_path) ? 2 : 0) + (packs_i8(s.ffn_path) ? 1 : 0);
    *w1_bytes = (size_t)s.num_experts * s.ffn * s.hidden * per;
    *w2_bytes = (size_t)s.num_experts * s.hidden * (s.ffn / 2) * per;
    return MOE_OK;
}

// The biased-byte part of a packed buffer: after the fp16 images (E*rows*cols*2
// bytes, a multiple of 1024 because N % 256 == 0 and H % 16 == 0) when the
// buffer holds both formats, else at its start.
static const void *packed_i8(const void *packed, int32_t path, int64_t E, int64_t rows,
                             int64_t cols) {
    return static_cast<const uint8_t *>(packed) + (packs_f16(path) ? (size_t)E * rows * cols * 2 : 0);
}

static bool use_small_path(int32_t path, int64_t rows, int64_t E) {
    if (path == MOE_FFN_PATH_SMALL) return true;
    if (path == MOE_FFN_PATH_LARGE || path == MOE_FFN_PATH_LARGE_PAIR) return false;
    return rows <= (int64_t)MOE_FFN_SMALL_ROWS_PER_EXPERT * E;
}

// Large-tile calls: AUTO and LARGE_PAIR take the SM-pair kernel (it falls back
// to one-SM tiles where no pair cluster fits), LARGE the one-SM kernel.
static moe_status run_gemm(bool small, int32_t path, Epi epi, const GemmArgs &g, cudaStream_t stream) {
    if (small) return launch_grouped_gemm_small(epi, g, stream);
    return launch_grouped_gemm(epi, g, stream,
                               path == MOE_FFN_PATH_LARGE_PAIR || path == MOE_FFN_PATH_AUTO);
}

moe_status moe_pack_weights(const moe_shape *shape, const int8_t *w1, const int8_t *w2,
                            void *w1_packed, void *w2_packed, cudaStream_t stream) {
    MOE_TRY(check_shape(shape, true));
    const moe_shape &s = *shape;
    if (!w1 || !w2 || !w1_packed || !w2_packed) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!aligned(w1, 16) || !aligned(w2, 16) || !aligned(w1_packed, kAlign) ||
        !aligned(w2_packed, kAlign))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    const int64_t E = s.num_experts, N = s.ffn, H = s.hidden, Nh = s.ffn / 2;
    const int32_t path = s.ffn_path;
    if (packs_f16(path)) {
        MOE_TRY(launch_pack_w1(w1, w1_packed, E, N, H, stream));
        MOE_TRY(launch_i8_to_f16(w2, w2_packed, E * H * Nh, stream));
    }
    if (packs_i8(path)) {
        MOE_TRY(launch_pack_w1_i8(w1, const_cast<void *>(packed_i8(w1_packed, path, E, N, H)), E,
                                  N, H, stream));
        MOE_TRY(launch_bias_i8(w2, const_cast<void *>(packed_i8(w2_packed, path, E, H, Nh)),
                               E * H * Nh, stream));
    }
    return MOE_OK;
}

// ---------------------------------------------------------------- grouped FFN
static moe_status run_ffn_core(const moe_shape &s, const Layout &L, void *ws,
                               const int32_t *offsets, const void *w1p, const float *scale1,
                               const void *w2p, const float *scale2, void *y,
                               cudaStream_t stream) {
    const int64_t cap = s.num_tokens * s.topk, Nh = s.ffn / 2;
    int32_t *status = at<int32_t>(ws, L.status);
    const bool small = use_small_path(s.ffn_path, cap, s.num_experts);
    GemmArgs g1{};
    g1.a_img = at<void>(ws, L.q1);
    g1.cap_rows = cap;
    g1.b_img = small ? packed_i8(w1p, s.ffn_path, s.num_experts, s.ffn, s.hidden) : w1p;
    g1.E = s.num_experts;
    g1.Nout = s.ffn;
    g1.Kd = s.hidden;
    g1.offsets = offsets;
    g1.sched = at<int32_t>(ws, L.sched);
    g1.g = at<float>(ws, L.g);
    g1.scale1 = scale1;
    g1.s1 = at<float>(ws, L.s1);
    g1.status = status;
    GemmArgs g2{};
    g2.a_img = at<void>(ws, L.q2);
    g2.cap_rows = cap;
    g2.b_img = small ? packed_i8(w2p, s.ffn_path, s.num_experts, s.hidden, Nh) : w2p;
    g2.E = s.num_experts;
    g2.Nout = s.hidden;
    g2.Kd = Nh;
    g2.offsets = offsets;
    g2.sched = at<int32_t>(ws, L.sched);
    g2.y = y;
    g2.scale2 = scale2;
    g2.s2 = at<float>(ws, L.s2);
    g2.status = status;
    MOE_TRY(run_gemm(small, s.ffn_path, Epi::SwiGLU, g1, stream));
    MOE_TRY(launch_quant2(at<float>(ws, L.g), offsets, s.num_experts, at<void>(ws, L.q2),
                          at<float>(ws, L.s2), cap, Nh, stream));
    return run_gemm(small, s.ffn_path, Epi::DequantBF16, g2, stream);
}

moe_status moe_grouped_ffn_workspace_size(const moe_shape *shape, size_t *bytes) {
    MOE_TRY(check_shape(shape, true));
    if (!bytes) return MOE_FAIL(MOE_ERR_NULLPTR);
    *bytes = layout_for(*shape, Op::Ffn).total;
    return MOE_OK;
}

moe_status moe_grouped_ffn(const moe_shape *shape, const void *expand_x,
                           const int32_t *expert_offsets, const void *w1_packed,
                           const float *scale1, const void *w2_packed, const float *scale2,
                           void *y, void *workspace, size_t workspace_bytes,
                           cudaStream_t stream) {
    MOE_TRY(check_shape(shape, true));
    const moe_shape &s = *shape;
    // with T == 0 the per-row arrays are empty and may be NULL
    const bool empty = s.num_tokens == 0;
    if (!expert_offsets || !w1_packed || !scale1 || !w2_packed || !scale2 || !workspace)
        return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && (!expand_x || !y)) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!aligned(expand_x, 16) || !aligned(y, 16) || !aligned(scale1, 16) || !aligned(scale2, 16) ||
        !aligned(w1_packed, kAlign) || !aligned(w2_packed, kAlign) || !aligned(workspace, kAlign))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    const Layout L = layout_for(s, Op::Ffn);
    if (workspace_bytes < L.total) return MOE_FAIL(MOE_ERR_WORKSPACE);
    if (s.num_tokens == 0) return MOE_OK;
    const int64_t cap = s.num_tokens * s.topk;
    MOE_TRY(launch_sched(expert_offsets, s.num_experts, at<int32_t>(workspace, L.sched),
                         at<int32_t>(workspace, L.status), stream));
    MOE_TRY(launch_quant_rows(expand_x, expert_offsets, s.num_experts, at<void>(workspace, L.q1),
                              at<float>(workspace, L.s1), cap, s.hidden, stream));
    return run_ffn_core(s, L, workspace, expert_offsets, w1_packed, scale1, w2_packed, scale2, y,
                        stream);
}

moe_status moe_grouped_ffn_q(const moe_shape *shape, const int8_t *expand_x,
                             const float *dynamic_scales, const int32_t *expert_offsets,
                             const void *w1_packed, const float *scale1, const void *w2_packed,
                             const float *scale2, void *y, void *workspace,
                             size_t workspace_bytes, cudaStream_t stream) {
    MOE_TRY(check_shape(shape, true));
    const moe_shape &s = *shape;
    const bool empty = s.num_tokens == 0;   // the per-row arrays may then be NULL
    if (!expert_offsets || !w1_packed || !scale1 || !w2_packed || !scale2 || !workspace)
        return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && (!expand_x || !dynamic_scales || !y)) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!aligned(expand_x, 16) || !aligned(y, 16) || !aligned(scale1, 16) || !aligned(scale2, 16) ||
        !aligned(w1_packed, kAlign) || !aligned(w2_packed, kAlign) || !aligned(workspace, kAlign))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    const Layout L = layout_for(s, Op::Ffn);
    if (workspace_bytes < L.total) return MOE_FAIL(MOE_ERR_WORKSPACE);
    if (s.num_tokens == 0) return MOE_OK;
    const int64_t cap = s.num_tokens * s.topk;
    MOE_TRY(launch_sched(expert_offsets, s.num_experts, at<int32_t>(workspace, L.sched),
                         at<int32_t>(workspace, L.status), stream));
    MOE_TRY(launch_rows_i8_to_f16(expand_x, dynamic_scales, expert_offsets, s.num_experts,
                                  at<void>(workspace, L.q1), at<float>(workspace, L.s1), cap,
                                  s.hidden, stream));
    return run_ffn_core(s, L, workspace, expert_offsets, w1_packed, scale1, w2_packed, scale2, y,
                        stream);
}

// ---------------------------------------------------------------- whole layer
moe_status moe_layer_workspace_size(const moe_shape *shape, size_t *bytes) {
    MOE_TRY(check_shape(shape, true));
    if (!bytes) return MOE_FAIL(MOE_ERR_NULLPTR);
    *bytes = layout_for(*shape, Op::Layer).total;
    return MOE_OK;
}

moe_status moe_layer(const moe_shape *shape, const void *x, const int32_t *expert_ids,
                     const float *expert_scales, const uint8_t *x_active_mask,
                     const void *shared_expert_x, const void *w1_packed, const float *scale1,
                     const void *w2_packed, const float *scale2, void *x_out, void *workspace,
                     size_t workspace_bytes, cudaStream_t stream) {
    MOE_TRY(check_shape(shape, true));
    const moe_shape &s = *shape;
    // with T == 0 the per-token and per-route arrays are empty and may be NULL
    const bool empty = s.num_tokens == 0;
    if (!w1_packed || !scale1 || !w2_packed || !scale2 || !workspace) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && (!x || !expert_ids || !expert_scales || !x_out)) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && s.has_shared && !shared_expert_x) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!s.has_shared && shared_expert_x) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    if (!empty && s.mask_kind != 0 && !x_active_mask) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (s.mask_kind == 0 && x_active_mask) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    if (!aligned(x, 16) || !aligned(x_out, 16) || !aligned(scale1, 16) || !aligned(scale2, 16) ||
        (shared_expert_x && !aligned(shared_expert_x, 16)) || !aligned(w1_packed, kAlign) ||
        !aligned(w2_packed, kAlign) || !aligned(workspace, kAlign) || !aligned(expert_ids, 4) ||
        !aligned(expert_scales, 4))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    const Layout L = layout_for(s, Op::Layer);
    if (workspace_bytes < L.total) return MOE_FAIL(MOE_ERR_WORKSPACE);
    const int64_t cap = s.num_tokens * s.topk;
    RouteDev r = route_dev(s, expert_ids, x_active_mask, workspace, L);
    int32_t *route_row = at<int32_t>(workspace, L.route_row);
    int32_t *offsets = at<int32_t>(workspace, L.offsets);
    MOE_TRY(launch_route_fused(r, route_chunks(s), at<int64_t>(workspace, L.counts), offsets,
                               at<int32_t>(workspace, L.recv_cum), at<int32_t>(workspace, L.sched),
                               route_row, stream));
    if (s.num_tokens == 0) return MOE_OK;
    MOE_TRY(launch_quant_scatter(r, x, route_row, at<int32_t>(workspace, L.assist),
                                 at<void>(workspace, L.q1), at<float>(workspace, L.s1), s.hidden,
                                 stream));
    void *y = at<void>(workspace, L.y);
    MOE_TRY(run_ffn_core(s, L, workspace, offsets, w1_packed, scale1, w2_packed, scale2, y, stream));
    return launch_combine(y, route_row, expert_scales, x_active_mask, s.mask_kind, shared_expert_x,
                          s.copy_experts > 0 ? x : nullptr, s.zero_experts + s.copy_experts > 0,
                          x_out, s.num_tokens, s.topk, s.hidden, cap,
                          at<int32_t>(workspace, L.status), stream);
}

moe_status moe_stage_views_get(const moe_shape *shape, int for_layer, void *workspace,
                               size_t workspace_bytes, moe_stage_views *v) {
    MOE_TRY(check_shape(shape, true));
    if (!workspace || !v) return MOE_FAIL(MOE_ERR_NULLPTR);
    const Layout L = layout_for(*shape, for_layer ? Op::Layer : Op::Ffn);
    if (workspace_bytes < L.total) return MOE_FAIL(MOE_ERR_WORKSPACE);
    memset(v, 0, sizeof *v);
    if (for_layer) {
        v->route_row = at<int32_t>(workspace, L.route_row);
        v->assist = at<int32_t>(workspace, L.assist);
        v->expert_offsets = at<int32_t>(workspace, L.offsets);
        v->expert_token_nums = at<int64_t>(workspace, L.counts);
        v->ep_recv_counts = at<int32_t>(workspace, L.recv_cum);
        v->y = at<void>(workspace, L.y);
    }
    v->q1 = at<void>(workspace, L.q1);
    v->s1 = at<float>(workspace, L.s1);
    v->g = at<float>(workspace, L.g);
    v->q2 = at<void>(workspace, L.q2);
    v->s2 = at<float>(workspace, L.s2);
    return MOE_OK;
}

// ---------------------------------------------------------------- plain grouped GEMM
static Layout gemm_layout(int64_t rows, int64_t E, int64_t N, int64_t Kd) {
    Layout L;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        size_t a = off;
        off = align_up(off + (bytes ? bytes : 1), kAlign);
        return a;
    };
    L.status = take(4);
    L.sched = take((size_t)(E + 1) * sizeof(int32_t));
    L.a_img = take((size_t)rows * Kd * 2);
    L.w_img = take((size_t)E * N * Kd * 2);
    L.total = off;
    return L;
}

moe_status moe_grouped_gemm_s32_workspace_size(int64_t rows, int64_t E, int64_t N, int64_t Kd,
                                               size_t *bytes) {
    if (!bytes) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (rows < 0 || rows > INT32_MAX || E < 1 || E > kMaxExperts || N < 8 || N % 8 != 0 || Kd < 8 ||
        Kd % 8 != 0 || N > (1 << 20) || Kd > 131072)
        return MOE_FAIL(MOE_ERR_SHAPE);
    *bytes = gemm_layout(rows, E, N, Kd).total;
    return MOE_OK;
}

moe_status moe_grouped_gemm_s32(int64_t rows, int64_t E, int64_t N, int64_t Kd,
                                const int32_t *expert_offsets, const int8_t *A, const int8_t *W,
                                int32_t *C, int path, void *workspace, size_t workspace_bytes,
                                cudaStream_t stream) {
    size_t need = 0;
    MOE_TRY(moe_grouped_gemm_s32_workspace_size(rows, E, N, Kd, &need));
    if (!expert_offsets || !A || !W || !C || !workspace) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!aligned(A, 16) || !aligned(W, 16) || !aligned(C, 16) || !aligned(workspace, kAlign))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    if (workspace_bytes < need) return MOE_FAIL(MOE_ERR_WORKSPACE);
    if (path < MOE_FFN_PATH_AUTO || path > MOE_FFN_PATH_LARGE_PAIR) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    if (path == MOE_FFN_PATH_SMALL && Kd % 16 != 0) return MOE_FAIL(MOE_ERR_SHAPE);
    const bool small = Kd % 16 == 0 && use_small_path(path, rows, E);
    if (rows == 0) return MOE_OK;
    const Layout L = gemm_layout(rows, E, N, Kd);
    MOE_TRY(launch_sched(expert_offsets, E, at<int32_t>(workspace, L.sched),
                         at<int32_t>(workspace, L.status), stream));
    MOE_TRY(launch_i8_to_f16(A, at<void>(workspace, L.a_img), rows * Kd, stream));
    if (small)
        MOE_TRY(launch_bias_i8(W, at<void>(workspace, L.w_img), E * N * Kd, stream));
    else
        MOE_TRY(launch_i8_to_f16(W, at<void>(workspace, L.w_img), E * N * Kd, stream));
    GemmArgs g{};
    g.a_img = at<void>(workspace, L.a_img);
    g.cap_rows = rows;
    g.b_img = at<void>(workspace, L.w_img);
    g.E = E;
    g.Nout = N;
    g.Kd = Kd;
    g.offsets = expert_offsets;
    g.sched = at<int32_t>(workspace, L.sched);
    g.c_s32 = C;
    g.status = at<int32_t>(workspace, L.status);
    return run_gemm(small, path, Epi::S32, g, stream);
}

}  // extern "C"
