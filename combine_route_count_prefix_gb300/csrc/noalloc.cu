// noalloc.cu -- moe_dispatch_noalloc: dispatch for callers that cannot
// allocate device memory.
//
// moe_dispatch needs a caller-provided workspace for its routing scratch (the
// per-chunk expert histograms, the per-chunk invalid-id flags and the status
// word).  Some callers have no way to provide one: a runtime whose device
// memory is planned once at load time and may not grow afterwards, a plugin
// inside a host framework that exposes no allocator, or code on a latency
// path where an allocation (and the synchronisation it can imply) is not
// allowed.  For them this entry point keeps the scratch in a fixed array in
// the library's own device memory instead.
//
// The array is a file-scope __device__ variable, so every GPU that loads the
// library holds it (kNoAllocScratchBytes plus a small header) until the
// process exits.  Host code cannot use the array's name as a device address;
// the address is looked up once per device with cudaGetSymbolAddress, on the
// first call made while that device is current, and cached.  That first call
// must therefore happen before any stream capture on that device.
//
// Every call shares the one array.  The routing kernels overwrite every
// scratch entry they read (histograms, flags and the status word are written
// before they are read in each call), so nothing has to be cleared between
// calls; but two calls whose kernels overlap on the GPU (different streams,
// or different host threads) race on the array and give wrong results.
#include "common.cuh"

#include <mutex>

namespace moe {
namespace {

// Scratch limit: histograms plus flags, in int32 entries.
constexpr size_t kNoAllocScratchEntries = 262144;                 // 1 MiB
constexpr size_t kNoAllocHeaderBytes = 256;                       // status word
constexpr size_t kNoAllocScratchBytes =
    kNoAllocHeaderBytes + kNoAllocScratchEntries * sizeof(int32_t);

static __device__ __align__(256) uint8_t g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mu;
void *g_noalloc_addr[kMaxDevices] = {nullptr};

// Device address of the scratch array for the current device (set-up on the
// first call per device).
moe_status noalloc_scratch(uint8_t **out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_FAIL(MOE_ERR_CUDA);
    std::lock_guard<std::mutex> lk(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) {
            cudaGetLastError();
            return MOE_FAIL(MOE_ERR_CUDA);
        }
        g_noalloc_addr[dev] = p;
    }
    *out = static_cast<uint8_t *>(g_noalloc_addr[dev]);
    return MOE_OK;
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

size_t moe_dispatch_noalloc_scratch_bytes(void) { return kNoAllocScratchBytes; }

moe_status moe_dispatch_noalloc(const moe_shape *shape, const void *x, const int32_t *expert_ids,
                                const uint8_t *x_active_mask, void *expand_x, int32_t *assist,
                                int64_t *expert_token_nums, int32_t *expert_offsets,
                                int32_t *ep_recv_counts, int32_t *route_row,
                                cudaStream_t stream) {
    MOE_TRY(check_shape(shape, false));
    const moe_shape &s = *shape;
    const bool empty = s.num_tokens == 0;
    if (!expert_token_nums || !expert_offsets || !ep_recv_counts) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && (!expert_ids || !assist || !route_row)) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && expand_x && !x) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (!empty && s.mask_kind != 0 && !x_active_mask) return MOE_FAIL(MOE_ERR_NULLPTR);
    if (s.mask_kind == 0 && x_active_mask) return MOE_FAIL(MOE_ERR_PARAM_INVALID);
    // the same alignment rules as moe_dispatch: 16-byte row vectors, 8-byte
    // counts, 4-byte indices
    auto misaligned = [](const void *ptr, uintptr_t a) { return ((uintptr_t)ptr % a) != 0; };
    if (expand_x && (misaligned(x, 16) || misaligned(expand_x, 16))) return MOE_FAIL(MOE_ERR_ALIGNMENT);
    if (misaligned(expert_ids, 4) || misaligned(assist, 4) || misaligned(expert_token_nums, 8) ||
        misaligned(expert_offsets, 4) || misaligned(ep_recv_counts, 4) || misaligned(route_row, 4))
        return MOE_FAIL(MOE_ERR_ALIGNMENT);
    const int64_t chunks = route_chunks(s);
    const size_t entries = (size_t)(chunks * s.num_experts + chunks);
    if (entries > kNoAllocScratchEntries) return MOE_FAIL(MOE_ERR_TOO_LARGE);

    uint8_t *scratch = nullptr;
    MOE_TRY(noalloc_scratch(&scratch));

    RouteDev r;
    r.ids = expert_ids;
    r.mask = x_active_mask;
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
    r.status = reinterpret_cast<int32_t *>(scratch);
    r.hist = reinterpret_cast<int32_t *>(scratch + kNoAllocHeaderBytes);
    r.bad = r.hist + chunks * s.num_experts;
    r.rows_final = 0;
    MOE_TRY(launch_route_fused(r, chunks, expert_token_nums, expert_offsets, ep_recv_counts,
                               nullptr, route_row, stream));
    if (expand_x) return launch_dispatch_rows(r, x, route_row, assist, expand_x, s.hidden, stream);
    return launch_route_resolve(r, route_row, assist, stream);
}

}  // extern "C"
