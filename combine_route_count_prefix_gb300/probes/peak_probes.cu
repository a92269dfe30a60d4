// peak_probes.cu -- instruction-rate probes behind the roofline denominators
// (a measurement tool built and run by `bench.py --peak-probes`; not part of
// the library).
//
//   mma_s8   the legacy warp-level int8 tensor instruction (mma.sync m16n8k32,
//            int8 x int8 -> int32), the exact int8 path that sm_103a still
//            offers besides tcgen05: many warps per SM, eight independent
//            accumulator chains per warp, operands in registers, so the rate is
//            the instruction's own.
//   copy     a streaming device-to-device copy (16-byte vectors, grid-stride),
//            to set beside the measured HBM peak.
//   link     the host link with pinned (mapped) host memory, one 29.4 MB tensor
//            (2048 x 7168 bf16) per copy: DMA host-to-device, device-to-host and
//            both at once on two streams, and the same copy kernel reading the
//            host buffer directly, the bound of a step whose inputs start on the
//            host.
//
// Prints one JSON object on stdout.
#include <cstdint>
#include <cstdio>
#include <cuda_runtime.h>

#define CK(x)                                                                          \
    do {                                                                               \
        cudaError_t e_ = (x);                                                          \
        if (e_ != cudaSuccess) {                                                       \
            fprintf(stderr, "%s: %s (line %d)\n", #x, cudaGetErrorString(e_), __LINE__); \
            return 1;                                                                  \
        }                                                                              \
    } while (0)

constexpr int kChains = 8;

__global__ void __launch_bounds__(256) k_mma_s8(int iters, int32_t *out) {
    // operand fragments: any values; they stay in registers
    const uint32_t t = threadIdx.x * 2654435761u + blockIdx.x;
    const uint32_t a0 = t, a1 = t ^ 0x5a5a5a5au, a2 = t * 3u, a3 = t + 0x01010101u;
    const uint32_t b0 = t ^ 0x33333333u, b1 = t * 7u;
    int32_t acc[kChains][4];
#pragma unroll
    for (int c = 0; c < kChains; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[c][j] = 0;
    for (int i = 0; i < iters; ++i) {
#pragma unroll
        for (int c = 0; c < kChains; ++c)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, "
                "{%8,%9}, {%0,%1,%2,%3};"
                : "+r"(acc[c][0]), "+r"(acc[c][1]), "+r"(acc[c][2]), "+r"(acc[c][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int32_t s = 0;
#pragma unroll
    for (int c = 0; c < kChains; ++c)
#pragma unroll
        for (int j = 0; j < 4; ++j) s += acc[c][j];
    out[blockIdx.x * blockDim.x + threadIdx.x] = s;   // keeps the chains live
}

__global__ void k_copy(const uint4 *__restrict__ src, uint4 *__restrict__ dst, size_t n) {
    for (size_t i = blockIdx.x * (size_t)blockDim.x + threadIdx.x; i < n;
         i += (size_t)gridDim.x * blockDim.x)
        dst[i] = src[i];
}

int main() {
    int sms = 0, dev = 0;
    CK(cudaGetDevice(&dev));
    CK(cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev));
    cudaEvent_t a, b;
    CK(cudaEventCreate(&a));
    CK(cudaEventCreate(&b));

    // ---- mma.sync int8
    const int blocks = sms * 8, threads = 256, iters = 4096;
    int32_t *out = nullptr;
    CK(cudaMalloc(&out, (size_t)blocks * threads * sizeof(int32_t)));
    k_mma_s8<<<blocks, threads>>>(64, out);   // warm-up
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    float best_ms = 1e30f;
    for (int r = 0; r < 5; ++r) {
        CK(cudaEventRecord(a));
        k_mma_s8<<<blocks, threads>>>(iters, out);
        CK(cudaEventRecord(b));
        CK(cudaEventSynchronize(b));
        CK(cudaGetLastError());
        float ms = 0;
        CK(cudaEventElapsedTime(&ms, a, b));
        if (ms < best_ms) best_ms = ms;
    }
    const double warps = (double)blocks * threads / 32;
    const double ops = warps * iters * kChains * (2.0 * 16 * 8 * 32);
    const double mma_tops = ops / (best_ms * 1e-3) / 1e12;

    // ---- copy, 2 GiB each way
    const size_t bytes = (size_t)2 << 30;
    void *src = nullptr, *dst = nullptr;
    CK(cudaMalloc(&src, bytes));
    CK(cudaMalloc(&dst, bytes));
    CK(cudaMemset(src, 1, bytes));
    const size_t n16 = bytes / 16;
    k_copy<<<sms * 4, 512>>>((const uint4 *)src, (uint4 *)dst, n16);
    CK(cudaGetLastError());
    CK(cudaDeviceSynchronize());
    float copy_ms = 1e30f;
    for (int r = 0; r < 5; ++r) {
        CK(cudaEventRecord(a));
        k_copy<<<sms * 4, 512>>>((const uint4 *)src, (uint4 *)dst, n16);
        CK(cudaEventRecord(b));
        CK(cudaEventSynchronize(b));
        CK(cudaGetLastError());
        float ms = 0;
        CK(cudaEventElapsedTime(&ms, a, b));
        if (ms < copy_ms) copy_ms = ms;
    }
    const double copy_gbs = 2.0 * bytes / (copy_ms * 1e-3) / 1e9;
    CK(cudaFree(src));
    CK(cudaFree(dst));

    // ---- host link
    const size_t lb = (size_t)2048 * 7168 * 2;
    void *h_in = nullptr, *h_out = nullptr, *dh_in = nullptr, *d_a = nullptr, *d_b = nullptr;
    CK(cudaHostAlloc(&h_in, lb, cudaHostAllocMapped));
    CK(cudaHostAlloc(&h_out, lb, cudaHostAllocMapped));
    CK(cudaHostGetDevicePointer(&dh_in, h_in, 0));
    CK(cudaMalloc(&d_a, lb));
    CK(cudaMalloc(&d_b, lb));
    CK(cudaMemset(d_b, 2, lb));
    for (size_t i = 0; i < lb; ++i) ((unsigned char *)h_in)[i] = (unsigned char)i;
    cudaStream_t s0, s1;
    CK(cudaStreamCreateWithFlags(&s0, cudaStreamNonBlocking));
    CK(cudaStreamCreateWithFlags(&s1, cudaStreamNonBlocking));
    cudaEvent_t join;
    CK(cudaEventCreateWithFlags(&join, cudaEventDisableTiming));
    // kind 0: DMA in, 1: DMA out, 2: both (two streams), 3: copy kernel reading host memory
    double link_gbs[4];
    for (int kind = 0; kind < 4; ++kind) {
        float best = 1e30f;
        for (int r = 0; r < 8; ++r) {   // the first three runs are warm-up
            CK(cudaEventRecord(a, s0));
            if (kind == 0 || kind == 2) CK(cudaMemcpyAsync(d_a, h_in, lb, cudaMemcpyHostToDevice, s0));
            if (kind == 1) CK(cudaMemcpyAsync(h_out, d_b, lb, cudaMemcpyDeviceToHost, s0));
            if (kind == 2) {
                CK(cudaStreamWaitEvent(s1, a, 0));   // starts with the copy in: both run together
                CK(cudaMemcpyAsync(h_out, d_b, lb, cudaMemcpyDeviceToHost, s1));
                CK(cudaEventRecord(join, s1));
                CK(cudaStreamWaitEvent(s0, join, 0));
            }
            if (kind == 3) k_copy<<<sms * 2, 512, 0, s0>>>((const uint4 *)dh_in, (uint4 *)d_a, lb / 16);
            CK(cudaEventRecord(b, s0));
            CK(cudaEventSynchronize(b));
            CK(cudaGetLastError());
            float ms = 0;
            CK(cudaEventElapsedTime(&ms, a, b));
            if (r >= 3 && ms < best) best = ms;
        }
        link_gbs[kind] = (kind == 2 ? 2.0 : 1.0) * lb / (best * 1e-3) / 1e9;
    }
    CK(cudaMemcpy(h_out, d_a, lb, cudaMemcpyDeviceToHost));   // the direct read delivered the host bytes
    for (size_t i = 0; i < lb; i += 4093)
        if (((unsigned char *)h_out)[i] != (unsigned char)i) {
            fprintf(stderr, "host-read copy mismatch at %zu\n", i);
            return 1;
        }

    printf("{\"sms\": %d, \"mma_sync_s8_tops\": %.1f, \"mma_sync_s8_ms\": %.3f, "
           "\"copy_gbs\": %.1f, \"copy_ms\": %.3f, \"link_h2d_dma_gbs\": %.1f, "
           "\"link_d2h_dma_gbs\": %.1f, \"link_bidir_dma_gbs\": %.1f, "
           "\"link_h2d_sm_gbs\": %.1f, \"link_bytes\": %zu}\n",
           sms, mma_tops, best_ms, copy_gbs, copy_ms, link_gbs[0], link_gbs[1], link_gbs[2],
           link_gbs[3], lb);
    CK(cudaFree(out));
    CK(cudaFree(d_a));
    CK(cudaFree(d_b));
    CK(cudaFreeHost(h_in));
    CK(cudaFreeHost(h_out));
    return 0;
}
