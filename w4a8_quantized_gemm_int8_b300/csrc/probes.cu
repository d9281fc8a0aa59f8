// Measurement kernels for the benchmark (test hooks, not part of the layer):
//  - the INT8 tensor rate this GPU offers to a register-only loop of the
//    legacy mma.sync.m16n8k32 s8 instruction (sm_103a has no integer kind of
//    tcgen05.mma), the denominator of "% INT8 peak";
//  - a plain streaming read of a buffer, launched like the GEMV (programmatic
//    dependent launch, two CTAs per SM), the ceiling a decode GEMV of the
//    same bytes is compared with.
#include <cuda_runtime.h>
#include <cstdint>

#include "device_common.cuh"
#include "kernels.h"

namespace cider {
namespace {

constexpr int kMmaThreads = 128;  // four warps per block
constexpr int kMmaChains = 8;     // independent accumulators per warp

// Each warp runs kMmaChains independent chains of `iters` MMAs (16 x 8 x 32
// INT8 products into int32, 8192 operations each) on register operands, and
// folds its accumulators into sink[thread].
__global__ void __launch_bounds__(kMmaThreads) int8_mma_loop_kernel(int64_t iters, int32_t* sink) {
    const uint32_t t = threadIdx.x + 1u;
    const uint32_t a0 = t * 0x01010101u, a1 = a0 ^ 0x5A5A5A5Au, a2 = a0 + 3u, a3 = a1 * 7u;
    const uint32_t b0 = t * 0x02030405u, b1 = b0 ^ 0x3C3C3C3Cu;
    int32_t c[kMmaChains][4] = {};
    for (int64_t i = 0; i < iters; ++i) {
#pragma unroll
        for (int j = 0; j < kMmaChains; ++j)
            asm volatile(
                "mma.sync.aligned.m16n8k32.row.col.s32.s8.s8.s32 {%0, %1, %2, %3}, "
                "{%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
                : "+r"(c[j][0]), "+r"(c[j][1]), "+r"(c[j][2]), "+r"(c[j][3])
                : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    int32_t s = 0;
#pragma unroll
    for (int j = 0; j < kMmaChains; ++j) s ^= c[j][0] ^ c[j][1] ^ c[j][2] ^ c[j][3];
    sink[blockIdx.x * kMmaThreads + threadIdx.x] = s;
}

constexpr int kReadThreads = 512;
constexpr int kReadUnroll = 4;

// Streams `n16` 16-byte vectors with kReadUnroll loads in flight per thread
// and folds them into one word per block (so the loads are not removed).
__global__ void __launch_bounds__(kReadThreads) read_bytes_kernel(const uint4* __restrict__ src,
                                                                  int64_t n16, uint32_t* sink) {
    grid_dep_wait();
    grid_dep_launch();
    const int64_t stride = (int64_t)gridDim.x * kReadThreads;
    uint32_t acc = 0;
    for (int64_t i0 = (int64_t)blockIdx.x * kReadThreads + threadIdx.x; i0 < n16;
         i0 += kReadUnroll * stride) {
        uint4 v[kReadUnroll];
#pragma unroll
        for (int u = 0; u < kReadUnroll; ++u) {
            const int64_t i = i0 + u * stride;
            v[u] = (i < n16) ? __ldg(src + i) : make_uint4(0u, 0u, 0u, 0u);
        }
#pragma unroll
        for (int u = 0; u < kReadUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) acc ^= __shfl_xor_sync(0xffffffffu, acc, o);
    __shared__ uint32_t red[kReadThreads / 32];
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = acc;
    __syncthreads();
    if (threadIdx.x == 0) {
        uint32_t r = 0;
        for (int w = 0; w < kReadThreads / 32; ++w) r ^= red[w];
        sink[blockIdx.x] = r;
    }
}

}  // namespace

cudaError_t launch_int8_mma_loop(int blocks, int64_t iters, int32_t* sink, cudaStream_t stream) {
    if (blocks <= 0 || iters <= 0) return cudaErrorInvalidValue;
    int8_mma_loop_kernel<<<blocks, kMmaThreads, 0, stream>>>(iters, sink);
    return cudaGetLastError();
}

cudaError_t launch_read_bytes(const void* src, int64_t bytes, int grid, uint32_t* sink,
                              cudaStream_t stream) {
    if (bytes <= 0 || bytes % 16 != 0 || grid <= 0) return cudaErrorInvalidValue;
    return launch_pdl(read_bytes_kernel, grid, kReadThreads, 0, stream,
                      static_cast<const uint4*>(src), bytes / 16, sink);
}

}  // namespace cider
