// Symmetric min-max quantization kernels (activations per token, weights per
// output channel or per group, INT4 packing) and the operand-image kernels
// that widen INT8 / INT4 codes to exact fp16 integers for the tensor cores.
//
// Definition (Cider README, section "Quantization"): activations are
// symmetric INT8 per token; W8A8 weights symmetric INT8 per channel or per
// group of 64/128; W4A8 weights symmetric INT4 stored with zero point 8.
// Scale = absmax / qmax (fp32, IEEE division), code = clamp(rint(x / scale))
// with ties to even, an all-zero block has scale 0 and codes 0.
#include <cuda_fp16.h>
#include <algorithm>
#include <cstdint>

#include "device_common.cuh"
#include "host_once.h"
#include "kernels.h"

namespace cider {

namespace {

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

// One code: clamp(rint(x / s), -qmax, qmax); s == 0 only for all-zero blocks
// (quant_code in device_common.cuh; r = quant_recip(s)).
__device__ __forceinline__ int quant_one(float x, float s, float r, int qmax) {
    return quant_code(x, s, r, qmax);
}

template <QuantOut OUT>
__device__ __forceinline__ void store_codes8(void* out, int64_t elem, const int (&q)[8]) {
    if constexpr (OUT == QuantOut::kInt8) {
        uint32_t lo = (uint32_t)(q[0] & 0xFF) | ((uint32_t)(q[1] & 0xFF) << 8) |
                      ((uint32_t)(q[2] & 0xFF) << 16) | ((uint32_t)(q[3] & 0xFF) << 24);
        uint32_t hi = (uint32_t)(q[4] & 0xFF) | ((uint32_t)(q[5] & 0xFF) << 8) |
                      ((uint32_t)(q[6] & 0xFF) << 16) | ((uint32_t)(q[7] & 0xFF) << 24);
        *reinterpret_cast<uint2*>(static_cast<int8_t*>(out) + elem) = make_uint2(lo, hi);
    } else if constexpr (OUT == QuantOut::kF16) {
        __half2 h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
            h[i] = __halves2half2(__int2half_rn(q[2 * i]), __int2half_rn(q[2 * i + 1]));
        *reinterpret_cast<uint4*>(static_cast<__half*>(out) + elem) =
            *reinterpret_cast<const uint4*>(h);
    } else {  // kInt4: nibble = code + 8, element 2j in the low nibble of byte j
        uint32_t w = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) w |= (uint32_t)((q[i] + 8) & 0xF) << (4 * i);
        *reinterpret_cast<uint32_t*>(static_cast<uint8_t*>(out) + elem / 2) = w;
    }
}

template <QuantOut OUT>
__device__ __forceinline__ void store_code1(void* out, int64_t elem, int q) {
    if constexpr (OUT == QuantOut::kInt8) {
        static_cast<int8_t*>(out)[elem] = (int8_t)q;
    } else if constexpr (OUT == QuantOut::kF16) {
        static_cast<__half*>(out)[elem] = __int2half_rn(q);
    }
}

// One warp per (row, group). Vector path: 16-byte loads of 8 fp16 (or bf16)
// values; requires K % 8 == 0 and gs % 8 == 0 (the host checks alignment).
template <typename T, QuantOut OUT>
__global__ void __launch_bounds__(256) quant_groups_vec_kernel(const T* __restrict__ src,
                                                               int64_t rows, int64_t K, int64_t gs,
                                                               int qmax, void* __restrict__ out,
                                                               float* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t G = K / gs;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    const int64_t nvec = gs >> 3;
    for (int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         item < rows * G; item += nwarps) {
        const int64_t row = item / G, g = item - row * G;
        const int64_t base = row * K + g * gs;
        const uint4* p = reinterpret_cast<const uint4*>(src + base);
        float amax = 0.0f;
        for (int64_t v = lane; v < nvec; v += 32) amax = fmaxf(amax, vec8_absmax<T>(__ldg(p + v)));
        amax = warp_max(amax);
        const float s = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, (float)qmax);
        const float r = quant_recip(s);
        if (lane == 0) scales[item] = s;
        for (int64_t v = lane; v < nvec; v += 32) {
            uint4 u = __ldg(p + v);
            const T* h = reinterpret_cast<const T*>(&u);
            int q[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) q[i] = quant_one(elem_to_float(h[i]), s, r, qmax);
            store_codes8<OUT>(out, base + v * 8, q);
        }
    }
}

// One pass per row (groups of the whole row, gs == K): each row is read once
// into registers (VPT 16-byte vectors per thread, all loads issued before any
// use), reduced to its absmax, and quantized from the registers. WPR = 1: one
// warp per row (K <= 256 * VPT); WPR = 8: the whole 256-thread block per row
// (K <= 2048 * VPT). Same arithmetic as quant_groups_vec_kernel.
template <typename T, QuantOut OUT, int VPT, int WPR>
__device__ __forceinline__ void quant_rows_reg_body(const T* __restrict__ src, int64_t rows,
                                                    int64_t K, int qmax, void* __restrict__ out,
                                                    float* __restrict__ scales, int block,
                                                    int nblocks) {
    static_assert(WPR == 1 || WPR == 8, "one warp or one block per row");
    __shared__ float red_s[8];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    constexpr int kRowsPerBlock = 8 / WPR;
    constexpr int kThreadsPerRow = 32 * WPR;
    const int t = (WPR == 1) ? lane : threadIdx.x;
    const int64_t nvec = K >> 3;
    for (int64_t row = (int64_t)block * kRowsPerBlock + (WPR == 1 ? warp : 0); row < rows;
         row += (int64_t)nblocks * kRowsPerBlock) {
        const uint4* p = reinterpret_cast<const uint4*>(src + row * K);
        uint4 v[VPT];
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t c = t + (int64_t)i * kThreadsPerRow;
            v[i] = (c < nvec) ? __ldg(p + c) : make_uint4(0u, 0u, 0u, 0u);
        }
        float amax = 0.0f;
#pragma unroll
        for (int i = 0; i < VPT; ++i) amax = fmaxf(amax, vec8_absmax<T>(v[i]));
        amax = warp_max(amax);
        if constexpr (WPR == 8) {
            if (lane == 0) red_s[warp] = amax;
            __syncthreads();
#pragma unroll
            for (int w = 0; w < 8; ++w) amax = fmaxf(amax, red_s[w]);
            __syncthreads();  // red_s is reused by the next row
        }
        const float s = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, (float)qmax);
        const float r = quant_recip(s);
        if (t == 0) scales[row] = s;
        // Codes by the reciprocal screen (quant_code); a warp in which any
        // lane has a value near a rounding boundary redoes that vector with
        // the correctly rounded division (a warp-uniform branch, rarely taken).
        // Padding vectors hold zeros, so every lane votes on every vector.
#pragma unroll
        for (int i = 0; i < VPT; ++i) {
            const int64_t c = t + (int64_t)i * kThreadsPerRow;
            const T* h = reinterpret_cast<const T*>(&v[i]);
            int q[8];
            bool near = false;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const float tq = __fmul_rn(elem_to_float(h[j]), r);
                const float rq = rintf(tq);
                near |= !(fabsf(tq - rq) < 0.5f - 0x1p-12f);
                q[j] = (int)rq;
            }
            if (__any_sync(0xffffffffu, near)) {
#pragma unroll
                for (int j = 0; j < 8; ++j)
                    q[j] = (s == 0.0f) ? 0 : __float2int_rn(__fdiv_rn(elem_to_float(h[j]), s));
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) q[j] = max(-qmax, min(qmax, q[j]));
            if (c < nvec) store_codes8<OUT>(out, row * K + c * 8, q);
        }
    }
}

template <typename T, QuantOut OUT, int VPT, int WPR>
__global__ void __launch_bounds__(256) quant_rows_reg_kernel(const T* __restrict__ src,
                                                             int64_t rows, int64_t K, int qmax,
                                                             void* __restrict__ out,
                                                             float* __restrict__ scales) {
    grid_dep_wait();
    grid_dep_launch();
    quant_rows_reg_body<T, OUT, VPT, WPR>(src, rows, K, qmax, out, scales, blockIdx.x, gridDim.x);
}

// Scalar fallback for shapes the vector path does not take (int8 / fp16 out).
template <typename T, QuantOut OUT>
__global__ void __launch_bounds__(256) quant_groups_scalar_kernel(const T* __restrict__ src,
                                                                  int64_t rows, int64_t K,
                                                                  int64_t gs, int qmax,
                                                                  void* __restrict__ out,
                                                                  float* __restrict__ scales) {
    const int lane = threadIdx.x & 31;
    const int64_t G = K / gs;
    const int64_t nwarps = (int64_t)gridDim.x * (blockDim.x >> 5);
    for (int64_t item = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
         item < rows * G; item += nwarps) {
        const int64_t row = item / G, g = item - row * G;
        const int64_t base = row * K + g * gs;
        float amax = 0.0f;
        for (int64_t k = lane; k < gs; k += 32) amax = fmaxf(amax, fabsf(elem_to_float(src[base + k])));
        amax = warp_max(amax);
        const float s = (amax == 0.0f) ? 0.0f : __fdiv_rn(amax, (float)qmax);
        const float r = quant_recip(s);
        if (lane == 0) scales[item] = s;
        for (int64_t k = lane; k < gs; k += 32)
            store_code1<OUT>(out, base + k, quant_one(elem_to_float(src[base + k]), s, r, qmax));
    }
}

// Percentile-clipped scales (weight preparation, offline): one block per
// (row, group). The |w| of the group, as fp32 bit patterns (which order like
// the values for non-negative numbers), are sorted in shared memory with a
// bitonic network (padding sorts last); the clip value is the pct-th
// percentile by linear interpolation between order statistics (position
// (n - 1) pct / 100, in fp64, rounded to fp32); scale = clip / qmax and codes
// clamp(rint(w / scale)). Requires gs % 8 == 0 (8-element vectors).
template <typename T, QuantOut OUT>
__global__ void __launch_bounds__(256) quant_groups_pct_kernel(const T* __restrict__ src,
                                                               int64_t rows, int64_t K,
                                                               int64_t gs, int qmax, double pct,
                                                               int npad, void* __restrict__ out,
                                                               float* __restrict__ scales) {
    extern __shared__ uint32_t keys[];
    __shared__ float clip_s;
    const int64_t G = K / gs;
    const int64_t item = blockIdx.x;
    if (item >= rows * G) return;
    const int64_t row = item / G, g = item - row * G;
    const int64_t base = row * K + g * gs;
    for (int i = threadIdx.x; i < npad; i += blockDim.x)
        keys[i] = (i < gs) ? __float_as_uint(fabsf(elem_to_float(src[base + i]))) : 0xFFFFFFFFu;
    __syncthreads();
    for (int k = 2; k <= npad; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            for (int i = threadIdx.x; i < npad; i += blockDim.x) {
                const int ixj = i ^ j;
                if (ixj > i) {
                    const uint32_t a = keys[i], b = keys[ixj];
                    if ((a > b) == ((i & k) == 0)) {
                        keys[i] = b;
                        keys[ixj] = a;
                    }
                }
            }
            __syncthreads();
        }
    }
    if (threadIdx.x == 0) {
        const double h = (double)(gs - 1) * pct / 100.0;
        const int64_t i = (int64_t)floor(h);
        const double lo = (double)__uint_as_float(keys[i]);
        const double c =
            (i + 1 < gs) ? lo + (h - (double)i) * ((double)__uint_as_float(keys[i + 1]) - lo) : lo;
        clip_s = (float)c;
    }
    __syncthreads();
    const float clip = clip_s;
    const float s = (clip == 0.0f) ? 0.0f : __fdiv_rn(clip, (float)qmax);
    if (threadIdx.x == 0) scales[item] = s;
    for (int64_t v = threadIdx.x; v < gs / 8; v += blockDim.x) {
        int q[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const float x = elem_to_float(src[base + 8 * v + j]);
            int c = (s == 0.0f) ? 0 : __float2int_rn(__fdiv_rn(x, s));
            q[j] = max(-qmax, min(qmax, c));
        }
        store_codes8<OUT>(out, base + 8 * v, q);
    }
}

// INT8 codes -> exact fp16 integers (operand image), 16 codes per thread step,
// four steps' loads in flight per thread.
__device__ __forceinline__ void widen_i8_body(const int8_t* __restrict__ src, int64_t n16,
                                              __half* __restrict__ dst, int block, int nblocks) {
    constexpr int U = 4;
    const int64_t stride = (int64_t)nblocks * blockDim.x;
    for (int64_t i0 = (int64_t)block * blockDim.x + threadIdx.x; i0 < n16; i0 += U * stride) {
        int4 u[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * stride;
            if (i < n16) u[k] = __ldg(reinterpret_cast<const int4*>(src) + i);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * stride;
            if (i >= n16) break;
            const int8_t* b = reinterpret_cast<const int8_t*>(&u[k]);
            __half2 h[8];
#pragma unroll
            for (int j = 0; j < 8; ++j)
                h[j] = __halves2half2(__short2half_rn(b[2 * j]), __short2half_rn(b[2 * j + 1]));
            uint4* d = reinterpret_cast<uint4*>(dst) + 2 * i;
            d[0] = *reinterpret_cast<const uint4*>(&h[0]);
            d[1] = *reinterpret_cast<const uint4*>(&h[4]);
        }
    }
}

// Packed INT4 (nibble = code + 8, element 2j in the low nibble of byte j) ->
// exact fp16 integers, 32 codes (16 bytes) per thread step, four steps' loads
// in flight per thread.
__device__ __forceinline__ void widen_i4_body(const uint8_t* __restrict__ src, int64_t n16,
                                              __half* __restrict__ dst, int block, int nblocks) {
    constexpr int U = 4;
    const int64_t stride = (int64_t)nblocks * blockDim.x;
    for (int64_t i0 = (int64_t)block * blockDim.x + threadIdx.x; i0 < n16; i0 += U * stride) {
        uint4 u[U];
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * stride;
            if (i < n16) u[k] = __ldg(reinterpret_cast<const uint4*>(src) + i);
        }
#pragma unroll
        for (int k = 0; k < U; ++k) {
            const int64_t i = i0 + k * stride;
            if (i >= n16) break;
            const uint8_t* b = reinterpret_cast<const uint8_t*>(&u[k]);
            __half2 h[16];
#pragma unroll
            for (int j = 0; j < 16; ++j)
                h[j] = __halves2half2(__short2half_rn((short)(b[j] & 0xF) - 8),
                                      __short2half_rn((short)(b[j] >> 4) - 8));
            uint4* d = reinterpret_cast<uint4*>(dst) + 4 * i;
#pragma unroll
            for (int j = 0; j < 4; ++j) d[j] = *reinterpret_cast<const uint4*>(&h[4 * j]);
        }
    }
}

__global__ void __launch_bounds__(256) widen_i8_kernel(const int8_t* __restrict__ src, int64_t n16,
                                                       __half* __restrict__ dst) {
    grid_dep_wait();
    grid_dep_launch();
    widen_i8_body(src, n16, dst, blockIdx.x, gridDim.x);
}

__global__ void __launch_bounds__(256) widen_i4_kernel(const uint8_t* __restrict__ src,
                                                       int64_t n16, __half* __restrict__ dst) {
    grid_dep_wait();
    grid_dep_launch();
    widen_i4_body(src, n16, dst, blockIdx.x, gridDim.x);
}

// Both operand images of the tensor-core GEMM in one launch: blocks
// [0, a_blocks) quantize the activation rows into exact fp16 codes and their
// scales; the remaining blocks widen the weight codes (INT8 or packed INT4)
// into exact fp16 integers. The two jobs are independent and share the GPU.
struct ImagesArgs {
    const void* x;  // fp16 or bf16 [M, K] (kernel template parameter)
    int64_t M, K;
    __half* a_img;
    float* s_a;
    const void* w;
    int64_t n16;      // 16-byte weight chunks
    __half* b_img;
    int a_blocks;
    const float* s_w;  // per-group weight scales [N, G] (NULL: nothing to transpose)
    float* s_wT;       // their group-major copy [G, N]
    int64_t N, G;
};

// Group-major copy of per-group scales: s_wT[g, n] = s_w[n, g] (writes
// coalesced along n), so the GEMM epilogue fetches one group's scales for a
// run of output channels as contiguous bytes.
__device__ __forceinline__ void transpose_scales_body(const float* __restrict__ s_w,
                                                      float* __restrict__ s_wT, int64_t N,
                                                      int64_t G, int block, int nblocks) {
    const int64_t total = N * G;
    for (int64_t i = (int64_t)block * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)nblocks * blockDim.x) {
        const int64_t g = i / N, n = i - g * N;
        s_wT[i] = __ldg(s_w + n * G + g);
    }
}

template <typename T, int VPT, int WPR, int BITS>
__global__ void __launch_bounds__(256) operand_images_kernel(const ImagesArgs a) {
    grid_dep_wait();
    grid_dep_launch();
    if ((int)blockIdx.x < a.a_blocks) {
        quant_rows_reg_body<T, QuantOut::kF16, VPT, WPR>(static_cast<const T*>(a.x), a.M, a.K, 127,
                                                         a.a_img, a.s_a,
                                                       blockIdx.x, a.a_blocks);
    } else {
        const int wb = blockIdx.x - a.a_blocks, nwb = gridDim.x - a.a_blocks;
        if constexpr (BITS == 8)
            widen_i8_body(static_cast<const int8_t*>(a.w), a.n16, a.b_img, wb, nwb);
        else
            widen_i4_body(static_cast<const uint8_t*>(a.w), a.n16, a.b_img, wb, nwb);
        if (a.s_wT) transpose_scales_body(a.s_w, a.s_wT, a.N, a.G, wb, nwb);
    }
}

int grid_for(int64_t work_items, int per_block, int num_sms) {
    int64_t b = (work_items + per_block - 1) / per_block;
    int64_t cap = (int64_t)num_sms * 16;
    if (b > cap) b = cap;
    if (b < 1) b = 1;
    return (int)b;
}

}  // namespace

namespace {

template <typename T, QuantOut OUT>
cudaError_t launch_rows_reg_t(const T* src, int64_t rows, int64_t K, int qmax, void* out,
                              float* scales, int num_sms, cudaStream_t stream) {
    const int64_t nvec = K / 8;
    const int64_t cap = (int64_t)num_sms * 8;  // 8 resident blocks of 256 threads per SM
    const int g1 = (int)std::min<int64_t>((rows + 7) / 8, cap);
    const int g8 = (int)std::min<int64_t>(rows, cap);
    // Few rows: a block of eight warps per row (see launch_images_t).
    if (rows <= (int64_t)num_sms * 4) {
        if (nvec <= 256 * 2)
            return launch_pdl(quant_rows_reg_kernel<T, OUT, 2, 8>, g8, 256, 0, stream, src, rows,
                              K, qmax, out, scales);
        if (nvec <= 256 * 4)
            return launch_pdl(quant_rows_reg_kernel<T, OUT, 4, 8>, g8, 256, 0, stream, src, rows,
                              K, qmax, out, scales);
        if (nvec <= 256 * 8)
            return launch_pdl(quant_rows_reg_kernel<T, OUT, 8, 8>, g8, 256, 0, stream, src, rows,
                              K, qmax, out, scales);
    }
    if (nvec <= 32 * 4)
        return launch_pdl(quant_rows_reg_kernel<T, OUT, 4, 1>, g1, 256, 0, stream, src, rows, K,
                          qmax, out, scales);
    if (nvec <= 32 * 8)
        return launch_pdl(quant_rows_reg_kernel<T, OUT, 8, 1>, g1, 256, 0, stream, src, rows, K,
                          qmax, out, scales);
    if (nvec <= 32 * 12)
        return launch_pdl(quant_rows_reg_kernel<T, OUT, 12, 1>, g1, 256, 0, stream, src, rows, K,
                          qmax, out, scales);
    if (nvec <= 32 * 16)
        return launch_pdl(quant_rows_reg_kernel<T, OUT, 16, 1>, g1, 256, 0, stream, src, rows, K,
                          qmax, out, scales);
    if (nvec <= 256 * 8)
        return launch_pdl(quant_rows_reg_kernel<T, OUT, 8, 8>, g8, 256, 0, stream, src, rows, K,
                          qmax, out, scales);
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t launch_quant_rows_reg(const T* src, int64_t rows, int64_t K, int qmax,
                                  QuantOut out_kind, void* out, float* scales, int num_sms,
                                  cudaStream_t stream) {
    if (out_kind == QuantOut::kInt8)
        return launch_rows_reg_t<T, QuantOut::kInt8>(src, rows, K, qmax, out, scales, num_sms,
                                                     stream);
    if (out_kind == QuantOut::kF16)
        return launch_rows_reg_t<T, QuantOut::kF16>(src, rows, K, qmax, out, scales, num_sms,
                                                    stream);
    return cudaErrorNotSupported;
}

template <typename T>
cudaError_t launch_quant_groups_t(const T* src, int64_t rows, int64_t K, int64_t gs, int qmax,
                                  QuantOut out_kind, void* out, float* scales, int num_sms,
                                  cudaStream_t stream) {
    const int64_t items = rows * (K / gs);
    const bool vec = (K % 8 == 0) && (gs % 8 == 0) &&
                     (reinterpret_cast<uintptr_t>(src) % 16 == 0) &&
                     (reinterpret_cast<uintptr_t>(out) % 16 == 0);
    const int grid = grid_for(items, 8, num_sms);
    if (vec && gs == K && out_kind != QuantOut::kInt4 && K <= 16384) {
        cudaError_t e = launch_quant_rows_reg<T>(src, rows, K, qmax, out_kind, out, scales,
                                                 num_sms, stream);
        if (e != cudaErrorNotSupported) return e;
    }
    if (vec) {
        switch (out_kind) {
            case QuantOut::kInt8:
                quant_groups_vec_kernel<T, QuantOut::kInt8>
                    <<<grid, 256, 0, stream>>>(src, rows, K, gs, qmax, out, scales);
                break;
            case QuantOut::kF16:
                quant_groups_vec_kernel<T, QuantOut::kF16>
                    <<<grid, 256, 0, stream>>>(src, rows, K, gs, qmax, out, scales);
                break;
            case QuantOut::kInt4:
                quant_groups_vec_kernel<T, QuantOut::kInt4>
                    <<<grid, 256, 0, stream>>>(src, rows, K, gs, qmax, out, scales);
                break;
        }
    } else {
        switch (out_kind) {
            case QuantOut::kInt8:
                quant_groups_scalar_kernel<T, QuantOut::kInt8>
                    <<<grid, 256, 0, stream>>>(src, rows, K, gs, qmax, out, scales);
                break;
            case QuantOut::kF16:
                quant_groups_scalar_kernel<T, QuantOut::kF16>
                    <<<grid, 256, 0, stream>>>(src, rows, K, gs, qmax, out, scales);
                break;
            case QuantOut::kInt4:
                return cudaErrorInvalidValue;  // packing needs the vector path
        }
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_quant_groups(const void* src, ElemType src_type, int64_t rows, int64_t K,
                                int64_t gs, int qmax, QuantOut out_kind, void* out,
                                float* scales, int num_sms, cudaStream_t stream) {
    if (src_type == ElemType::kBF16)
        return launch_quant_groups_t(static_cast<const __nv_bfloat16*>(src), rows, K, gs, qmax,
                                     out_kind, out, scales, num_sms, stream);
    return launch_quant_groups_t(static_cast<const __half*>(src), rows, K, gs, qmax, out_kind,
                                 out, scales, num_sms, stream);
}

namespace {

// Largest sort buffer of the clipped quantizer: groups of up to 16384
// elements, padded to a power of two, 4 bytes each.
constexpr int kPctMaxSmem = 16384 * 4;

template <typename T, QuantOut OUT>
cudaError_t launch_pct_out(const T* p, int64_t rows, int64_t K, int64_t gs, int qmax, double pct,
                           int npad, size_t smem, void* out, float* scales, int64_t items,
                           cudaStream_t stream) {
    auto kern = quant_groups_pct_kernel<T, OUT>;
    // Opt in once per device to the largest buffer any call needs, so that
    // concurrent calls with different group sizes never lower it.
    static PerDevice<int> attr;
    const cudaError_t e = attr.get([&](int&) {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    kPctMaxSmem);
    });
    if (e != cudaSuccess) return e;
    kern<<<(unsigned)items, 256, smem, stream>>>(p, rows, K, gs, qmax, pct, npad, out, scales);
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_pct(const T* p, int64_t rows, int64_t K, int64_t gs, int qmax, double pct,
                       int npad, size_t smem, QuantOut out_kind, void* out, float* scales,
                       int64_t items, cudaStream_t stream) {
    if (smem > (size_t)kPctMaxSmem) return cudaErrorInvalidValue;
    if (out_kind == QuantOut::kInt8)
        return launch_pct_out<T, QuantOut::kInt8>(p, rows, K, gs, qmax, pct, npad, smem, out,
                                                  scales, items, stream);
    return launch_pct_out<T, QuantOut::kInt4>(p, rows, K, gs, qmax, pct, npad, smem, out, scales,
                                              items, stream);
}

}  // namespace

cudaError_t launch_quant_groups_pct(const void* src, ElemType src_type, int64_t rows, int64_t K,
                                    int64_t gs, int qmax, double pct, QuantOut out_kind,
                                    void* out, float* scales, cudaStream_t stream) {
    if (gs <= 0 || K % gs != 0 || gs % 8 != 0 || gs > 16384 || !(pct > 0.0) || pct > 100.0 ||
        out_kind == QuantOut::kF16)
        return cudaErrorInvalidValue;
    const int64_t items = rows * (K / gs);
    if (items <= 0 || items > INT32_MAX) return cudaErrorInvalidValue;
    int npad = 1;
    while (npad < gs) npad <<= 1;
    const size_t smem = (size_t)npad * 4;
    if (src_type == ElemType::kBF16)
        return launch_pct<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(src), rows, K, gs,
                                         qmax, pct, npad, smem, out_kind, out, scales, items,
                                         stream);
    return launch_pct<__half>(static_cast<const __half*>(src), rows, K, gs, qmax, pct, npad, smem,
                              out_kind, out, scales, items, stream);
}

cudaError_t launch_widen_i8(const int8_t* src, int64_t n, __half* dst, int num_sms,
                            cudaStream_t stream) {
    if (n % 16 != 0) return cudaErrorInvalidValue;
    const int64_t n16 = n / 16;
    return launch_pdl(widen_i8_kernel, grid_for(n16, 256 * 4, num_sms), 256, 0, stream, src, n16,
                      dst);
}

cudaError_t launch_widen_i4(const uint8_t* src, int64_t n_codes, __half* dst, int num_sms,
                            cudaStream_t stream) {
    if (n_codes % 32 != 0) return cudaErrorInvalidValue;
    const int64_t n16 = n_codes / 32;
    return launch_pdl(widen_i4_kernel, grid_for(n16, 256 * 4, num_sms), 256, 0, stream, src, n16,
                      dst);
}

namespace {

template <typename T, int BITS>
cudaError_t launch_images_t(const ImagesArgs& a0, int64_t nvec, int num_sms, cudaStream_t stream) {
    ImagesArgs a = a0;
    int64_t b_blocks = std::min<int64_t>((a.n16 + 256 * 4 - 1) / (256 * 4), (int64_t)num_sms * 4);
    if (b_blocks == 0 && a.s_wT) b_blocks = std::min<int64_t>(grid_for(a.N * a.G, 256, num_sms), num_sms);
    auto go = [&](auto kern, int64_t a_blocks) {
        a.a_blocks = (int)a_blocks;
        return launch_pdl(kern, (unsigned)(a_blocks + b_blocks), 256, 0, stream, a);
    };
    const int64_t g1 = std::min<int64_t>((a.M + 7) / 8, (int64_t)num_sms * 3);
    const int64_t g8 = std::min<int64_t>(a.M, (int64_t)num_sms * 4);
    // Few rows: a block of eight warps per row, so that the rows' loads are
    // spread over many SMs (one warp per row left most SMs idle and took
    // about 7 us at 128 x 2560).
    if (a.M <= (int64_t)num_sms * 4) {
        if (nvec <= 256 * 2) return go(operand_images_kernel<T, 2, 8, BITS>, g8);
        if (nvec <= 256 * 4) return go(operand_images_kernel<T, 4, 8, BITS>, g8);
        if (nvec <= 256 * 8) return go(operand_images_kernel<T, 8, 8, BITS>, g8);
    }
    if (nvec <= 32 * 4) return go(operand_images_kernel<T, 4, 1, BITS>, g1);
    if (nvec <= 32 * 8) return go(operand_images_kernel<T, 8, 1, BITS>, g1);
    if (nvec <= 32 * 12) return go(operand_images_kernel<T, 12, 1, BITS>, g1);
    if (nvec <= 32 * 16) return go(operand_images_kernel<T, 16, 1, BITS>, g1);
    return go(operand_images_kernel<T, 8, 8, BITS>, g8);
}

}  // namespace

__global__ void __launch_bounds__(256) transpose_scales_kernel(const float* __restrict__ s_w,
                                                               float* __restrict__ s_wT, int64_t N,
                                                               int64_t G) {
    grid_dep_wait();
    grid_dep_launch();
    transpose_scales_body(s_w, s_wT, N, G, blockIdx.x, gridDim.x);
}

cudaError_t launch_operand_images(const void* x, ElemType x_type, int64_t M, int64_t K,
                                  const void* w, int bits,
                                  int64_t N, __half* a_img, float* s_a, __half* b_img,
                                  const float* s_w, float* s_wT, int64_t G, int num_sms,
                                  cudaStream_t stream) {
    const int64_t nvec = K / 8;
    const int64_t codes_per_chunk = (bits == 8) ? 16 : 32;
    const bool fused = (K % 8 == 0) && nvec <= 256 * 8 &&
                       (reinterpret_cast<uintptr_t>(x) % 16 == 0) &&
                       (reinterpret_cast<uintptr_t>(a_img) % 16 == 0) &&
                       (w == nullptr || (N * K) % codes_per_chunk == 0);
    if (!fused) {
        cudaError_t e = launch_quant_groups(x, x_type, M, K, K, 127, QuantOut::kF16, a_img, s_a,
                                            num_sms, stream);
        if (e != cudaSuccess) return e;
        if (w != nullptr) {
            e = (bits == 8) ? launch_widen_i8(static_cast<const int8_t*>(w), N * K, b_img,
                                              num_sms, stream)
                            : launch_widen_i4(static_cast<const uint8_t*>(w), N * K, b_img,
                                              num_sms, stream);
            if (e != cudaSuccess) return e;
        }
        if (!s_wT) return e;
        return launch_pdl(transpose_scales_kernel, grid_for(N * G, 256, num_sms), 256, 0, stream,
                          s_w, s_wT, N, G);
    }
    const int64_t n16 = (w == nullptr) ? 0 : (N * K) / codes_per_chunk;
    ImagesArgs a{x, M, K, a_img, s_a, w, n16, b_img, 0, s_w, s_wT, N, G};
    if (x_type == ElemType::kBF16)
        return (bits == 8) ? launch_images_t<__nv_bfloat16, 8>(a, nvec, num_sms, stream)
                           : launch_images_t<__nv_bfloat16, 4>(a, nvec, num_sms, stream);
    return (bits == 8) ? launch_images_t<__half, 8>(a, nvec, num_sms, stream)
                       : launch_images_t<__half, 4>(a, nvec, num_sms, stream);
}

}  // namespace cider
