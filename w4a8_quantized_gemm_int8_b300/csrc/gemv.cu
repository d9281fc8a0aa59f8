// M = 1 INT8 GEMV: the decode-time path of the quantized linear layer.
//
// It computes the same function as the GEMM at M = 1 (the token is
// quantized per token to INT8, the int32 dot products are exact, the same
// dequant epilogue follows), so routing on M never changes a result. Cider
// README, section "Metal Kernel Pipeline", "Decode (M = 1)": a dedicated
// matrix-vector kernel; section "Quantization" for the arithmetic.
//
// B300 design: the op is a stream of N*K weight bytes (N*K/2 for INT4) from
// HBM. Each CTA first quantizes x into shared memory (x is a few KB and sits
// in L2; its first weight loads are already in flight meanwhile), then each
// warp walks whole weight rows with 16-byte coalesced loads, eight in flight
// per lane and the next block issued before the current one is consumed.
// Dot products use dp4a (4 x int8 -> int32); INT4 nibbles are widened to
// signed bytes in registers. Per-group partials are reduced across the lanes
// that hold one group, rescaled, and summed in ascending group order.
#include <cuda_fp16.h>
#include <cstdint>

#include "kernels.h"

namespace cider {
namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;
constexpr int kUnroll = 8;           // 16-byte chunks in flight per lane
constexpr int kMaxK = 16384;         // codes kept in shared memory
constexpr int kMaxGroups = kMaxK / 32;

struct Params {
    const __half* x;
    int K, N;
    const uint8_t* w;  // row-major, K bytes (int8) or K/2 bytes (int4) per row
    const float* s_w;
    int G;             // columns of s_w (1 for per-channel)
    int cpg;           // 16-byte chunks per group (per-group only)
    __half* y;
};

__device__ __forceinline__ uint4 ld_stream(const uint4* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ int dp4a(int a, int b, int c) { return __dp4a(a, b, c); }

// Packed INT4 word (elements 2j in low nibbles) -> two words of four signed
// bytes each, in element order, nibble b decoded as b - 8.
__device__ __forceinline__ void widen_nibbles(uint32_t wd, int& e0, int& e1) {
    const uint32_t lo = wd & 0x0F0F0F0Fu;
    const uint32_t hi = (wd >> 4) & 0x0F0F0F0Fu;
    e0 = (int)__vsub4(__byte_perm(lo, hi, 0x5140), 0x08080808u);
    e1 = (int)__vsub4(__byte_perm(lo, hi, 0x7362), 0x08080808u);
}

template <int BITS>
__device__ __forceinline__ int chunk_dot(const uint4& wv, const uint4* codes, int c) {
    if constexpr (BITS == 8) {
        const uint4 q = codes[c];
        int acc = dp4a((int)wv.x, (int)q.x, 0);
        acc = dp4a((int)wv.y, (int)q.y, acc);
        acc = dp4a((int)wv.z, (int)q.z, acc);
        return dp4a((int)wv.w, (int)q.w, acc);
    } else {
        const uint4 q0 = codes[2 * c], q1 = codes[2 * c + 1];
        int e0, e1, acc;
        widen_nibbles(wv.x, e0, e1);
        acc = dp4a(e0, (int)q0.x, 0);
        acc = dp4a(e1, (int)q0.y, acc);
        widen_nibbles(wv.y, e0, e1);
        acc = dp4a(e0, (int)q0.z, acc);
        acc = dp4a(e1, (int)q0.w, acc);
        widen_nibbles(wv.z, e0, e1);
        acc = dp4a(e0, (int)q1.x, acc);
        acc = dp4a(e1, (int)q1.y, acc);
        widen_nibbles(wv.w, e0, e1);
        acc = dp4a(e0, (int)q1.z, acc);
        return dp4a(e1, (int)q1.w, acc);
    }
}

template <int BITS, bool PG>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const Params p) {
    __shared__ __align__(16) int8_t codes_s[kMaxK];
    __shared__ float prod_s[PG ? kWarps : 1][PG ? kMaxGroups : 1];
    __shared__ float red_s[kWarps];
    __shared__ float sa_s;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int row_bytes = (BITS == 8) ? p.K : p.K / 2;
    const int nchunk = row_bytes / 16;
    const int row_stride = gridDim.x * kWarps;
    const uint4* codes = reinterpret_cast<const uint4*>(codes_s);

    // Block iterator over (row, first chunk) of this warp's work.
    int n = blockIdx.x * kWarps + warp;
    int c0 = 0;
    uint4 cur[kUnroll];
    auto load_block = [&](uint4 (&dst)[kUnroll], int rn, int rc0) {
        const uint4* row = reinterpret_cast<const uint4*>(p.w + (int64_t)rn * row_bytes);
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int c = rc0 + u * 32 + lane;
            if (c < nchunk) dst[u] = ld_stream(row + c);
        }
    };
    if (n < p.N) load_block(cur, n, 0);

    // ---- per-token quantization of x (each CTA, from L2) -------------------
    {
        const uint4* xv = reinterpret_cast<const uint4*>(p.x);
        const int nvec = p.K / 8;
        __half2 hm = __float2half2_rn(0.0f);
        for (int v = threadIdx.x; v < nvec; v += kThreads) {
            uint4 u = __ldg(xv + v);
            const __half2* h = reinterpret_cast<const __half2*>(&u);
#pragma unroll
            for (int i = 0; i < 4; ++i) hm = __hmax2(hm, __habs2(h[i]));
        }
        float m = fmaxf(__low2float(hm), __high2float(hm));
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) red_s[warp] = m;
        __syncthreads();
        if (threadIdx.x == 0) {
            float a = red_s[0];
            for (int w = 1; w < kWarps; ++w) a = fmaxf(a, red_s[w]);
            sa_s = (a == 0.0f) ? 0.0f : __fdiv_rn(a, 127.0f);
        }
        __syncthreads();
        const float s = sa_s;
        for (int v = threadIdx.x; v < nvec; v += kThreads) {
            uint4 u = __ldg(xv + v);
            const __half* h = reinterpret_cast<const __half*>(&u);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                int q = 0;
                if (s != 0.0f) {
                    q = __float2int_rn(__fdiv_rn(__half2float(h[i]), s));
                    q = q > 127 ? 127 : (q < -127 ? -127 : q);
                }
                if (i < 4)
                    lo |= (uint32_t)(q & 0xFF) << (8 * i);
                else
                    hi |= (uint32_t)(q & 0xFF) << (8 * (i - 4));
            }
            reinterpret_cast<uint2*>(codes_s)[v] = make_uint2(lo, hi);
        }
        __syncthreads();
    }
    const float s_a = sa_s;

    // ---- weight stream --------------------------------------------------------
    int lane_acc = 0;  // per-channel: this lane's share of the row's int32 sum
    while (n < p.N) {
        int nn = n, nc0 = c0 + kUnroll * 32;
        if (nc0 >= nchunk) {
            nn = n + row_stride;
            nc0 = 0;
        }
        uint4 nxt[kUnroll];
        if (nn < p.N) load_block(nxt, nn, nc0);

#pragma unroll
        for (int u = 0; u < kUnroll; ++u) {
            const int cbase = c0 + u * 32;  // warp-uniform
            if (cbase >= nchunk) break;
            const int c = cbase + lane;
            int part = (c < nchunk) ? chunk_dot<BITS>(cur[u], codes, c) : 0;
            if constexpr (!PG) {
                lane_acc += part;
            } else {
                for (int o = 1; o < p.cpg; o <<= 1) part += __shfl_xor_sync(0xffffffffu, part, o);
                if ((lane % p.cpg) == 0 && c < nchunk) {
                    const int g = c / p.cpg;
                    prod_s[warp][g] =
                        __fmul_rn(__int2float_rn(part), __ldg(p.s_w + (int64_t)n * p.G + g));
                }
            }
        }

        if (nc0 == 0) {  // row n complete
            if constexpr (!PG) {
                int a = lane_acc;
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) a += __shfl_xor_sync(0xffffffffu, a, o);
                if (lane == 0) {
                    const float t = __fmul_rn(__fmul_rn(__int2float_rn(a), s_a), __ldg(p.s_w + n));
                    p.y[n] = __float2half_rn(t);
                }
                lane_acc = 0;
            } else {
                __syncwarp();
                if (lane == 0) {
                    float f = 0.0f;
                    for (int g = 0; g < p.G; ++g) f = __fadd_rn(f, prod_s[warp][g]);
                    p.y[n] = __float2half_rn(__fmul_rn(f, s_a));
                }
                __syncwarp();
            }
        }
#pragma unroll
        for (int u = 0; u < kUnroll; ++u) cur[u] = nxt[u];
        n = nn;
        c0 = nc0;
    }
}

template <int BITS, bool PG>
cudaError_t launch_one(const Params& p, int num_sms, cudaStream_t stream) {
    int grid = num_sms * 2;
    const int rows_per_cta = kWarps;
    const int need = (p.N + rows_per_cta - 1) / rows_per_cta;
    if (need < grid) grid = need;
    gemv_kernel<BITS, PG><<<grid, kThreads, 0, stream>>>(p);
    return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, int num_sms, cudaStream_t stream) {
    if (a.K <= 0 || a.N <= 0 || a.K > kMaxK || a.N > INT32_MAX) return cudaErrorInvalidValue;
    if (a.bits != 8 && a.bits != 4) return cudaErrorInvalidValue;
    const int chunk_elems = (a.bits == 8) ? 16 : 32;
    if (a.K % chunk_elems != 0) return cudaErrorInvalidValue;
    Params p{};
    p.x = a.x;
    p.K = (int)a.K;
    p.N = (int)a.N;
    p.w = static_cast<const uint8_t*>(a.w);
    p.s_w = a.s_w;
    p.y = a.y;
    if (a.group_size == 0) {
        p.G = 1;
        p.cpg = 0;
    } else {
        if (a.group_size % chunk_elems != 0 || a.K % a.group_size != 0) return cudaErrorInvalidValue;
        p.G = (int)(a.K / a.group_size);
        p.cpg = a.group_size / chunk_elems;
        if (p.cpg > 32 || (p.cpg & (p.cpg - 1)) != 0 || p.G > kMaxGroups)
            return cudaErrorInvalidValue;
    }
    const bool pg = a.group_size != 0;
    if (a.bits == 8)
        return pg ? launch_one<8, true>(p, num_sms, stream) : launch_one<8, false>(p, num_sms, stream);
    return pg ? launch_one<4, true>(p, num_sms, stream) : launch_one<4, false>(p, num_sms, stream);
}

}  // namespace cider
