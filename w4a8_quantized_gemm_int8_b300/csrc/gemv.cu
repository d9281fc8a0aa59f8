// M = 1 INT8 GEMV: the decode-time path of the quantized linear layer.
//
// It computes the same function as the GEMM at M = 1 (the token is
// quantized per token to INT8, the int32 dot products are exact, the same
// dequant epilogue follows), so routing on M never changes a result. Cider
// README, section "Metal Kernel Pipeline", "Decode (M = 1)": a dedicated
// matrix-vector kernel; section "Quantization" for the arithmetic.
//
// B300 design: the op is a stream of N*K weight bytes (N*K/2 for INT4) from
// HBM, so the kernel is built to keep as many bytes in flight as HBM needs.
// Two CTAs per SM, each owning a contiguous slice of weight rows (row-major
// weights make the slice one contiguous byte range). Weights and their scales
// may be written by the kernel just before a GEMV (a weight-preparation
// call), so ahead of the wait on that kernel (programmatic dependent launch)
// the producer warp only prefetches its slice into L2; after the wait it
// stages the per-channel scales of its rows, then issues bulk
// asynchronous copies (cp.async.bulk, mbarrier completion) of whole groups of
// rows into a ring of shared-memory stages - one at once, the rest as soon as
// the consumers hold x (so x's load does not queue behind the copies); for
// the decode shapes the whole slice fits the ring. Sixteen consumer warps
// wait for the preceding kernel, quantize x into shared memory, then take
// rows from the landed stages: dp4a (4 x int8 -> int32) over 16-byte
// chunks, INT4 nibbles widened to signed bytes in registers. Per-group
// scales travel in the same stage as their rows (when 16-byte aligned); the
// per-group partials are rescaled and summed in ascending group order by one
// lane. Every mbarrier wait is bounded and reports to the device status word.
#include <cuda_fp16.h>
#include <cstdint>

#include "device_common.cuh"
#include "host_once.h"
#include "kernels.h"

namespace cider {
namespace {

constexpr int kConsumerWarps = 16;
constexpr int kConsumers = kConsumerWarps * 32;
constexpr int kThreads = kConsumers + 32;  // + one producer warp
constexpr int kMaxK = 16384;
constexpr int kStageTarget = 16384;        // weight bytes per stage (at least one row)
constexpr int kMaxStages = 32;
constexpr int kUnroll = 4;          // 16-byte chunks per lane loaded before use
constexpr int kXVec = kMaxK / 8 / kConsumers;  // 8-element x vectors per consumer thread
static_assert(kMaxK % (8 * kConsumers) == 0, "x vectors per thread");
constexpr int kEarlyStages = 1;  // copies issued before x is in registers

struct Params {
    const void* x;     // fp16 or bf16 (kernel template parameter)
    int K, N;
    const uint8_t* w;  // row-major, row_bytes per row
    const float* s_w;
    int G;             // columns of s_w (1 for per-channel)
    int cpg;           // 16-byte chunks per group (per-group only)
    void* y;           // fp16, or bf16 with y_bf16
    int y_bf16;
    int row_bytes;
    int rows_per_stage;
    int stage_bytes;     // weights + staged scales, 128-byte multiple
    int num_stages;      // ring depth
    int scales_staged;   // per-group scales copied with their rows
    int sw_in_smem;      // per-channel scales of the CTA's rows prefetched to shared memory
    int codes_off, prod_off, sw_off, bar_off, stage_off;
    uint64_t timeout_ns;
    unsigned long long* status;
};

enum : uint32_t {
    kSiteGemvProducerEmpty = 0x201,
    kSiteGemvConsumerFull = 0x202,
    kSiteGemvProducerDrain = 0x203,
    kSiteGemvScales = 0x204,
    kSiteGemvX = 0x205,
};

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

// ---- A16 mode: activations used as they are, weights dequantized ---------
// Two activations of type T packed in 32 bits -> fp32 (exact).
__device__ __forceinline__ float2 to_f2(uint32_t v, __half) {
    return __half22float2(*reinterpret_cast<const __half2*>(&v));
}
__device__ __forceinline__ float2 to_f2(uint32_t v, __nv_bfloat16) {
    return __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&v));
}

// Signed byte j of w -> fp32 (exact): the byte offset by 128 is placed under
// the exponent of 2^23 and the offset 2^23 + 128 subtracted.
__device__ __forceinline__ float byte_to_float(uint32_t w_biased, int j) {
    return __int_as_float((int)__byte_perm(w_biased, 0x4B000000u, 0x7540u | (uint32_t)j)) -
           8388736.0f;
}

// acc + the four codes of `w` (signed bytes, element order) times the four
// activations packed in x01, x23.
template <typename T>
__device__ __forceinline__ float dot4_f32(uint32_t w, uint32_t x01, uint32_t x23, float acc) {
    const uint32_t u = w ^ 0x80808080u;
    const float2 a = to_f2(x01, T()), b = to_f2(x23, T());
    acc = fmaf(a.x, byte_to_float(u, 0), acc);
    acc = fmaf(a.y, byte_to_float(u, 1), acc);
    acc = fmaf(b.x, byte_to_float(u, 2), acc);
    return fmaf(b.y, byte_to_float(u, 3), acc);
}

// fp32 dot product of one 16-byte weight chunk (16 INT8 or 32 INT4 codes)
// with the matching activations xs (16-byte vectors of 8 elements of T).
template <typename T, int BITS>
__device__ __forceinline__ float chunk_dot_a16(const uint4& wv, const uint4* xs, int c) {
    if constexpr (BITS == 8) {
        const uint4 x0 = xs[2 * c], x1 = xs[2 * c + 1];
        float acc = dot4_f32<T>(wv.x, x0.x, x0.y, 0.0f);
        acc = dot4_f32<T>(wv.y, x0.z, x0.w, acc);
        acc = dot4_f32<T>(wv.z, x1.x, x1.y, acc);
        return dot4_f32<T>(wv.w, x1.z, x1.w, acc);
    } else {
        const uint32_t wd[4] = {wv.x, wv.y, wv.z, wv.w};
        float acc = 0.0f;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint4 xv = xs[4 * c + i];
            int e0, e1;
            widen_nibbles(wd[i], e0, e1);
            acc = dot4_f32<T>((uint32_t)e0, xv.x, xv.y, acc);
            acc = dot4_f32<T>((uint32_t)e1, xv.z, xv.w, acc);
        }
        return acc;
    }
}

// One output element, rounded to nearest even as fp16 or bf16.
__device__ __forceinline__ void store_y(const Params& p, int n, float v) {
    if (p.y_bf16)
        static_cast<__nv_bfloat16*>(p.y)[n] = __float2bfloat16_rn(v);
    else
        static_cast<__half*>(p.y)[n] = __float2half_rn(v);
}

// A16 = false: the INT8 GEMV (x quantized per token, int32 dot products).
// A16 = true: the A16 decode product, y = sum_g s_w[n,g] sum_k x[k] code[n,k]
// with x used as it is and fp32 accumulation (no activation quantization).
template <typename T, int BITS, bool PG, bool A16>
__global__ void __launch_bounds__(kThreads, 2) gemv_kernel(const Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    int8_t* codes_s = reinterpret_cast<int8_t*>(smem + p.codes_off);
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* empty = full + kMaxStages;
    float* red_s = reinterpret_cast<float*>(empty + kMaxStages);  // [kConsumerWarps]
    volatile int* abort_flag = reinterpret_cast<volatile int*>(red_s + kConsumerWarps);
    uint64_t* sw_bar = reinterpret_cast<uint64_t*>(red_s + kConsumerWarps) + 1;
    uint64_t* x_bar = sw_bar + 1;
    uint8_t* stages = smem + p.stage_off;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // This CTA's rows: [n0, n0 + nrows), balanced over the grid.
    const int n0 = (int)(((int64_t)p.N * blockIdx.x) / gridDim.x);
    const int nrows = (int)(((int64_t)p.N * (blockIdx.x + 1)) / gridDim.x) - n0;
    const int R = p.rows_per_stage;
    const int nst = (nrows + R - 1) / R;
    const int NS = p.num_stages;

    if (threadIdx.x == kConsumers) {
        for (int s = 0; s < NS; ++s) {
            mbar_init(smem_u32(&full[s]), 1);
            mbar_init(smem_u32(&empty[s]), kConsumerWarps);
        }
        mbar_init(smem_u32(sw_bar), 1);
        mbar_init(smem_u32(x_bar), 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();

    float* sw_s = reinterpret_cast<float*>(smem + p.sw_off);
    if (warp == kConsumerWarps) {
        // ------------------------------ producer ------------------------------
        // Ahead of the dependency wait the CTA's weight slice (and staged
        // per-group scales) is only prefetched into L2, which returns no data:
        // the preceding kernel in the stream may be the one writing the
        // weights (a weight-preparation call), so every read that lands in
        // shared memory or registers comes after griddepcontrol.wait.
        if (lane == 0) {
            const uint8_t* src = p.w + (int64_t)n0 * p.row_bytes;
            for (int s = 0; s < nst; ++s) {
                const int rows = min(R, nrows - s * R);
                bulk_prefetch_l2(src + (int64_t)s * R * p.row_bytes, (uint32_t)rows * p.row_bytes);
            }
            if (p.scales_staged && nrows > 0)
                bulk_prefetch_l2(reinterpret_cast<const uint8_t*>(p.s_w) + (int64_t)n0 * p.G * 4,
                                 (uint32_t)nrows * p.G * 4);
        }
        grid_dep_wait();
        // Per-channel scales of the CTA's rows first: a small latency-bound
        // load that must not queue behind the bulk copies.
        if (!PG && p.sw_in_smem)
            for (int i = lane; i < nrows; i += 32) sw_s[i] = __ldg(p.s_w + n0 + i);
        __syncwarp();
        if (lane == 0) mbar_arrive(smem_u32(sw_bar));
        if (lane == 0) {
            const uint8_t* src = p.w + (int64_t)n0 * p.row_bytes;
            const uint8_t* ssrc =
                reinterpret_cast<const uint8_t*>(p.s_w) + (int64_t)n0 * p.G * 4;
            int issued = 0;
            for (int s = 0; s < nst; ++s) {
                // Past the first kEarlyStages copies, wait until the consumers
                // hold x: its load must not queue behind this CTA's bulk copies.
                if (s == kEarlyStages && !mbar_wait_bounded(smem_u32(x_bar), 0, p.timeout_ns,
                                                            abort_flag, p.status, kSiteGemvX))
                    break;
                const int slot = s % NS;
                const uint32_t use = (uint32_t)(s / NS);
                if (!mbar_wait_bounded(smem_u32(&empty[slot]), (use & 1u) ^ 1u, p.timeout_ns,
                                       abort_flag, p.status, kSiteGemvProducerEmpty))
                    break;
                const int rows = min(R, nrows - s * R);
                const uint32_t wbytes = (uint32_t)rows * p.row_bytes;
                const uint32_t sbytes = p.scales_staged ? (uint32_t)rows * p.G * 4 : 0u;
                const uint32_t fb = smem_u32(&full[slot]);
                uint8_t* dst = stages + (size_t)slot * p.stage_bytes;
                mbar_arrive_expect_tx(fb, wbytes + sbytes);
                bulk_load(smem_u32(dst), src + (int64_t)s * R * p.row_bytes, wbytes, fb);
                if (sbytes)
                    bulk_load(smem_u32(dst + (size_t)R * p.row_bytes),
                              ssrc + (int64_t)s * R * p.G * 4, sbytes, fb);
                issued = s + 1;
            }
            // No copy may still be landing when the CTA exits: wait for the
            // last use of every slot (immediate unless consumers gave up).
            for (int s = max(0, issued - NS); s < issued; ++s)
                if (!mbar_wait_drain(smem_u32(&full[s % NS]), (uint32_t)(s / NS) & 1u,
                                     p.timeout_ns))
                    report_device_error(p.status, kDevTimeout, kSiteGemvProducerDrain);
        }
        return;
    }

    // -------------------- per-token quantization of x ------------------------
    // Only the producer's L2 prefetch may run before the preceding kernel in
    // the stream has finished (programmatic dependent launch); x, weights,
    // scales and y are read or written only after this wait.
    grid_dep_wait();
    grid_dep_launch();
    {
        const uint4* xv = reinterpret_cast<const uint4*>(p.x);
        const int nvec = p.K / 8;
        uint4 xr[kXVec];
#pragma unroll
        for (int i = 0; i < kXVec; ++i) {
            const int v = threadIdx.x + i * kConsumers;
            xr[i] = (v < nvec) ? __ldg(xv + v) : make_uint4(0u, 0u, 0u, 0u);
        }
        if constexpr (A16) {
            // The activations go to shared memory as they are.
#pragma unroll
            for (int i = 0; i < kXVec; ++i) {
                const int v = threadIdx.x + i * kConsumers;
                if (v < nvec) reinterpret_cast<uint4*>(codes_s)[v] = xr[i];
            }
        }
        float m = 0.0f;
        if constexpr (!A16) {
#pragma unroll
            for (int i = 0; i < kXVec; ++i) m = fmaxf(m, vec8_absmax<T>(xr[i]));
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
        if (lane == 0) red_s[warp] = m;
        named_bar_sync(1, kConsumers);
        if (threadIdx.x == 0) mbar_arrive(smem_u32(x_bar));  // x is in registers: copies may go on
        float a = red_s[0];
#pragma unroll
        for (int w = 1; w < kConsumerWarps; ++w) a = fmaxf(a, red_s[w]);
        const float s = (a == 0.0f) ? 0.0f : __fdiv_rn(a, 127.0f);
        const float r = quant_recip(s);
#pragma unroll
        for (int i = 0; i < kXVec; ++i) {
            if constexpr (A16) break;
            const int v = threadIdx.x + i * kConsumers;
            if (v >= nvec) break;
            const T* h = reinterpret_cast<const T*>(&xr[i]);
            uint32_t lo = 0, hi = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const int q = quant_code(elem_to_float(h[j]), s, r, 127);
                if (j < 4)
                    lo |= (uint32_t)(q & 0xFF) << (8 * j);
                else
                    hi |= (uint32_t)(q & 0xFF) << (8 * (j - 4));
            }
            reinterpret_cast<uint2*>(codes_s)[v] = make_uint2(lo, hi);
        }
        named_bar_sync(1, kConsumers);
        if (!PG && p.sw_in_smem) {
            const bool ok = mbar_wait_bounded(smem_u32(sw_bar), 0, p.timeout_ns, abort_flag,
                                              p.status, kSiteGemvScales);
            if (!__all_sync(0xffffffffu, ok)) return;
        }
        const float s_a = s;  // every consumer thread holds the token scale

        // ------------------------------ weight rows ---------------------------
        const uint4* codes = reinterpret_cast<const uint4*>(codes_s);
        const int nchunk = p.row_bytes / 16;
        float* prod = PG ? reinterpret_cast<float*>(smem + p.prod_off) + warp * p.G : nullptr;
        for (int st = 0; st < nst; ++st) {
            const int slot = st % NS;
            const uint32_t use = (uint32_t)(st / NS);
            {
                const bool ok = mbar_wait_bounded(smem_u32(&full[slot]), use & 1u, p.timeout_ns,
                                                  abort_flag, p.status, kSiteGemvConsumerFull);
                if (!__all_sync(0xffffffffu, ok)) return;
            }
            const uint8_t* stage = stages + (size_t)slot * p.stage_bytes;
            const int rows = min(R, nrows - st * R);
            // Rows of the stage go to warps round-robin on the CTA-local row index.
            int j = (warp - (st * R) % kConsumerWarps + kConsumerWarps) % kConsumerWarps;
            for (; j < rows; j += kConsumerWarps) {
                const int n = n0 + st * R + j;
                const uint4* wrow = reinterpret_cast<const uint4*>(stage + (size_t)j * p.row_bytes);
                if constexpr (A16 && !PG) {
                    float acc = 0.0f;
                    for (int c0 = 0; c0 < nchunk; c0 += 32 * kUnroll) {  // warp-uniform
                        uint4 wv[kUnroll];
#pragma unroll
                        for (int u = 0; u < kUnroll; ++u) {
                            const int c = c0 + u * 32 + lane;
                            if (c < nchunk) wv[u] = wrow[c];
                        }
#pragma unroll
                        for (int u = 0; u < kUnroll; ++u) {
                            const int c = c0 + u * 32 + lane;
                            if (c < nchunk) acc += chunk_dot_a16<T, BITS>(wv[u], codes, c);
                        }
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                    if (lane == 0)
                        store_y(p, n, acc * (p.sw_in_smem ? sw_s[n - n0] : __ldg(p.s_w + n)));
                } else if constexpr (!PG) {
                    int acc = 0;
                    for (int c0 = 0; c0 < nchunk; c0 += 32 * kUnroll) {  // warp-uniform
                        uint4 wv[kUnroll];
#pragma unroll
                        for (int u = 0; u < kUnroll; ++u) {
                            const int c = c0 + u * 32 + lane;
                            if (c < nchunk) wv[u] = wrow[c];
                        }
#pragma unroll
                        for (int u = 0; u < kUnroll; ++u) {
                            const int c = c0 + u * 32 + lane;
                            if (c < nchunk) acc += chunk_dot<BITS>(wv[u], codes, c);
                        }
                    }
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                    if (lane == 0)
                        store_y(p, n,
                                __fmul_rn(__fmul_rn(__int2float_rn(acc), s_a),
                                          p.sw_in_smem ? sw_s[n - n0] : __ldg(p.s_w + n)));
                } else {
                    const float* srow =
                        p.scales_staged
                            ? reinterpret_cast<const float*>(stage + (size_t)R * p.row_bytes) + j * p.G
                            : p.s_w + (int64_t)n * p.G;
                    for (int c0 = 0; c0 < nchunk; c0 += 32 * kUnroll) {  // warp-uniform
                        uint4 wv[kUnroll];
#pragma unroll
                        for (int u = 0; u < kUnroll; ++u) {
                            const int c = c0 + u * 32 + lane;
                            if (c < nchunk) wv[u] = wrow[c];
                        }
#pragma unroll
                        for (int u = 0; u < kUnroll; ++u) {
                            const int c = c0 + u * 32 + lane;
                            if (c0 + u * 32 >= nchunk) break;  // warp-uniform
                            if constexpr (A16) {
                                float part = (c < nchunk) ? chunk_dot_a16<T, BITS>(wv[u], codes, c)
                                                          : 0.0f;
                                for (int o = 1; o < p.cpg; o <<= 1)
                                    part += __shfl_xor_sync(0xffffffffu, part, o);
                                if ((lane & (p.cpg - 1)) == 0 && c < nchunk)
                                    prod[c / p.cpg] = part * srow[c / p.cpg];
                            } else {
                                int part = (c < nchunk) ? chunk_dot<BITS>(wv[u], codes, c) : 0;
                                for (int o = 1; o < p.cpg; o <<= 1)
                                    part += __shfl_xor_sync(0xffffffffu, part, o);
                                if ((lane & (p.cpg - 1)) == 0 && c < nchunk) {
                                    const int g = c / p.cpg;
                                    prod[g] = __fmul_rn(__int2float_rn(part), srow[g]);
                                }
                            }
                        }
                    }
                    __syncwarp();
                    if (lane == 0) {
                        float f = 0.0f;
                        for (int g = 0; g < p.G; ++g) f = __fadd_rn(f, prod[g]);
                        store_y(p, n, A16 ? f : __fmul_rn(f, s_a));
                    }
                    __syncwarp();
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(smem_u32(&empty[slot]));
        }
    }
}

PerDevice<int> g_max_smem;  // opt-in shared memory per block, per device

template <typename T, int BITS, bool PG, bool A16>
cudaError_t launch_one(const Params& p, int grid, int smem, int max_smem, cudaStream_t stream) {
    auto kern = gemv_kernel<T, BITS, PG, A16>;
    static PerDevice<int> attr;  // opt-in to the device's whole per-block shared memory
    const cudaError_t e = attr.get([&](int&) {
        return cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, max_smem);
    });
    if (e != cudaSuccess) return e;
    return launch_pdl(kern, grid, kThreads, smem, stream, p);
}

template <typename T, bool A16>
cudaError_t launch_bits(const Params& p, int bits, bool pg, int grid, int smem, int max_smem,
                        cudaStream_t stream) {
    if (bits == 8)
        return pg ? launch_one<T, 8, true, A16>(p, grid, smem, max_smem, stream)
                  : launch_one<T, 8, false, A16>(p, grid, smem, max_smem, stream);
    return pg ? launch_one<T, 4, true, A16>(p, grid, smem, max_smem, stream)
              : launch_one<T, 4, false, A16>(p, grid, smem, max_smem, stream);
}

}  // namespace

cudaError_t launch_gemv(const GemvArgs& a, int num_sms, cudaStream_t stream) {
    if (a.K <= 0 || a.N <= 0 || a.K > kMaxK || a.N > INT32_MAX) return cudaErrorInvalidValue;
    if (a.bits != 8 && a.bits != 4) return cudaErrorInvalidValue;
    const int chunk_elems = (a.bits == 8) ? 16 : 32;
    if (a.K % chunk_elems != 0) return cudaErrorInvalidValue;
    int max_smem = 0;
    {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e == cudaSuccess)
            e = g_max_smem.get(dev, [dev](int& v) {
                return cudaDeviceGetAttribute(&v, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
            }, &max_smem);
        if (e != cudaSuccess) return e;
    }
    Params p{};
    p.x = a.x;
    p.K = (int)a.K;
    p.N = (int)a.N;
    p.w = static_cast<const uint8_t*>(a.w);
    p.s_w = a.s_w;
    p.y = a.y;
    p.y_bf16 = a.y_bf16;
    p.timeout_ns = a.timeout_ns;
    p.status = a.status;
    if (a.group_size == 0) {
        p.G = 1;
        p.cpg = 0;
    } else {
        if (a.group_size % chunk_elems != 0 || a.K % a.group_size != 0) return cudaErrorInvalidValue;
        p.G = (int)(a.K / a.group_size);
        p.cpg = a.group_size / chunk_elems;
        if (p.cpg > 32 || (p.cpg & (p.cpg - 1)) != 0) return cudaErrorInvalidValue;
    }
    const bool pg = a.group_size != 0;
    p.row_bytes = (a.bits == 8) ? p.K : p.K / 2;
    p.rows_per_stage = kStageTarget / p.row_bytes > 0 ? kStageTarget / p.row_bytes : 1;
    p.scales_staged = pg && (p.G % 4 == 0) && (reinterpret_cast<uintptr_t>(a.s_w) % 16 == 0);
    const int stage_payload =
        p.rows_per_stage * (p.row_bytes + (p.scales_staged ? p.G * 4 : 0));
    p.stage_bytes = (stage_payload + 127) & ~127;

    // Two CTAs per SM, each with at most half the shared memory: consecutive
    // GEMVs (programmatic dependent launch) then overlap on every SM, the
    // next one streaming its weights while the previous one finishes.
    const int grid = (int)(a.N < 2 * num_sms ? a.N : 2 * num_sms);
    const int max_rows = (int)((a.N + grid - 1) / grid);
    const int max_stages_needed = (max_rows + p.rows_per_stage - 1) / p.rows_per_stage;

    // Shared memory: codes | per-warp group products | barriers | stages.
    p.codes_off = 0;
    // x area: INT8 codes (K bytes), or the activations themselves in A16 mode
    p.prod_off = ((a.a16 ? 2 * p.K : p.K) + 127) & ~127;
    const int prod_bytes = pg ? ((kConsumerWarps * p.G * 4 + 127) & ~127) : 0;
    p.sw_off = p.prod_off + prod_bytes;
    p.sw_in_smem = !pg && max_rows <= 8192;
    const int sw_bytes = p.sw_in_smem ? ((max_rows * 4 + 127) & ~127) : 0;
    p.bar_off = p.sw_off + sw_bytes;
    const int bar_bytes = 2 * kMaxStages * 8 + kConsumerWarps * 4 + 32;  // + abort flag, 2 barriers
    p.stage_off = (p.bar_off + bar_bytes + 127) & ~127;
    const int budget = (max_smem / 2 - 1024) - p.stage_off;
    int ns = budget / p.stage_bytes;
    if (ns > kMaxStages) ns = kMaxStages;
    if (ns > max_stages_needed) ns = max_stages_needed;
    if (ns < 1) return cudaErrorInvalidValue;
    p.num_stages = ns;
    const int smem = p.stage_off + ns * p.stage_bytes;
    if (a.a16)
        return a.x_bf16
                   ? launch_bits<__nv_bfloat16, true>(p, a.bits, pg, grid, smem, max_smem, stream)
                   : launch_bits<__half, true>(p, a.bits, pg, grid, smem, max_smem, stream);
    return a.x_bf16
               ? launch_bits<__nv_bfloat16, false>(p, a.bits, pg, grid, smem, max_smem, stream)
               : launch_bits<__half, false>(p, a.bits, pg, grid, smem, max_smem, stream);
}

}  // namespace cider
