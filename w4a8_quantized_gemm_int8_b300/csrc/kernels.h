// Internal launcher declarations shared by the C-ABI layer and the kernel
// translation units (host side only; not part of the public interface).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "../../include/cider.h"

namespace cider {

// The quantized linear layer behind every layer entry point: argument
// checks, workspace carving (ws / ws_bytes: at least cider_workspace_bytes
// of the problem, else CIDER_ERR_WORKSPACE), then the kernels on `stream`.
// M == 1 runs the GEMV when route_m1_to_gemv is set, the tensor-core GEMM
// otherwise (the same results either way). x / y types: CIDER_DTYPE_*.
cider_status linear_call(const void* x, int32_t x_dtype, int64_t M, int64_t N, int64_t K,
                         const void* w, int bits, const float* s_w, int32_t gs, void* y,
                         int32_t y_dtype, void* ws, size_t ws_bytes, cudaStream_t stream,
                         bool route_m1_to_gemv);

// Launches `kern` with programmatic stream serialization: it may be scheduled
// while the preceding kernel in the stream is still running (that kernel
// allows it by executing griddepcontrol.launch_dependents); every kernel
// launched this way executes griddepcontrol.wait before its first access to
// memory that a preceding kernel may write.
template <typename... Params, typename... Args>
cudaError_t launch_pdl(void (*kern)(Params...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

enum class QuantOut : int { kInt8 = 0, kF16 = 1, kInt4 = 2 };

// 16-bit floating-point element type of activations (and of layer outputs).
enum class ElemType : int { kF16 = 0, kBF16 = 1 };

// Symmetric quantization of `rows` x K fp16 (or bf16) values in groups of
// `gs` consecutive elements of a row (gs == K: one group per row), scale =
// absmax / qmax; codes written as int8, as exact fp16 integers, or as packed
// nibbles (code + 8, two per byte). scales: [rows, K / gs].
cudaError_t launch_quant_groups(const void* src, ElemType src_type, int64_t rows, int64_t K,
                                int64_t gs, int qmax, QuantOut out_kind, void* out,
                                float* scales, int num_sms, cudaStream_t stream);

// Weight quantization with percentile-clipped scales (offline preparation):
// per block of gs elements (gs % 8 == 0, gs <= 16384), clip = the pct-th
// percentile of |w| (linear interpolation between order statistics), scale
// = clip / qmax; codes as int8 or packed nibbles (out_kind kInt8 / kInt4).
cudaError_t launch_quant_groups_pct(const void* src, ElemType src_type, int64_t rows, int64_t K,
                                    int64_t gs, int qmax, double pct, QuantOut out_kind,
                                    void* out, float* scales, cudaStream_t stream);

// Both operand images of the tensor-core GEMM in one launch: x fp16 [M,K] ->
// a_img (exact fp16 codes) + s_a, and weights (INT8 [N,K] or packed INT4
// [N,K/2]) -> b_img (exact fp16 integers; skipped when w is NULL); with s_wT
// non-NULL also the group-major copy s_wT [G,N] of per-group scales s_w
// [N,G]. Falls back to separate launches for shapes the fused kernel does
// not take.
cudaError_t launch_operand_images(const void* x, ElemType x_type, int64_t M, int64_t K,
                                  const void* w, int bits,
                                  int64_t N, __half* a_img, float* s_a, __half* b_img,
                                  const float* s_w, float* s_wT, int64_t G, int num_sms,
                                  cudaStream_t stream);

// Operand images: INT8 codes / packed INT4 nibbles -> exact fp16 integers.
cudaError_t launch_widen_i8(const int8_t* src, int64_t n, __half* dst, int num_sms,
                            cudaStream_t stream);
cudaError_t launch_widen_i4(const uint8_t* src, int64_t n_codes, __half* dst, int num_sms,
                            cudaStream_t stream);

// ---- tensor-core GEMM over fp16 operand images ------------------------------
enum class GemmMode : int {
    kPcF16 = 0,     // y = fp16(((float)acc * s_a[m]) * s_w[n])
    kPgF16 = 1,     // f = sum_g (float)P_g * s_w[n,g] (ascending g); y = fp16(f * s_a[m])
    kRawS32 = 2,    // out int32 [M,N] = acc
    kRawPgS32 = 3,  // out int32 [M,N,G] = P_g
};

struct GemmArgs {
    const __half* a_img;  // [M, K] fp16 codes (tokens)
    const __half* b_img;  // [N, K] fp16 codes (weights)
    int64_t M, N, K;
    int group_size;       // 0 for per-channel / raw totals
    const float* s_a;     // [M]
    const float* s_w;     // [N] or [N, K/gs]
    const float* s_wT;    // per-group scales group-major [K/gs, N] (optional; faster fetch)
    void* out;
    GemmMode mode;
    uint64_t timeout_ns;
    unsigned long long* status;  // device status word
    // Raw weight codes instead of b_img: INT8 [N, K] (b_bits 8) or packed
    // INT4 [N, K/2] (b_bits 4), widened on chip.
    const void* b_raw;
    int b_bits;
    int out_bf16;  // fp16-output modes: write bfloat16 instead of fp16
    // Stream-K scratch for per-channel layers of at most 128 tokens (NULL:
    // whole tiles per CTA): per CTA two int32 partial tiles of
    // stream_k_part_rows(M) x 128 (single-SM engine: [2][32][rows][4]; SM
    // pairs: [2][rows][128]), summed by a fix-up launch after the GEMM.
    int32_t* sk_part;
};

// Stream-K sizing: at most kStreamKMaxCtas CTAs share the k-blocks of all
// tiles; each keeps at most two partial tiles (its first and its last).
constexpr int kStreamKMaxCtas = 160;
inline int64_t stream_k_part_rows(int64_t M) { return M >= 128 ? 128 : (M + 31) / 32 * 32; }
inline size_t stream_k_part_bytes(int64_t M) {
    return (size_t)kStreamKMaxCtas * 2 * (size_t)stream_k_part_rows(M) * 128 * 4;
}

cudaError_t launch_gemm_tc(const GemmArgs& args, int num_sms, cudaStream_t stream);
// Same function on SM pairs with the raw weight codes (b_raw) widened on chip
// into tensor memory, where the tensor core reads them as its A operand; no
// weight image. INT8 per-group layers of more than 128 tokens (192-token
// tiles), and the few-token layers gemm_tw_takes_few_tokens picks (128-token
// tiles).
cudaError_t launch_gemm_tw(const GemmArgs& args, int num_sms, cudaStream_t stream);
// True when launch_gemm_tw is the better engine for a problem of at most 128
// tokens (raw INT8 / INT4 codes; per-channel, or per-group when its pair
// tiles occupy at least as many SMs as the single-SM engine's tiles).
bool gemm_tw_takes_few_tokens(const GemmArgs& args, int num_sms);
// Same function on SM pairs (cta_group::2, 256 x 256 tiles, or 256 x 192 for
// per-channel layers where that takes no more waves); for M > 128.
cudaError_t launch_gemm_tc_pair(const GemmArgs& args, int num_sms, cudaStream_t stream);
// Picks the engine for the problem: SM pairs for M > 128; for M <= 128 the
// raw-code pair kernel where gemm_tw_takes_few_tokens says so, single SMs
// otherwise (CIDER_GEMM_ENGINE=single|pair in the environment overrides:
// single keeps every M <= 128 problem on single SMs).
cudaError_t launch_gemm(const GemmArgs& args, int num_sms, cudaStream_t stream);
// True when launch_gemm takes an M > 128 engine (fp16 weight image, or raw
// codes for INT8 per-group); false for the few-token engines (raw codes).
bool gemm_uses_pair(int64_t M);
// True when the engine launch_gemm picks for `args` reads the group-major
// scale copy s_wT (per-group layers on the image pair kernel or on single
// SMs); the raw-code pair kernel reads s_w itself.
bool gemm_reads_scales_t(const GemmArgs& args, int num_sms);

// ---- M = 1 GEMV (quantizes x per CTA, int32 dot products, same epilogue) ----
struct GemvArgs {
    const void* x;       // [K] fp16, or bf16 with x_bf16
    int64_t K, N;
    const void* w;       // int8 [N, K] or packed int4 [N, K/2]
    const float* s_w;    // [N] or [N, K/gs]
    int bits;            // 8 or 4
    int group_size;      // 0, 64 or 128 (w4: 0 or 128, any multiple of 32)
    void* y;             // [N] fp16, or bf16 with y_bf16
    uint64_t timeout_ns;          // bound on every device-side wait
    unsigned long long* status;   // device status word
    int x_bf16;
    int y_bf16;
    int a16;     // A16 decode product: x used as it is, weights dequantized, fp32 sums
};

cudaError_t launch_gemv(const GemvArgs& args, int num_sms, cudaStream_t stream);

// ---- measurement kernels (benchmark test hooks) ----------------------------
// `blocks` blocks of 4 warps, each warp 8 x iters mma.sync.m16n8k32 s8
// instructions (8192 operations each); sink: blocks * 128 int32.
cudaError_t launch_int8_mma_loop(int blocks, int64_t iters, int32_t* sink, cudaStream_t stream);
// Streaming read of `bytes` (a multiple of 16, src 16-byte aligned) by `grid`
// blocks of 512 threads, launched like the GEMV; sink: grid words.
cudaError_t launch_read_bytes(const void* src, int64_t bytes, int grid, uint32_t* sink,
                              cudaStream_t stream);

// ---- device status --------------------------------------------------------
// Address of the current device's status word (looked up once per device).
cudaError_t device_status_ptr(unsigned long long** ptr);
cudaError_t read_and_clear_device_status(unsigned long long* value, cudaStream_t stream);
cudaError_t launch_wait_timeout_probe(uint64_t timeout_ns, cudaStream_t stream);

// Host-side encoder for a 2D fp16 row-major tile map (any swizzle mode).
CUresult encode_tmap_f16_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                            uint32_t box_rows, uint32_t box_cols, CUtensorMapSwizzle swizzle);

// Host-side encoder for a 2D byte tile map (unswizzled).
CUresult encode_tmap_u8_2d(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                           uint32_t box_rows, uint32_t box_cols);

// Host-side encoder for a 2D byte tile map with the given swizzle (the box's
// row of bytes must equal the swizzle span for the 32/64/128-byte modes).
CUresult encode_tmap_u8_2d_swizzled(CUtensorMap* map, const void* base, uint64_t rows,
                                    uint64_t cols, uint32_t box_rows, uint32_t box_cols,
                                    CUtensorMapSwizzle swizzle);

// Host-side encoder for a 2D fp16 K-major tile map with 128-byte swizzle.
CUresult encode_tmap_f16_kmajor(CUtensorMap* map, const void* base, uint64_t rows, uint64_t cols,
                                uint32_t box_rows, uint32_t box_cols);

}  // namespace cider
