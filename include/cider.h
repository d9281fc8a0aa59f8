/*
 * cider.h - C ABI of the B300 (sm_103a) quantized linear-layer library:
 * online per-token INT8 activation quantization, INT8 x INT8 -> INT32
 * matrix products with a fused dequant epilogue, for W8A8 per-channel,
 * W8A8 per-group and W4A8 weights, plus the M = 1 INT8 GEMV.
 *
 * The method is the one described for the "cider" project (Mininglamp-AI)
 * in its README and blog posts; each entry point names the passage that
 * defines it. The arithmetic, exactly:
 *   activations (README "Quantization", row "Activations: Symmetric INT8,
 *   Per-token"): s_a[m] = absmax_k |x[m,k]| / 127 (fp32 IEEE division),
 *   q[m,k] = clamp(rint(x[m,k] / s_a[m]), -127, 127) (IEEE division, ties
 *   to even); an all-zero row has s_a = 0 and q = 0; -128 never occurs.
 *   weights: the same with one scale per output channel, or per group of
 *   group_size consecutive k; INT4 uses qmax 7 and stores code + 8.
 *   products (row "Accumulation: INT32"): exact int32 sums.
 *   per-channel output (row "Output dequant: C_fp16 = C_int32 * s_act *
 *   s_weight"): y = fp16_rn(((float)acc * s_a[m]) * s_w[n]).
 *   per-group output: f = 0; for g = 0..K/gs-1: f = f + (float)P_g * s_w[n,g]
 *   (rounded product, rounded sum); y = fp16_rn(f * s_a[m]).
 *
 * Conventions for every call:
 *  - Tensors are row-major and contiguous. fp16 tensors are IEEE binary16.
 *    Weights are stored [N = out_features, K = in_features], so the layer
 *    computes y[M,N] = x[M,K] . W^T.
 *  - Unless a comment says "host", every pointer is a device pointer owned
 *    by the caller; the library never allocates, frees, or keeps them.
 *    Pointers must be 16-byte aligned. Each buffer must hold at least the
 *    elements its comment states for the sizes passed (the library sees
 *    only pointers and cannot check this; the Python binding checks tensor
 *    shapes before every call).
 *  - `stream` is a cudaStream_t (NULL = the legacy default stream). Calls
 *    only enqueue work on it and return without synchronizing, except
 *    cider_device_status, which synchronizes the stream.
 *  - Return value: CIDER_OK, or the first error found. Argument checks run
 *    before any work is enqueued; a call that returns an error has enqueued
 *    nothing (except CIDER_ERR_CUDA raised by a launch).
 *  - The library is stateless apart from per-device caches of launch
 *    attributes and the device status word; calls are thread-safe for
 *    distinct streams.
 *  - NaN / Inf inputs are outside the contract.
 */
#ifndef CIDER_H
#define CIDER_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define CIDER_API __attribute__((visibility("default")))
#else
#define CIDER_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef enum cider_status {
    CIDER_OK = 0,
    CIDER_ERR_INVALID_ARG = 1, /* null pointer, size <= 0, negative group size */
    CIDER_ERR_UNSUPPORTED = 2, /* shape, group size, alignment or device not handled */
    CIDER_ERR_CUDA = 3,        /* a CUDA runtime call or kernel launch failed */
    CIDER_ERR_TIMEOUT = 4,     /* a bounded device-side wait gave up (see cider_device_status) */
    CIDER_ERR_WORKSPACE = 5    /* workspace pointer missing or smaller than required */
} cider_status;

#define CIDER_ABI_VERSION 3

/* Element types of activations and layer outputs (README roadmap: automatic
 * dtype handling, float16 / bfloat16). Both convert exactly to fp32; an
 * output is the fp32 epilogue value rounded to nearest even in that type. */
#define CIDER_DTYPE_F16 0
#define CIDER_DTYPE_BF16 1

/* Human-readable name of a status code (static string, never NULL). */
CIDER_API const char* cider_status_string(cider_status status);

/* CIDER_ABI_VERSION of the built library. */
CIDER_API int cider_abi_version(void);

/*
 * Per-token symmetric INT8 activation quantization.
 * README "Quantization" (row "Activations") and "Metal Kernel Pipeline",
 * prefill step 1 ("FP16 activations -> INT8 + per-token scales").
 *   x_f16 [M,K] fp16 in; q [M,K] int8 out; s_a [M] fp32 out.
 * Any K >= 1 (16-byte-aligned rows take a vectorized path).
 */
CIDER_API cider_status cider_quantize_act(const void* x_f16, int64_t M, int64_t K, int8_t* q, float* s_a,
                                void* stream);

/*
 * Offline INT8 weight quantization (README "Low-Level API":
 * quantize_weight_int8; "W8A8 Quantization Granularity" table).
 *   w_f16 [N,K] fp16 in; wq [N,K] int8 out;
 *   s_w out: [N] fp32 for group_size 0 (per output channel), else
 *   [N, K/group_size] fp32 (group g covers k in [g*gs, (g+1)*gs)).
 * group_size: 0 or any divisor of K.
 */
CIDER_API cider_status cider_quantize_weight_int8(const void* w_f16, int64_t N, int64_t K,
                                        int32_t group_size, int8_t* wq, float* s_w, void* stream);

/*
 * Offline INT4 weight quantization and packing (README "Low-Level API":
 * pack_weight_int4; "Quantization" row "W4A8 weights: Symmetric INT4
 * (zp=8)"). Codes in [-7, 7] with scale absmax/7; nibble = code + 8; byte j
 * of a row holds element 2j in its low nibble and 2j+1 in its high nibble.
 *   w_f16 [N,K] fp16 in; wp [N, K/2] uint8 out; s_w as above.
 * K % 8 == 0; group_size 0 or a divisor of K that is a multiple of 8.
 */
CIDER_API cider_status cider_pack_weight_int4(const void* w_f16, int64_t N, int64_t K, int32_t group_size,
                                    uint8_t* wp, float* s_w, void* stream);

/*
 * Weight preparation with percentile-clipped scales (README "LLM
 * Quantization" note: besides min-max, "the 99th percentile method
 * (clip_percentile=99.9)"). Per block (output channel for group_size 0,
 * else each group of group_size along K) the clip value is the
 * clip_percentile-th percentile of |w| by linear interpolation between order
 * statistics (position (n - 1) * p / 100 in the sorted |w|), scale = clip /
 * qmax (127 for bits 8, 7 for bits 4), codes clamp(rint(w / scale)): values
 * beyond the clip saturate. clip_percentile 100 equals min-max.
 *   w [N,K] fp16 (w_dtype CIDER_DTYPE_F16) or bf16; wq out: int8 [N,K] (bits
 *   8) or packed uint8 [N,K/2] (bits 4, nibble = code + 8, element 2j low);
 *   s_w out [N] or [N, K/gs] fp32.
 * clip_percentile in (0, 100]; block size a multiple of 8 and <= 16384;
 * w and wq 16-byte aligned.
 */
CIDER_API cider_status cider_quantize_weight_clipped(const void* w, int32_t w_dtype, int64_t N,
                                                     int64_t K, int32_t group_size, int32_t bits,
                                                     double clip_percentile, void* wq,
                                                     float* s_w, void* stream);

/*
 * Bytes of device workspace the GEMM calls below need for this problem:
 * group_size 0 (per channel) or the per-group size, then bits 8 or 4 (the
 * order of the layer calls' own arguments). The workspace holds the fp16
 * image of the quantized activations (the codes as exact fp16 integers) and
 * the per-token scales; for M > 128, except for INT8 per-group layers (whose
 * weights are widened on chip), an fp16 image of the weight codes; for
 * per-group layers that read one, a group-major copy of the weight scales;
 * and for per-channel layers of at most 128 tokens, whose k-blocks are
 * shared out evenly among the SMs, int32 partial output tiles (up to
 * 2 * 160 tiles of 128 columns and min(M rounded up to 32, 128) rows) that
 * a fix-up launch sums exactly. Returns 0 when M == 1 (the GEMV path needs
 * none) and on invalid sizes (including a group_size that does not divide
 * K).
 */
CIDER_API size_t cider_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t group_size,
                                       int32_t bits);

/*
 * W8A8 per-channel linear layer: quantize x per token, int32 GEMM with wq,
 * y = fp16(((float)acc * s_a[m]) * s_w[n]).
 * README "Metal Kernel Pipeline" (prefill: quantize_per_token then
 * matmul_fused_dequant), "Quantization" table.
 *   x_f16 [M,K] fp16; wq [N,K] int8; s_w [N] fp32; y_f16 [M,N] fp16 out;
 *   ws / ws_bytes: device workspace of at least
 *   cider_workspace_bytes(M, N, K, 0, 8) bytes (may be NULL if that is 0).
 * K % 16 == 0. M == 1 runs the GEMV (same results).
 */
CIDER_API cider_status cider_w8a8_gemm_pc(const void* x_f16, int64_t M, int64_t N, int64_t K,
                                const int8_t* wq, const float* s_w, void* y_f16, void* ws,
                                size_t ws_bytes, void* stream);

/*
 * W8A8 per-group linear layer: as above with s_w [N, K/group_size]; each
 * group's int32 partial is rescaled and summed in ascending group order, the
 * token scale applied last. README "W8A8 Quantization Granularity" (one
 * scale per 64 / 128 elements), "Quantization" table.
 * group_size: a multiple of 64 dividing K, at most 1024 for M > 1 (a group's
 * partial must stay exact in the tensor core's fp32 accumulator); 64 and 128
 * are the pages' sizes. Larger groups give CIDER_ERR_UNSUPPORTED.
 */
CIDER_API cider_status cider_w8a8_gemm_pg(const void* x_f16, int64_t M, int64_t N, int64_t K,
                                const int8_t* wq, const float* s_w, int32_t group_size,
                                void* y_f16, void* ws, size_t ws_bytes, void* stream);

/*
 * W4A8 linear layer: packed INT4 weights wp [N, K/2] (as written by
 * cider_pack_weight_int4) are unpacked to INT8 codes before the product
 * (README "Modes", W4A8 compute path "Unpack -> TensorOps"), then the
 * per-channel (group_size 0, s_w [N]) or per-group (s_w [N, K/gs]) layer.
 * K % 32 == 0; group_size 0 or a multiple of 64 dividing K (at most 1024
 * for M > 1).
 */
CIDER_API cider_status cider_w4a8_gemm(const void* x_f16, int64_t M, int64_t N, int64_t K,
                             const uint8_t* wp, const float* s_w, int32_t group_size, void* y_f16,
                             void* ws, size_t ws_bytes, void* stream);

/*
 * The linear layer for either activation / output element type: as
 * cider_w8a8_gemm_pc (bits 8, group_size 0), cider_w8a8_gemm_pg (bits 8,
 * group_size > 0) or cider_w4a8_gemm (bits 4), with x [M,K] of element type
 * x_dtype and y [M,N] written as y_dtype (CIDER_DTYPE_F16 or
 * CIDER_DTYPE_BF16; any combination). The quantization reads each element's
 * exact fp32 value; the epilogue is the same fp32 arithmetic, rounded to the
 * output type. M == 1 runs the GEMV. Same workspace, alignment and shape
 * rules as the fp16 entry points; an unknown dtype or bits gives
 * CIDER_ERR_INVALID_ARG.
 */
CIDER_API cider_status cider_linear(const void* x, int32_t x_dtype, int64_t M, int64_t N,
                                    int64_t K, const void* w, int32_t bits, const float* s_w,
                                    int32_t group_size, void* y, int32_t y_dtype, void* ws,
                                    size_t ws_bytes, void* stream);

/*
 * cider_quantize_act for either element type of x (CIDER_DTYPE_F16 or
 * CIDER_DTYPE_BF16): per-token INT8 codes q [M,K] and scales s_a [M] of the
 * exact fp32 values.
 */
CIDER_API cider_status cider_quantize_act_ex(const void* x, int32_t x_dtype, int64_t M, int64_t K,
                                             int8_t* q, float* s_a, void* stream);

/*
 * A16 decode matrix-vector product (README "Metal Kernel Pipeline", decode:
 * a matrix-vector kernel "with on-the-fly weight dequantization (no
 * activation quantization needed)"): y[n] = sum_g s_w[n,g] * sum_{k in g}
 * x[k] * code[n,k], with x [K] used as it is (fp16 or bf16, x_dtype), the
 * weight codes dequantized on the fly, fp32 accumulation, y [N] written as
 * y_dtype. A floating-point sum: its result agrees with the exact value
 * within the fp32 accumulation bound, not bit for bit with another order.
 * Weights, scales and limits as cider_int8_gemv. Needs no workspace.
 */
CIDER_API cider_status cider_a16_gemv(const void* x, int32_t x_dtype, int64_t K, int64_t N,
                                      const void* w, int32_t bits, const float* s_w,
                                      int32_t group_size, void* y, int32_t y_dtype, void* stream);

/*
 * M = 1 INT8 GEMV (README "Metal Kernel Pipeline", "Decode (M = 1)").
 * Computes exactly the GEMM's function at M = 1: the single token is
 * quantized per token to INT8, products are exact int32, then the same
 * per-channel or per-group epilogue.
 *   x_f16 [K] fp16; w: int8 [N,K] (bits 8) or packed uint8 [N, K/2]
 *   (bits 4); s_w [N] or [N, K/gs]; y_f16 [N] fp16 out.
 * K <= 16384; bits 8: K % 16 == 0, group_size 0 or a multiple of 16
 * dividing K (at most 32 chunks of 16 per group, a power of two);
 * bits 4: K % 32 == 0, group_size 0 or a multiple of 32 likewise.
 * Needs no workspace.
 */
CIDER_API cider_status cider_int8_gemv(const void* x_f16, int64_t K, int64_t N, const void* w,
                             const float* s_w, int32_t bits, int32_t group_size, void* y_f16,
                             void* stream);

/*
 * cider_w8a8_gemm_pc without a caller workspace, for callers that cannot
 * allocate device memory (for example code running under a framework that
 * owns every device allocation through its own pool, or a latency-critical
 * loop that must not pay cudaMalloc's implicit synchronization). The pages
 * describe no counterpart of this entry point.
 *   Same arguments, layouts and result as cider_w8a8_gemm_pc minus ws /
 *   ws_bytes; M == 1 is computed by the tensor-core GEMM (no GEMV routing,
 *   same bits). The scratch (fp16 operand images of the codes and the
 *   token scales, 2*M*K + 4*M + 2*N*K bytes, each part rounded up to 256)
 *   comes from one 64 MiB array compiled into the library
 *   (CIDER_STATIC_SCRATCH_BYTES); larger problems return
 *   CIDER_ERR_WORKSPACE and enqueue nothing. The call allocates nothing.
 *   The first call on a device looks up the array's device address with
 *   that device current; make that first call before any stream capture.
 *   All calls on a device share the array: calls whose execution overlaps
 *   on the GPU (other streams, other threads) race and must be serialized.
 *   Every GPU that loads the library keeps the array until the process
 *   exits.
 */
#define CIDER_STATIC_SCRATCH_BYTES (64u << 20)
CIDER_API cider_status cider_w8a8_gemm_pc_noalloc(const void* x_f16, int64_t M, int64_t N,
                                                  int64_t K, const int8_t* wq, const float* s_w,
                                                  void* y_f16, void* stream);

/*
 * The three stages the GEMM entry points above run, exposed so a caller can
 * time them separately or keep a weight image across calls. The tensor
 * cores of sm_103a have no integer MMA kind, so the library multiplies the
 * INT8 codes held exactly as fp16 integers (every code in [-127, 127] is an
 * fp16 value) and folds the fp32 accumulator into int32 every <= 1024 k,
 * which keeps every partial sum exact.
 *
 * cider_act_image: per-token INT8 quantization of x_f16 [M,K] (same codes
 *   and scales as cider_quantize_act), writing each code as an fp16 integer
 *   into a_img [M,K] fp16, and s_a [M] fp32. K % 8 == 0.
 * cider_weight_image: INT8 codes [N,K] (bits 8) or packed INT4 [N,K/2]
 *   (bits 4) -> b_img [N,K] fp16 integers. N*K % 32 == 0.
 * cider_gemm_images: the tensor-core GEMM with the fused dequant epilogue on
 *   the two images: y [M,N] fp16 from a_img [M,K], s_a [M], b_img [N,K] and
 *   s_w ([N] for group_size 0, else [N, K/gs], gs a multiple of 64 dividing
 *   K, at most 1024). K % 16 == 0; any M >= 1 (no GEMV routing).
 */
CIDER_API cider_status cider_act_image(const void* x_f16, int64_t M, int64_t K, void* a_img,
                                       float* s_a, void* stream);
CIDER_API cider_status cider_weight_image(const void* w, int64_t N, int64_t K, int32_t bits,
                                          void* b_img, void* stream);
CIDER_API cider_status cider_gemm_images(const void* a_img, const float* s_a, const void* b_img,
                                         const float* s_w, int64_t M, int64_t N, int64_t K,
                                         int32_t group_size, void* y_f16, void* stream);

/*
 * Test hook, not for users: the raw int32 products of the tensor-core GEMM
 * engine on pre-quantized codes, for the bit-exact INT32 contract.
 *   q [M,K] int8; w int8 [N,K] (bits 8) or packed [N, K/2] (bits 4);
 *   out int32: [M,N] totals for group_size 0, else per-group partials
 *   [M, N, K/group_size]. Workspace as cider_workspace_bytes(max(M,2), N, K, 0, bits).
 */
CIDER_API cider_status cider_test_gemm_s32(const int8_t* q, const void* w, int64_t M, int64_t N, int64_t K,
                                 int32_t bits, int32_t group_size, int32_t* out, void* ws,
                                 size_t ws_bytes, void* stream);

/*
 * Measurement hook, not for users: the INT8 tensor rate available to a
 * register-only loop of the legacy mma.sync.m16n8k32 s8 instruction (sm_103a
 * has no integer kind of tcgen05.mma), the denominator the benchmark uses
 * for "% INT8 peak". Launches `blocks` blocks of 4 warps; each warp executes
 * 8 * iters MMAs of 16 x 8 x 32 products (8192 operations each), so the call
 * performs blocks * 4 * 8 * iters * 8192 operations. sink: blocks * 128
 * int32 (device), written with a fold of the accumulators.
 */
CIDER_API cider_status cider_test_int8_mma_loop(int32_t blocks, int64_t iters, int32_t* sink,
                                               void* stream);

/*
 * Measurement hook, not for users: a plain streaming read of `bytes` bytes
 * at src (device, 16-byte aligned, bytes a multiple of 16), launched as the
 * GEMV is (two blocks per SM, programmatic dependent launch), the ceiling a
 * decode GEMV of the same bytes is compared with. sink: 2 * (number of SMs)
 * uint32 (device).
 */
CIDER_API cider_status cider_test_read_bytes(const void* src, int64_t bytes, uint32_t* sink,
                                            void* stream);

/*
 * Synchronizes `stream`, then reads and clears the device status word of the
 * current device. Returns CIDER_ERR_TIMEOUT if a bounded device-side wait
 * (mbarrier poll) gave up since the last read, CIDER_OK otherwise. If
 * site != NULL (host pointer), *site receives the recorded wait site.
 */
CIDER_API cider_status cider_device_status(void* stream, uint32_t* site);

/*
 * Test hook, not for users: launches a one-thread kernel that waits on an
 * mbarrier nothing arrives at, with a bound of timeout_ns; the kernel then
 * returns normally and cider_device_status reports CIDER_ERR_TIMEOUT.
 * Checks the give-up path without hanging or faulting the GPU.
 */
CIDER_API cider_status cider_test_wait_timeout(int64_t timeout_ns, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* CIDER_H */
