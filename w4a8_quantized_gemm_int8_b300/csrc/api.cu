// C ABI of the library (declared in include/cider.h): argument checks,
// workspace carving, routing (M == 1 -> GEMV) and kernel launches.
#include <cuda_runtime.h>
#include <cstdint>

#include "../../include/cider.h"
#include "device_common.cuh"
#include "host_once.h"
#include "kernels.h"

namespace {

using namespace cider;

constexpr uint64_t kWaitTimeoutNs = 2000000000ull;  // 2 s bound on every device-side wait
PerDevice<int> g_num_sms;

cider_status num_sms(int* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CIDER_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CIDER_ERR_UNSUPPORTED;
    const cudaError_t e = g_num_sms.get(dev, [dev](int& v) {
        return cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    }, out);
    return e == cudaSuccess ? CIDER_OK : CIDER_ERR_CUDA;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

constexpr size_t align256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

cider_status from_cuda(cudaError_t e) {
    if (e == cudaSuccess) return CIDER_OK;
    if (e == cudaErrorInvalidValue) {
        cudaGetLastError();  // a launcher's own argument rejection, nothing launched
        return CIDER_ERR_UNSUPPORTED;
    }
    return CIDER_ERR_CUDA;
}

struct Workspace {
    __half* a_img;
    float* s_a;
    __half* b_img;  // fp16 weight image (SM-pair engine, image path only)
    float* s_wT;    // per-group scales, group-major (per-group, engines that read it)
    int32_t* sk_part;  // stream-K partial tiles (M <= 128, per channel)
};

// Weight operand of the SM-pair engine (M > 128): INT8 per-group layers take
// the raw codes, widened on chip into tensor memory (gemm_tw.cu); the other
// layers take an fp16 weight image written by the operand-image launch
// (gemm_tc2.cu). Measured on B300 at M = 4096 (public call): per-group gs 64
// 362 us raw against 493 us with the image, gs 128 295 against 315; per
// channel 200 against 160 and W4A8 gs 128 (M = 8192) 537 against 442 - the
// raw engine widens each weight k-block once per 192-token tile, the image
// once per call. Layers of at most 128 tokens always take raw codes.
bool pair_uses_image(int64_t M, int64_t gs, int bits) {
    return gemm_uses_pair(M) && !(gs > 0 && bits == 8);
}

// Group-major scale copy: read by the single-SM engine and by the image
// pair kernel in per-group mode (for M <= 128 allocated whichever engine
// the launch picks; written only when that engine reads it).
bool uses_scales_t(int64_t M, int64_t gs, int bits) {
    return gs > 0 && (!gemm_uses_pair(M) || pair_uses_image(M, gs, bits));
}

// Per-channel layers of at most 128 tokens may split the k-blocks of all
// tiles over the SMs or SM pairs (stream-K) and need its scratch.
bool uses_stream_k(int64_t M, int64_t gs) { return gs == 0 && !gemm_uses_pair(M); }

// a_img [M,K] fp16 | s_a [M] fp32 | b_img [N,K] fp16 (image path) |
// s_wT [K/gs, N] fp32 (uses_scales_t) | stream-K partial tiles (uses_stream_k)
size_t workspace_bytes(int64_t M, int64_t N, int64_t K, int64_t gs, int bits) {
    const size_t b = pair_uses_image(M, gs, bits) ? align256((size_t)N * K * 2) : 0;
    const size_t t = uses_scales_t(M, gs, bits) ? align256((size_t)(K / gs) * N * 4) : 0;
    const size_t sk = uses_stream_k(M, gs) ? align256(stream_k_part_bytes(M)) : 0;
    return align256((size_t)M * K * 2) + align256((size_t)M * 4) + b + t + sk;
}

Workspace carve(void* ws, int64_t M, int64_t N, int64_t K, int64_t gs, int bits) {
    uint8_t* p = static_cast<uint8_t*>(ws);
    Workspace w;
    w.a_img = reinterpret_cast<__half*>(p);
    p += align256((size_t)M * K * 2);
    w.s_a = reinterpret_cast<float*>(p);
    p += align256((size_t)M * 4);
    w.b_img = nullptr;
    if (pair_uses_image(M, gs, bits)) {
        w.b_img = reinterpret_cast<__half*>(p);
        p += align256((size_t)N * K * 2);
    }
    w.s_wT = nullptr;
    if (uses_scales_t(M, gs, bits)) {
        w.s_wT = reinterpret_cast<float*>(p);
        p += align256((size_t)(K / gs) * N * 4);
    }
    w.sk_part = uses_stream_k(M, gs) ? reinterpret_cast<int32_t*>(p) : nullptr;
    return w;
}

bool valid_group(int32_t gs, int64_t K, int multiple) {
    return gs == 0 || (gs > 0 && gs % multiple == 0 && K % gs == 0);
}

// Shared body of the three GEMM entry points.
bool valid_dtype(int32_t d) { return d == CIDER_DTYPE_F16 || d == CIDER_DTYPE_BF16; }

ElemType elem(int32_t d) { return d == CIDER_DTYPE_BF16 ? ElemType::kBF16 : ElemType::kF16; }

}  // namespace

// Shared body of the layer entry points (x / y element types: CIDER_DTYPE_*);
// declared in kernels.h.
cider_status cider::linear_call(const void* x, int32_t x_dtype, int64_t M, int64_t N, int64_t K,
                                const void* w, int bits, const float* s_w, int32_t gs, void* y,
                                int32_t y_dtype, void* ws, size_t ws_bytes, cudaStream_t stream,
                                bool route_m1_to_gemv) {
    if (!valid_dtype(x_dtype) || !valid_dtype(y_dtype)) return CIDER_ERR_INVALID_ARG;
    if (!x || !w || !s_w || !y) return CIDER_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || gs < 0) return CIDER_ERR_INVALID_ARG;
    if (K % 16 != 0 || (bits == 4 && K % 32 != 0)) return CIDER_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w) || !aligned16(y) || !aligned16(s_w))
        return CIDER_ERR_UNSUPPORTED;
    if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;

    if (M == 1 && route_m1_to_gemv) {  // decode: the GEMV computes the same function
        if (K > 16384 || !valid_group(gs, K, bits == 8 ? 16 : 32)) return CIDER_ERR_UNSUPPORTED;
        unsigned long long* status = nullptr;
        if (device_status_ptr(&status) != cudaSuccess) return CIDER_ERR_CUDA;
        GemvArgs g{x, K, N, w, s_w, bits, gs, y, kWaitTimeoutNs, status,
                   x_dtype == CIDER_DTYPE_BF16, y_dtype == CIDER_DTYPE_BF16};
        return from_cuda(launch_gemv(g, sms, stream));
    }
    // A group's partial sum must stay exact in the tensor core's fp32
    // accumulator: at most 1024 products of magnitude <= 127^2.
    if (!valid_group(gs, K, 64) || gs > 1024) return CIDER_ERR_UNSUPPORTED;
    const size_t need = workspace_bytes(M, N, K, gs, bits);
    if (!ws || ws_bytes < need) return CIDER_ERR_WORKSPACE;
    if (!aligned16(ws)) return CIDER_ERR_UNSUPPORTED;
    unsigned long long* status = nullptr;
    if (device_status_ptr(&status) != cudaSuccess) return CIDER_ERR_CUDA;

    Workspace wsp = carve(ws, M, N, K, gs, bits);
    const bool img = wsp.b_img != nullptr;
    GemmArgs a{};
    a.a_img = wsp.a_img;
    a.b_img = wsp.b_img;
    a.b_raw = img ? nullptr : w;
    a.b_bits = bits;
    a.M = M;
    a.N = N;
    a.K = K;
    a.group_size = gs;
    a.s_a = wsp.s_a;
    a.s_w = s_w;
    a.s_wT = wsp.s_wT;
    a.out = y;
    a.mode = (gs == 0) ? GemmMode::kPcF16 : GemmMode::kPgF16;
    a.timeout_ns = kWaitTimeoutNs;
    a.status = status;
    a.out_bf16 = (y_dtype == CIDER_DTYPE_BF16);
    a.sk_part = wsp.sk_part;
    // The group-major scale copy only where the chosen engine reads it.
    float* s_wT = (wsp.s_wT && gemm_reads_scales_t(a, sms)) ? wsp.s_wT : nullptr;
    a.s_wT = s_wT;
    // The activation image (fp16 codes and token scales), and the fp16
    // weight image where the engine takes one, in one launch; the other
    // engines widen the raw weight codes on chip.
    cudaError_t e = launch_operand_images(x, elem(x_dtype), M, K, img ? w : nullptr, bits, N,
                                          wsp.a_img, wsp.s_a, wsp.b_img, s_w, s_wT,
                                          gs > 0 ? K / gs : 1, sms, stream);
    if (e != cudaSuccess) return from_cuda(e);
    return from_cuda(launch_gemm(a, sms, stream));
}

namespace {

cider_status gemm_common(const void* x, int32_t x_dtype, int64_t M, int64_t N, int64_t K,
                         const void* w, int bits, const float* s_w, int32_t gs, void* y,
                         int32_t y_dtype, void* ws, size_t ws_bytes, cudaStream_t stream) {
    return linear_call(x, x_dtype, M, N, K, w, bits, s_w, gs, y, y_dtype, ws, ws_bytes, stream,
                       true);
}

}  // namespace

extern "C" {

const char* cider_status_string(cider_status status) {
    switch (status) {
        case CIDER_OK: return "CIDER_OK";
        case CIDER_ERR_INVALID_ARG: return "CIDER_ERR_INVALID_ARG";
        case CIDER_ERR_UNSUPPORTED: return "CIDER_ERR_UNSUPPORTED";
        case CIDER_ERR_CUDA: return "CIDER_ERR_CUDA";
        case CIDER_ERR_TIMEOUT: return "CIDER_ERR_TIMEOUT";
        case CIDER_ERR_WORKSPACE: return "CIDER_ERR_WORKSPACE";
        default: return "CIDER_ERR_UNKNOWN";
    }
}

int cider_abi_version(void) { return CIDER_ABI_VERSION; }

cider_status cider_quantize_act(const void* x_f16, int64_t M, int64_t K, int8_t* q, float* s_a,
                                void* stream) {
    if (!x_f16 || !q || !s_a) return CIDER_ERR_INVALID_ARG;
    if (M <= 0 || K <= 0) return CIDER_ERR_INVALID_ARG;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    return from_cuda(launch_quant_groups(x_f16, ElemType::kF16, M, K, K, 127,
                                         QuantOut::kInt8, q, s_a, sms,
                                         static_cast<cudaStream_t>(stream)));
}

cider_status cider_quantize_weight_int8(const void* w_f16, int64_t N, int64_t K,
                                        int32_t group_size, int8_t* wq, float* s_w,
                                        void* stream) {
    if (!w_f16 || !wq || !s_w) return CIDER_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || group_size < 0) return CIDER_ERR_INVALID_ARG;
    if (group_size != 0 && K % group_size != 0) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    const int64_t gs = group_size ? group_size : K;
    return from_cuda(launch_quant_groups(w_f16, ElemType::kF16, N, K, gs, 127,
                                         QuantOut::kInt8, wq, s_w, sms,
                                         static_cast<cudaStream_t>(stream)));
}

cider_status cider_pack_weight_int4(const void* w_f16, int64_t N, int64_t K, int32_t group_size,
                                    uint8_t* wp, float* s_w, void* stream) {
    if (!w_f16 || !wp || !s_w) return CIDER_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || group_size < 0) return CIDER_ERR_INVALID_ARG;
    if (K % 8 != 0 || !valid_group(group_size, K, 8)) return CIDER_ERR_UNSUPPORTED;
    if (!aligned16(w_f16) || !aligned16(wp)) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    const int64_t gs = group_size ? group_size : K;
    return from_cuda(launch_quant_groups(w_f16, ElemType::kF16, N, K, gs, 7,
                                         QuantOut::kInt4, wp, s_w, sms,
                                         static_cast<cudaStream_t>(stream)));
}

cider_status cider_quantize_weight_clipped(const void* w, int32_t w_dtype, int64_t N, int64_t K,
                                           int32_t group_size, int32_t bits,
                                           double clip_percentile, void* wq, float* s_w,
                                           void* stream) {
    if (!w || !wq || !s_w) return CIDER_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || group_size < 0 || !valid_dtype(w_dtype)) return CIDER_ERR_INVALID_ARG;
    if (bits != 8 && bits != 4) return CIDER_ERR_INVALID_ARG;
    if (!(clip_percentile > 0.0) || clip_percentile > 100.0) return CIDER_ERR_INVALID_ARG;
    const int64_t gs = group_size ? group_size : K;
    if (K % gs != 0 || gs % 8 != 0 || gs > 16384) return CIDER_ERR_UNSUPPORTED;
    if (!aligned16(w) || !aligned16(wq)) return CIDER_ERR_UNSUPPORTED;
    if (N * (K / gs) > INT32_MAX) return CIDER_ERR_UNSUPPORTED;
    return from_cuda(launch_quant_groups_pct(w, elem(w_dtype), N, K, gs, bits == 8 ? 127 : 7,
                                             clip_percentile,
                                             bits == 8 ? QuantOut::kInt8 : QuantOut::kInt4, wq,
                                             s_w, static_cast<cudaStream_t>(stream)));
}

size_t cider_workspace_bytes(int64_t M, int64_t N, int64_t K, int32_t group_size, int32_t bits) {
    if (M <= 1 || N <= 0 || K <= 0 || (bits != 8 && bits != 4)) return 0;
    if (group_size < 0 || (group_size > 0 && K % group_size != 0)) return 0;
    return workspace_bytes(M, N, K, group_size, bits);
}

cider_status cider_w8a8_gemm_pc(const void* x_f16, int64_t M, int64_t N, int64_t K,
                                const int8_t* wq, const float* s_w, void* y_f16, void* ws,
                                size_t ws_bytes, void* stream) {
    return gemm_common(x_f16, CIDER_DTYPE_F16, M, N, K, wq, 8, s_w, 0, y_f16, CIDER_DTYPE_F16,
                       ws, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

cider_status cider_w8a8_gemm_pg(const void* x_f16, int64_t M, int64_t N, int64_t K,
                                const int8_t* wq, const float* s_w, int32_t group_size,
                                void* y_f16, void* ws, size_t ws_bytes, void* stream) {
    if (group_size <= 0) return CIDER_ERR_INVALID_ARG;
    return gemm_common(x_f16, CIDER_DTYPE_F16, M, N, K, wq, 8, s_w, group_size, y_f16,
                       CIDER_DTYPE_F16, ws, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

cider_status cider_w4a8_gemm(const void* x_f16, int64_t M, int64_t N, int64_t K,
                             const uint8_t* wp, const float* s_w, int32_t group_size, void* y_f16,
                             void* ws, size_t ws_bytes, void* stream) {
    return gemm_common(x_f16, CIDER_DTYPE_F16, M, N, K, wp, 4, s_w, group_size, y_f16,
                       CIDER_DTYPE_F16, ws, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

cider_status cider_linear(const void* x, int32_t x_dtype, int64_t M, int64_t N, int64_t K,
                          const void* w, int32_t bits, const float* s_w, int32_t group_size,
                          void* y, int32_t y_dtype, void* ws, size_t ws_bytes, void* stream) {
    if (bits != 8 && bits != 4) return CIDER_ERR_INVALID_ARG;
    return gemm_common(x, x_dtype, M, N, K, w, bits, s_w, group_size, y, y_dtype, ws, ws_bytes,
                       static_cast<cudaStream_t>(stream));
}

cider_status cider_quantize_act_ex(const void* x, int32_t x_dtype, int64_t M, int64_t K,
                                   int8_t* q, float* s_a, void* stream) {
    if (!x || !q || !s_a) return CIDER_ERR_INVALID_ARG;
    if (M <= 0 || K <= 0 || !valid_dtype(x_dtype)) return CIDER_ERR_INVALID_ARG;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    return from_cuda(launch_quant_groups(x, elem(x_dtype), M, K, K, 127, QuantOut::kInt8, q, s_a,
                                         sms, static_cast<cudaStream_t>(stream)));
}

cider_status cider_int8_gemv(const void* x_f16, int64_t K, int64_t N, const void* w,
                             const float* s_w, int32_t bits, int32_t group_size, void* y_f16,
                             void* stream) {
    if (!x_f16 || !w || !s_w || !y_f16) return CIDER_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || group_size < 0) return CIDER_ERR_INVALID_ARG;
    if (bits != 8 && bits != 4) return CIDER_ERR_INVALID_ARG;
    if (K > 16384 || K % (bits == 8 ? 16 : 32) != 0) return CIDER_ERR_UNSUPPORTED;
    if (!valid_group(group_size, K, bits == 8 ? 16 : 32)) return CIDER_ERR_UNSUPPORTED;
    if (!aligned16(x_f16) || !aligned16(w)) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    unsigned long long* status = nullptr;
    if (device_status_ptr(&status) != cudaSuccess) return CIDER_ERR_CUDA;
    GemvArgs g{x_f16, K, N, w, s_w, bits, group_size, y_f16, kWaitTimeoutNs, status, 0, 0};
    return from_cuda(launch_gemv(g, sms, static_cast<cudaStream_t>(stream)));
}

cider_status cider_a16_gemv(const void* x, int32_t x_dtype, int64_t K, int64_t N, const void* w,
                            int32_t bits, const float* s_w, int32_t group_size, void* y,
                            int32_t y_dtype, void* stream) {
    if (!x || !w || !s_w || !y) return CIDER_ERR_INVALID_ARG;
    if (K <= 0 || N <= 0 || group_size < 0) return CIDER_ERR_INVALID_ARG;
    if (bits != 8 && bits != 4) return CIDER_ERR_INVALID_ARG;
    if (!valid_dtype(x_dtype) || !valid_dtype(y_dtype)) return CIDER_ERR_INVALID_ARG;
    if (K > 16384 || K % (bits == 8 ? 16 : 32) != 0) return CIDER_ERR_UNSUPPORTED;
    if (!valid_group(group_size, K, bits == 8 ? 16 : 32)) return CIDER_ERR_UNSUPPORTED;
    if (!aligned16(x) || !aligned16(w)) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    unsigned long long* status = nullptr;
    if (device_status_ptr(&status) != cudaSuccess) return CIDER_ERR_CUDA;
    GemvArgs g{x, K, N, w, s_w, bits, group_size, y, kWaitTimeoutNs, status,
               x_dtype == CIDER_DTYPE_BF16, y_dtype == CIDER_DTYPE_BF16, 1};
    return from_cuda(launch_gemv(g, sms, static_cast<cudaStream_t>(stream)));
}

cider_status cider_act_image(const void* x_f16, int64_t M, int64_t K, void* a_img, float* s_a,
                             void* stream) {
    if (!x_f16 || !a_img || !s_a) return CIDER_ERR_INVALID_ARG;
    if (M <= 0 || K <= 0) return CIDER_ERR_INVALID_ARG;
    if (K % 8 != 0 || !aligned16(x_f16) || !aligned16(a_img)) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    return from_cuda(launch_quant_groups(x_f16, ElemType::kF16, M, K, K, 127,
                                         QuantOut::kF16, a_img, s_a, sms,
                                         static_cast<cudaStream_t>(stream)));
}

cider_status cider_weight_image(const void* w, int64_t N, int64_t K, int32_t bits, void* b_img,
                                void* stream) {
    if (!w || !b_img) return CIDER_ERR_INVALID_ARG;
    if (N <= 0 || K <= 0 || (bits != 8 && bits != 4)) return CIDER_ERR_INVALID_ARG;
    if ((N * K) % 32 != 0 || !aligned16(w) || !aligned16(b_img)) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    return from_cuda(bits == 8 ? launch_widen_i8(static_cast<const int8_t*>(w), N * K,
                                                 static_cast<__half*>(b_img), sms, s)
                               : launch_widen_i4(static_cast<const uint8_t*>(w), N * K,
                                                 static_cast<__half*>(b_img), sms, s));
}

cider_status cider_gemm_images(const void* a_img, const float* s_a, const void* b_img,
                               const float* s_w, int64_t M, int64_t N, int64_t K,
                               int32_t group_size, void* y_f16, void* stream) {
    if (!a_img || !s_a || !b_img || !s_w || !y_f16) return CIDER_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || group_size < 0) return CIDER_ERR_INVALID_ARG;
    if (K % 16 != 0 || !valid_group(group_size, K, 64) || group_size > 1024)
        return CIDER_ERR_UNSUPPORTED;
    if (!aligned16(a_img) || !aligned16(b_img) || !aligned16(y_f16) || !aligned16(s_w))
        return CIDER_ERR_UNSUPPORTED;
    if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    unsigned long long* status = nullptr;
    if (device_status_ptr(&status) != cudaSuccess) return CIDER_ERR_CUDA;
    GemmArgs a{};
    a.a_img = static_cast<const __half*>(a_img);
    a.b_img = static_cast<const __half*>(b_img);
    a.M = M;
    a.N = N;
    a.K = K;
    a.group_size = group_size;
    a.s_a = s_a;
    a.s_w = s_w;
    a.out = y_f16;
    a.mode = (group_size == 0) ? GemmMode::kPcF16 : GemmMode::kPgF16;
    a.timeout_ns = kWaitTimeoutNs;
    a.status = status;
    return from_cuda(launch_gemm(a, sms, static_cast<cudaStream_t>(stream)));
}

cider_status cider_test_gemm_s32(const int8_t* q, const void* w, int64_t M, int64_t N, int64_t K,
                                 int32_t bits, int32_t group_size, int32_t* out, void* ws,
                                 size_t ws_bytes, void* stream) {
    if (!q || !w || !out) return CIDER_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0 || group_size < 0 || (bits != 8 && bits != 4))
        return CIDER_ERR_INVALID_ARG;
    if (K % 32 != 0 || !valid_group(group_size, K, 64) || group_size > 1024)
        return CIDER_ERR_UNSUPPORTED;
    if (!aligned16(q) || !aligned16(w) || !aligned16(out)) return CIDER_ERR_UNSUPPORTED;
    const int64_t Mw = M < 2 ? 2 : M;
    if (!ws || ws_bytes < workspace_bytes(Mw, N, K, group_size, bits)) return CIDER_ERR_WORKSPACE;
    if (!aligned16(ws)) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    unsigned long long* status = nullptr;
    if (device_status_ptr(&status) != cudaSuccess) return CIDER_ERR_CUDA;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    Workspace wsp = carve(ws, Mw, N, K, group_size, bits);
    cudaError_t e = launch_widen_i8(q, M * K, wsp.a_img, sms, s);
    if (e != cudaSuccess) return from_cuda(e);
    if (wsp.b_img) {
        e = (bits == 8) ? launch_widen_i8(static_cast<const int8_t*>(w), N * K, wsp.b_img, sms, s)
                        : launch_widen_i4(static_cast<const uint8_t*>(w), N * K, wsp.b_img, sms, s);
        if (e != cudaSuccess) return from_cuda(e);
    }
    GemmArgs a{};
    a.a_img = wsp.a_img;
    a.b_img = wsp.b_img;
    a.b_raw = wsp.b_img ? nullptr : w;
    a.b_bits = bits;
    a.M = M;
    a.N = N;
    a.K = K;
    a.group_size = group_size;
    a.s_a = nullptr;
    a.s_w = nullptr;
    a.out = out;
    a.mode = (group_size == 0) ? GemmMode::kRawS32 : GemmMode::kRawPgS32;
    a.timeout_ns = kWaitTimeoutNs;
    a.status = status;
    return from_cuda(launch_gemm(a, sms, s));
}

cider_status cider_test_int8_mma_loop(int32_t blocks, int64_t iters, int32_t* sink,
                                      void* stream) {
    if (blocks <= 0 || iters <= 0 || !sink) return CIDER_ERR_INVALID_ARG;
    return from_cuda(launch_int8_mma_loop(blocks, iters, sink, static_cast<cudaStream_t>(stream)));
}

cider_status cider_test_read_bytes(const void* src, int64_t bytes, uint32_t* sink, void* stream) {
    if (!src || !sink || bytes <= 0) return CIDER_ERR_INVALID_ARG;
    if (bytes % 16 != 0 || !aligned16(src)) return CIDER_ERR_UNSUPPORTED;
    int sms = 0;
    cider_status st = num_sms(&sms);
    if (st != CIDER_OK) return st;
    return from_cuda(launch_read_bytes(src, bytes, 2 * sms, sink,
                                       static_cast<cudaStream_t>(stream)));
}

cider_status cider_device_status(void* stream, uint32_t* site) {
    unsigned long long v = 0;
    if (read_and_clear_device_status(&v, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return CIDER_ERR_CUDA;
    if (site) *site = static_cast<uint32_t>(v & 0xFFFFFFFFu);
    if ((v >> 32) == kDevTimeout) return CIDER_ERR_TIMEOUT;
    return v == 0 ? CIDER_OK : CIDER_ERR_CUDA;
}

cider_status cider_test_wait_timeout(int64_t timeout_ns, void* stream) {
    if (timeout_ns <= 0 || timeout_ns > 10000000000ll) return CIDER_ERR_INVALID_ARG;
    return from_cuda(launch_wait_timeout_probe((uint64_t)timeout_ns,
                                               static_cast<cudaStream_t>(stream)));
}

}  // extern "C"
