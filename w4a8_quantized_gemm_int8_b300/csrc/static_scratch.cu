// cider_w8a8_gemm_pc_noalloc: the W8A8 per-channel linear layer for callers
// that cannot allocate device memory.
//
// cider_w8a8_gemm_pc needs a caller-provided workspace (the fp16 operand
// images of the activation and weight codes, and the per-token scales).
// Some callers cannot call cudaMalloc at all: for example code hosted by a
// framework that owns every device allocation through its own pool and
// forbids others, or a latency-critical loop where cudaMalloc's implicit
// device synchronization is not acceptable. This variant takes its scratch
// from a fixed-size array compiled into the library instead.
//
// The array: kStaticScratchBytes (64 MiB) of device memory, file scope,
// shared by every call on a device and kept by every GPU that loads it until
// the process exits. Problems whose scratch would exceed it are rejected
// with CIDER_ERR_WORKSPACE before anything is enqueued.
//
// Host code cannot use the array's name as a device address (in host code
// it names a host-side stand-in), so the device address is looked up once
// per device, with that device current, by the first call on that device;
// that first call should therefore happen before any stream capture.
//
// Every call overwrites the parts of the array it reads (the kernels write
// the operand images and scales before the GEMM reads them, and rows beyond
// M are zero-filled by the tensor loads, not read from the array), so stale
// contents from an earlier call never matter. Calls whose execution overlaps
// on the GPU (different streams, or different host threads) share the array
// and race: serialize them.
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "../../include/cider.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;
constexpr uint64_t kWaitTimeoutNs = 2000000000ull;
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

constexpr size_t round256(size_t v) { return (v + 255) & ~static_cast<size_t>(255); }

// Device address of the array on the current device (looked up once).
cider_status scratch_address(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return CIDER_ERR_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return CIDER_ERR_UNSUPPORTED;
    std::lock_guard<std::mutex> lock(g_scratch_mutex);
    if (g_scratch_addr[dev] == nullptr) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_static_scratch) != cudaSuccess || p == nullptr)
            return CIDER_ERR_CUDA;
        g_scratch_addr[dev] = p;
    }
    *out = g_scratch_addr[dev];
    return CIDER_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

extern "C" cider_status cider_w8a8_gemm_pc_noalloc(const void* x_f16, int64_t M, int64_t N,
                                                   int64_t K, const int8_t* wq, const float* s_w,
                                                   void* y_f16, void* stream) {
    using namespace cider;
    if (!x_f16 || !wq || !s_w || !y_f16) return CIDER_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0) return CIDER_ERR_INVALID_ARG;
    if (K % 16 != 0) return CIDER_ERR_UNSUPPORTED;
    if (!aligned16(x_f16) || !aligned16(wq) || !aligned16(s_w) || !aligned16(y_f16))
        return CIDER_ERR_UNSUPPORTED;
    if (M > (1 << 30) || N > (1 << 30) || K > (1 << 30)) return CIDER_ERR_UNSUPPORTED;
    // Layout inside the array: a_img [M,K] fp16 | s_a [M] fp32 | b_img [N,K]
    // fp16 (only for the SM-pair engine; the single-SM engine reads wq itself).
    const bool img = gemm_uses_pair(M);
    const size_t a_bytes = round256((size_t)M * K * 2);
    const size_t s_bytes = round256((size_t)M * 4);
    const size_t b_bytes = img ? round256((size_t)N * K * 2) : 0;
    if (a_bytes + s_bytes + b_bytes > kStaticScratchBytes) return CIDER_ERR_WORKSPACE;

    void* base = nullptr;
    cider_status st = scratch_address(&base);
    if (st != CIDER_OK) return st;
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return CIDER_ERR_CUDA;
    unsigned long long* status = nullptr;
    if (device_status_ptr(&status) != cudaSuccess) return CIDER_ERR_CUDA;

    uint8_t* p = static_cast<uint8_t*>(base);
    __half* a_img = reinterpret_cast<__half*>(p);
    float* s_a = reinterpret_cast<float*>(p + a_bytes);
    __half* b_img = img ? reinterpret_cast<__half*>(p + a_bytes + s_bytes) : nullptr;
    cudaStream_t s = static_cast<cudaStream_t>(stream);

    cudaError_t e = launch_operand_images(x_f16, ElemType::kF16, M, K,
                                          img ? wq : nullptr, 8, N, a_img, s_a, b_img, nullptr,
                                          nullptr, 1, sms, s);
    if (e == cudaSuccess) {
        GemmArgs a{};
        a.a_img = a_img;
        a.b_img = b_img;
        a.b_raw = img ? nullptr : wq;
        a.b_bits = 8;
        a.M = M;
        a.N = N;
        a.K = K;
        a.group_size = 0;
        a.s_a = s_a;
        a.s_w = s_w;
        a.out = y_f16;
        a.mode = GemmMode::kPcF16;
        a.timeout_ns = kWaitTimeoutNs;
        a.status = status;
        e = launch_gemm(a, sms, s);
    }
    if (e == cudaSuccess) return CIDER_OK;
    if (e == cudaErrorInvalidValue) {
        cudaGetLastError();
        return CIDER_ERR_UNSUPPORTED;
    }
    return CIDER_ERR_CUDA;
}
