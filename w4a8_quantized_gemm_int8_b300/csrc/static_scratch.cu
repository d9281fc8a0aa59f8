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
// The call is cider_w8a8_gemm_pc's own layer body (the same checks, the same
// workspace layout and the same kernels) with the array as its workspace;
// only M == 1 differs: it runs the tensor-core GEMM instead of the GEMV (the
// same results). Every call overwrites the parts of the array it reads (the
// kernels write the operand images and scales before the GEMM reads them,
// and rows beyond M are zero-filled by the tensor loads, not read from the
// array), so stale contents from an earlier call never matter. Calls whose
// execution overlaps on the GPU (different streams, or different host
// threads) share the array and race: serialize them.
#include <cuda_runtime.h>
#include <cstdint>
#include <mutex>

#include "../../include/cider.h"
#include "kernels.h"

namespace {

constexpr size_t kStaticScratchBytes = size_t(64) << 20;
static_assert(kStaticScratchBytes == CIDER_STATIC_SCRATCH_BYTES, "size stated in cider.h");
constexpr int kMaxDevices = 64;

static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

std::mutex g_scratch_mutex;
void* g_scratch_addr[kMaxDevices] = {};

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

}  // namespace

extern "C" cider_status cider_w8a8_gemm_pc_noalloc(const void* x_f16, int64_t M, int64_t N,
                                                   int64_t K, const int8_t* wq, const float* s_w,
                                                   void* y_f16, void* stream) {
    if (!x_f16 || !wq || !s_w || !y_f16) return CIDER_ERR_INVALID_ARG;
    if (M <= 0 || N <= 0 || K <= 0) return CIDER_ERR_INVALID_ARG;
    // Problems whose scratch exceeds the array are refused before the
    // address lookup (the layer body checks the size again, M == 1 included).
    if (M > 1 && cider_workspace_bytes(M, N, K, 0, 8) > kStaticScratchBytes)
        return CIDER_ERR_WORKSPACE;
    void* base = nullptr;
    const cider_status st = scratch_address(&base);
    if (st != CIDER_OK) return st;
    return cider::linear_call(x_f16, CIDER_DTYPE_F16, M, N, K, wq, 8, s_w, 0, y_f16,
                              CIDER_DTYPE_F16, base, kStaticScratchBytes,
                              static_cast<cudaStream_t>(stream), false);
}
