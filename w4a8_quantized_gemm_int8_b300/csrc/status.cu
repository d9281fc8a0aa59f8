// The device status word that bounded waits report to, and a small kernel
// whose mbarrier wait is never satisfied (used by the test suite to check,
// without hanging or faulting the GPU, that a wait gives up and reports).
#include <cuda_runtime.h>
#include <cstdint>

#include "device_common.cuh"
#include "host_once.h"
#include "kernels.h"

namespace cider {

namespace {
__device__ unsigned long long g_status_word = 0;

// One thread initialises an mbarrier that expects one arrival, never arrives,
// and waits on it with the bounded wait. It returns normally after
// `timeout_ns`, leaving kDevTimeout in the status word.
__global__ void wait_timeout_probe_kernel(uint64_t timeout_ns, unsigned long long* status) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        fence_mbar_init();
        (void)mbar_wait_bounded(smem_u32(&bar), 0, timeout_ns, &abort_flag, status, 0x901);
    }
}

PerDevice<unsigned long long*> g_status_ptr;
}  // namespace

cudaError_t device_status_ptr(unsigned long long** ptr) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    return g_status_ptr.get(dev, [](unsigned long long*& v) {
        void* p = nullptr;
        const cudaError_t r = cudaGetSymbolAddress(&p, g_status_word);
        v = static_cast<unsigned long long*>(p);
        return r;
    }, ptr);
}

cudaError_t read_and_clear_device_status(unsigned long long* value, cudaStream_t stream) {
    unsigned long long* dptr = nullptr;
    cudaError_t e = device_status_ptr(&dptr);
    if (e != cudaSuccess) return e;
    e = cudaStreamSynchronize(stream);
    if (e != cudaSuccess) return e;
    unsigned long long v = 0;
    e = cudaMemcpy(&v, dptr, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return e;
    if (v != 0) {
        const unsigned long long zero = 0;
        e = cudaMemcpy(dptr, &zero, sizeof zero, cudaMemcpyHostToDevice);
        if (e != cudaSuccess) return e;
    }
    *value = v;
    return cudaSuccess;
}

cudaError_t launch_wait_timeout_probe(uint64_t timeout_ns, cudaStream_t stream) {
    unsigned long long* dptr = nullptr;
    cudaError_t e = device_status_ptr(&dptr);
    if (e != cudaSuccess) return e;
    wait_timeout_probe_kernel<<<1, 32, 0, stream>>>(timeout_ns, dptr);
    return cudaGetLastError();
}

}  // namespace cider
