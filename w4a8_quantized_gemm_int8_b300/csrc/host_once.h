// Once-per-device host-side setup shared by the launchers: kernel attributes
// (dynamic shared memory opt-in), device properties and occupancy figures.
// CUDA function attributes and device properties belong to a device, so each
// value is kept per device. Whichever thread asks first computes it, under
// std::call_once for that device's slot; later callers, on any thread, see
// the first call's status and value.
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace cider {

constexpr int kMaxDevices = 64;  // device ordinals handled (0 .. kMaxDevices - 1)

// The calling thread's current device, or -1 when there is none or its
// ordinal is kMaxDevices or more.
inline int current_device() {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
    return dev;
}

template <class T>
class PerDevice {
  public:
    // Runs init(value&) -> cudaError_t once for device `dev` and returns its
    // status; *out (if given) receives the value. Later calls for the same
    // device return the first call's status and value without running init.
    // An ordinal outside [0, kMaxDevices) returns cudaErrorInvalidDevice.
    template <class F>
    cudaError_t get(int dev, F&& init, T* out = nullptr) {
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        std::call_once(once_[dev], [&] { err_[dev] = init(val_[dev]); });
        if (out != nullptr) *out = val_[dev];
        return err_[dev];
    }

    // The same for the calling thread's current device.
    template <class F>
    cudaError_t get(F&& init, T* out = nullptr) {
        return get(current_device(), init, out);
    }

  private:
    std::once_flag once_[kMaxDevices];
    cudaError_t err_[kMaxDevices] = {};
    T val_[kMaxDevices] = {};
};

}  // namespace cider
