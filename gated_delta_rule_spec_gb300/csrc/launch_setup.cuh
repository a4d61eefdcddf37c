// launch_setup.cuh -- per-device launch set-up of a kernel, kept between calls:
// the SM count (read once) and the dynamic shared-memory limit (raised only
// when a call needs more than an earlier one), so that a launch costs no
// attribute calls once a device has seen its shapes.
#pragma once

#include <cstddef>
#include <mutex>

#include <cuda_runtime.h>

namespace gdnspec {

constexpr int kSetupDevices = 64;

// One record per kernel (a function-local static next to its launch).
struct KernelSetup {
    std::mutex mu;
    int sms[kSetupDevices] = {};           // 0 until the device is set up
    size_t smem_set[kSetupDevices] = {};   // dynamic shared-memory limit set so far
};

// On the current device: make sure `kern` may use `smem` bytes of dynamic
// shared memory and return the device's SM count.
inline cudaError_t kernel_setup(KernelSetup &ks, const void *kern, size_t smem, int *sms_out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= kSetupDevices) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(ks.mu);
    if (!ks.sms[dev]) {
        int sms = 0;
        if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
        ks.sms[dev] = sms;
    }
    if (smem > ks.smem_set[dev]) {
        if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem)) != cudaSuccess)
            return e;
        ks.smem_set[dev] = smem;
    }
    *sms_out = ks.sms[dev];
    return cudaSuccess;
}

}  // namespace gdnspec
