// launch_setup.cuh -- launch helpers of the non-verify kernels: the per-device
// set-up of a kernel, kept between calls (the SM count, read once, and the
// dynamic shared-memory limit, raised only when a call needs more than an
// earlier one), so that a launch costs no attribute calls once a device has
// seen its shapes; and programmatic dependent launch for the short kernels
// of a step.
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

// Programmatic dependent launch, for the short kernels that follow one
// another in a step (commit, fold, cursor move): such a kernel may start while
// the kernel before it in the stream is finishing, and calls grid_dep_wait()
// before its first global memory access (it returns once every grid the
// kernel depends on has completed and its memory is visible; at once for a
// kernel launched without the attribute).  grid_dep_launch() lets the next
// kernel start its own launch early; only the commit and the cursor move call
// it, right after their wait, so at most two neighbouring kernels overlap.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                             Args &&...args) {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args &&>(args)...);
}

}  // namespace gdnspec
