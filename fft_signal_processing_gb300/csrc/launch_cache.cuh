// Per-device launch configuration of one kernel instantiation: its shared-memory attributes are
// set and its resident CTAs per SM and the device's SM count are queried on the first launch on
// each device, then reused.  A mutex serialises that set-up and every lookup, so host threads
// may launch the same kernel concurrently (each launcher owns one LaunchCache as a
// function-local static, whose construction C++ makes thread-safe).
#pragma once

#include <cuda_runtime.h>

#include <mutex>

namespace gbfft {

struct LaunchGeom {
    int per_sm = 0;   // resident CTAs per SM (persistent kernels; 0 where unused)
    int num_sms = 0;  // SMs of the device
};

class LaunchCache {
public:
    // setup(dev, &geom) runs once per device, with that device current; it returns
    // cudaSuccess after filling geom, and is run again on a later call if it failed.
    template <class Setup>
    cudaError_t get(Setup setup, LaunchGeom* out) {
        int dev = 0;
        cudaError_t e = cudaGetDevice(&dev);
        if (e != cudaSuccess) return e;
        if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
        std::lock_guard<std::mutex> lock(mu_);
        if (!ready_[dev]) {
            LaunchGeom g;
            e = setup(dev, &g);
            if (e != cudaSuccess) return e;
            geom_[dev] = g;
            ready_[dev] = true;
        }
        *out = geom_[dev];
        return cudaSuccess;
    }

private:
    static constexpr int kMaxDevices = 64;
    std::mutex mu_;
    bool ready_[kMaxDevices] = {};
    LaunchGeom geom_[kMaxDevices];
};

// The set-up of a persistent kernel: dynamic shared memory up to `smem` bytes, the largest
// shared-memory carveout, and the occupancy that sizes its grid.
template <class K>
cudaError_t setup_persistent(K kern, int threads, size_t smem, int dev, LaunchGeom* g) {
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, 100);
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&g->per_sm, kern, threads, smem);
    if (e == cudaSuccess) e = cudaDeviceGetAttribute(&g->num_sms, cudaDevAttrMultiProcessorCount, dev);
    if (e == cudaSuccess && g->per_sm < 1) e = cudaErrorInvalidConfiguration;
    return e;
}

}  // namespace gbfft
