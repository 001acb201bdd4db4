// Kernel launches that opt in to programmatic dependent launch: the kernel may
// start while its predecessor in the stream is still running; everything it
// reads from earlier kernels comes after grid_dep_wait().
#pragma once

#include <cuda_runtime.h>
#include <stdlib.h>

#include <atomic>
#include <mutex>

namespace tq {

// One-time set-up of a kernel per device (its shared-memory attribute, the
// device's SM count ...), done for the device current at the call and kept
// for that device; safe when several threads launch at once.
constexpr int kMaxDevices = 64;
struct PerDevice {
  std::atomic<int> ready[kMaxDevices];
  int value[kMaxDevices];
  std::mutex mu;
};

// Runs setup(dev, value) once per device; *out (if not null) receives the
// value it stored.
template <typename F>
cudaError_t per_device(PerDevice& pd, int* out, F&& setup) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  if (!pd.ready[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(pd.mu);
    if (!pd.ready[dev].load(std::memory_order_relaxed)) {
      int v = 0;
      e = setup(dev, v);
      if (e != cudaSuccess) return e;
      pd.value[dev] = v;
      pd.ready[dev].store(1, std::memory_order_release);
    }
  }
  if (out != nullptr) *out = pd.value[dev];
  return cudaSuccess;
}

inline bool pdl_enabled() {
  // TQ_PDL=0 turns programmatic dependent launch off (for A/B timing)
  static const int on = [] {
    const char* v = getenv("TQ_PDL");
    return (v != nullptr && v[0] == '0') ? 0 : 1;
  }();
  return on != 0;
}

template <typename... KArgs, typename... Args>
cudaError_t launch_k(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                     Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// Same, with a 1-D thread-block cluster of `cluster` CTAs along x.
template <typename... KArgs, typename... Args>
cudaError_t launch_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, int cluster,
                           cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = pdl_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace tq
