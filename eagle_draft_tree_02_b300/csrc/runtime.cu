// Host-side runtime helpers shared by the launch code.
#include <cuda_runtime.h>

#include <map>
#include <mutex>
#include <utility>

#include "common.cuh"

namespace e3 {

// The dynamic shared-memory limit is an attribute of a kernel on one device,
// so it is raised once per (device, kernel) -- a process that drives several
// GPUs, or one whose host threads share the library, gets it on each device.
bool smem_limit(const void* kernel, int bytes) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, int> done;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_pair(dev, kernel);
  auto it = done.find(key);
  if (it != done.end() && it->second >= bytes) return true;
  if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  done[key] = bytes;
  return true;
}

}  // namespace e3
