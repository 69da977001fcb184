// Host-side state kept per device: the SM count and the dynamic shared-memory limit already
// raised for each kernel.  cudaFuncSetAttribute acts on the current device only, so a kernel
// launched on a second GPU of the same process needs its own opt-in; both tables are keyed by
// the device ordinal and guarded by one mutex (several host threads may launch at once).
#include <map>
#include <mutex>
#include <utility>

#include "internal.cuh"

namespace moe {
namespace {

std::mutex g_mu;
std::map<int, int> g_sm_count;                           // device -> SM count
std::map<std::pair<int, const void*>, int> g_smem;       // (device, kernel) -> bytes opted in

}  // namespace

cudaError_t current_sm_count(int* n) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_sm_count.find(dev);
  if (it == g_sm_count.end()) {
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (v <= 0) return cudaErrorInvalidDevice;
    it = g_sm_count.emplace(dev, v).first;
  }
  *n = it->second;
  return cudaSuccess;
}

cudaError_t ensure_dynamic_smem(const void* kernel, int bytes) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  int& have = g_smem[{dev, kernel}];
  if (have >= bytes) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e == cudaSuccess) have = bytes;
  return e;
}

}  // namespace moe
