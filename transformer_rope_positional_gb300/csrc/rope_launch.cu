// Launch bookkeeping shared by the kernels' launchers: the launch counter,
// the SM count, occupancy-sized persistent grids and the dynamic shared
// memory opt-in.
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "rope_launch.h"

namespace rope {

namespace {
std::atomic<uint64_t> g_launches{0};  // every kernel launch of the library
constexpr int kMaxDevices = 64;
std::once_flag g_sm_once[kMaxDevices];
int g_sm_count[kMaxDevices];
}  // namespace

void count_launch() { g_launches.fetch_add(1, std::memory_order_relaxed); }

uint64_t launch_count() { return g_launches.load(std::memory_order_relaxed); }

int sm_count() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 148;
  std::call_once(g_sm_once[dev], [dev] {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
    g_sm_count[dev] = n;
  });
  return g_sm_count[dev];
}

cudaError_t opt_in_shared(const void* kernel, size_t smem) {
  static std::mutex mu;
  static std::map<std::pair<int, const void*>, size_t> granted;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(mu);
  size_t& have = granted[std::make_pair(dev, kernel)];
  if (have >= smem) return cudaSuccess;
  e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (e == cudaSuccess) have = smem;
  return e;
}

int resident_blocks(const void* kernel, int threads, size_t smem) {
  static std::mutex mu;
  static std::map<std::tuple<int, const void*, int, size_t>, int> cache;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) dev = -1;
  const auto key = std::make_tuple(dev, kernel, threads, smem);
  {
    std::lock_guard<std::mutex> lock(mu);
    auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  int n = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem) != cudaSuccess || n < 1) {
    (void)cudaGetLastError();  // do not leave a sticky-looking error for the launch check
    n = 1;
  }
  std::lock_guard<std::mutex> lock(mu);
  cache[key] = n;
  return n;
}

}  // namespace rope
