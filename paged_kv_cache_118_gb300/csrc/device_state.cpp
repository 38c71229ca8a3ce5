// Per-device launch state of the pagedkv kernels: SM counts and the dynamic
// shared-memory attribute a kernel needs, looked up once per device (and
// kernel) rather than once per process, so that a process may use several GPUs.
#include <cuda.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "pkv_host.h"

namespace pkv {

namespace {
std::mutex g_mu;
std::map<int, int> g_sms;                                      // device -> SM count
std::map<std::tuple<int, const void*, int>, int> g_occupancy;  // (device, kernel, smem) -> CTAs/SM
std::map<std::pair<int, const void*>, int> g_smem_limit;        // (device, kernel) -> limit set

template <typename F>
F driver_entry(const char* name, int version) {
  void* f = nullptr;
  cudaDriverEntryPointQueryResult q{};
  if (cudaGetDriverEntryPointByVersion(name, &f, version, cudaEnableDefault, &q) != cudaSuccess ||
      q != cudaDriverEntryPointSuccess)
    return nullptr;
  return reinterpret_cast<F>(f);
}
}  // namespace

bool current_context_id(unsigned long long* id) {
  static const auto get_current = driver_entry<PFN_cuCtxGetCurrent_v4000>("cuCtxGetCurrent", 4000);
  static const auto get_id = driver_entry<PFN_cuCtxGetId_v12000>("cuCtxGetId", 12000);
  *id = 0;
  if (get_current == nullptr || get_id == nullptr) return false;
  CUcontext ctx = nullptr;
  if (get_current(&ctx) != CUDA_SUCCESS) return false;
  if (ctx == nullptr) return true;                 // no context current on this thread yet
  return get_id(ctx, id) == CUDA_SUCCESS;
}

cudaError_t device_sm_count(int* sms) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  auto it = g_sms.find(dev);
  if (it == g_sms.end()) {
    int v = 0;
    e = cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    if (v < 1) return cudaErrorInvalidDevice;
    it = g_sms.emplace(dev, v).first;
  }
  *sms = it->second;
  return cudaSuccess;
}

cudaError_t prepare_kernel(const void* kernel, int threads, int smem_bytes, int* ctas_per_sm) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  std::lock_guard<std::mutex> lock(g_mu);
  // The limit only ever grows: a launch with less shared memory than the
  // limit is fine, one with more is refused.
  int& limit = g_smem_limit[std::make_pair(dev, kernel)];
  if (smem_bytes > limit) {
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
    if (e != cudaSuccess) return e;
    limit = smem_bytes;
  }
  const auto key = std::make_tuple(dev, kernel, smem_bytes);
  auto it = g_occupancy.find(key);
  if (it == g_occupancy.end()) {
    int blocks = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&blocks, kernel, threads, smem_bytes);
    if (e != cudaSuccess) return e;
    it = g_occupancy.emplace(key, blocks).first;
  }
  if (ctas_per_sm != nullptr) *ctas_per_sm = it->second;
  return cudaSuccess;
}

}  // namespace pkv
