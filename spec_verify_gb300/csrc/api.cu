// Library-wide entry points (status strings, version) and host launch helpers.
#include <cuda_runtime.h>

#include <stdlib.h>

#include <map>
#include <tuple>
#include <mutex>
#include <utility>

#include "launch.h"
#include "smp.h"

namespace smp {

static thread_local int g_last_cuda_error = 0;

__global__ void clear_status_kernel(int32_t* status) {
  asm volatile("griddepcontrol.launch_dependents;");
  asm volatile("griddepcontrol.wait;" ::: "memory");
  if (threadIdx.x == 0) *status = 0;
}

smp_status clear_status(int32_t* status, cudaStream_t stream) {
  LaunchShape ls;
  ls.pdl = true;
  int32_t* arg = status;
  const cudaError_t err =
      launch_cluster(reinterpret_cast<const void*>(&clear_status_kernel), dim3(1), dim3(32), ls, stream, &arg);
  if (err != cudaSuccess) return fail_cuda(err);
  return SMP_OK;
}

smp_status fail_cuda(cudaError_t err) {
  g_last_cuda_error = int(err);
  return SMP_ERR_CUDA;
}

int current_device() {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess) return -1;
  return dev;
}

int device_sms(int dev) {
  static std::mutex mu;
  static std::map<int, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  auto it = cache.find(dev);
  if (it != cache.end()) return it->second;
  int sms = 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    sms = 1;
  cache[dev] = sms;
  return sms;
}

int forced_cluster() {
  const char* v = getenv("SMP_FORCE_CLUSTER");
  if (!v) return 0;
  const int c = atoi(v);
  return (c == 1 || c == 2 || c == 4 || c == 8 || c == 16) ? c : 0;
}

bool verbose() { return getenv("SMP_VERBOSE") != nullptr; }

uint64_t wait_limit_ns() {
  const char* v = getenv("SMP_WAIT_LIMIT_NS");
  if (v && *v) {
    char* end = nullptr;
    const unsigned long long n = strtoull(v, &end, 10);
    if (end && *end == '\0') return uint64_t(n);
  }
  return 2000000000ull;
}

cudaError_t prepare_kernel(const void* kernel, int dev, const LaunchShape& ls) {
  static std::mutex mu;
  static std::map<std::pair<const void*, int>, std::pair<size_t, int>> done;
  std::lock_guard<std::mutex> lock(mu);
  auto& slot = done[{kernel, dev}];
  if (slot.first < ls.smem) {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, int(ls.smem));
    if (err != cudaSuccess) return err;
    slot.first = ls.smem;
  }
  if (ls.cluster > 8 && slot.second == 0) {
    cudaError_t err = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (err != cudaSuccess) return err;
    slot.second = 1;
  }
  return cudaSuccess;
}

cudaError_t max_active_clusters(const void* kernel, int dev, const LaunchShape& ls, int* out) {
  static std::mutex mu;
  static std::map<std::tuple<const void*, int, int, size_t>, int> cache;
  std::lock_guard<std::mutex> lock(mu);
  const auto key = std::make_tuple(kernel, dev, ls.cluster, ls.smem);
  auto it = cache.find(key);
  if (it != cache.end()) {
    *out = it->second;
    return cudaSuccess;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(unsigned(ls.cluster) * 64u);
  cfg.blockDim = dim3(256);
  cfg.dynamicSmemBytes = ls.smem;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(ls.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  const cudaError_t err = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg);
  if (err != cudaSuccess) return err;
  cache[key] = n;
  *out = n;
  return cudaSuccess;
}

}  // namespace smp

extern "C" const char* smp_status_string(smp_status s) {
  switch (s) {
    case SMP_OK: return "SMP_OK";
    case SMP_ERR_INVALID_ARG: return "SMP_ERR_INVALID_ARG: a pointer is NULL or misaligned, or a size is out of range";
    case SMP_ERR_DTYPE: return "SMP_ERR_DTYPE: dtype must be SMP_F32 or SMP_BF16";
    case SMP_ERR_CUDA: return "SMP_ERR_CUDA: a CUDA runtime call failed (smp_last_cuda_error has the code)";
    case SMP_ERR_UNSUPPORTED: return "SMP_ERR_UNSUPPORTED: the vocabulary is larger than the kernels support";
    case SMP_ERR_WORKSPACE: return "SMP_ERR_WORKSPACE: the workspace is NULL, misaligned or too small";
  }
  return "unknown smp_status";
}

extern "C" int32_t smp_last_cuda_error(void) { return smp::g_last_cuda_error; }

extern "C" int32_t smp_abi_version(void) { return SMP_ABI_VERSION; }
