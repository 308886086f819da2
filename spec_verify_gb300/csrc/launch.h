// Host-side launch helpers: device queries, per-kernel attributes and
// cluster launches through cudaLaunchKernelEx.
#pragma once

#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <mutex>

#include "smp.h"

namespace smp {

constexpr size_t kSliceTargetBytes = 48 * 1024;   // preferred slice per CTA
constexpr size_t kSliceMinBytes = 8 * 1024;       // smallest slice worth a CTA
constexpr size_t kMaxDynamicSmem = 200 * 1024;

struct LaunchShape {
  int cluster = 1;   // CTAs per row
  int slice = 0;     // elements per CTA
  size_t smem = 0;   // dynamic shared memory per CTA
  bool pdl = false;  // programmatic launch: the kernel may start before the previous kernel on the
                     // stream ends, and waits for it (griddepcontrol.wait) before touching memory
};

// Records `err` as the last CUDA error of this thread and returns SMP_ERR_CUDA.
smp_status fail_cuda(cudaError_t err);

// Clears the device status word with a one-CTA kernel launched as a
// programmatic dependent of the previous kernel on `stream`: it lets the next
// kernel be scheduled at once and waits for the previous one before the store.
// Kernels launched after it with LaunchShape::pdl must call
// grid_dependency_wait() before they touch memory.
smp_status clear_status(int32_t* status, cudaStream_t stream);

// Current device, or -1 if it cannot be queried.
int current_device();

// Number of SMs of `dev` (cached).
int device_sms(int dev);

// Cluster size forced through the environment variable SMP_FORCE_CLUSTER
// (1, 2, 4, 8 or 16; used by tests to show that results do not depend on the
// launch shape), or 0.
int forced_cluster();

// True when the environment variable SMP_VERBOSE is set: launch shapes are
// printed to stderr.
bool verbose();

// Time limit, in nanoseconds, of one bounded device wait: the environment
// variable SMP_WAIT_LIMIT_NS when it holds a number (0 gives up at the first
// poll that finds the awaited data missing, which lets a test see the
// expiry path on normal inputs), else 2 s.
uint64_t wait_limit_ns();

// Sets the dynamic shared memory limit and, for clusters above 8, the
// non-portable cluster size attribute of `kernel` (once per device and size).
cudaError_t prepare_kernel(const void* kernel, int dev, const LaunchShape& ls);

// Number of clusters of shape `ls` that can be resident at once (cached).
cudaError_t max_active_clusters(const void* kernel, int dev, const LaunchShape& ls, int* out);

// Launches `kernel(*args)` with a cluster of ls.cluster CTAs along x.
template <typename Args>
cudaError_t launch_cluster(const void* kernel, dim3 grid, dim3 block, const LaunchShape& ls,
                           cudaStream_t stream, Args* args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = ls.smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = unsigned(ls.cluster);
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  unsigned n = 1;
  if (ls.pdl) {
    attr[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[n].val.programmaticStreamSerializationAllowed = 1;
    ++n;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  void* params[1] = {args};
  return cudaLaunchKernelExC(&cfg, kernel, params);
}

}  // namespace smp
