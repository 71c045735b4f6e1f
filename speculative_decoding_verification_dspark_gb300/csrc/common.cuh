// Shared helpers for the dspark kernels (device side and launch side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <mutex>

#include "dspark.h"

namespace dspark {

// One-time host set-up per device (kernel attributes, occupancy queries, symbol
// addresses): fn() runs once for each device, with that device current, and its
// result is kept.  Safe when several host threads make their first call at once.
constexpr int kMaxDevices = 64;
template <class T>
struct PerDevice {
  std::once_flag flag[kMaxDevices];
  T value[kMaxDevices] = {};
};
// The current device's value, computed by fn() on first use; `fail` when the
// current device cannot be read or is out of range.
template <class T, class Fn>
T once_per_device(PerDevice<T>& pd, T fail, Fn&& fn) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return fail;
  std::call_once(pd.flag[dev], [&] { pd.value[dev] = fn(); });
  return pd.value[dev];
}

// Device error word: one per device, owned by api.cu.  Kernels receive its
// address as an argument so that no translation unit needs relocatable code.
unsigned int* device_error_word();

__device__ __forceinline__ void raise_error(unsigned int* err, unsigned int bits) {
  if (err) atomicOr(err, bits);
}

__host__ __device__ constexpr int ceil_div(int a, int b) { return (a + b - 1) / b; }

// Largest index i in [0, n) with cu[i] <= x, for an ascending cu[0..n].
__device__ __forceinline__ int upper_segment(const int32_t* cu, int n, int x) {
  int lo = 0, hi = n;  // invariant: cu[lo] <= x < cu[hi]
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (cu[mid] <= x) lo = mid; else hi = mid;
  }
  return lo;
}

int num_sms_cached();

// Programmatic dependent launch.  Every kernel of the library is launched with
// launch_pdl, may therefore start while the kernel before it in the stream is
// still running, and calls pdl_wait() before it touches global memory that
// earlier work writes or reads.  pdl_release() lets the next kernel start
// launching (its own pdl_wait() still waits for this grid to complete).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_release() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Set (for the calling host thread) while a graph is captured without programmatic
// dependencies: the launches below are then ordinary stream-ordered launches.
inline thread_local bool g_no_pdl = false;

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_no_pdl ? 0 : 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch_pdl with thread-block clusters of cluster_x CTAs along x.
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl_cluster(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                                      cudaStream_t stream, int cluster_x, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cluster_x;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = g_no_pdl ? 1 : 2;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace dspark
