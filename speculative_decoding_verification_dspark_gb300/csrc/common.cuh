// Shared helpers for the dspark kernels (device side and launch side).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "dspark.h"

namespace dspark {

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

}  // namespace dspark

#define DSPARK_LAUNCH_CHECK()                                  \
  do {                                                         \
    cudaError_t e__ = cudaGetLastError();                      \
    if (e__ != cudaSuccess) return DSPARK_ECUDA;                \
  } while (0)
