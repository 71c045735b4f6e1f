// Calibration of the confidence head from the verification step's own outcomes
// (DevPress/CSDN article on DSpark in SGLang, section 5 "可观测性": per-request
// confidence and calibration metrics such as ECE; "DSpark：投机解码与生产级 Serving
// 学习笔记", section 07: the cumulative survival a_j predicts that prefix 1..j is
// accepted, and Sequential Temperature Scaling a_hat_j = sigmoid(logit(a_j) / T_j)
// calibrates it).
//
//   calib_collect_kernel  one CTA: per draft position j, the verified requests (j <
//                         w_r, or j < gamma in cap-accept mode) in request order
//                         append (a, a_hat, y = [j < cap_r]) to position j's sample
//                         store; offsets by block-wide exclusive scans, so the store
//                         is filled deterministically, step after step.
//   calib_ece_*_kernel    equal-width bins of the stored a_hat: per-CTA bins in shared
//                         memory over a slice of the samples, fp64 atomics into the
//                         outputs, then ECE = (1/N) sum_b |sum y - sum a_hat|.
//   sts_fit_kernel        one CTA per position: z = logit(a) in fp64 once into the
//                         workspace (kept as fp32), then bisections of log(1/T) on
//                         the derivative of the binary cross-entropy,
//                         sum (sigmoid(z/T) - y) z: sigmoid on the SFU, per-thread
//                         fp32 partial sums, fixed-order fp64 block reduction.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kCollectThreads = 1024;  // one thread per request (B <= 1024)
constexpr int kFitThreads = 1024;
constexpr int kEceThreads = 512;
constexpr double kLogBetaLo = -4.1588830833596715;  // log(1/64)
constexpr double kLogBetaHi = 4.1588830833596715;   // log(64)

__device__ __forceinline__ int warp_scan_incl(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

}  // namespace

__global__ void __launch_bounds__(kCollectThreads)
    calib_collect_kernel(const float* __restrict__ survival, const float* __restrict__ a_hat,
                         const int32_t* __restrict__ windows, const int32_t* __restrict__ cap_len,
                         int mode, int B, int gamma, float* __restrict__ s_a,
                         float* __restrict__ s_ahat, int8_t* __restrict__ s_y,
                         int32_t* __restrict__ count, int cap) {
  pdl_release();
  pdl_wait();  // survival, windows and cap_len come from the step's kernels
  __shared__ int s_warp[32];
  __shared__ int s_base;
  const int r = threadIdx.x;
  int v = 0, c = 0;
  if (r < B) {
    v = mode == DSPARK_CAP_ACCEPT ? gamma : windows[r];
    v = v < 0 ? 0 : (v > gamma ? gamma : v);
    c = cap_len[r];
  }
  const int nwarps = blockDim.x >> 5;
  for (int j = 0; j < gamma; ++j) {
    const int flag = (r < B && j < v) ? 1 : 0;
    const int incl = warp_scan_incl(flag);
    if ((r & 31) == 31) s_warp[r >> 5] = incl;
    if (r == 0) s_base = count[j];
    __syncthreads();
    if (r < 32) {
      int w = r < nwarps ? s_warp[r] : 0;
      w = warp_scan_incl(w);
      s_warp[r] = w;
    }
    __syncthreads();
    const int excl = ((r >> 5) ? s_warp[(r >> 5) - 1] : 0) + incl - flag;
    const int total = s_warp[nwarps - 1];
    const long long pos = static_cast<long long>(s_base) + excl;
    if (flag && pos < cap) {
      const long long at = static_cast<long long>(j) * cap + pos;
      s_a[at] = survival[r * gamma + j];
      s_ahat[at] = a_hat[r * gamma + j];
      s_y[at] = (j + 1 <= c) ? 1 : 0;
    }
    __syncthreads();
    if (r == 0) count[j] = s_base + total;  // samples seen; the store keeps the first cap
    __syncthreads();
  }
}

// ECE in three launches: zero the bins, accumulate (many CTAs, bins privatised in
// shared memory, then fp64 atomics into the outputs), finish (one thread).
__global__ void calib_ece_zero_kernel(int n_bins, int32_t* __restrict__ bin_n,
                                      double* __restrict__ bin_p, double* __restrict__ bin_y) {
  pdl_release();
  pdl_wait();
  for (int b = threadIdx.x; b < n_bins; b += blockDim.x) {
    bin_n[b] = 0;
    bin_p[b] = 0.0;
    bin_y[b] = 0.0;
  }
}

__global__ void __launch_bounds__(kEceThreads)
    calib_ece_kernel(const float* __restrict__ s_ahat, const int8_t* __restrict__ s_y,
                     const int32_t* __restrict__ count, int cap, int gamma, int n_bins,
                     int32_t* __restrict__ bin_n, double* __restrict__ bin_p,
                     double* __restrict__ bin_y) {
  pdl_release();
  pdl_wait();
  // bin sums of a_hat in fixed point (units of 2^-32, a_hat rounded to them): integer
  // additions are exact in any order, and so are the fp64 additions of the per-CTA
  // sums below 2^21 per bin -- the totals do not depend on the atomics' order
  __shared__ int h_n[DSPARK_MAX_ECE_BINS];
  __shared__ unsigned long long h_p[DSPARK_MAX_ECE_BINS];
  __shared__ int h_y[DSPARK_MAX_ECE_BINS];
  for (int b = threadIdx.x; b < n_bins; b += blockDim.x) {
    h_n[b] = 0;
    h_p[b] = 0ull;
    h_y[b] = 0;
  }
  __syncthreads();
  const int stride = gridDim.x * blockDim.x;
  for (int j = 0; j < gamma; ++j) {
    const int n = min(count[j], cap);
    for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < n; i += stride) {
      const float p = s_ahat[static_cast<long long>(j) * cap + i];
      int b = static_cast<int>(floor(static_cast<double>(p) * n_bins));  // exact product
      b = b < 0 ? 0 : (b >= n_bins ? n_bins - 1 : b);
      const double pc = p < 0.f ? 0.0 : (p > 1.f ? 1.0 : static_cast<double>(p));
      atomicAdd(&h_n[b], 1);
      atomicAdd(&h_p[b], __double2ull_rn(pc * 4294967296.0));
      atomicAdd(&h_y[b], static_cast<int>(s_y[static_cast<long long>(j) * cap + i]));
    }
  }
  __syncthreads();
  for (int b = threadIdx.x; b < n_bins; b += blockDim.x) {
    if (h_n[b] == 0) continue;
    atomicAdd(&bin_n[b], h_n[b]);
    atomicAdd(&bin_p[b], static_cast<double>(h_p[b]) * 2.3283064365386963e-10);  // 2^-32
    atomicAdd(&bin_y[b], static_cast<double>(h_y[b]));
  }
}

__global__ void calib_ece_finish_kernel(int n_bins, const int32_t* __restrict__ bin_n,
                                        const double* __restrict__ bin_p,
                                        const double* __restrict__ bin_y, double* __restrict__ ece) {
  pdl_release();
  pdl_wait();
  if (threadIdx.x == 0) {
    long long N = 0;
    double e = 0.0;
    for (int b = 0; b < n_bins; ++b) {
      N += bin_n[b];
      e += fabs(bin_y[b] - bin_p[b]);
    }
    *ece = N > 0 ? e / static_cast<double>(N) : 0.0;
  }
}

__global__ void __launch_bounds__(kFitThreads)
    sts_fit_kernel(const float* __restrict__ s_a, const int8_t* __restrict__ s_y,
                   const int32_t* __restrict__ count, int cap, int iters,
                   float* __restrict__ zbuf, float* __restrict__ temps) {
  pdl_release();
  pdl_wait();
  __shared__ double red[kFitThreads / 32];
  __shared__ double s_lo, s_hi;
  __shared__ int s_usable;
  const int j = blockIdx.x;
  const int n = min(count[j], cap);
  const long long base = static_cast<long long>(j) * cap;
  // z = logit(a) in fp64 once, kept as fp32 (a <= 0 or a >= 1: infinite logit, left
  // out as NaN)
  int usable = 0;
  for (int i = threadIdx.x; i < n; i += blockDim.x) {
    const double a = static_cast<double>(s_a[base + i]);
    const bool ok = a > 0.0 && a < 1.0;
    zbuf[base + i] = ok ? static_cast<float>(log(a) - log1p(-a)) : __int_as_float(0x7fc00000);
    usable += ok ? 1 : 0;
  }
  usable = __syncthreads_count(usable > 0);
  if (threadIdx.x == 0) {
    s_lo = kLogBetaLo;
    s_hi = kLogBetaHi;
    s_usable = usable;
  }
  __syncthreads();
  if (s_usable == 0) {
    if (threadIdx.x == 0) temps[j] = 1.f;
    return;
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  for (int it = 0; it < iters; ++it) {
    const double mid = 0.5 * (s_lo + s_hi);
    const float beta = static_cast<float>(exp(mid));
    // derivative of the loss at beta: per-thread fp32 partial sums (sigmoid on the
    // SFU), summed in fp64 across the block in a fixed order
    float g = 0.f;
    for (int i = threadIdx.x; i < n; i += blockDim.x) {
      const float z = zbuf[base + i];
      if (z == z) {
        const float sig = 1.f / (1.f + __expf(-beta * z));
        g = fmaf(sig - static_cast<float>(s_y[base + i]), z, g);
      }
    }
    double gd = static_cast<double>(g);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) gd += __shfl_xor_sync(0xffffffffu, gd, o);
    if (lane == 0) red[warp] = gd;
    __syncthreads();
    if (threadIdx.x == 0) {
      double t = 0.0;
      for (int w = 0; w < kFitThreads / 32; ++w) t += red[w];
      if (t > 0.0) s_hi = mid;
      else s_lo = mid;
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) temps[j] = static_cast<float>(1.0 / exp(0.5 * (s_lo + s_hi)));
}

int launch_calib_collect(const float* survival, const float* a_hat, const int32_t* windows,
                         const int32_t* cap_len, int mode, int B, int gamma, float* s_a,
                         float* s_ahat, int8_t* s_y, int32_t* count, int cap,
                         cudaStream_t stream) {
  return launch_pdl(calib_collect_kernel, dim3(1), dim3(kCollectThreads), 0, stream, survival,
                    a_hat, windows, cap_len, mode, B, gamma, s_a, s_ahat, s_y, count, cap) ==
                 cudaSuccess
             ? DSPARK_OK
             : DSPARK_ECUDA;
}

int launch_calib_ece(const float* s_ahat, const int8_t* s_y, const int32_t* count, int cap,
                     int gamma, int n_bins, int32_t* bin_n, double* bin_p, double* bin_y,
                     double* ece, cudaStream_t stream) {
  const long long work = static_cast<long long>(gamma) * cap;  // samples the store can hold
  long long grid = (work + kEceThreads * 16 - 1) / (kEceThreads * 16);
  const int sms = num_sms_cached();
  if (grid > 2LL * sms) grid = 2LL * sms;
  if (grid < 1) grid = 1;
  if (launch_pdl(calib_ece_zero_kernel, dim3(1), dim3(256), 0, stream, n_bins, bin_n, bin_p,
                 bin_y) != cudaSuccess ||
      launch_pdl(calib_ece_kernel, dim3(static_cast<int>(grid)), dim3(kEceThreads), 0, stream,
                 s_ahat, s_y, count, cap, gamma, n_bins, bin_n, bin_p, bin_y) != cudaSuccess ||
      launch_pdl(calib_ece_finish_kernel, dim3(1), dim3(32), 0, stream, n_bins, bin_n, bin_p,
                 bin_y, ece) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}

int launch_sts_fit(const float* s_a, const int8_t* s_y, const int32_t* count, int cap, int gamma,
                   int iters, float* zbuf, float* temps, cudaStream_t stream) {
  return launch_pdl(sts_fit_kernel, dim3(gamma), dim3(kFitThreads), 0, stream, s_a, s_y, count,
                    cap, iters, zbuf, temps) == cudaSuccess
             ? DSPARK_OK
             : DSPARK_ECUDA;
}

}  // namespace dspark
