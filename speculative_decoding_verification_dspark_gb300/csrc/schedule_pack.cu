// Confidence scheduling and ragged packing.
//
// schedule_kernel (one CTA of 1024 threads):
//   * one thread per request: c_k (sigmoid of the confidence logit, fp64 then one
//     fp32 rounding), prefix survival a_j = prod_{i<=j} c_i as an fp32 running
//     product, Sequential Temperature Scaling a_hat_j = sigmoid(logit(a_j)/T_j)
//     in fp64 rounded to fp32, clamped non-increasing in j
//     ("DSpark：投机解码与生产级 Serving 学习笔记", section 07 Confidence Head);
//   * a bitonic sort of the <= 4096 (a_hat, request, position) keys in shared
//     memory, survival descending, ties by request then position;
//   * the greedy of section 08.3 (add candidates while expected throughput
//     E / T(M) rises, stop at the first that does not; M = bs + K as in the
//     CSDN article's additive cost model): fp64 block-wide prefix sums give E
//     before every candidate, each candidate's decision is evaluated in
//     parallel, and the first failing index is a block-wide minimum.
// pack_kernel (one CTA): exclusive scan of the per-request row counts
//   (cu_seqlens), tier selection, and per-row request / position / token
//   ("DFlash 到 DSpark in SGLang", section "Ragged verify under full CUDA graphs").

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kSchedThreads = 1024;
constexpr int kPerThread = DSPARK_MAX_CANDS / kSchedThreads;  // 4

__device__ __forceinline__ double warp_incl_scan(double v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    double u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

__device__ __forceinline__ int warp_incl_scan_i(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

}  // namespace

__global__ void __launch_bounds__(kSchedThreads)
    schedule_kernel(const float* __restrict__ conf, int conf_is_logit,
                    const float* __restrict__ sts_temp, const float* __restrict__ cost, int B,
                    int gamma, int max_tokens, int mode, int32_t* __restrict__ windows,
                    float* __restrict__ a_hat, int32_t* __restrict__ M_out,
                    double* __restrict__ E_out) {
  __shared__ unsigned long long keys[DSPARK_MAX_CANDS];
  __shared__ double s_warp[32];
  __shared__ int s_first;
  __shared__ int s_win[DSPARK_MAX_B];
  const int tid = threadIdx.x;
  const int n = B * gamma;
  int npow = 1;
  while (npow < n) npow <<= 1;

  if (tid == 0) s_first = n;
  for (int r = tid; r < B; r += blockDim.x) {
    float acc = 0.f, prev = 0.f;
    for (int j = 0; j < gamma; ++j) {
      const float x = conf[r * gamma + j];
      float c = x;
      if (conf_is_logit) {
        const double z = static_cast<double>(x);
        c = __double2float_rn(1.0 / (1.0 + exp(-z)));
      }
      acc = (j == 0) ? c : __fmul_rn(acc, c);
      const double a = static_cast<double>(acc);
      double y;
      if (a <= 0.0) {
        y = 0.0;
      } else if (a >= 1.0) {
        y = 1.0;
      } else {
        const double t = (log(a) - log1p(-a)) / static_cast<double>(sts_temp[j]);
        y = 1.0 / (1.0 + exp(-t));
      }
      float v = __double2float_rn(y);
      if (j > 0 && v > prev) v = prev;
      prev = v;
      a_hat[r * gamma + j] = v;
      keys[r * gamma + j] = (static_cast<unsigned long long>(~__float_as_uint(v)) << 32) |
                            (static_cast<unsigned>(r) << 16) | static_cast<unsigned>(j);
    }
    s_win[r] = 0;
  }
  for (int i = n + tid; i < npow; i += blockDim.x) keys[i] = ~0ull;
  __syncthreads();

  // bitonic sort, ascending keys = survival descending
  for (int k = 2; k <= npow; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      for (int i = tid; i < npow; i += blockDim.x) {
        const int ixj = i ^ j;
        if (ixj > i) {
          const unsigned long long a = keys[i], b = keys[ixj];
          const bool up = (i & k) == 0;
          if ((a > b) == up) {
            keys[i] = b;
            keys[ixj] = a;
          }
        }
      }
      __syncthreads();
    }
  }

  // E_k = B + sum_{i<k} a_hat(i), fp64, thread owns 4 consecutive candidates
  double v[kPerThread];
  double local = 0.0;
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int k = tid * kPerThread + q;
    v[q] = (k < n) ? static_cast<double>(__uint_as_float(~static_cast<unsigned>(keys[k] >> 32)))
                   : 0.0;
    local += v[q];
  }
  double incl = warp_incl_scan(local);
  if ((tid & 31) == 31) s_warp[tid >> 5] = incl;
  __syncthreads();
  if (tid < 32) {
    double w = s_warp[tid];
    w = warp_incl_scan(w);
    s_warp[tid] = w;
  }
  __syncthreads();
  const double warp_off = (tid >> 5) ? s_warp[(tid >> 5) - 1] : 0.0;
  const double total = s_warp[31];
  double E = static_cast<double>(B) + warp_off + (incl - local);

  const bool greedy = (mode != DSPARK_STATIC);
  int first_fail = n;
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int k = tid * kPerThread + q;
    if (greedy && k < n && first_fail == n) {
      const int M = B + k;
      bool ok = (M + 1 <= max_tokens);
      if (ok) {
        const double lhs = (E + v[q]) / static_cast<double>(cost[M + 1]);
        const double rhs = E / static_cast<double>(cost[M]);
        ok = lhs > rhs;
      }
      if (!ok) first_fail = k;
    }
    E += v[q];
  }
  if (first_fail < n) atomicMin(&s_first, first_fail);
  __syncthreads();
  const int kstar = greedy ? s_first : n;

  for (int k = tid; k < kstar; k += blockDim.x) {
    const int r = static_cast<int>((keys[k] >> 16) & 0xFFFFu);
    atomicAdd(&s_win[r], 1);
  }
  // E before candidate k*: the owning thread recomputes it
  if (kstar < n && kstar / kPerThread == tid) {
    double e = static_cast<double>(B) + warp_off + (incl - local);
    for (int q = 0; q < kstar % kPerThread; ++q) e += v[q];
    *E_out = e;
  }
  if (kstar >= n && tid == 0) *E_out = static_cast<double>(B) + total;
  __syncthreads();
  for (int r = tid; r < B; r += blockDim.x) windows[r] = greedy ? s_win[r] : gamma;
  if (tid == 0) *M_out = B + kstar;
}

__global__ void __launch_bounds__(1024)
    pack_kernel(const int32_t* __restrict__ windows, const int32_t* __restrict__ ctx_len,
                const int32_t* __restrict__ anchor, const int32_t* __restrict__ draft_tok,
                const int32_t* __restrict__ tiers, int n_tiers, int B, int gamma, int mode,
                int max_rows, int32_t* __restrict__ cu_seqlens, int32_t* __restrict__ M_out,
                int32_t* __restrict__ tier_out, int32_t* __restrict__ row_req,
                int32_t* __restrict__ row_pos, int32_t* __restrict__ row_tok,
                unsigned int* __restrict__ err) {
  __shared__ int s_cu[DSPARK_MAX_B + 1];
  __shared__ int s_warp[32];
  __shared__ int s_tier;
  const int tid = threadIdx.x;
  int cnt = 0;
  if (tid < B) {
    int w = windows[tid];
    if (w < 0 || w > gamma) {
      raise_error(err, DSPARK_DEVERR_BAD_INPUT);
      w = w < 0 ? 0 : gamma;
    }
    cnt = 1 + (mode == DSPARK_CAP_ACCEPT ? gamma : w);
  }
  const int incl = warp_incl_scan_i(cnt);
  if ((tid & 31) == 31) s_warp[tid >> 5] = incl;
  __syncthreads();
  if (tid < 32) {
    int w = s_warp[tid];
    w = warp_incl_scan_i(w);
    s_warp[tid] = w;
  }
  __syncthreads();
  const int off = ((tid >> 5) ? s_warp[(tid >> 5) - 1] : 0) + incl;
  if (tid < B) s_cu[tid + 1] = off;
  if (tid == 0) s_cu[0] = 0;
  __syncthreads();
  const int M = s_cu[B];
  if (tid == 0) {
    int tier = M;
    for (int i = 0; i < n_tiers; ++i) {
      if (tiers[i] >= M) {
        tier = tiers[i];
        break;
      }
    }
    s_tier = tier;
    *M_out = M;
    *tier_out = tier;
    if (tier > max_rows) raise_error(err, DSPARK_DEVERR_ROWS_OVERFLOW);
  }
  for (int i = tid; i <= B; i += blockDim.x) cu_seqlens[i] = s_cu[i];
  __syncthreads();
  const int limit = s_tier < max_rows ? s_tier : max_rows;
  for (int row = tid; row < limit; row += blockDim.x) {
    if (row < M) {
      const int r = upper_segment(s_cu, B, row);
      const int i = row - s_cu[r];
      row_req[row] = r;
      row_pos[row] = ctx_len[r] + i;
      row_tok[row] = (i == 0) ? anchor[r] : draft_tok[r * gamma + i - 1];
    } else {
      row_req[row] = -1;
      row_pos[row] = -1;
      row_tok[row] = -1;
    }
  }
}

int launch_schedule(const float* conf, int conf_is_logit, const float* sts_temp,
                    const float* cost_table, int B, int gamma, int max_tokens, int mode,
                    int32_t* windows, float* a_hat, int32_t* M_out, double* E_out,
                    cudaStream_t stream) {
  schedule_kernel<<<1, kSchedThreads, 0, stream>>>(conf, conf_is_logit, sts_temp, cost_table, B,
                                                   gamma, max_tokens, mode, windows, a_hat, M_out,
                                                   E_out);
  DSPARK_LAUNCH_CHECK();
  return DSPARK_OK;
}

int launch_pack(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out, int32_t* tier_out,
                int32_t* row_req, int32_t* row_pos, int32_t* row_tok, cudaStream_t stream) {
  pack_kernel<<<1, 1024, 0, stream>>>(windows, ctx_len, anchor, draft_tok, tiers, n_tiers, B, gamma,
                                      mode, max_rows, cu_seqlens, M_out, tier_out, row_req, row_pos,
                                      row_tok, device_error_word());
  DSPARK_LAUNCH_CHECK();
  return DSPARK_OK;
}

}  // namespace dspark
