// Confidence scheduling and ragged packing.
//
// calibrate_kernel (one warp per request, many CTAs): c_k (sigmoid of the
//   confidence logit, fp64 then one fp32 rounding), prefix survival
//   a_j = prod_{i<=j} c_i as fp32 products in left-to-right order, Sequential
//   Temperature Scaling a_hat_j = sigmoid(logit(a_j)/T_j) in fp64 rounded to fp32,
//   clamped non-increasing in j ("DSpark：投机解码与生产级 Serving 学习笔记",
//   section 07 Confidence Head).  FP64 is slow on this part, so these run spread
//   over the whole GPU rather than in the sorting CTA.
// greedy_kernel (one CTA of 1024 threads): a bitonic sort of the <= 4096
//   (a_hat, request, position) keys, survival descending, ties by request then
//   position; the greedy of section 08.3 (add candidates while expected
//   throughput E / T(M) rises, stop at the first that does not; M = bs + K as in
//   the CSDN article's additive cost model): fp64 block-wide prefix sums give E
//   before every candidate, each candidate's test is evaluated in parallel, and
//   the first failing index is a block-wide minimum.
// pack_kernel (one CTA): exclusive scan of the per-request row counts
//   (cu_seqlens), tier selection, and per-row request / position / token
//   ("DFlash 到 DSpark in SGLang", section "Ragged verify under full CUDA graphs").

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn.h"
#include "common.cuh"
#include "kernels.h"
#include "worklist.cuh"

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

// Calibration: one warp per request, lane j = position j (gamma <= 32).  The fp64
// transcendentals of every position run in parallel across warps and CTAs;
// lane j forms a_j = ((c_0 c_1) c_2 ... c_j) with the fp32 products taken in that
// left-to-right order; the clamp to a non-increasing sequence is an (exact)
// inclusive min-scan over the lanes.
__global__ void __launch_bounds__(64)
    calibrate_kernel(const float* __restrict__ conf, int conf_is_logit,
                     const float* __restrict__ sts_temp, int B, int gamma,
                     float* __restrict__ a_hat, float* __restrict__ survival) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  const int r = blockIdx.x * 2 + (threadIdx.x >> 5);
  const int j = threadIdx.x & 31;
  if (r >= B) return;  // warp-uniform
  float c = 1.f;
  if (j < gamma) {
    const float x = conf[r * gamma + j];
    c = x;
    if (conf_is_logit) c = __double2float_rn(1.0 / (1.0 + exp(-static_cast<double>(x))));
  }
  float a = 0.f;
  for (int i = 0; i < gamma; ++i) {
    const float ci = __shfl_sync(0xffffffffu, c, i);
    if (i == 0) a = ci;
    else if (i <= j) a = __fmul_rn(a, ci);
  }
  if (survival && j < gamma) survival[r * gamma + j] = a;  // uncalibrated, for refits
  float v = 1.f;
  if (j < gamma) {
    const double ad = static_cast<double>(a);
    double y;
    if (ad <= 0.0) {
      y = 0.0;
    } else if (ad >= 1.0) {
      y = 1.0;
    } else {
      const double t = (log(ad) - log1p(-ad)) / static_cast<double>(sts_temp[j]);
      y = 1.0 / (1.0 + exp(-t));
    }
    v = __double2float_rn(y);
  }
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const float u = __shfl_up_sync(0xffffffffu, v, o);
    if (j >= o) v = fminf(v, u);
  }
  if (j < gamma) a_hat[r * gamma + j] = v;
}

// Compare-exchange of register slots A < B (indices tid + A*T < tid + B*T) in
// bitonic stage k.
template <int A, int Bq>
__device__ __forceinline__ void bitonic_slots(unsigned long long (&kv)[4], int tid, int T, int k) {
  const bool asc = ((tid + A * T) & k) == 0;
  const unsigned long long a = kv[A], b = kv[Bq];
  if ((a > b) == asc) {
    kv[A] = b;
    kv[Bq] = a;
  }
}

// Greedy window choice over the calibrated survival (one CTA, one thread per
// candidate up to 1024): bitonic sort of the <= 4096 (a_hat, request, position)
// keys, fp64 block-wide prefix sums of a_hat in sorted order (E before each
// candidate), every candidate's throughput test in parallel, first failure by a
// block minimum.
__global__ void __launch_bounds__(kSchedThreads)
    greedy_kernel(const float* __restrict__ a_hat, const float* __restrict__ cost, int B,
                  int gamma, int max_tokens, int mode, int32_t* __restrict__ windows,
                  int32_t* __restrict__ M_out, double* __restrict__ E_out) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  __shared__ unsigned long long keys[DSPARK_MAX_CANDS];
  __shared__ double s_warp[32];
  __shared__ int s_first;
  __shared__ int s_win[DSPARK_MAX_B];
  const int tid = threadIdx.x;
  const int n = B * gamma;
  int npow = 1;
  while (npow < n) npow <<= 1;

  if (tid == 0) s_first = n;
  for (int r = tid; r < B; r += blockDim.x) s_win[r] = 0;
  // Bitonic sort, ascending keys = survival descending.  Thread t holds the keys
  // at t + q*T (T = blockDim.x, q < npow/T) in registers: pairs at distance < 32
  // are exchanged by shuffles, at distance >= T inside the thread, and only the
  // distances 32..T/2 go through shared memory.
  const int T = blockDim.x;
  if (npow < T) npow = T;  // at least one key per thread (padding keys sort last)
  const int m = npow / T;  // 1, 2 or 4 (npow <= T * kPerThread, T >= 32)
  unsigned long long kv[kPerThread];
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int k = tid + q * T;
    unsigned long long key = ~0ull;
    if (q < m && k < n) {
      const int r = k / gamma, j = k - r * gamma;
      key = (static_cast<unsigned long long>(~__float_as_uint(a_hat[k])) << 32) |
            (static_cast<unsigned>(r) << 16) | static_cast<unsigned>(j);
    }
    kv[q] = key;
  }
  for (int k = 2; k <= npow; k <<= 1) {
    for (int j = k >> 1; j > 0; j >>= 1) {
      if (j >= T) {  // partner in this thread: slot q ^ (j / T), j / T = 1 or 2
        if (j == T) {
          bitonic_slots<0, 1>(kv, tid, T, k);
          if (m > 2) bitonic_slots<2, 3>(kv, tid, T, k);
        } else {
          bitonic_slots<0, 2>(kv, tid, T, k);
          bitonic_slots<1, 3>(kv, tid, T, k);
        }
      } else if (j >= 32) {  // partner in another warp: through shared memory
#pragma unroll
        for (int q = 0; q < kPerThread; ++q)
          if (q < m) keys[tid + q * T] = kv[q];
        __syncthreads();
#pragma unroll
        for (int q = 0; q < kPerThread; ++q) {
          if (q < m) {
            const int i = tid + q * T;
            const unsigned long long p = keys[i ^ j];
            const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
            kv[q] = keep_min ? (kv[q] < p ? kv[q] : p) : (kv[q] > p ? kv[q] : p);
          }
        }
        __syncthreads();
      } else {  // partner lane ^ j of this warp
#pragma unroll
        for (int q = 0; q < kPerThread; ++q) {
          if (q < m) {  // uniform over the block
            const int i = tid + q * T;
            const unsigned long long p = __shfl_xor_sync(0xffffffffu, kv[q], j);
            const bool keep_min = ((i & j) == 0) == ((i & k) == 0);
            kv[q] = keep_min ? (kv[q] < p ? kv[q] : p) : (kv[q] > p ? kv[q] : p);
          }
        }
      }
    }
  }
#pragma unroll
  for (int q = 0; q < kPerThread; ++q)
    if (q < m) keys[tid + q * T] = kv[q];
  __syncthreads();

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
  const int nwarps = blockDim.x >> 5;
  double incl = warp_incl_scan(local);
  if ((tid & 31) == 31) s_warp[tid >> 5] = incl;
  __syncthreads();
  if (tid < 32) {
    double w = tid < nwarps ? s_warp[tid] : 0.0;
    w = warp_incl_scan(w);
    s_warp[tid] = w;
  }
  __syncthreads();
  const double warp_off = (tid >> 5) ? s_warp[(tid >> 5) - 1] : 0.0;
  const double total = s_warp[nwarps - 1];
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
        // throughput E/T(M) rises iff (E + a) T[M] > E T[M+1]  (T > 0)
        const double lhs = __dmul_rn(E + v[q], static_cast<double>(cost[M]));
        const double rhs = __dmul_rn(E, static_cast<double>(cost[M + 1]));
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
    if (r < B) atomicAdd(&s_win[r], 1);
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

// The pack of one step, by every thread of a 1024-thread CTA.  Besides the device
// outputs it can publish the tier to a pinned host word (ts.host) and select the
// matching body of a step graph's switch node (ts.use): body i for tiers[i], body
// n_tiers for a batch above every tier (run unpadded), none if it overflows max_rows.
__device__ inline void pack_body(const TierSel ts, const int32_t* __restrict__ windows,
                                 const int32_t* __restrict__ ctx_len,
                                 const int32_t* __restrict__ anchor,
                                 const int32_t* __restrict__ draft_tok,
                                 const int32_t* __restrict__ tiers, int n_tiers, int B, int gamma,
                                 int mode, int max_rows, int32_t* __restrict__ cu_seqlens,
                                 int32_t* __restrict__ M_out, int32_t* __restrict__ tier_out,
                                 int32_t* __restrict__ row_req, int32_t* __restrict__ row_pos,
                                 int32_t* __restrict__ row_tok, unsigned int* __restrict__ err) {
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
    int body = n_tiers;
    for (int i = 0; i < n_tiers; ++i)
      if (tiers[i] == tier) {
        body = i;
        break;
      }
    if (tier > max_rows) {
      raise_error(err, DSPARK_DEVERR_ROWS_OVERFLOW);
      body = n_tiers + 1;  // no body: the rest of the step is skipped
    }
    if (ts.host) *reinterpret_cast<volatile int32_t*>(ts.host) = tier;
    if (ts.use) cudaGraphSetConditional(ts.handle, static_cast<unsigned int>(body));
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

__global__ void __launch_bounds__(1024)
    pack_kernel(const int32_t* __restrict__ windows, const int32_t* __restrict__ ctx_len,
                const int32_t* __restrict__ anchor, const int32_t* __restrict__ draft_tok,
                const int32_t* __restrict__ tiers, int n_tiers, int B, int gamma, int mode,
                int max_rows, int32_t* __restrict__ cu_seqlens, int32_t* __restrict__ M_out,
                int32_t* __restrict__ tier_out, int32_t* __restrict__ row_req,
                int32_t* __restrict__ row_pos, int32_t* __restrict__ row_tok,
                const TierSel ts, unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  pack_body(ts, windows, ctx_len, anchor, draft_tok, tiers, n_tiers, B, gamma, mode, max_rows,
            cu_seqlens, M_out, tier_out, row_req, row_pos, row_tok, err);
}

// Pack, then the attention work list of the same step from the cu_seqlens just
// written (this CTA's own global writes, visible to it after the barrier): one kernel
// fewer between the step's schedule and its attention.
struct PackPlanArgs {
  int attn_max_rows, Hkv, parts, rows_per_tile, nk, ncta, max_splits, rotate, max_items;
  attn::AttnItem* items;
  int* item_begin;
  attn::SplitGroup* groups;
};

__global__ void __launch_bounds__(1024)
    pack_plan_kernel(const int32_t* __restrict__ windows, const int32_t* __restrict__ ctx_len,
                     const int32_t* __restrict__ anchor, const int32_t* __restrict__ draft_tok,
                     const int32_t* __restrict__ tiers, int n_tiers, int B, int gamma, int mode,
                     int max_rows, int32_t* __restrict__ cu_seqlens, int32_t* __restrict__ M_out,
                     int32_t* __restrict__ tier_out, int32_t* __restrict__ row_req,
                     int32_t* __restrict__ row_pos, int32_t* __restrict__ row_tok,
                     const PackPlanArgs a, const TierSel ts, unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  pack_body(ts, windows, ctx_len, anchor, draft_tok, tiers, n_tiers, B, gamma, mode, max_rows,
            cu_seqlens, M_out, tier_out, row_req, row_pos, row_tok, err);
  __syncthreads();  // cu_seqlens (global, written above by this CTA) is complete
  extern __shared__ __align__(16) uint8_t pack_plan_smem[];
  attn::WorkListSmem& S = *reinterpret_cast<attn::WorkListSmem*>(pack_plan_smem);
  attn::build_work_list(S, ctx_len, cu_seqlens, B, a.attn_max_rows, a.Hkv, a.parts,
                        a.rows_per_tile, a.nk, a.ncta, a.max_splits, a.rotate, a.max_items, a.items,
                        a.item_begin, a.groups, err);
}

int launch_schedule(const float* conf, int conf_is_logit, const float* sts_temp,
                    const float* cost_table, int B, int gamma, int max_tokens, int mode,
                    int32_t* windows, float* a_hat, float* survival, int32_t* M_out,
                    double* E_out, cudaStream_t stream) {
  if (launch_pdl(calibrate_kernel, dim3(ceil_div(B, 2)), dim3(64), 0, stream, conf, conf_is_logit,
                 sts_temp, B, gamma, a_hat, survival) != cudaSuccess)
    return DSPARK_ECUDA;
  int npow = 1;
  while (npow < B * gamma) npow <<= 1;
  // one sorting key per thread up to 1024 keys (two or four beyond), at least a warp
  const int threads = npow < 32 ? 32 : (npow > kSchedThreads ? kSchedThreads : npow);
  if (launch_pdl(greedy_kernel, dim3(1), dim3(threads), 0, stream, a_hat, cost_table, B, gamma,
                 max_tokens, mode, windows, M_out, E_out) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}

int launch_pack_plan(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                     const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                     int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out,
                     int32_t* tier_out, int32_t* row_req, int32_t* row_pos, int32_t* row_tok,
                     int attn_max_rows, int Hkv, int max_splits, const attn::Plan& pl,
                     void* attn_ws, const TierSel& ts, cudaStream_t stream) {
  static PerDevice<bool> configured;
  const int smem = static_cast<int>(sizeof(attn::WorkListSmem));
  if (!once_per_device(configured, false, [&] {
        return cudaFuncSetAttribute(pack_plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    smem) == cudaSuccess;
      }))
    return DSPARK_ECUDA;
  uint8_t* w = static_cast<uint8_t*>(attn_ws);
  PackPlanArgs a;
  a.attn_max_rows = attn_max_rows;
  a.Hkv = Hkv;
  a.parts = pl.parts;
  a.rows_per_tile = pl.rows_per_tile;
  a.nk = pl.nk;
  a.ncta = pl.ncta;
  a.max_splits = max_splits < 2 ? 2 : (max_splits > 32 ? 32 : max_splits);
  a.rotate = pl.mla ? 1 : 0;  // as the attention call's own work list
  a.max_items = pl.max_items > 0x7fffffff ? 0x7fffffff : static_cast<int>(pl.max_items);
  a.items = reinterpret_cast<attn::AttnItem*>(w + pl.off_items);
  a.item_begin = reinterpret_cast<int*>(w + pl.off_begin);
  a.groups = reinterpret_cast<attn::SplitGroup*>(w + pl.off_groups);
  if (launch_pdl(pack_plan_kernel, dim3(1), dim3(1024), smem, stream, windows, ctx_len, anchor,
                 draft_tok, tiers, n_tiers, B, gamma, mode, max_rows, cu_seqlens, M_out, tier_out,
                 row_req, row_pos, row_tok, a, ts, device_error_word()) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}

int launch_pack(const int32_t* windows, const int32_t* ctx_len, const int32_t* anchor,
                const int32_t* draft_tok, const int32_t* tiers, int n_tiers, int B, int gamma,
                int mode, int max_rows, int32_t* cu_seqlens, int32_t* M_out, int32_t* tier_out,
                int32_t* row_req, int32_t* row_pos, int32_t* row_tok, const TierSel& ts,
                cudaStream_t stream) {
  if (launch_pdl(pack_kernel, dim3(1), dim3(1024), 0, stream, windows, ctx_len, anchor, draft_tok,
                 tiers, n_tiers, B, gamma, mode, max_rows, cu_seqlens, M_out, tier_out, row_req,
                 row_pos, row_tok, ts, device_error_word()) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}

}  // namespace dspark
