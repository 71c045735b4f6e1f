// Confidence scheduling and ragged packing.
//
// calibrate_kernel (one warp of floor(32/gamma) requests per CTA): c_k (sigmoid of the
//   confidence logit, fp64 then one fp32 rounding), prefix survival
//   a_j = prod_{i<=j} c_i as fp32 products in left-to-right order, Sequential
//   Temperature Scaling a_hat_j = sigmoid(logit(a_j)/T_j) in fp64 rounded to fp32,
//   clamped non-increasing in j ("DSpark：投机解码与生产级 Serving 学习笔记",
//   section 07 Confidence Head).  FP64 is slow on this part, so these run spread
//   over the whole GPU rather than in the sorting CTA.
// greedy_kernel (one CTA of up to 1024 threads): the <= 4096 (a_hat, request,
//   position) candidates ordered survival descending, ties by request then
//   position, by merging the per-request runs (each already in order); the greedy
//   of section 08.3 (add candidates while expected
//   throughput E / T(M) rises, stop at the first that does not; M = bs + K as in
//   the CSDN article's additive cost model): exact fixed-point block-wide prefix
//   sums give E before every candidate, each candidate's test is evaluated in
//   parallel (fp32 with a proven error bound, fp64 for near-ties), and the first
//   failing index is a block-wide minimum.
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

__device__ __forceinline__ int warp_incl_scan_i(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

__device__ __forceinline__ long long warp_incl_scan_ll(long long v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const long long u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// A fixed-point E (units 2^-50) as fp64 (rounded once).
__device__ __forceinline__ double fx_to_double(long long e) {
  return __ll2double_rn(e) * 8.8817841970012523e-16;  // 2^-50, exact scaling
}

// Does the throughput E / T(M) rise with the candidate: (E + a) T[M] > E T[M+1]
// (T > 0), E in units of 2^-50?  In fp32 first: E32 = fl(E), l = fl(fl(E32 + a) T[M]),
// r = fl(E32 T[M+1]) are each within 3 * 2^-24 (relative) of the exact products, so a
// gap beyond 2^-20 decides the exact comparison; otherwise the test is taken in fp64
// as written (E rounded once to fp64), like a plain fp64 evaluation.
__device__ __forceinline__ bool throughput_rises(long long E, float a, float tm, float tm1) {
  const float e32 = __ll2float_rn(E) * 8.8817841970012523e-16f;  // 2^-50
  const float l = __fmul_rn(__fadd_rn(e32, a), tm);
  const float r = __fmul_rn(e32, tm1);
  if (l > r * (1.0f + 9.5367431640625e-07f)) return true;   // 1 + 2^-20
  if (l < r * (1.0f - 9.5367431640625e-07f)) return false;
  const double e = fx_to_double(E);
  return __dmul_rn(e + static_cast<double>(a), static_cast<double>(tm)) >
         __dmul_rn(e, static_cast<double>(tm1));
}

}  // namespace

// Calibration by one warp of floor(32 / gamma) requests: request g * rpw + s on
// lanes s * gamma .. s * gamma + gamma - 1, lane s * gamma + j = position j.  The
// fp64 transcendentals of all its lanes run in parallel (fp64 work is counted per
// warp instruction, so filling the lanes divides it); lane j forms
// a_j = ((c_0 c_1) c_2 ... c_j) with the fp32 products taken in that left-to-right
// order; the clamp to a non-increasing sequence is an (exact) inclusive min-scan
// within the request's lanes.
__device__ __forceinline__ int requests_per_warp(int gamma) { return 32 / gamma; }

__device__ __forceinline__ void calibrate_group(int g, int B, const float* __restrict__ conf,
                                                int conf_is_logit,
                                                const float* __restrict__ sts_temp, int gamma,
                                                float* __restrict__ a_hat,
                                                float* __restrict__ survival) {
  const int lane = threadIdx.x & 31;
  const int rpw = requests_per_warp(gamma);
  const int seg = lane / gamma, j = lane - seg * gamma, base = seg * gamma;
  const int r = g * rpw + seg;
  const bool live = seg < rpw && r < B;  // this lane holds (r, j)
  float c = 1.f;
  if (live) {
    const float x = conf[r * gamma + j];
    c = x;
    if (conf_is_logit) c = __double2float_rn(1.0 / (1.0 + exp(-static_cast<double>(x))));
  }
  float a = 0.f;
  for (int i = 0; i < gamma; ++i) {
    const float ci = __shfl_sync(0xffffffffu, c, (base + i) & 31);
    if (i == 0) a = ci;
    else if (i <= j) a = __fmul_rn(a, ci);
  }
  if (live && survival) survival[r * gamma + j] = a;  // uncalibrated, for refits
  float v = 1.f;
  if (live) {
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
    if (j >= o) v = fminf(v, u);  // lane - o is in the same request
  }
  if (live) a_hat[r * gamma + j] = v;
}

// One warp per CTA (fp64 throughput is per SM on this part: one calibrating warp per
// SM is the fastest arrangement), floor(32 / gamma) requests per warp.
__global__ void __launch_bounds__(32)
    calibrate_kernel(const float* __restrict__ conf, int conf_is_logit,
                     const float* __restrict__ sts_temp, int B, int gamma,
                     float* __restrict__ a_hat, float* __restrict__ survival) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  calibrate_group(blockIdx.x, B, conf, conf_is_logit, sts_temp, gamma, a_hat, survival);
}

// Greedy window choice over the calibrated survival (one CTA): the candidates in
// order (run merging, below), E before every candidate by an exact fixed-point
// block-wide prefix sum, every candidate's throughput test in parallel, the first
// failure by a block minimum.
// One CTA of T threads (a multiple of 32, npow(B*gamma) clamped to 32..1024); each
// thread holds four consecutive candidates in the scan and the tests.
// Ordering buffers (dynamic shared memory): values and candidate indices, two each.
struct SortSmem {
  float val[2][DSPARK_MAX_CANDS];
  uint16_t idx[2][DSPARK_MAX_CANDS];
};

__global__ void __launch_bounds__(kSchedThreads)
    greedy_kernel(const float* __restrict__ a_hat, const float* __restrict__ cost, int B,
                  int gamma, int max_tokens, int mode, int32_t* __restrict__ windows,
                  int32_t* __restrict__ M_out, double* __restrict__ E_out) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  extern __shared__ __align__(16) uint8_t greedy_smem[];
  SortSmem& ss = *reinterpret_cast<SortSmem*>(greedy_smem);
  float (&s_val)[2][DSPARK_MAX_CANDS] = ss.val;
  uint16_t (&s_idx)[2][DSPARK_MAX_CANDS] = ss.idx;
  __shared__ long long s_warp[32];
  __shared__ int s_first;
  __shared__ int s_win[DSPARK_MAX_B];
  const int tid = threadIdx.x;
  const int T = blockDim.x;
  const int n = B * gamma;

  if (tid == 0) s_first = n;
  for (int r = tid; r < B; r += blockDim.x) s_win[r] = 0;
  // Order: a_hat descending, ties by request then position.  Each request's gamma
  // candidates are already in that order (a_hat is non-increasing in j), so the runs
  // of 1, 2, 4, ... requests are merged pairwise: an element of the left run moves
  // past the right run's elements that are strictly larger, an element of the right
  // run past the left run's elements that are larger or equal (ties: lower request
  // first) -- one binary search each, all elements of a level in parallel.
  for (int k = tid; k < n; k += blockDim.x) {
    s_val[0][k] = a_hat[k];
    s_idx[0][k] = static_cast<uint16_t>(k);
  }
  __syncthreads();
  int src = 0;
  for (int run = gamma; run < n; run <<= 1, src ^= 1) {
    const float* sv = s_val[src];
    const uint16_t* si = s_idx[src];
    for (int k = tid; k < n; k += blockDim.x) {
      const int p0 = (k / (2 * run)) * (2 * run);
      const int b0 = min(p0 + run, n), b1 = min(p0 + 2 * run, n);
      const float x = sv[k];
      int lo, hi;  // binary search in the other run
      if (k < b0) {
        lo = b0; hi = b1;  // first right element <= x
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (sv[mid] > x) lo = mid + 1; else hi = mid;
        }
        const int pos = p0 + (k - p0) + (lo - b0);
        s_val[src ^ 1][pos] = x;
        s_idx[src ^ 1][pos] = si[k];
      } else {
        lo = p0; hi = b0;  // first left element < x
        while (lo < hi) {
          const int mid = (lo + hi) >> 1;
          if (sv[mid] >= x) lo = mid + 1; else hi = mid;
        }
        const int pos = p0 + (k - b0) + (lo - p0);
        s_val[src ^ 1][pos] = x;
        s_idx[src ^ 1][pos] = si[k];
      }
    }
    __syncthreads();
  }
  const float* sorted_val = s_val[src];
  const uint16_t* sorted_idx = s_idx[src];

  // E_k = B + sum_{i<k} a_hat(i) as an exact integer sum in units of 2^-50 (each
  // a_hat rounded to that unit, error <= 2^-51 per term; E < 2^13 fits int64): no
  // fp64 arithmetic, and the same value in any summation order.  Thread owns 4
  // consecutive candidates.
  constexpr float kFx = 1125899906842624.0f;  // 2^50
  long long v[kPerThread];
  float av[kPerThread];
  long long local = 0;
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int k = tid * kPerThread + q;
    av[q] = k < n ? sorted_val[k] : 0.f;
    v[q] = __float2ll_rn(av[q] * kFx);  // exact scaling by a power of two
    local += v[q];
  }
  const int nwarps = T >> 5;
  long long incl = warp_incl_scan_ll(local);
  if ((tid & 31) == 31) s_warp[tid >> 5] = incl;
  __syncthreads();
  if (tid < 32) {
    long long w = tid < nwarps ? s_warp[tid] : 0ll;
    w = warp_incl_scan_ll(w);
    s_warp[tid] = w;
  }
  __syncthreads();
  const long long warp_off = (tid >> 5) ? s_warp[(tid >> 5) - 1] : 0ll;
  const long long total = s_warp[nwarps - 1];
  const long long e0 = (static_cast<long long>(B) << 50) + warp_off + (incl - local);
  long long E = e0;

  const bool greedy = (mode != DSPARK_STATIC);
  int first_fail = n;
#pragma unroll
  for (int q = 0; q < kPerThread; ++q) {
    const int k = tid * kPerThread + q;
    if (greedy && k < n && first_fail == n) {
      const int M = B + k;
      bool ok = (M + 1 <= max_tokens);
      if (ok) ok = throughput_rises(E, av[q], cost[M], cost[M + 1]);
      if (!ok) first_fail = k;
    }
    E += v[q];
  }
  if (first_fail < n) atomicMin(&s_first, first_fail);
  __syncthreads();
  const int kstar = greedy ? s_first : n;

  if (greedy) {
    for (int k = tid; k < kstar; k += blockDim.x) atomicAdd(&s_win[sorted_idx[k] / gamma], 1);
  }
  // E before candidate k*: the owning thread recomputes it
  if (kstar < n && kstar / kPerThread == tid) {
    long long e = e0;
    for (int q = 0; q < kstar % kPerThread; ++q) e += v[q];
    *E_out = fx_to_double(e);
  }
  if (kstar >= n && tid == 0) *E_out = fx_to_double((static_cast<long long>(B) << 50) + total);
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
  __shared__ int s_tiers[DSPARK_MAX_TIERS];
  const int tid = threadIdx.x;
  // the tiers, one load per thread beside the windows' (the tier search below then
  // reads shared memory instead of a chain of global loads)
  if (tid < n_tiers) s_tiers[tid] = tiers[tid];
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
      if (s_tiers[i] >= M) {
        tier = s_tiers[i];
        break;
      }
    }
    s_tier = tier;
    *M_out = M;
    *tier_out = tier;
    int body = n_tiers;
    for (int i = 0; i < n_tiers; ++i)
      if (s_tiers[i] == tier) {
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
  if (launch_pdl(calibrate_kernel, dim3(ceil_div(B, 32 / gamma)), dim3(32), 0, stream, conf,
                 conf_is_logit, sts_temp, B, gamma, a_hat, survival) != cudaSuccess)
    return DSPARK_ECUDA;
  int npow = 1;
  while (npow < B * gamma) npow <<= 1;
  // one sorting key per thread up to 1024 keys (two or four beyond), at least a warp
  const int threads = npow < 32 ? 32 : (npow > kSchedThreads ? kSchedThreads : npow);
  static PerDevice<bool> configured;
  const int smem = static_cast<int>(sizeof(SortSmem));
  if (!once_per_device(configured, false, [&] {
        return cudaFuncSetAttribute(greedy_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                    smem) == cudaSuccess;
      }))
    return DSPARK_ECUDA;
  if (launch_pdl(greedy_kernel, dim3(1), dim3(threads), smem, stream, a_hat, cost_table, B, gamma,
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
