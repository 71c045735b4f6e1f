// Prefix speculative-sampling acceptance, bonus/correction token and the c* label.
//
// Sources: "DSpark：投机解码与生产级 Serving 学习笔记" section 02 (acceptance is a
// prefix: after the first rejection every later draft is discarded) and section
// 07 (c*_k = 1 - 1/2 ||p_d,k - p_t,k||_1); "DFlash 到 DSpark in SGLang" sections
// "Background" (the verify forward also yields a bonus token) and "Confidence
// scheduler 与 verify 模式" (cap-accept verifies the block, commits to the window).
//
// Three kernels:
//   accept_test_kernel   one warp per request, one lane per position: the fp32 test
//                        u*p_d(d_j) <= p_t(d_j) over the verified positions ->
//                        committed length, cap, and which packed row is sampled
//                        (residual or target).
//   accept_vocab_kernel  persistent grid over (packed row, vocab chunk): one pass of
//                        128-bit coalesced loads of p_t and p_d computes the partial
//                        L1 distance for c*, and on the sampled row the partial
//                        exponential-race argmax (w_v / e_v, lowest index on ties)
//                        for both the residual max(0, p_t - p_d) and p_t itself.
//   accept_final_kernel  one warp per request: fixed-order fp64 sums of the chunk
//                        partials (c*) and the chunk-ordered argmax (token).

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

constexpr int kVocabThreads = 256;
constexpr int kChunk = 8192;  // vocabulary entries per work item (32 per thread)

struct RowInfo {        // per request
  int commit, cap, sample_row, residual;
};

struct __align__(16) Partial {  // per (packed row, chunk)
  double l1;
  float key_res;
  int idx_res;
  float key_t;
  int idx_t;
};

__device__ __forceinline__ float ld_p(const float* p, long long i) { return __ldg(p + i); }
__device__ __forceinline__ float ld_p(const __nv_bfloat16* p, long long i) {
  return __bfloat162float(p[i]);
}

template <class T>
struct Vec8;  // eight consecutive probabilities as fp32
template <>
struct Vec8<float> {
  __device__ static void load(const float* p, float (&x)[8]) {
    const float4 a = __ldcs(reinterpret_cast<const float4*>(p));
    const float4 b = __ldcs(reinterpret_cast<const float4*>(p) + 1);
    x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
    x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
  }
};
template <>
struct Vec8<__nv_bfloat16> {
  __device__ static void load(const __nv_bfloat16* p, float (&x)[8]) {
    const uint4 u = __ldcs(reinterpret_cast<const uint4*>(p));
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      x[2 * i] = __uint_as_float(w[i] << 16);
      x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
    }
  }
};

__device__ __forceinline__ void better(float& k, int& i, float k2, int i2) {
  if (k2 > k || (k2 == k && i2 < i)) {
    k = k2;
    i = i2;
  }
}

}  // namespace

// One warp per request, lane j = draft position j+1: every test's two gathers are
// issued at once; the accepted prefix is the run of set bits from lane 0.
template <class T>
__global__ void __launch_bounds__(128)
    accept_test_kernel(const T* __restrict__ p_t, const T* __restrict__ p_d, int V,
                       const int32_t* __restrict__ draft_tok, const float* __restrict__ uniforms,
                       const int32_t* __restrict__ windows, const int32_t* __restrict__ cu,
                       int mode, int B, int gamma, int max_rows, int32_t* __restrict__ accept_len,
                       int32_t* __restrict__ cap_len, RowInfo* __restrict__ info,
                       unsigned int* __restrict__ err) {
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (cu[B] > max_rows) {  // packed rows beyond the caller's buffers: report, touch nothing
    if (r == 0 && lane == 0) raise_error(err, DSPARK_DEVERR_ROWS_OVERFLOW);
    return;
  }
  if (r >= B) return;  // warp-uniform
  const int w = windows[r];
  const int base = cu[r];
  const int n_rows = cu[r + 1] - base;
  int test_len = (mode == DSPARK_CAP_ACCEPT) ? gamma : w;
  if (test_len > n_rows - 1) test_len = n_rows - 1;
  bool acc = false;
  if (lane < test_len) {
    const int x = draft_tok[r * gamma + lane];
    if (x < 0 || x >= V) {
      raise_error(err, DSPARK_DEVERR_BAD_INPUT);  // an out-of-range draft is rejected
    } else {
      const float pt = ld_p(p_t, (long long)(base + lane) * V + x);
      const float pd = ld_p(p_d, ((long long)r * gamma + lane) * V + x);
      acc = __fmul_rn(uniforms[r * gamma + lane], pd) <= pt;
    }
  }
  const unsigned ok = __ballot_sync(0xffffffffu, acc);
  const unsigned in_range = test_len >= 32 ? 0xffffffffu : ((1u << test_len) - 1u);
  const unsigned rejected = ~ok & in_range;
  const int L = rejected ? __ffs(rejected) - 1 : test_len;
  if (lane == 0) {
    const int commit = L < w ? L : w;
    RowInfo ri;
    ri.commit = commit;
    ri.cap = L;
    ri.sample_row = commit;
    ri.residual = commit < w ? 1 : 0;
    info[r] = ri;
    accept_len[r] = commit;
    cap_len[r] = L;
  }
}

template <class T>
__global__ void __launch_bounds__(kVocabThreads)
    accept_vocab_kernel(const T* __restrict__ p_t, const T* __restrict__ p_d,
                        const float* __restrict__ exp_noise, int V, int n_chunks,
                        const int32_t* __restrict__ cu, int B, int gamma, int max_rows,
                        const RowInfo* __restrict__ info, Partial* __restrict__ part) {
  __shared__ double s_l1[kVocabThreads / 32];
  __shared__ float s_kr[kVocabThreads / 32], s_kt[kVocabThreads / 32];
  __shared__ int s_ir[kVocabThreads / 32], s_it[kVocabThreads / 32];
  const int M = cu[B];
  if (M > max_rows) return;  // reported by the test kernel
  const long long n_items = (long long)M * n_chunks;
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  for (long long item = blockIdx.x; item < n_items; item += gridDim.x) {
    const int row = static_cast<int>(item / n_chunks);
    const int ch = static_cast<int>(item % n_chunks);
    const int r = upper_segment(cu, B, row);
    const int j = row - cu[r];
    const RowInfo ri = info[r];
    const bool do_l1 = j < gamma;
    const bool do_samp = j == ri.sample_row;
    if (!do_l1 && !do_samp) continue;  // block-uniform
    const bool need_d = do_l1 || (do_samp && ri.residual);
    const T* pt_row = p_t + (long long)row * V;
    const T* pd_row = p_d + ((long long)r * gamma + (j < gamma ? j : 0)) * V;
    const float* e_row = exp_noise + (long long)r * V;
    const int v0 = ch * kChunk;
    const int v1 = (v0 + kChunk < V) ? v0 + kChunk : V;
    float l1 = 0.f;
    float kr = -1.f, kt = -1.f;
    int ir = 0x7fffffff, it_ = 0x7fffffff;
    for (int v = v0 + threadIdx.x * 8; v < v1; v += kVocabThreads * 8) {
      float a[8], d[8];
      Vec8<T>::load(pt_row + v, a);
      if (need_d) {
        Vec8<T>::load(pd_row + v, d);
      } else {
#pragma unroll
        for (int q = 0; q < 8; ++q) d[q] = 0.f;
      }
      if (do_l1) {
#pragma unroll
        for (int q = 0; q < 8; ++q) l1 += fabsf(d[q] - a[q]);
      }
      if (do_samp) {
        const float4 e0 = __ldcs(reinterpret_cast<const float4*>(e_row + v));
        const float4 e1 = __ldcs(reinterpret_cast<const float4*>(e_row + v) + 1);
        const float e[8] = {e0.x, e0.y, e0.z, e0.w, e1.x, e1.y, e1.z, e1.w};
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float kq = __fdiv_rn(a[q], e[q]);
          if (kq > kt) { kt = kq; it_ = v + q; }
          if (ri.residual) {
            const float res = fmaxf(__fsub_rn(a[q], d[q]), 0.f);
            const float rq = __fdiv_rn(res, e[q]);
            if (rq > kr) { kr = rq; ir = v + q; }
          }
        }
      }
    }
    // block reduction (fixed tree: deterministic)
    double l1d = static_cast<double>(l1);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      l1d += __shfl_xor_sync(0xffffffffu, l1d, o);
      better(kr, ir, __shfl_xor_sync(0xffffffffu, kr, o), __shfl_xor_sync(0xffffffffu, ir, o));
      better(kt, it_, __shfl_xor_sync(0xffffffffu, kt, o), __shfl_xor_sync(0xffffffffu, it_, o));
    }
    if (lane == 0) {
      s_l1[wid] = l1d;
      s_kr[wid] = kr; s_ir[wid] = ir;
      s_kt[wid] = kt; s_it[wid] = it_;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      Partial pp;
      pp.l1 = 0.0;
      pp.key_res = -1.f; pp.idx_res = 0x7fffffff;
      pp.key_t = -1.f; pp.idx_t = 0x7fffffff;
      for (int q = 0; q < kVocabThreads / 32; ++q) {
        pp.l1 += s_l1[q];
        better(pp.key_res, pp.idx_res, s_kr[q], s_ir[q]);
        better(pp.key_t, pp.idx_t, s_kt[q], s_it[q]);
      }
      part[(long long)row * n_chunks + ch] = pp;
    }
    __syncthreads();
  }
}

__global__ void __launch_bounds__(128)
    accept_final_kernel(const int32_t* __restrict__ cu, int B, int gamma, int max_rows,
                        int n_chunks, const RowInfo* __restrict__ info,
                        const Partial* __restrict__ part, int32_t* __restrict__ out_tok,
                        float* __restrict__ cstar, int32_t* __restrict__ fallback) {
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (r >= B || cu[B] > max_rows) return;
  const int base = cu[r];
  const int n_rows = cu[r + 1] - base;
  const RowInfo ri = info[r];
  for (int j = lane; j < gamma; j += 32) {
    float c = __int_as_float(0x7fc00000);  // NaN: no target row for this position
    if (j < n_rows) {
      double s = 0.0;
      for (int ch = 0; ch < n_chunks; ++ch) s += part[(long long)(base + j) * n_chunks + ch].l1;
      c = __double2float_rn(1.0 - 0.5 * s);
    }
    cstar[r * gamma + j] = c;
  }
  if (lane == 0) {
    const long long prow = (long long)(base + ri.sample_row) * n_chunks;
    float kr = -1.f, kt = -1.f;
    int ir = 0x7fffffff, it_ = 0x7fffffff;
    for (int ch = 0; ch < n_chunks; ++ch) {
      const Partial p = part[prow + ch];
      better(kr, ir, p.key_res, p.idx_res);
      better(kt, it_, p.key_t, p.idx_t);
    }
    int tok = it_, fb = 0;
    if (ri.residual) {
      if (kr > 0.f) tok = ir;
      else fb = 1;
    }
    out_tok[r] = tok;
    if (fallback) fallback[r] = fb;
  }
}

size_t accept_workspace(int B, int max_rows, int V) {
  const int n_chunks = ceil_div(V, kChunk);
  size_t a = ((size_t)B * sizeof(RowInfo) + 255) & ~size_t(255);
  return a + (size_t)max_rows * n_chunks * sizeof(Partial);
}

// Scratch of dspark_accept_noalloc: a fixed array in the library image, one per
// device.  Its address is looked up once per device, with that device current.
static __device__ __align__(256) unsigned char g_accept_scratch[DSPARK_ACCEPT_NOALLOC_SCRATCH_BYTES];

void* accept_fixed_scratch() {
  constexpr int kMaxDevices = 64;
  static std::atomic<void*> addr[kMaxDevices];
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  void* p = addr[dev].load(std::memory_order_acquire);
  if (p == nullptr) {
    if (cudaGetSymbolAddress(&p, g_accept_scratch) != cudaSuccess) return nullptr;
    addr[dev].store(p, std::memory_order_release);
  }
  return p;
}

int launch_accept(const void* p_t, const void* p_d, int pdt, int V, const int32_t* draft_tok,
                  const float* uniforms, const float* exp_noise, const int32_t* windows,
                  const int32_t* cu, int mode, int B, int gamma, int max_rows, int32_t* accept_len,
                  int32_t* cap_len, int32_t* out_tok, float* cstar, int32_t* fallback, void* ws,
                  cudaStream_t stream) {
  const int n_chunks = ceil_div(V, kChunk);
  RowInfo* info = static_cast<RowInfo*>(ws);
  Partial* part = reinterpret_cast<Partial*>(static_cast<uint8_t*>(ws) +
                                             (((size_t)B * sizeof(RowInfo) + 255) & ~size_t(255)));
  unsigned int* err = device_error_word();
  const int sms = num_sms_cached();
  const long long max_items = (long long)max_rows * n_chunks;
  long long grid = (long long)sms * 8;
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  if (pdt == DSPARK_F32) {
    const float* t = static_cast<const float*>(p_t);
    const float* d = static_cast<const float*>(p_d);
    accept_test_kernel<float><<<ceil_div(B * 32, 128), 128, 0, stream>>>(
        t, d, V, draft_tok, uniforms, windows, cu, mode, B, gamma, max_rows, accept_len, cap_len, info,
        err);
    DSPARK_LAUNCH_CHECK();
    accept_vocab_kernel<float><<<(int)grid, kVocabThreads, 0, stream>>>(t, d, exp_noise, V, n_chunks,
                                                                        cu, B, gamma, max_rows, info,
                                                                        part);
  } else {
    const __nv_bfloat16* t = static_cast<const __nv_bfloat16*>(p_t);
    const __nv_bfloat16* d = static_cast<const __nv_bfloat16*>(p_d);
    accept_test_kernel<__nv_bfloat16><<<ceil_div(B * 32, 128), 128, 0, stream>>>(
        t, d, V, draft_tok, uniforms, windows, cu, mode, B, gamma, max_rows, accept_len, cap_len, info,
        err);
    DSPARK_LAUNCH_CHECK();
    accept_vocab_kernel<__nv_bfloat16><<<(int)grid, kVocabThreads, 0, stream>>>(
        t, d, exp_noise, V, n_chunks, cu, B, gamma, max_rows, info, part);
  }
  DSPARK_LAUNCH_CHECK();
  accept_final_kernel<<<ceil_div(B * 32, 128), 128, 0, stream>>>(cu, B, gamma, max_rows, n_chunks,
                                                                 info, part, out_tok, cstar, fallback);
  DSPARK_LAUNCH_CHECK();
  return DSPARK_OK;
}

}  // namespace dspark
