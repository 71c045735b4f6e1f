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
//   accept_vocab_kernel  persistent, one CTA per SM over (packed row, vocab chunk)
//                        items: bulk copies stream p_t, p_d and the noise row through
//                        a shared-memory ring; one pass computes the partial L1
//                        distance for c*, and on the sampled row the partial
//                        exponential-race argmax (w_v / e_v, lowest index on ties)
//                        for both the residual max(0, p_t - p_d) and p_t itself.
//   accept_final_kernel  one block per request: fixed-order fp64 sums of the chunk
//                        partials (c*, a warp per row) and the argmax over the
//                        chunk partials (token), with the p_t race behind a
//                        residual that has no positive entry.
//
// Race rule (the Gumbel-max draw as an exponential race): key w_v / e_v in fp32,
// lowest index on ties; an entry with w_v = 0 has log w_v = -inf and never wins.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dspark {

namespace {

constexpr int kChunk = 8192;  // vocabulary entries per work item (32 per thread)

struct RowInfo {        // per request
  int commit, cap, sample_row, residual;
};

// row_desc flags: low 16 bits = position j of the row in its request's segment
constexpr int kRowL1 = 1 << 16;        // c* needs this row's L1 distance
constexpr int kRowSample = 1 << 17;    // the token is drawn on this row
constexpr int kRowResidual = 1 << 18;  // ... from max(0, p_t - p_d) (a correction)

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

// Race key of an entry whose weight is not positive: -inf, below every live key.
// Bests start at kDead with index kNoIndex, and entries are taken on a strict
// comparison, so a dead entry is never taken and a row with no positive weight
// ends with index kNoIndex (reading A11: such an entry never wins).
constexpr float kDead = -__builtin_huge_valf();
constexpr int kNoIndex = 0x7fffffff;

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
                       int2* __restrict__ row_desc, int* __restrict__ claim,
                       unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (blockIdx.x == 0 && threadIdx.x == 0) *claim = 0;  // the vocabulary pass's item counter
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
  // what the vocabulary pass does on each of this request's packed rows
  const int commit = __shfl_sync(0xffffffffu, L < w ? L : w, 0);
  for (int j = lane; j < n_rows; j += 32) {
    int flags = j;
    if (j < gamma) flags |= kRowL1;
    if (j == commit) flags |= kRowSample | (commit < w ? kRowResidual : 0);
    row_desc[base + j] = make_int2(r, flags);
  }
}

// ---------------------------------------------------------------- vocabulary pass
// Persistent, one CTA per SM over a contiguous range of (packed row, 8192-entry
// chunk) items.  One thread streams the rows the method needs (p_t always, p_d for
// c* rows and corrections, the noise row on the sampled row) with bulk copies into a
// shared-memory ring of whole items (noise into a ring of its own), running ahead
// across items; sixteen consumer warps reduce each slot from shared memory; a reducer
// warp combines the sixteen warps' results of an item into its partial.  A slot holds
// the item's 8192 entries of each probability row: 32 KB copies per row in fp32 (a
// single issuing thread streams 32 KB copies about 15% faster than 16 KB ones), 16 KB
// in bf16.  fp32 takes three slots and one noise slot, bf16 five and two: 224 KB.
template <int ES> struct RingGeom;
template <> struct RingGeom<4> { static constexpr int kStages = 3, kNoise = 1; };
template <> struct RingGeom<2> { static constexpr int kStages = 5, kNoise = 2; };
constexpr int kMaxVStages = 5;
constexpr int kRingBytes = 224 * 1024;        // main ring, then the noise ring
constexpr int kConsumerWarps = 16;
constexpr int kProducerWarp = 16, kReducerWarp = 17;
constexpr int kVocabCtaThreads = 18 * 32;
constexpr uint64_t kDrainWaitNs = 2000000000ull;  // draining own copies: always 2 s

struct WarpPart {
  double l1;
  float kr, kt;
  int ir, it;
  int pad[2];
};

struct VocabSmem {
  uint8_t ring[kRingBytes];  // RingGeom<ES>::kStages slots of p_t | p_d, then noise slots
  WarpPart red[2][kConsumerWarps];
  int4 meta[kMaxVStages];  // item, sub-chunk | sub-chunks << 8, request, row flags
  uint64_t full[kMaxVStages], empty[kMaxVStages], nempty[4], red_full[2], red_free[2];
  uint64_t never;  // a barrier nothing arrives at (the wait probe)
  int abort_flag;
};

// Bounded wait: false once this CTA aborts (another role's wait ran out, or this
// one ran past wait_ns, which then raises DSPARK_DEVERR_WAIT_TIMEOUT).
__device__ __forceinline__ bool vwait(uint32_t bar, uint32_t parity, volatile int* abort_flag,
                                      unsigned int* err, uint64_t wait_ns) {
  if (ptx::mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = ptx::globaltimer_ns();
  uint32_t n = 0;
  while (!ptx::mbar_try_wait(bar, parity)) {
    if ((++n & 31u) == 0) {
      if (*abort_flag) return false;
      if (ptx::globaltimer_ns() - t0 > wait_ns) {
        *abort_flag = 1;
        raise_error(err, DSPARK_DEVERR_WAIT_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

// Work of row `row` of the packed batch, decoded from the test kernel's descriptor.
struct RowWork {
  int r, j;
  bool l1, samp, residual, need_d;
};
__device__ __forceinline__ RowWork decode_row(int2 d) {
  RowWork w;
  w.r = d.x;
  w.j = d.y & 0xffff;
  w.l1 = (d.y & kRowL1) != 0;
  w.samp = (d.y & kRowSample) != 0;
  w.residual = (d.y & kRowResidual) != 0;
  w.need_d = w.l1 || w.residual;
  return w;
}

// x[q] for a run-time q without dynamic indexing (keeps x in registers).
__device__ __forceinline__ float pick8(const float (&x)[8], int q) {
  float v = x[0];
#pragma unroll
  for (int i = 1; i < 8; ++i) v = q == i ? x[i] : v;
  return v;
}

// Approximate reciprocal (hardware, relative error well below 2^-20 for normal e).
__device__ __forceinline__ float approx_rcp(float x) {
  float y;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
// Keys are >= 0.  The approximate quotient a * rcp.approx(e) is within 2^-21 of
// the exact one (relative).  Once some entry's approximate key is K, the final
// maximum is at least K (1 - 2^-21); an entry whose approximate key is at or
// below K (1 - 2^-15) has an exact key below K (1 - 2^-16), whose rounding is
// strictly below the final maximum: it can neither win nor tie.
constexpr float kFilter = 1.0f - 1.0f / 32768.0f;
constexpr float kHuge = 3.0e38f;  // marks an entry that must take the exact path

template <class T>
__device__ __forceinline__ void smem_vec8(const uint8_t* p, float (&x)[8]);
template <>
__device__ __forceinline__ void smem_vec8<float>(const uint8_t* p, float (&x)[8]) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 16);
  x[0] = a.x; x[1] = a.y; x[2] = a.z; x[3] = a.w;
  x[4] = b.x; x[5] = b.y; x[6] = b.z; x[7] = b.w;
}
template <>
__device__ __forceinline__ void smem_vec8<__nv_bfloat16>(const uint8_t* p, float (&x)[8]) {
  const uint4 u = *reinterpret_cast<const uint4*>(p);
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    x[2 * i] = __uint_as_float(w[i] << 16);
    x[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <class T>
__global__ void __launch_bounds__(kVocabCtaThreads, 1)
    accept_vocab_kernel(const T* __restrict__ p_t, const T* __restrict__ p_d,
                        const float* __restrict__ exp_noise, int V, int n_chunks,
                        const int32_t* __restrict__ cu, int B, int gamma, int max_rows,
                        const int2* __restrict__ row_desc, Partial* __restrict__ part,
                        int* __restrict__ claim, unsigned int* __restrict__ err,
                        uint64_t wait_ns, int probe) {
  extern __shared__ __align__(128) uint8_t vsmem_raw[];
  VocabSmem& S = *reinterpret_cast<VocabSmem*>(vsmem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  pdl_release();
  pdl_wait();  // row descriptors come from the test kernel
  const int M = cu[B];
  if (M > max_rows) return;  // reported by the test kernel (block-uniform)
  // items round-robin over the CTAs: the chunks of one row (and so the costlier
  // sampled rows) spread over many SMs
  const long long n_items = (long long)M * n_chunks;
  volatile int* abort_flag = &S.abort_flag;
  constexpr int ES = static_cast<int>(sizeof(T));
  constexpr int kSubT = kChunk;                         // entries per slot: one item
  constexpr int kRowB = kSubT * ES;                     // one probability row in a slot
  constexpr int kVStages = RingGeom<ES>::kStages;
  constexpr int kNStages = RingGeom<ES>::kNoise;         // noise slots
  constexpr int kNoiseOff = kVStages * 2 * kRowB;
  static_assert(kNoiseOff + kNStages * kSubT * 4 <= kRingBytes && kVStages <= kMaxVStages,
                "ring");
  if (threadIdx.x == 0) {
    S.abort_flag = 0;
    for (int s = 0; s < kVStages; ++s) {
      ptx::mbar_init(ptx::smem_addr(&S.full[s]), 1);
      ptx::mbar_init(ptx::smem_addr(&S.empty[s]), kConsumerWarps);
    }
    for (int s = 0; s < 4; ++s) ptx::mbar_init(ptx::smem_addr(&S.nempty[s]), kConsumerWarps);
    for (int p = 0; p < 2; ++p) {
      ptx::mbar_init(ptx::smem_addr(&S.red_full[p]), kConsumerWarps);
      ptx::mbar_init(ptx::smem_addr(&S.red_free[p]), 1);
    }
    ptx::mbar_init(ptx::smem_addr(&S.never), 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  auto n_sub_of = [&](int ch) {
    const int len = min(kChunk, V - ch * kChunk);
    return (len + kSubT - 1) / kSubT;
  };

  if (warp == kProducerWarp) {
    // Items are claimed one at a time from a counter shared by all CTAs (the costlier
    // sampled rows then balance out); each stage carries its item in meta[].
    if (lane == 0) {
      int g = 0, gn = 0;  // main-ring and noise-ring sub-chunks issued
      bool ok = true, marker = false;
      // the wait probe (a failure-detection test): a wait that must run out
      if (probe) ok = vwait(ptx::smem_addr(&S.never), 0, abort_flag, err, wait_ns);
      long long item = ok ? atomicAdd(claim, 1) : n_items;
      while (ok) {
        long long next = n_items;
        RowWork w{};
        bool work = false;
        int2 desc = make_int2(0, 0);
        if (item < n_items) {
          next = atomicAdd(claim, 1);  // taken ahead: its latency hides behind this item
          desc = row_desc[item / n_chunks];
          w = decode_row(desc);
          work = w.l1 || w.samp;
          if (w.r < 0 || w.r >= B || w.j < 0 || w.j > gamma) {
            // not a descriptor the test kernel writes: touch no row, report
            raise_error(err, DSPARK_DEVERR_BAD_INPUT);
            work = false;
          }
        }
        const int s = g % kVStages;
        if (item < n_items && !work) {  // nothing to do on this row: next claim
          item = next;
          continue;
        }
        const int row = static_cast<int>(item / n_chunks), ch = static_cast<int>(item % n_chunks);
        const int ns = item < n_items ? n_sub_of(ch) : 1;
        for (int sb = 0; sb < ns; ++sb, ++g) {
          const int st = g % kVStages;
          if (g >= kVStages &&
              !vwait(ptx::smem_addr(&S.empty[st]), ((g / kVStages) - 1) & 1, abort_flag, err, wait_ns)) {
            ok = false;
            break;
          }
          const uint32_t full = ptx::smem_addr(&S.full[st]);
          if (item >= n_items) {  // end marker: a stage without data
            S.meta[st] = make_int4(-1, 0, 0, 0);
            ptx::mbar_arrive(full);
            marker = true;
            ok = false;  // done
            break;
          }
          const int sn = gn % kNStages;
          if (w.samp && gn >= kNStages &&
              !vwait(ptx::smem_addr(&S.nempty[sn]), ((gn / kNStages) - 1) & 1, abort_flag, err, wait_ns)) {
            ok = false;
            break;
          }
          const T* pt_row = p_t + (long long)row * V;
          const T* pd_row = p_d + ((long long)w.r * gamma + (w.j < gamma ? w.j : 0)) * V;
          const float* e_row = exp_noise + (long long)w.r * V;
          const int v0 = ch * kChunk + sb * kSubT;
          const uint32_t len = static_cast<uint32_t>(min(kSubT, V - v0));
          const uint32_t base = ptx::smem_addr(S.ring + st * 2 * kRowB);
          const uint32_t bytes = len * ES * (w.need_d ? 2u : 1u) + (w.samp ? len * 4u : 0u);
          S.meta[st] = make_int4(static_cast<int>(item), sb | (ns << 8), w.r, desc.y);
          ptx::mbar_expect_tx(full, bytes);
          ptx::bulk_load_g2s(base, pt_row + v0, len * ES, full);
          if (w.need_d) ptx::bulk_load_g2s(base + kRowB, pd_row + v0, len * ES, full);
          if (w.samp) {
            ptx::bulk_load_g2s(ptx::smem_addr(S.ring + kNoiseOff + sn * kSubT * 4), e_row + v0,
                               len * 4, full);
            ++gn;
          }
          ptx::mbar_arrive(full);
        }
        (void)s;
        item = next;
      }
      // Never leave copies in flight: wait for the last data phase of every ring slot
      // (on the fixed drain limit, also after an abort).  The slot the end marker
      // reused held a stage the consumers had already released (the empty wait
      // before the marker), and its barrier has moved past that phase: skipped.
      const int first = g - kVStages > 0 ? g - kVStages : 0;
      for (int gg = first; gg < g; ++gg) {
        if (marker && gg % kVStages == g % kVStages) continue;
        const uint32_t bar = ptx::smem_addr(&S.full[gg % kVStages]);
        const uint32_t par = (gg / kVStages) & 1;
        const uint64_t t0 = ptx::globaltimer_ns();
        while (!ptx::mbar_try_wait(bar, par)) {
          if (ptx::globaltimer_ns() - t0 > kDrainWaitNs) {
            raise_error(err, DSPARK_DEVERR_WAIT_TIMEOUT);
            break;
          }
        }
      }
    }
  } else if (warp == kReducerWarp) {
    // the consumer warps' results of an item -> its partial (fixed order: deterministic)
    int n_it = 0;
    bool ok = true;
    while (ok) {
      const int p = n_it & 1;
      ok = vwait(ptx::smem_addr(&S.red_full[p]), (n_it >> 1) & 1, abort_flag, err, wait_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int item = S.red[p][0].pad[0];
      if (item < 0) break;  // the consumers are done
      if (lane == 0) {
        Partial pp;
        pp.l1 = 0.0;
        pp.key_res = kDead; pp.idx_res = kNoIndex;
        pp.key_t = kDead; pp.idx_t = kNoIndex;
        for (int q = 0; q < kConsumerWarps; ++q) {
          const WarpPart& wp = S.red[p][q];
          pp.l1 += wp.l1;
          better(pp.key_res, pp.idx_res, wp.kr, wp.ir);
          better(pp.key_t, pp.idx_t, wp.kt, wp.it);
        }
        part[item] = pp;  // item = row * n_chunks + chunk
        ptx::mbar_arrive(ptx::smem_addr(&S.red_free[p]));
      }
      __syncwarp();
      ++n_it;
    }
  } else {
    // consumers: thread t owns entries 8t..8t+7 of each sub-chunk; the stages' meta[]
    // gives their items
    int g = 0, gn = 0, n_it = 0;
    bool ok = true;
    float l1 = 0.f, kbest = kDead, thr = -1.f;
    int ibest = kNoIndex;
    while (ok) {
      const int s = g % kVStages;
      ok = vwait(ptx::smem_addr(&S.full[s]), (g / kVStages) & 1, abort_flag, err, wait_ns);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      const int4 m = S.meta[s];
      if (m.x < 0) {  // end: tell the reducer
        const int p = n_it & 1;
        if (n_it >= 2) {
          ok = vwait(ptx::smem_addr(&S.red_free[p]), ((n_it >> 1) - 1) & 1, abort_flag, err, wait_ns);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        if (lane == 0) {
          S.red[p][warp].pad[0] = -1;
          ptx::mbar_arrive(ptx::smem_addr(&S.red_full[p]));
        }
        break;
      }
      const int sb = m.y & 0xff, ns = m.y >> 8;
      RowWork w;
      w.r = m.z;
      w.j = m.w & 0xffff;
      w.l1 = (m.w & kRowL1) != 0;
      w.samp = (m.w & kRowSample) != 0;
      w.residual = (m.w & kRowResidual) != 0;
      w.need_d = w.l1 || w.residual;
      const int ch = m.x % n_chunks;
      if (sb == 0) {
        l1 = 0.f;
        kbest = kDead;
        ibest = kNoIndex;
        thr = -1.f;
      }
      {
        const int v0 = ch * kChunk + sb * kSubT;
        const int len = min(kSubT, V - v0);
        const uint8_t* st = S.ring + s * 2 * kRowB;
        const int sn = gn % kNStages;
        const uint8_t* nz = S.ring + kNoiseOff + sn * kSubT * 4;
#pragma unroll
        for (int k = 0; k < kSubT / (kConsumerWarps * 32 * 8); ++k) {
          const int e = (k * kConsumerWarps * 32 + threadIdx.x) * 8;
          const bool valid = e < len;
          float a[8], d[8], en[8], ka[8];
#pragma unroll
          for (int q = 0; q < 8; ++q) { a[q] = 0.f; d[q] = 0.f; en[q] = 1.f; ka[q] = kDead; }
          if (valid) {
            smem_vec8<T>(st + e * ES, a);
            if (w.need_d) smem_vec8<T>(st + kRowB + e * ES, d);
            if (w.l1) {
#pragma unroll
              for (int q = 0; q < 8; ++q) l1 += fabsf(d[q] - a[q]);
            }
            if (w.samp) {
              // race weights: the residual max(0, p_t - p_d) for a correction, p_t
              // for a bonus token (the p_t race behind an all-zero residual is
              // left to the final kernel)
              smem_vec8<float>(nz + e * 4, en);
#pragma unroll
              for (int q = 0; q < 8; ++q) {
                if (w.residual) a[q] = fmaxf(__fsub_rn(a[q], d[q]), 0.f);
                const float inv = approx_rcp(en[q]);
                // a weight that is not positive never wins (log 0 = -inf in the
                // Gumbel form); e beyond the reciprocal's range forces the exact path
                ka[q] = !(a[q] > 0.f) ? kDead : (inv == 0.f ? kHuge : a[q] * inv);
              }
            }
          }
          if (w.samp) {  // warp-uniform
            // Raise the filter to just below the warp's largest approximate key:
            // the final maximum is at least that key's exact value.
            float mt = ka[0];
#pragma unroll
            for (int q = 1; q < 8; ++q) mt = fmaxf(mt, ka[q]);
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) mt = fmaxf(mt, __shfl_xor_sync(0xffffffffu, mt, o));
            // (a zero maximum leaves the filter: live entries whose key rounds to 0
            // still reach the exact path; dead entries never pass it)
            if (mt < kHuge && mt > 0.f) thr = fmaxf(thr, mt * kFilter);
            // A lane visits its entries in increasing index order and keeps the first
            // strict maximum of its rounded keys fl(w / e); an entry at or below the
            // filter has fl(w / e) strictly below the final maximum, so only the few
            // others take the exact division.
            unsigned cand = 0;
#pragma unroll
            for (int q = 0; q < 8; ++q)
              if (valid && ka[q] > thr) cand |= 1u << q;
#pragma unroll 1
            for (; cand; cand &= cand - 1) {
              const int q = __ffs(cand) - 1;
              const float kq = __fdiv_rn(pick8(a, q), pick8(en, q));
              if (kq > kbest) { kbest = kq; ibest = v0 + e + q; }
            }
          }
        }
        __syncwarp();
        if (lane == 0) {
          ptx::mbar_arrive(ptx::smem_addr(&S.empty[s]));
          if (w.samp) ptx::mbar_arrive(ptx::smem_addr(&S.nempty[sn]));
        }
        if (w.samp) ++gn;
      }
      ++g;
      if (sb != ns - 1) continue;
      // item done: warp results to the reducer
      float kr = kDead, kt = kDead;
      int ir = kNoIndex, it_ = kNoIndex;
      if (w.residual) { kr = kbest; ir = ibest; } else { kt = kbest; it_ = ibest; }
      double l1d = static_cast<double>(l1);
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        l1d += __shfl_xor_sync(0xffffffffu, l1d, o);
        better(kr, ir, __shfl_xor_sync(0xffffffffu, kr, o), __shfl_xor_sync(0xffffffffu, ir, o));
        better(kt, it_, __shfl_xor_sync(0xffffffffu, kt, o), __shfl_xor_sync(0xffffffffu, it_, o));
      }
      const int p = n_it & 1;
      // slot p was last read by the reducer for item n_it - 2
      if (n_it >= 2) {
        ok = vwait(ptx::smem_addr(&S.red_free[p]), ((n_it >> 1) - 1) & 1, abort_flag, err, wait_ns);
        ok = __all_sync(0xffffffffu, ok);
        if (!ok) break;
      }
      if (lane == 0) {
        WarpPart& wp = S.red[p][warp];
        wp.l1 = l1d;
        wp.kr = kr; wp.ir = ir;
        wp.kt = kt; wp.it = it_;
        wp.pad[0] = m.x;
        ptx::mbar_arrive(ptx::smem_addr(&S.red_full[p]));
      }
      __syncwarp();
      ++n_it;
    }
  }
  __syncthreads();
}

// One block per request: warp w sums the chunk partials of c* rows w, w + 8, ...
// (lanes over chunks, a fixed shuffle tree: deterministic), warp 0 also takes the
// token from the sampled row's partials.
template <class T>
__global__ void __launch_bounds__(256)
    accept_final_kernel(const T* __restrict__ p_t, const float* __restrict__ exp_noise, int V,
                        const int32_t* __restrict__ cu, int B, int gamma, int max_rows,
                        int n_chunks, const RowInfo* __restrict__ info,
                        const Partial* __restrict__ part, int32_t* __restrict__ out_tok,
                        float* __restrict__ cstar, int32_t* __restrict__ fallback) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  const int r = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (r >= B || cu[B] > max_rows) return;  // block-uniform
  const int base = cu[r];
  const int n_rows = cu[r + 1] - base;
  for (int j = warp; j < gamma; j += 8) {
    float c = __int_as_float(0x7fc00000);  // NaN: no target row for this position
    if (j < n_rows) {
      double s = 0.0;
      for (int ch = lane; ch < n_chunks; ch += 32) s += part[(long long)(base + j) * n_chunks + ch].l1;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      c = __double2float_rn(1.0 - 0.5 * s);
    }
    if (lane == 0) cstar[r * gamma + j] = c;
  }
  if (warp != 0) return;
  const RowInfo ri = info[r];
  // token: the sampled row's race maximum over the chunk partials (max, then lowest
  // index: order-independent)
  const long long prow = (long long)(base + ri.sample_row) * n_chunks;
  float k = kDead;
  int idx = kNoIndex;
  for (int ch = lane; ch < n_chunks; ch += 32) {
    const Partial p = part[prow + ch];
    if (ri.residual) better(k, idx, p.key_res, p.idx_res);
    else better(k, idx, p.key_t, p.idx_t);
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1)
    better(k, idx, __shfl_xor_sync(0xffffffffu, k, o), __shfl_xor_sync(0xffffffffu, idx, o));
  int fb = 0;
  if (ri.residual && idx == kNoIndex) {
    // A residual with no positive entry (reachable only through rounding): the
    // token is drawn from p_t on the same row with the same noise; the vocabulary
    // pass raced only the residual there, so this warp races p_t.
    fb = 1;
    k = kDead;
    const long long trow = (long long)(base + ri.sample_row) * V;
    for (int v = lane; v < V; v += 32) {
      const float p = ld_p(p_t, trow + v);
      const float kq = p > 0.f ? __fdiv_rn(p, exp_noise[(long long)r * V + v]) : kDead;
      if (kq > k) { k = kq; idx = v; }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1)
      better(k, idx, __shfl_xor_sync(0xffffffffu, k, o), __shfl_xor_sync(0xffffffffu, idx, o));
  }
  if (lane == 0) {
    // no positive weight on the raced row at all: the lowest index (undefined draw)
    out_tok[r] = idx == kNoIndex ? 0 : idx;
    if (fallback) fallback[r] = fb;
  }
}

// The acceptance pass's wait limit per device (0: the default 2 s), and the wait
// probe (a failure-detection test: the pass first waits on a barrier nothing
// arrives at).
namespace {
constexpr uint64_t kDefaultWaitNs = 2000000000ull;
std::atomic<unsigned long long> g_accept_wait_ns[kMaxDevices];
std::atomic<int> g_accept_wait_probe[kMaxDevices];
}  // namespace

uint64_t accept_wait_limit_ns() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return kDefaultWaitNs;
  const unsigned long long v = g_accept_wait_ns[dev].load(std::memory_order_relaxed);
  return v ? v : kDefaultWaitNs;
}

int set_accept_wait_limit_ns(unsigned long long ns) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSPARK_ECUDA;
  g_accept_wait_ns[dev].store(ns, std::memory_order_relaxed);
  return DSPARK_OK;
}

int accept_wait_probe() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  return g_accept_wait_probe[dev].load(std::memory_order_relaxed);
}

int set_accept_wait_probe(int on) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return DSPARK_ECUDA;
  g_accept_wait_probe[dev].store(on ? 1 : 0, std::memory_order_relaxed);
  return DSPARK_OK;
}

bool vocab_configure() {
  static PerDevice<bool> done;
  return once_per_device(done, false, [] {
    const int bytes = static_cast<int>(sizeof(VocabSmem));
    return cudaFuncSetAttribute(accept_vocab_kernel<float>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess &&
           cudaFuncSetAttribute(accept_vocab_kernel<__nv_bfloat16>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, bytes) == cudaSuccess;
  });
}

// workspace: RowInfo[B] | claim counter | int2 row_desc[max_rows] | Partial[max_rows][n_chunks]
size_t accept_workspace(int B, int max_rows, int V) {
  const int n_chunks = ceil_div(V, kChunk);
  const size_t a = ((size_t)B * sizeof(RowInfo) + 255) & ~size_t(255);
  const size_t b = ((size_t)max_rows * sizeof(int2) + 255) & ~size_t(255);
  return a + 256 + b + (size_t)max_rows * n_chunks * sizeof(Partial);
}

// Scratch of dspark_accept_noalloc: a fixed array in the library image, one per
// device.  Its address is looked up once per device, with that device current.
static __device__ __align__(256) unsigned char g_accept_scratch[DSPARK_ACCEPT_NOALLOC_SCRATCH_BYTES];

void* accept_fixed_scratch() {
  static PerDevice<void*> addr;
  return once_per_device(addr, static_cast<void*>(nullptr), [] {
    void* p = nullptr;
    return cudaGetSymbolAddress(&p, g_accept_scratch) == cudaSuccess ? p : nullptr;
  });
}

// Block-accept estimate, thread per request: in compact mode a request whose whole
// window was accepted is tested at position w + 1 on its bonus row (the target row of
// that position, packed row cu[r] + w) against the drafter's row w + 1, as a
// full-block verification would test it; the cap is then w (rejected) or lies in
// [w + 1, gamma].  Otherwise the cap is the accepted length (compact) or cap_len.
template <class T>
__global__ void __launch_bounds__(128)
    accept_estimate_kernel(const T* __restrict__ p_t, const T* __restrict__ p_d, int V,
                           const int32_t* __restrict__ draft_tok, const float* __restrict__ uniforms,
                           const int32_t* __restrict__ windows, const int32_t* __restrict__ cu,
                           const int32_t* __restrict__ accept_len, const int32_t* __restrict__ cap_len,
                           int mode, int B, int gamma, int max_rows, int32_t* __restrict__ cap_lo,
                           int32_t* __restrict__ cap_hi, unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // the acceptance's outputs
  const int r = blockIdx.x * blockDim.x + threadIdx.x;
  if (r >= B) return;
  if (mode != DSPARK_COMPACT) {
    cap_lo[r] = cap_len[r];
    cap_hi[r] = cap_len[r];
    return;
  }
  const int w = windows[r], L = accept_len[r];
  int lo = L, hi = L;
  if (L >= w && w < gamma) {
    const int row = cu[r] + w;
    const int x = w >= 0 ? draft_tok[r * gamma + w] : -1;
    if (w < 0 || row >= cu[r + 1] || row >= max_rows || x < 0 || x >= V) {
      raise_error(err, DSPARK_DEVERR_BAD_INPUT);
    } else {
      const float pt = ld_p(p_t, (long long)row * V + x);
      const float pd = ld_p(p_d, ((long long)r * gamma + w) * V + x);
      if (__fmul_rn(uniforms[r * gamma + w], pd) <= pt) {
        lo = w + 1;
        hi = gamma;
      } else {
        lo = hi = w;
      }
    }
  }
  cap_lo[r] = lo;
  cap_hi[r] = hi;
}

int launch_accept_estimate(const void* p_t, const void* p_d, int pdt, int V,
                           const int32_t* draft_tok, const float* uniforms, const int32_t* windows,
                           const int32_t* cu, const int32_t* accept_len, const int32_t* cap_len,
                           int mode, int B, int gamma, int max_rows, int32_t* cap_lo,
                           int32_t* cap_hi, cudaStream_t stream) {
  unsigned int* err = device_error_word();
  const dim3 grid(ceil_div(B, 128)), block(128);
  cudaError_t e;
  if (pdt == DSPARK_F32)
    e = launch_pdl(accept_estimate_kernel<float>, grid, block, 0, stream,
                   static_cast<const float*>(p_t), static_cast<const float*>(p_d), V, draft_tok,
                   uniforms, windows, cu, accept_len, cap_len, mode, B, gamma, max_rows, cap_lo,
                   cap_hi, err);
  else
    e = launch_pdl(accept_estimate_kernel<__nv_bfloat16>, grid, block, 0, stream,
                   static_cast<const __nv_bfloat16*>(p_t), static_cast<const __nv_bfloat16*>(p_d),
                   V, draft_tok, uniforms, windows, cu, accept_len, cap_len, mode, B, gamma,
                   max_rows, cap_lo, cap_hi, err);
  return e == cudaSuccess ? DSPARK_OK : DSPARK_ECUDA;
}

int launch_accept(const void* p_t, const void* p_d, int pdt, int V, const int32_t* draft_tok,
                  const float* uniforms, const float* exp_noise, const int32_t* windows,
                  const int32_t* cu, int mode, int B, int gamma, int max_rows, int32_t* accept_len,
                  int32_t* cap_len, int32_t* out_tok, float* cstar, int32_t* fallback, void* ws,
                  cudaStream_t stream) {
  const int n_chunks = ceil_div(V, kChunk);
  RowInfo* info = static_cast<RowInfo*>(ws);
  const size_t off_claim = ((size_t)B * sizeof(RowInfo) + 255) & ~size_t(255);
  int* claim = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + off_claim);
  const size_t off_desc = off_claim + 256;
  int2* row_desc = reinterpret_cast<int2*>(static_cast<uint8_t*>(ws) + off_desc);
  Partial* part = reinterpret_cast<Partial*>(
      static_cast<uint8_t*>(ws) + off_desc + (((size_t)max_rows * sizeof(int2) + 255) & ~size_t(255)));
  unsigned int* err = device_error_word();
  const int sms = num_sms_cached();
  const long long max_items = (long long)max_rows * n_chunks;
  long long grid = sms;  // persistent, one CTA per SM
  if (grid > max_items) grid = max_items;
  if (grid < 1) grid = 1;
  if (!vocab_configure()) return DSPARK_ECUDA;
  const uint64_t wait_ns = accept_wait_limit_ns();
  const int probe = accept_wait_probe();
  if (pdt == DSPARK_F32) {
    const float* t = static_cast<const float*>(p_t);
    const float* d = static_cast<const float*>(p_d);
    if (launch_pdl(accept_test_kernel<float>, dim3(ceil_div(B * 32, 128)), dim3(128), 0, stream, t,
                   d, V, draft_tok, uniforms, windows, cu, mode, B, gamma, max_rows, accept_len,
                   cap_len, info, row_desc, claim, err) != cudaSuccess)
      return DSPARK_ECUDA;
    if (launch_pdl(accept_vocab_kernel<float>, dim3((int)grid), dim3(kVocabCtaThreads),
                   sizeof(VocabSmem), stream, t, d, exp_noise, V, n_chunks, cu, B, gamma, max_rows,
                   row_desc, part, claim, err, wait_ns, probe) != cudaSuccess)
      return DSPARK_ECUDA;
  } else {
    const __nv_bfloat16* t = static_cast<const __nv_bfloat16*>(p_t);
    const __nv_bfloat16* d = static_cast<const __nv_bfloat16*>(p_d);
    if (launch_pdl(accept_test_kernel<__nv_bfloat16>, dim3(ceil_div(B * 32, 128)), dim3(128), 0,
                   stream, t, d, V, draft_tok, uniforms, windows, cu, mode, B, gamma, max_rows,
                   accept_len, cap_len, info, row_desc, claim, err) != cudaSuccess)
      return DSPARK_ECUDA;
    if (launch_pdl(accept_vocab_kernel<__nv_bfloat16>, dim3((int)grid), dim3(kVocabCtaThreads),
                   sizeof(VocabSmem), stream, t, d, exp_noise, V, n_chunks, cu, B, gamma, max_rows,
                   row_desc, part, claim, err, wait_ns, probe) != cudaSuccess)
      return DSPARK_ECUDA;
  }
  cudaError_t e;
  if (pdt == DSPARK_F32)
    e = launch_pdl(accept_final_kernel<float>, dim3(B), dim3(256), 0, stream,
                   static_cast<const float*>(p_t), exp_noise, V, cu, B, gamma, max_rows, n_chunks,
                   info, part, out_tok, cstar, fallback);
  else
    e = launch_pdl(accept_final_kernel<__nv_bfloat16>, dim3(B), dim3(256), 0, stream,
                   static_cast<const __nv_bfloat16*>(p_t), exp_noise, V, cu, B, gamma, max_rows,
                   n_chunks, info, part, out_tok, cstar, fallback);
  if (e != cudaSuccess) return DSPARK_ECUDA;
  return DSPARK_OK;
}

}  // namespace dspark
