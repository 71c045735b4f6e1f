// Draft-side sampling with a Markov head: one persistent kernel per draft block.
//
// What it computes ("DSpark：投机解码与生产级 Serving 学习笔记", section 05 "Core
// Innovation A", 5.1-5.3: the parallel backbone gives base logits U_1..U_gamma for the
// whole block and a sequential head adds a transition bias of the previous token,
// B(x_{k-1}, v) ~ (W1 W2)[x_{k-1}, v] with rank 256; "DFlash 到 DSpark in SGLang",
// section "Zero-overhead scheduling 与 kernel": the drafter's sampling path folded
// into fused kernels).  For k = 1..gamma and every request r at once:
//     logit  = U[r, k] + W1[x_{k-1}] . W2                (x_0 = the anchor token)
//     p_d[r, k] = softmax(logit)
//     x_k = argmax_v p_d[r, k, v] / e[r, k, v]            (exponential race, lowest index on ties)
// The race needs no normalisation (p/e and exp(logit)/e order the vocabulary alike): each
// thread keeps its best as the fraction 2^(x_best - m) / e_best against its running
// maximum m, compared by cross-multiplication; p_d itself is written normalised.
//
// Layout of the work: the vocabulary is cut into 128-entry tiles, each CTA (one per SM,
// a cooperative launch) owns the tiles t = blockIdx.x + i * gridDim.x for the whole
// block, and one tcgen05 product per tile gives the bias of all requests at once:
//     D [128 vocab x N requests] = W2 tile^T [128 x 256] . H^T [256 x N]
// with W2's tile (MN-major) streamed by TMA and H = the W1 rows of the previous tokens
// (K-major) gathered into shared memory.  D stays in TMEM (two positions' worth), so
// the logits are read from HBM as U once and p is written once.
//
// Roles in each CTA: a W2 producer (TMA), a U / e producer (TMA, boxes of npad requests
// x 128 vocabulary entries; they depend on no token, so they stream ahead), the MMA
// issuer, a sequencer warp and sixteen epilogue warps (thread = vocabulary entry, eight
// request columns).
// Per position k:
//   epilogue  A(k): logit = D + U per tile (stored back into TMEM in the log2 domain), a
//             running (max, sum) per request and the race, then the CTA's (max, sum) and
//             race winner per request published (a partial array, and an atomic maximum
//             on a packed key/index word per request), and the grid barrier's arrival;
//             then C(k-1): (M, S) of the previous position from every CTA's partials in
//             one fixed order (every CTA normalises with the same numbers) and
//             p = 2^(logit - M - log2 S) written out
//   sequencer waits for the barrier, reads the tokens x_k from the words, copies their
//             W1 rows (one bulk copy per request) and lays them out as H for position
//             k+1, which starts its products: the next position's chain runs while the
//             epilogue normalises the previous one.
// The W2 ring also runs ahead across positions.  W2 is loaded with an evict-last L2
// policy and the streamed U, e and p with evict-first accesses, so W2 stays in L2
// across the block.  Every wait is bounded in time (DSPARK_DEVERR_WAIT_TIMEOUT).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include "attn.h"
#include "common.cuh"
#include "kernels.h"
#include "ptx.cuh"

namespace dspark {
namespace md {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kR = 256;                           // rank of the head (the MMA's K)
constexpr int kMV = 128;                          // vocabulary entries per tile (the MMA's M)
constexpr int kMaxG = 32;                         // requests per launch (the MMA's N <= 32)
constexpr int kMaxTilesPerCta = 16;
constexpr int kKH = kR / 2;                       // K rows per W2 stage
constexpr int kStage = kMV * kKH * 2;             // 32 KB: [2 vocabulary halves][128 K rows][64]
constexpr int kStageHalf = kStage / 2;
constexpr int kStages = 3;                        // W2 ring: one and a half tiles
constexpr int kUStage = 2 * kMaxG * kMV * 4;      // 32 KB: U then e, [rows][128 vocab] fp32
constexpr int kUStages = 3;                       // U / e ring
constexpr int kHBytes = kMaxG * kR * 2;           // 16 KB: [4 K blocks][32 rows][64 K]
constexpr int kEpiWarps = 16;                     // four per TMEM lane quadrant
constexpr int kCols = 8;                          // request columns per epilogue thread
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kSeqWarp = 3;                       // warp 0 W2, 1 MMA, 2 U / e, 3 sequencer
constexpr int kEpiWarp0 = 4;                      // 4..11 epilogue
constexpr int kThreads = kEpiWarp0 * 32 + kEpiThreads;
constexpr int OFF_RING = 0;
constexpr int OFF_URING = OFF_RING + kStages * kStage;
constexpr int OFF_H = OFF_URING + kUStages * kUStage;
// the W1 rows of the next tokens as copied (row r at r * 512 bytes), before the
// sequencer lays them out as H; the epilogue's reduction scratch shares it (float2
// st[4][32], float key[4][32], int idx[4][32]): the scratch is read before the CTA
// arrives at a position's barrier and the rows are copied after that barrier
constexpr int OFF_STG = OFF_H + kHBytes;
constexpr int OFF_RED = OFF_STG;
constexpr int OFF_BAR = OFF_STG + kHBytes;
// full[3], empty[3], u_full[3], u_empty[3], h_full, start_done, last_done, stg_full,
// acc_full[16], tfree[16]
constexpr int N_BARS = 2 * kStages + 2 * kUStages + 4 + 2 * kMaxTilesPerCta;
constexpr int OFF_COL = OFF_BAR + 384;            // float (M + log2 S)[32]
constexpr int OFF_MISC = OFF_COL + 256;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
static_assert(N_BARS * 8 <= 384, "barrier area");
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
constexpr int kMaxGrid = 256;                     // the partial reduction reads 8 per lane
constexpr int kNoIndex = 0x7fffffff;
constexpr float kLog2e = 1.4426950408889634f;

struct Params {
  const __nv_bfloat16* W1;   // [V, 256]
  const int32_t* anchor;     // [G] (the launch's request rows)
  int32_t* draft_tok;        // [G, gamma]
  float* p_draft;            // [G, gamma, V]
  float2* part;              // [3][kMaxG][grid]: each CTA's (max, sum), log2 domain
  unsigned long long* word;  // [3][kMaxG]: packed race maximum per request
  unsigned int* gbar;        // grid barrier word (low 31 bits zero between barriers)
  unsigned int* err;
  int g0;                    // first request row of the launch (U and e are read by map)
  int G, npad, gamma, V, n_tiles, n_my_max;
  uint32_t tmem_cols;
};

struct Ctx {
  volatile int* abort_flag;
  unsigned int* err;
};

// Waits sleep in the barrier (up to 20 us at a time) between checks of the abort flag
// and of the time limit.
constexpr uint32_t kSleepNs = 20000;
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctx& cx) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kSleepNs)) return true;
    if (*cx.abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *cx.abort_flag = 1;
      raise_error(cx.err, DSPARK_DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
}
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Ctx& cx) {
  const bool ok = wait_bar(bar, parity, cx);
  return __all_sync(0xffffffffu, ok);
}
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, unsigned int* err) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      raise_error(err, DSPARK_DEVERR_WAIT_TIMEOUT);
      return;
    }
  }
}

// Named barrier of the epilogue warps; returns the OR of `pred` over them.
__device__ __forceinline__ bool epi_sync_or(bool pred) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.or.pred q, 1, %2, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"(pred ? 1u : 0u), "n"(kEpiThreads)
      : "memory");
  return r != 0u;
}

// Grid barrier over the co-resident CTAs: the word's top bit flips once all have
// arrived (CTA 0 adds 2^31 - (n - 1), the others 1; the low bits return to zero).
// The first arrival of a launch reads the word to learn the top bit; barrier b of the
// launch then ends when the top bit equals that bit ^ ((b + 1) & 1).
__device__ __forceinline__ unsigned int grid_arrive_first(unsigned int* w, bool master,
                                                          unsigned int n) {
  __threadfence();
  return atomicAdd(w, master ? 0x80000000u - (n - 1u) : 1u) >> 31;
}
__device__ __forceinline__ void grid_arrive(unsigned int* w, bool master, unsigned int n) {
  const unsigned int inc = master ? 0x80000000u - (n - 1u) : 1u;
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(w), "r"(inc) : "memory");
}
__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int* p) {
  unsigned int v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ bool grid_wait(const unsigned int* w, unsigned int top, const Ctx& cx) {
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while ((ld_acquire_gpu(w) >> 31) != top) {
    if ((++n & 15u) == 0) {
      if (*cx.abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        raise_error(cx.err, DSPARK_DEVERR_WAIT_TIMEOUT);
        return false;
      }
    }
  }
  return true;
}

__device__ __forceinline__ uint32_t sw128_off(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ float exp2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// (m, s) with s a sum of 2^(x - m): the merge of two such pairs (m = -inf: empty).
__device__ __forceinline__ void merge_ms(float& m, float& s, float m2, float s2) {
  const float mm = fmaxf(m, m2);
  // 2^(m - mm) and 2^(m2 - mm) with an empty side (-inf) giving 0, never NaN
  const float e1 = m == -INFINITY ? 0.f : exp2_approx(m - mm);
  const float e2 = m2 == -INFINITY ? 0.f : exp2_approx(m2 - mm);
  s = s * e1 + s2 * e2;
  m = mm;
}
__device__ __forceinline__ void better(float& k, int& i, float k2, int i2) {
  const bool b = k2 > k || (k2 == k && i2 < i);
  k = b ? k2 : k;
  i = b ? i2 : i;
}
// A race result as one word whose unsigned maximum is the winner: the key's bits mapped
// to an order-preserving unsigned in the high half, the complement of the index in the
// low half; 0 = nothing (no candidate, or a NaN key).
__device__ __forceinline__ unsigned long long race_word(float key, int idx) {
  if (idx == kNoIndex || key != key) return 0ull;
  uint32_t u = __float_as_uint(key);
  u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
  return (static_cast<unsigned long long>(u) << 32) | static_cast<uint32_t>(~idx);
}

__global__ void __launch_bounds__(kThreads, 1)
    markov_draft_kernel(const __grid_constant__ CUtensorMap tm_w2,
                        const __grid_constant__ CUtensorMap tm_u,
                        const __grid_constant__ CUtensorMap tm_e, const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = smem_raw + (base - raw);
  auto bar = [&](int i) { return base + OFF_BAR + 8 * i; };
  auto full = [&](int s) { return bar(s); };
  auto empty = [&](int s) { return bar(kStages + s); };
  auto u_full = [&](int s) { return bar(2 * kStages + s); };
  auto u_empty = [&](int s) { return bar(2 * kStages + kUStages + s); };
  const uint32_t h_full = bar(2 * kStages + 2 * kUStages);
  const uint32_t start_done = h_full + 8;  // the race words are clear everywhere
  const uint32_t last_done = h_full + 16;  // the last position's barrier has completed
  const uint32_t stg_full = h_full + 24;   // the W1 rows have landed
  auto acc_full = [&](int i) { return bar(2 * kStages + 2 * kUStages + 4 + i); };
  auto tfree = [&](int i) { return bar(2 * kStages + 2 * kUStages + 4 + kMaxTilesPerCta + i); };
  float2* red_st = reinterpret_cast<float2*>(bp + OFF_RED);        // [4][32]
  float* red_key = reinterpret_cast<float*>(bp + OFF_RED + 1024);  // [4][32]
  int* red_idx = reinterpret_cast<int*>(bp + OFF_RED + 1536);      // [4][32]
  float* colM = reinterpret_cast<float*>(bp + OFF_COL);  // [32]: M + log2 S, log2 domain
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bp + OFF_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bp + OFF_MISC + 16);
  const Ctx cx{abort_flag, prm.err};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nb = gridDim.x;
  const int n_my = (prm.n_tiles - 1 - (int)blockIdx.x) / nb + 1;  // grid <= n_tiles
  const int gamma = prm.gamma, V = prm.V, npad = prm.npad, G = prm.G;
  const uint32_t ubox = static_cast<uint32_t>(npad) * kMV * 4;    // one U (or e) box
  const bool master = blockIdx.x == 0;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int s = 0; s < kUStages; ++s) {
      mbar_init(u_full(s), 1);
      mbar_init(u_empty(s), kEpiWarps);
    }
    mbar_init(h_full, 1);
    mbar_init(start_done, 1);
    mbar_init(last_done, 1);
    mbar_init(stg_full, 1);
    for (int i = 0; i < kMaxTilesPerCta; ++i) {
      mbar_init(acc_full(i), 1);
      mbar_init(tfree(i), kEpiWarps);
    }
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) prefetch_tensormap(&tm_w2);
  if (warp == 2 && lane == 0) {
    prefetch_tensormap(&tm_u);
    prefetch_tensormap(&tm_e);
  }
  if (warp == 1) {
    tmem_alloc(smem_addr(tmem_slot), prm.tmem_cols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int total = gamma * n_my;  // (position, tile) pairs, position-major

  if (warp == 0) {
    // ---------------- W2 tiles of every position, in K halves, through the ring (kept in L2)
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_last();
      int issued = 0;
      for (int q = 0; q < 2 * total; ++q) {
        const int s = q % kStages;
        if (q >= kStages && !wait_bar(empty(s), ((q / kStages) - 1) & 1, cx)) break;
        const int t = (int)blockIdx.x + ((q >> 1) % n_my) * nb, kh = q & 1;
        const uint32_t dst = base + OFF_RING + s * kStage;
        mbar_arrive_expect_tx(full(s), kStage);
        tma_load_2d_hint(dst, &tm_w2, full(s), t * kMV, kh * kKH, pol);
        tma_load_2d_hint(dst + kStageHalf, &tm_w2, full(s), t * kMV + 64, kh * kKH, pol);
        issued = q + 1;
      }
      // no copy left in flight
      for (int q = issued > kStages ? issued - kStages : 0; q < issued; ++q)
        drain_bar(full(q % kStages), (q / kStages) & 1, prm.err);
    }
  } else if (warp == 2) {
    // ---------------- U and e boxes [npad rows x 128 vocab] of every (position, tile)
    if (lane == 0) {
      const uint64_t pol = l2_policy_evict_first();
      int issued = 0;
      for (int q = 0; q < total; ++q) {
        const int s = q % kUStages;
        if (q >= kUStages && !wait_bar(u_empty(s), ((q / kUStages) - 1) & 1, cx)) break;
        const int t = (int)blockIdx.x + (q % n_my) * nb, k = q / n_my;
        const uint32_t dst = base + OFF_URING + s * kUStage;
        mbar_arrive_expect_tx(u_full(s), 2 * ubox);
        tma_load_3d_hint(dst, &tm_u, u_full(s), t * kMV, k, prm.g0, pol);
        tma_load_3d_hint(dst + kUStage / 2, &tm_e, u_full(s), t * kMV, k, prm.g0, pol);
        issued = q + 1;
      }
      for (int q = issued > kUStages ? issued - kUStages : 0; q < issued; ++q)
        drain_bar(u_full(q % kUStages), (q / kUStages) & 1, prm.err);
    }
  } else if (warp == 1) {
    // ---------------- MMA: D[128 x npad] = W2 tile^T . H^T, one product per tile
    const uint32_t idesc = idesc_bf16_f32(kMV, npad, 1, 0);
    int last_i = -1, last_k = 0;
    bool ok = true;
    for (int k = 0; k < gamma && ok; ++k) {
      if (!wait_warp(h_full, k & 1, cx)) break;
      tc_fence_after();
      for (int i = 0; i < n_my && ok; ++i) {
        // TMEM half k & 1 of tile i was last read by the normalisation of position k - 2
        if (k >= 2 && !wait_warp(tfree(i), k & 1, cx)) {
          ok = false;
          break;
        }
        const uint32_t d = tmem + static_cast<uint32_t>(((k & 1) * prm.n_my_max + i) * npad);
        for (int kh = 0; kh < 2; ++kh) {
          const int q = 2 * (k * n_my + i) + kh, s = q % kStages;
          if (!wait_warp(full(s), (q / kStages) & 1, cx)) {
            ok = false;
            break;
          }
          if (lane == 0) {
            tc_fence_after();
            const uint32_t a0 = base + OFF_RING + s * kStage;
#pragma unroll
            for (int kk = 0; kk < kKH / 16; ++kk) {
              // A: 16 K rows of 128 bytes per step, the two 64-wide vocabulary halves apart
              const uint64_t a = smem_desc(a0 + kk * 2048, kStageHalf, 1024, SW_128B);
              // B: K-major rows of the gathered H, four 64-wide K blocks of npad rows
              const int kg = kh * (kKH / 16) + kk;
              const uint64_t b = smem_desc(base + OFF_H + (kg >> 2) * (npad * 128) + (kg & 3) * 32,
                                           16, 1024, SW_128B);
              umma_bf16(d, a, b, idesc, (kh | kk) ? 1u : 0u);
            }
            if (kh == 1) umma_commit(acc_full(i));
            umma_commit(empty(s));
          }
          __syncwarp();
        }
        last_i = i;
        last_k = k;
      }
    }
    // every product issued has completed before TMEM is released
    if (lane == 0 && last_i >= 0) drain_bar(acc_full(last_i), last_k & 1, prm.err);
    __syncwarp();
  } else if (warp == kSeqWarp) {
    // ---------------- sequencer: the grid barriers, the tokens, H for the next position
    // H = the W1 rows of the previous tokens (k = 0: the anchors), K-major with the
    // 128-byte swizzle; rows G..npad-1 zero.  Lane r < G holds request r's token and
    // copies its row with one bulk copy (the copy engine takes the 32 scattered rows at
    // once); the warp then lays the rows out, lane = 16-byte piece.
    int n_gather = 0;
    auto gather = [&](int tok) -> bool {
      if (lane == 0) mbar_arrive_expect_tx(stg_full, static_cast<uint32_t>(G) * (kR * 2));
      __syncwarp();
      if (lane < G)
        bulk_load_g2s(base + OFF_STG + lane * (kR * 2), prm.W1 + (long long)tok * kR, kR * 2, stg_full);
      if (!wait_warp(stg_full, n_gather & 1, cx)) return false;
      ++n_gather;
      const uint4* stg = reinterpret_cast<const uint4*>(bp + OFF_STG) + lane;
      uint8_t* hb = bp + OFF_H + (lane >> 3) * (npad * 128);
      for (int r0 = 0; r0 < npad; r0 += 8) {  // eight rows in flight per lane
        uint4 v[8];
#pragma unroll
        for (int j = 0; j < 8; ++j)
          v[j] = r0 + j < G ? stg[(r0 + j) * (kR * 2 / 16)] : make_uint4(0, 0, 0, 0);
#pragma unroll
        for (int j = 0; j < 8; ++j)
          *reinterpret_cast<uint4*>(hb + sw128_off(r0 + j, lane & 7)) = v[j];
      }
      fence_proxy_async_smem();  // H is read by the tensor cores, the staging rewritten by copies
      __syncwarp();
      if (lane == 0) mbar_arrive(h_full);
      return true;
    };
    auto checked = [&](int x) {
      if (x < 0 || x >= V) {
        raise_error(prm.err, DSPARK_DEVERR_BAD_INPUT);
        return 0;
      }
      return x;
    };
    // start: CTA 0 clears the race words of positions 0..2 (later ones are cleared as they
    // are retired), then every CTA arrives at the launch's first barrier
    if (master)
      for (int j = lane; j < 3 * kMaxG; j += 32) prm.word[j] = 0ull;
    __syncwarp();
    unsigned int top0 = 0;  // the barrier word's top bit before this launch's first barrier
    if (lane == 0) top0 = grid_arrive_first(prm.gbar, master, nb);
    top0 = __shfl_sync(0xffffffffu, top0, 0);
    bool ok = gather(lane < G ? checked(prm.anchor[lane]) : 0);
    if (ok && lane == 0) {
      ok = grid_wait(prm.gbar, top0 ^ 1u, cx);
      if (ok) mbar_arrive(start_done);
    }
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;  // (a failed gather fails on every lane)
    for (int k = 0; k < gamma && ok; ++k) {
      // barrier k + 1 of the launch: every CTA has published position k
      if (lane == 0) ok = grid_wait(prm.gbar, top0 ^ static_cast<unsigned int>(k & 1), cx);
      ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      if (!ok) break;
      int tok = 0;
      if (lane < G) {
        const unsigned long long w = __ldcg(prm.word + (k % 3) * kMaxG + lane);
        tok = w == 0ull ? 0 : static_cast<int>(~static_cast<uint32_t>(w));
        if (master) {
          prm.draft_tok[lane * gamma + k] = tok;
          // position k-1's words are read by every CTA; they serve position k+2 next
          if (k >= 1) prm.word[((k + 2) % 3) * kMaxG + lane] = 0ull;
        }
      }
      if (master) __threadfence();  // cleared before this CTA's next arrival
      if (k + 1 < gamma) {
        ok = gather(tok);
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(last_done);
      }
    }
    if (!ok) *abort_flag = 1;
  } else {
    // ---------------- epilogue: thread = vocabulary entry, 16 request columns per warp
    const int ew = warp - kEpiWarp0;
    const int qd = warp & 3;  // TMEM lane quadrant
    const int h = ew >> 2;    // request columns 8h .. 8h + 7
    const int c0 = kCols * h;
    const int et = threadIdx.x - kEpiWarp0 * 32;
    const bool has_cols = c0 < G;
    const int vq = 32 * qd + lane;
    const uint32_t tl = tmem + (static_cast<uint32_t>(32 * qd) << 16) + c0;
    const long long rstride = (long long)gamma * V;
    auto tmem_col = [&](int k, int i) {
      return tl + static_cast<uint32_t>(((k & 1) * prm.n_my_max + i) * npad);
    };

    // (M, S) of position k from every CTA's partial, in one fixed order (warp w takes the
    // requests w and w + 16; all of its loads are issued first)
    auto row_stats = [&](int k) {
      const float2* pk = prm.part + (size_t)(k % 3) * kMaxG * nb;
      float2 pv[2][8];
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = ew + kEpiWarps * cc;
#pragma unroll
        for (int r = 0; r < 8; ++r) {
          const int j = lane + 32 * r;
          pv[cc][r] = (c < G && j < nb) ? __ldcg(pk + (size_t)c * nb + j) : make_float2(-INFINITY, 0.f);
        }
      }
#pragma unroll
      for (int cc = 0; cc < 2; ++cc) {
        const int c = ew + kEpiWarps * cc;
        float mx = -INFINITY;
#pragma unroll
        for (int r = 0; r < 8; ++r) mx = fmaxf(mx, pv[cc][r].x);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
        float sum = 0.f;
#pragma unroll
        for (int r = 0; r < 8; ++r)
          if (pv[cc][r].x != -INFINITY) sum += pv[cc][r].y * exp2_approx(pv[cc][r].x - mx);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
        if (lane == 0 && c < G) colM[c] = mx + log2f(sum);  // p = 2^(x - M - log2 S)
      }
    };

    // p = 2^(logit - M - log2 S) of position k, from TMEM (the next tile's columns load while
    // this one's are written out); each tile's columns are released to the products of
    // position k + 2
    auto normalise = [&](int k) {
      float a[kCols], an[kCols], cm[kCols];
      if (has_cols) {
        tmem_ld8(tmem_col(k, 0), an);
#pragma unroll
        for (int c = 0; c < kCols; ++c) cm[c] = colM[(c0 + c) < G ? c0 + c : 0];
      }
      const bool full = c0 + kCols <= G;
      for (int i = 0; i < n_my; ++i) {
        if (has_cols) {
          tmem_wait_ld8(an);
#pragma unroll
          for (int c = 0; c < kCols; ++c) a[c] = an[c];
          if (i + 1 < n_my) tmem_ld8(tmem_col(k, i + 1), an);
          float* out = prm.p_draft + (long long)k * V + ((int)blockIdx.x + i * nb) * kMV + vq;
          if (full) {
#pragma unroll
            for (int c = 0; c < kCols; ++c)
              __stcs(out + (c0 + c) * rstride, exp2_approx(a[c] - cm[c]));
          } else {
#pragma unroll
            for (int c = 0; c < kCols; ++c)
              if (c0 + c < G) __stcs(out + (c0 + c) * rstride, exp2_approx(a[c] - cm[c]));
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tfree(i));
      }
    };

    bool stop = false;
    for (int k = 0; k < gamma && !stop; ++k) {
      // ---- A(k): per request the running max m and sum s of 2^(x - m), and the race
      // kept as the fraction bn / bd = 2^(x_best - m) / e_best (no division, no log)
      float m[kCols], s[kCols], bn[kCols], bd[kCols];
      int ib[kCols];
#pragma unroll
      for (int c = 0; c < kCols; ++c) {
        m[c] = -INFINITY;
        s[c] = 0.f;
        bn[c] = 0.f;
        bd[c] = 1.f;
        ib[c] = kNoIndex;
      }
      bool ok = wait_warp(acc_full(0), k & 1, cx);
      float a[kCols], an[kCols];
      if (ok) {
        tc_fence_after();
        if (has_cols) tmem_ld8(tmem_col(k, 0), an);
      }
      for (int i = 0; i < n_my && ok; ++i) {
        const int q = k * n_my + i, us = q % kUStages;
        if (i + 1 < n_my && !wait_warp(acc_full(i + 1), k & 1, cx)) {
          ok = false;
          break;
        }
        if (!wait_warp(u_full(us), (q / kUStages) & 1, cx)) {
          ok = false;
          break;
        }
        tc_fence_after();
        if (has_cols) {
          tmem_wait_ld8(an);
#pragma unroll
          for (int c = 0; c < kCols; ++c) a[c] = an[c];
          if (i + 1 < n_my) tmem_ld8(tmem_col(k, i + 1), an);
          const int v = ((int)blockIdx.x + i * nb) * kMV + vq;
          const float* su = reinterpret_cast<const float*>(bp + OFF_URING + us * kUStage) + vq;
          const float* se = su + kUStage / 8;
          // one entry of request column c: logit -> log2 domain, running (max, sum), race
          auto entry = [&](int c) {
            const int col = c0 + c;
            const float x2 = (a[c] + su[col * kMV]) * kLog2e;
            const float e = se[col * kMV];
            const float d = x2 - m[c];
            const float ex = exp2_approx(-fabsf(d));
            const bool up = d > 0.f;  // a new maximum rescales the sum and the numerator
            s[c] = up ? fmaf(s[c], ex, 1.f) : s[c] + ex;
            bn[c] = up ? bn[c] * ex : bn[c];
            m[c] = up ? x2 : m[c];
            const float w = up ? 1.f : ex;
            const bool win = w * bd[c] > bn[c] * e;  // w / e beats bn / bd; ties keep the lowest index
            bn[c] = win ? w : bn[c];
            bd[c] = win ? e : bd[c];
            ib[c] = win ? v : ib[c];
            a[c] = x2;
          };
          if (c0 + kCols <= G) {
#pragma unroll
            for (int c = 0; c < kCols; ++c) entry(c);
          } else {
#pragma unroll
            for (int c = 0; c < kCols; ++c)
              if (c0 + c < G) entry(c);
          }
          tmem_st8(tmem_col(k, i), a);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(u_empty(us));  // this warp is done with the boxes
      }
      if (has_cols) tmem_wait_ld8(an);
      tmem_wait_st();
      if (ok && has_cols) {
        // the race in the log2 domain: key = m + log2(bn / bd); no candidate: -inf
        float kb[kCols];
#pragma unroll
        for (int c = 0; c < kCols; ++c)
          kb[c] = bn[c] > 0.f ? m[c] + (__log2f(bn[c]) - __log2f(bd[c])) : -INFINITY;
        // lane l ends with request column c0 + (l & 7): halving exchanges over lane bits
        // 2, 1, 0, then lanes that hold the same column merge over bits 3 and 4
#pragma unroll
        for (int o = kCols / 2; o > 0; o >>= 1) {
          const bool upper = (lane & o) != 0;
#pragma unroll
          for (int j = 0; j < o; ++j) {
            const float sm = upper ? m[j] : m[j + o], ss = upper ? s[j] : s[j + o];
            const float sk = upper ? kb[j] : kb[j + o];
            const int si = upper ? ib[j] : ib[j + o];
            const float rm = __shfl_xor_sync(0xffffffffu, sm, o), rs = __shfl_xor_sync(0xffffffffu, ss, o);
            const float rk = __shfl_xor_sync(0xffffffffu, sk, o);
            const int ri = __shfl_xor_sync(0xffffffffu, si, o);
            float km = upper ? m[j + o] : m[j], ks = upper ? s[j + o] : s[j];
            float kk2 = upper ? kb[j + o] : kb[j];
            int ki = upper ? ib[j + o] : ib[j];
            merge_ms(km, ks, rm, rs);
            better(kk2, ki, rk, ri);
            m[j] = km;
            s[j] = ks;
            kb[j] = kk2;
            ib[j] = ki;
          }
        }
#pragma unroll
        for (int o = kCols; o < 32; o <<= 1) {
          const float rm = __shfl_xor_sync(0xffffffffu, m[0], o), rs = __shfl_xor_sync(0xffffffffu, s[0], o);
          const float rk = __shfl_xor_sync(0xffffffffu, kb[0], o);
          const int ri = __shfl_xor_sync(0xffffffffu, ib[0], o);
          merge_ms(m[0], s[0], rm, rs);
          better(kb[0], ib[0], rk, ri);
        }
        if (lane < kCols) {
          const int col = c0 + lane;
          red_st[qd * kMaxG + col] = make_float2(m[0], s[0]);
          red_key[qd * kMaxG + col] = kb[0];
          red_idx[qd * kMaxG + col] = ib[0];
        }
      }
      stop = epi_sync_or(!ok || *abort_flag);
      if (stop) break;
      // the race words are clear in every CTA's view before the first race
      if (k == 0) {
        const bool ok0 = wait_warp(start_done, 0, cx);
        stop = epi_sync_or(!ok0);
        if (stop) break;
      }
      if (et < G) {
        float pm = -INFINITY, ps = 0.f, pkey = -INFINITY;
        int pidx = kNoIndex;
#pragma unroll
        for (int w = 0; w < 4; ++w) {
          const float2 st = red_st[w * kMaxG + et];
          merge_ms(pm, ps, st.x, st.y);
          better(pkey, pidx, red_key[w * kMaxG + et], red_idx[w * kMaxG + et]);
        }
        // three buffers: a CTA still reading position k's partials has not arrived at
        // barrier k + 3, which precedes every write of position k + 3's
        prm.part[(size_t)(k % 3) * kMaxG * nb + (size_t)et * nb + blockIdx.x] = make_float2(pm, ps);
        const unsigned long long wv = race_word(pkey, pidx);
        if (wv) atomicMax(prm.word + (k % 3) * kMaxG + et, wv);
      }
      fence_proxy_async_smem();  // the scratch is overwritten by the next rows' copies
      epi_sync_or(false);
      // barrier k + 1 of the launch (the first one was the start's)
      if (et == 0) grid_arrive(prm.gbar, master, nb);
      // ---- C(k-1) while the sequencer runs position k's barrier and position k+1's
      // gather: position k-1's partials are complete (its barrier preceded the
      // products of position k)
      if (k >= 1) {
        row_stats(k - 1);
        epi_sync_or(false);
        normalise(k - 1);
      }
    }
    if (!stop) {
      // the last position: its barrier is the sequencer's last wait
      const bool okl = wait_warp(last_done, 0, cx);
      stop = epi_sync_or(!okl);
      if (!stop) {
        row_stats(gamma - 1);
        epi_sync_or(false);
        normalise(gamma - 1);
      }
    }
    if (stop) *abort_flag = 1;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, prm.tmem_cols);
}

struct Geometry {
  int nb, n_tiles, n_my_max, g_max;
};

// Grid and request-group size for a vocabulary of V (a multiple of 128).
bool geometry(int V, Geometry* g) {
  const int sms = num_sms_cached();
  if (sms <= 0 || V < kMV || V % kMV) return false;
  g->n_tiles = V / kMV;
  g->nb = g->n_tiles < sms ? g->n_tiles : sms;
  if (g->nb > kMaxGrid) g->nb = kMaxGrid;
  g->n_my_max = ceil_div(g->n_tiles, g->nb);
  if (g->n_my_max > kMaxTilesPerCta) return false;
  // TMEM: two positions x n_my_max tiles x N columns <= 512, N a multiple of 16
  int gm = (256 / g->n_my_max) & ~15;
  g->g_max = gm < kMaxG ? gm : kMaxG;
  return g->g_max >= 16;
}

bool configure() {
  static PerDevice<bool> done;
  return once_per_device(done, false, [] {
    int dev = 0, coop = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return false;
    if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop)
      return false;
    if (cudaFuncSetAttribute(markov_draft_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             SMEM_BYTES) != cudaSuccess)
      return false;
    int per_sm = 0;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, markov_draft_kernel, kThreads,
                                                         SMEM_BYTES) == cudaSuccess &&
           per_sm >= 1;
  });
}

constexpr size_t kWordsOff = 256;
constexpr size_t kPartOff = kWordsOff + 3 * kMaxG * sizeof(unsigned long long);

}  // namespace md

bool markov_supported(int V, int* group) {
  md::Geometry g;
  if (!md::geometry(V, &g)) return false;
  if (group) *group = g.g_max;
  return true;
}

// The same for every device: the partial array is sized for the largest grid (256).
size_t markov_workspace(int V) {
  if (V < md::kMV || V % md::kMV) return 0;
  return md::kPartOff + (size_t)3 * md::kMaxG * md::kMaxGrid * sizeof(float2);
}

int launch_markov_draft(const float* U, const void* W1, const void* W2, const int32_t* anchor,
                        const float* exp_noise, int B, int gamma, int V, int32_t* draft_tok,
                        float* p_draft, void* ws, cudaStream_t stream) {
  using namespace md;
  Geometry geo;
  if (!geometry(V, &geo)) return DSPARK_EUNSUPPORTED;
  if (!configure()) return DSPARK_ECUDA;
  CUtensorMap tm_w2;
  {
    const uint64_t dims[2] = {(uint64_t)V, (uint64_t)kR};
    const uint64_t strides[1] = {(uint64_t)V * 2};
    const uint32_t box[2] = {64u, (uint32_t)kKH};
    if (!attn::gqa::encode_bf16_map(&tm_w2, W2, 2, dims, strides, box)) return DSPARK_ECUDA;
  }
  uint8_t* w = static_cast<uint8_t*>(ws);
  for (int g0 = 0; g0 < B; g0 += geo.g_max) {
    const int G = B - g0 < geo.g_max ? B - g0 : geo.g_max;
    const int npad = (G + 15) & ~15;
    // U and e as [B][gamma][V] fp32: boxes of 128 vocabulary entries x 1 position x npad rows
    CUtensorMap tm_u, tm_e;
    {
      const uint64_t dims[3] = {(uint64_t)V, (uint64_t)gamma, (uint64_t)B};
      const uint64_t strides[2] = {(uint64_t)V * 4, (uint64_t)gamma * V * 4};
      const uint32_t box[3] = {(uint32_t)kMV, 1u, (uint32_t)npad};
      if (!attn::gqa::encode_f32_map(&tm_u, U, 3, dims, strides, box) ||
          !attn::gqa::encode_f32_map(&tm_e, exp_noise, 3, dims, strides, box))
        return DSPARK_ECUDA;
    }
    Params prm;
    const size_t roff = (size_t)g0 * gamma * V;
    prm.g0 = g0;
    prm.W1 = static_cast<const __nv_bfloat16*>(W1);
    prm.anchor = anchor + g0;
    prm.draft_tok = draft_tok + (size_t)g0 * gamma;
    prm.p_draft = p_draft + roff;
    prm.part = reinterpret_cast<float2*>(w + kPartOff);
    prm.word = reinterpret_cast<unsigned long long*>(w + kWordsOff);
    prm.gbar = reinterpret_cast<unsigned int*>(w);
    prm.err = device_error_word();
    prm.G = G;
    prm.npad = npad;
    prm.gamma = gamma;
    prm.V = V;
    prm.n_tiles = geo.n_tiles;
    prm.n_my_max = geo.n_my_max;
    uint32_t cols = 32;
    while (cols < (uint32_t)(2 * geo.n_my_max * prm.npad)) cols <<= 1;
    prm.tmem_cols = cols;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(geo.nb);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = SMEM_BYTES;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeCooperative;
    attr[0].val.cooperative = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (cudaLaunchKernelEx(&cfg, markov_draft_kernel, tm_w2, tm_u, tm_e, prm) != cudaSuccess) return DSPARK_ECUDA;
  }
  return DSPARK_OK;
}

}  // namespace dspark
