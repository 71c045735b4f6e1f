// Varlen verify attention, GQA shape (head dim 128), keys on the MMA's M side.
//
// What it computes ("DFlash 到 DSpark in SGLang", section "Ragged verify under
// full CUDA graphs": each packed verify token attends only to its own request's
// KV, causal inside the block): for packed row cu_seqlens[r] + i and query head
// h of KV group kvh, o = softmax(scale q.K^T) V over the ctx_len[r] committed keys
// (paged) followed by block rows 0..i; lse = log-sum-exp.
//
// Why transposed: a verify step has few query rows per (request, KV head) -- the
// window's 1 + w rows times the group's G heads, typically 10-40 -- against
// thousands of keys.  With keys on the M side (128 TMEM lanes) and the query rows
// on N (NT = 32, 64 or 128 columns), every tensor-core row and every softmax
// thread does useful work, and the exp count per key scales with the real row
// count instead of a padded 128.
//
//   S^T [128 keys x NT rows] = K_tile [128 x 128] . Q^T           (tcgen05, TMEM)
//   O^T [128 d    x NT rows] += V_tile^T . P^T                    (tcgen05, TMEM)
//
// Warp roles (one CTA per SM, persistent over its stream-K range of the work list):
//   warp 0     K producer: TMA tiled loads (128-byte swizzle, no multicast) of the
//              context pages holding at least one visible key and of the block's
//              own rows; keys past the visible range are left as they are (the
//              softmax masks them by index)
//   warp 1     V producer: TMA for every full 16-key chunk; the one partial chunk
//              of a tile by plain loads with zeros past the visible keys.  Chunks
//              past the visible keys are neither loaded nor multiplied (PV skips
//              them), so no stale value reaches O
//   warp 2     Q loader: the next item's query tile into the second Q buffer
//              while the current item runs
//   warp 3     MMA issuer (one lane) + TMEM owner.  O^T is double-buffered in
//              TMEM, so the next item's products start while the epilogue of the
//              last one still reads its O^T
//   warps 4-7  softmax: thread = key (TMEM lane).  Per tile: per-row max by a
//              warp transpose-reduction and one cross-warp exchange through an
//              mbarrier, lazy rescale of O^T when a row's max grows by > 2^8,
//              exp2 on the SFU, P^T to shared memory in bf16, per-row sums by a
//              second transpose-reduction of the bf16 P the PV product multiplies
//              (so the weights applied to V are exactly the normalised rounded P).
//              Epilogue: O / l, lse.
//   warps 8-11 (128-column tile only) a second softmax warpgroup: warps 4-7 own
//              query columns 0-63 and warps 8-11 columns 64-127, each with its
//              own half of P^T, its own PV product (N = 64) and its own share
//              of the epilogue staging.  A half with no rows in an item only
//              releases S^T; the PV product of that half is skipped.
// Every wait is bounded in time (DSPARK_DEVERR_WAIT_TIMEOUT on expiry).

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"
#include "common.cuh"
#include "ptx.cuh"

namespace dspark {
namespace attn {
namespace gqa {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kKT = 128;              // keys per tile (MMA M)
constexpr int kD = 128;               // head dim
constexpr int kStages = 2;
constexpr int kKWarp = 0;
constexpr int kVWarp = 1;
constexpr int kQWarp = 2;
constexpr int kMmaWarp = 3;
constexpr int kSoftmaxWarp0 = 4;
constexpr int kTileHalf = kKT * 128;  // one 64-wide column block of a [128 x 128] bf16 tile
constexpr int kKVBytes = 2 * kTileHalf;
constexpr int kStageBytes = 2 * kKVBytes;  // K and V
constexpr int kChunkRows = 16;             // V chunk = PV k-step; also the block-row box
constexpr int kSmemItems = 32;             // work items of a CTA kept in shared memory

template <int NT_>
struct Cfg {
  static constexpr int NT = NT_;                         // query rows (N)
  static constexpr int Q_CB = NT * 128;                  // one 64-wide column block of Q
  static constexpr int Q_BYTES = 2 * Q_CB;
  static constexpr int Q_BUFS = NT <= 64 ? 2 : 1;
  static constexpr int P_ROW = NT <= 64 ? NT * 2 : 128;  // bytes per key row of one P block
  static constexpr int P_BLOCKS = NT <= 64 ? 1 : NT / 64;
  static constexpr int P_BYTES = kKT * NT * 2;
  static constexpr int P_BUFS = NT <= 64 ? 2 : 1;
  static constexpr SwizzleMode P_SW = NT == 32 ? SW_64B : SW_128B;
  static constexpr int G32 = NT / 32;                    // 32-row groups
  // softmax warpgroups: the 128-column tile has two, each owning 64 query rows (its own
  // half of P^T, released to its own PV product)
  static constexpr int WGS = NT == 128 ? 2 : 1;
  static constexpr int THREADS = (4 + 4 * WGS) * 32;
  static constexpr int G32_WG = G32 / WGS;               // 32-row groups per warpgroup
  static constexpr int PH = WGS;                          // P^T halves with their own barriers
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_STAGE = OFF_Q + Q_BUFS * Q_BYTES;
  static constexpr int OFF_P = OFF_STAGE + kStages * kStageBytes;
  static constexpr int OFF_RED = OFF_P + P_BUFS * P_BYTES;         // float wmax[2][4][NT]
  static constexpr int OFF_REF = OFF_RED + 2 * 4 * NT * 4;         // float mref[4][NT], alpha[4][NT]
  static constexpr int OFF_LS = OFF_REF + 2 * 4 * NT * 4;          // float lsum[4][NT]
  static constexpr int OFF_MT = OFF_LS + 4 * NT * 4;               // float mtrue[4][NT]
  static constexpr int OFF_OVER = OFF_MT + 4 * NT * 4;              // int over[2][WGS][4]
  static constexpr int OFF_ITEMS = OFF_OVER + 32 * WGS;             // AttnItem[kSmemItems]
  static constexpr int OFF_BAR = OFF_ITEMS + kSmemItems * (int)sizeof(AttnItem);
  // k_full[2], k_empty[2], v_full[2], v_empty[2], s_full[2], s_free[2], o_free[2];
  // per warpgroup xw[2], xs[2], ep[2], stg_full, stg_free; p_full[PB][PH],
  // p_empty[PB][PH], q_full[QB], q_empty[QB]
  static constexpr int N_BARS = 14 + 8 * WGS + 2 * P_BUFS * PH + 2 * Q_BUFS;
  // epilogue: O / l is staged row-major (512 B per query row) in the P buffers, each
  // warpgroup in its own share of them
  static constexpr int STG_BYTES_WG = P_BUFS * P_BYTES / WGS;
  static constexpr int STG_ROWS = STG_BYTES_WG / (kD * 4);
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;
  static constexpr int TMEM_S = 0;          // S^T, two buffers of NT columns
  static constexpr int TMEM_O = 2 * NT;     // O^T, two buffers of NT columns
  static constexpr int TMEM_COLS = 4 * NT <= 128 ? 128 : (4 * NT <= 256 ? 256 : 512);
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(NT == 32 || NT == 64 || NT == 128, "query tile");
  static_assert(NT != 128 || P_BUFS == 1, "the 128-column tile's halves count phases on one P buffer");
};

struct Ctx {
  volatile int* abort_flag;
  unsigned int* err;
};

// Waits sleep in the barrier (up to 20 us at a time, so that a waiting warp takes no
// issue slots from the softmax warp beside it) between checks of the abort flag and of
// the time limit.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctx& cx) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, 20000)) return true;
    if (*cx.abort_flag) return false;
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      *cx.abort_flag = 1;
      raise_error(cx.err, DSPARK_DEVERR_WAIT_TIMEOUT);
      return false;
    }
  }
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

// warp-uniform bounded wait (every lane polls; all agree on the outcome)
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Ctx& cx) {
  bool ok = wait_bar(bar, parity, cx);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t sw128_off(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
__device__ __forceinline__ uint32_t sw64_off(int row, int chunk) {
  return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}

// Warp transpose-reduction: lane l holds v[0..31] (one value per query row for
// its key); returns op over all 32 lanes of v[l], i.e. the reduction for row l.
template <bool MAX, int W>
__device__ __forceinline__ void transpose_step(float (&v)[32], int lane) {
  const bool hi = (lane & W) != 0;
#pragma unroll
  for (int i = 0; i < W; ++i) {
    const float send = hi ? v[i] : v[i + W];
    const float keep = hi ? v[i + W] : v[i];
    const float got = __shfl_xor_sync(0xffffffffu, send, W);
    v[i] = MAX ? fmaxf(keep, got) : keep + got;
  }
}
template <bool MAX>
__device__ __forceinline__ float transpose_reduce(float (&v)[32], int lane) {
  transpose_step<MAX, 16>(v, lane);
  transpose_step<MAX, 8>(v, lane);
  transpose_step<MAX, 4>(v, lane);
  transpose_step<MAX, 2>(v, lane);
  transpose_step<MAX, 1>(v, lane);
  return v[0];
}

template <int NT>
struct Layout {
  uint32_t base;
  __device__ uint32_t q(int b) const { return base + Cfg<NT>::OFF_Q + b * Cfg<NT>::Q_BYTES; }
  __device__ uint32_t stage(int s) const { return base + Cfg<NT>::OFF_STAGE + s * kStageBytes; }
  __device__ uint32_t pbuf(int b) const { return base + Cfg<NT>::OFF_P + b * Cfg<NT>::P_BYTES; }
  __device__ uint32_t bar(int i) const { return base + Cfg<NT>::OFF_BAR + 8 * i; }
  __device__ uint32_t k_full(int s) const { return bar(s); }
  __device__ uint32_t k_empty(int s) const { return bar(2 + s); }
  __device__ uint32_t v_full(int s) const { return bar(4 + s); }
  __device__ uint32_t v_empty(int s) const { return bar(6 + s); }
  __device__ uint32_t s_full(int b) const { return bar(8 + b); }
  __device__ uint32_t s_free(int b) const { return bar(10 + b); }
  __device__ uint32_t o_free(int b) const { return bar(12 + b); }
  // per softmax warpgroup w
  __device__ uint32_t xw(int w, int b) const { return bar(14 + 8 * w + b); }
  __device__ uint32_t xs(int w, int b) const { return bar(14 + 8 * w + 2 + b); }
  __device__ uint32_t ep(int w, int b) const { return bar(14 + 8 * w + 4 + b); }
  __device__ uint32_t stg_full(int w) const { return bar(14 + 8 * w + 6); }
  __device__ uint32_t stg_free(int w) const { return bar(14 + 8 * w + 7); }
  static constexpr int P0 = 14 + 8 * Cfg<NT>::WGS;
  // P buffer b, half h (the 128-column tile's halves; one half otherwise)
  __device__ uint32_t p_full(int b, int h) const { return bar(P0 + b * Cfg<NT>::PH + h); }
  __device__ uint32_t p_empty(int b, int h) const {
    return bar(P0 + Cfg<NT>::P_BUFS * Cfg<NT>::PH + b * Cfg<NT>::PH + h);
  }
  __device__ uint32_t q_full(int b) const { return bar(P0 + 2 * Cfg<NT>::P_BUFS * Cfg<NT>::PH + b); }
  __device__ uint32_t q_empty(int b) const {
    return bar(P0 + 2 * Cfg<NT>::P_BUFS * Cfg<NT>::PH + Cfg<NT>::Q_BUFS + b);
  }
};

// Work item `it` of this CTA: from shared memory for the first kSmemItems items.
__device__ __forceinline__ AttnItem fetch_item(const AttnItem* s_items, const AttnItem* g_items,
                                               int it, int it_begin) {
  const int k = it - it_begin;
  return k < kSmemItems ? s_items[k] : g_items[it];
}

// Keys of tile t of a request that a query row can see at all: the cache tile's
// keys below ctx, or the block tile's rows below n_r.
__device__ __forceinline__ int visible_keys(int t, int ct, int ctx, int n_r) {
  const int v = t < ct ? ctx - t * kKT : n_r - (t - ct) * kKT;
  return v < kKT ? v : kKT;
}

struct Params {
  const __nv_bfloat16* q;
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  const __nv_bfloat16* k_cache;
  const __nv_bfloat16* v_cache;
  const int32_t* page_table;
  const int32_t* ctx_len;
  const int32_t* cu_seqlens;
  const AttnItem* items;
  const int* item_begin;  // [gridDim.x + 1]: CTA c runs items [item_begin[c], item_begin[c+1])
  float* out;
  float* lse;
  float* ws_o;
  float* ws_lse;
  unsigned int* err;
  int max_pages, B, Hq, Hkv, page_size, log2_page, max_rows, n_pages;
  float scale_log2;
};

template <int NT>
__global__ void __launch_bounds__(Cfg<NT>::THREADS, 1)
    verify_attn_gqa_kernel(const __grid_constant__ CUtensorMap tm_k,
                           const __grid_constant__ CUtensorMap tm_v,
                           const __grid_constant__ CUtensorMap tm_kn,
                           const __grid_constant__ CUtensorMap tm_vn, const Params prm) {
  using C = Cfg<NT>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = smem_raw + (base - raw);
  const Layout<NT> L{base};
  float* s_wmax = reinterpret_cast<float*>(bp + C::OFF_RED);       // [2][4][NT]
  float* s_mref = reinterpret_cast<float*>(bp + C::OFF_REF);       // [4][NT]
  float* s_alpha = s_mref + 4 * NT;                                 // [4][NT]
  float* s_lsum = reinterpret_cast<float*>(bp + C::OFF_LS);        // [4][NT]
  AttnItem* s_items = reinterpret_cast<AttnItem*>(bp + C::OFF_ITEMS);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bp + C::OFF_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bp + C::OFF_MISC + 16);
  const Ctx cx{abort_flag, prm.err};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int b = 0; b < 2; ++b) {
      mbar_init(L.k_full(b), 1);
      mbar_init(L.k_empty(b), 1);
      mbar_init(L.v_full(b), 1);
      mbar_init(L.v_empty(b), 1);
      mbar_init(L.s_full(b), 1);
      mbar_init(L.s_free(b), 4 * C::WGS);
      mbar_init(L.o_free(b), 4 * C::WGS);
      for (int w = 0; w < C::WGS; ++w) {
        mbar_init(L.xw(w, b), 4);
        mbar_init(L.xs(w, b), 4);
        mbar_init(L.ep(w, b), 4);
      }
    }
    for (int w = 0; w < C::WGS; ++w) {
      mbar_init(L.stg_full(w), 4);
      mbar_init(L.stg_free(w), 1);
    }
    for (int b = 0; b < C::P_BUFS; ++b)
      for (int h = 0; h < C::PH; ++h) {
        mbar_init(L.p_full(b, h), 4);
        mbar_init(L.p_empty(b, h), 1);
      }
    for (int b = 0; b < C::Q_BUFS; ++b) {
      mbar_init(L.q_full(b), 1);
      mbar_init(L.q_empty(b), 1);
    }
    fence_mbar_init();
  }
  if (warp == kKWarp && lane == 0) {
    prefetch_tensormap(&tm_k);
    prefetch_tensormap(&tm_kn);
  }
  if (warp == kVWarp && lane == 0) {
    prefetch_tensormap(&tm_v);
    prefetch_tensormap(&tm_vn);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  pdl_release();
  pdl_wait();  // the work list and the step's inputs come from earlier kernels
  const int it_begin = prm.item_begin[blockIdx.x];
  const int it_end = prm.item_begin[blockIdx.x + 1];
  {
    const int n_s = min(kSmemItems, it_end - it_begin);
    constexpr int kWords = (int)(sizeof(AttnItem) / sizeof(uint4));
    for (int i = threadIdx.x; i < n_s * kWords; i += C::THREADS)
      reinterpret_cast<uint4*>(s_items)[i] = reinterpret_cast<const uint4*>(prm.items + it_begin)[i];
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int G = prm.Hq / prm.Hkv;
  const int P = prm.page_size;
  const int lp = prm.log2_page;

  if (warp == kKWarp || warp == kVWarp) {
    // ------------------------------------------------------------- producers
    // Each stream has its own two-slot ring: a K slot is released as soon as QK^T of
    // its tile completes, so the next K tiles (and with them QK^T and the softmax)
    // run ahead of the V stream.  Lane j holds page-table slot win_base + j of the
    // current request.
    const bool is_v = warp == kVWarp;
    const CUtensorMap* tm_c = is_v ? &tm_v : &tm_k;
    const CUtensorMap* tm_n = is_v ? &tm_vn : &tm_kn;
    // K boxes follow the page (up to a tile); V boxes are 16-key chunks
    const int box_rows = is_v ? kChunkRows : (P < kKT ? P : kKT);
    int g = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it) {
      const AttnItem item = fetch_item(s_items, prm.items, it, it_begin);
      const int r = item.r;
      const int ctx = item.ctx;
      const int c0 = item.c0;
      const int n_r = item.n_r;
      const int ct = ceil_div(ctx, kKT);
      const int32_t* ptab = prm.page_table + (long long)r * prm.max_pages;
      int win_base = -1, win_page = 0;
      for (int t = item.tb; t < item.te; ++t, ++g) {
        const int s = g % kStages;
        const uint32_t full = is_v ? L.v_full(s) : L.k_full(s);
        if (g >= kStages) {
          ok = wait_warp(is_v ? L.v_empty(s) : L.k_empty(s), ((g / kStages) - 1) & 1, cx);
          if (!ok) break;
        }
        const uint32_t dst0 = L.stage(s) + (is_v ? kKVBytes : 0);
        const int vis = visible_keys(t, ct, ctx, n_r);  // >= 1
        // boxes copied by TMA: K every box with a visible key, V every 16-key chunk
        // with one (the MMA warp zeroes the V rows past them); cache boxes are
        // box_rows keys, block-row boxes kChunkRows rows
        const int rows_box = t < ct ? box_rows : kChunkRows;
        const int nb = ceil_div(vis, rows_box);
        if (lane == 0) mbar_expect_tx(full, nb * 2 * rows_box * 128);
        __syncwarp();
        if (t < ct) {
          const int slot0 = (t * kKT) >> lp;
          const int nslot = ceil_div(kKT, P);
          if (win_base < 0 || slot0 + nslot > win_base + 32) {
            win_base = slot0;
            const int sl = win_base + lane;
            int pg = (sl << lp) < ctx ? ptab[sl] : 0;
            if ((sl << lp) < ctx && (pg < 0 || pg >= prm.n_pages)) {
              raise_error(prm.err, DSPARK_DEVERR_BAD_INPUT);
              pg = -1;
            }
            win_page = pg;
          }
          // lane = (box, column block), one copy each; every copied box starts at a
          // visible key, so its page-table slot is a valid one
          for (int base_l = 0; base_l < 2 * nb; base_l += 32) {
            const int o = base_l + lane;
            const int bx = o >> 1, cb = o & 1;
            const int kg = t * kKT + bx * box_rows;
            const int src_lane = bx < nb ? ((kg >> lp) - win_base) & 31 : 0;
            const int page = __shfl_sync(0xffffffffu, win_page, src_lane);  // converged
            if (bx < nb)
              tma_load_4d(dst0 + cb * kTileHalf + bx * box_rows * 128, tm_c, full, cb * 64,
                          item.kvh, kg & (P - 1), page);
          }
        } else {
          // block tile: the request's own rows b0.., 16-row boxes of the packed buffer
          const int b0 = (t - ct) * kKT;
          if (lane < 2 * nb) {
            const int bx = lane >> 1, cb = lane & 1;
            tma_load_3d(dst0 + cb * kTileHalf + bx * kChunkRows * 128, tm_n, full, cb * 64, item.kvh,
                        c0 + b0 + bx * kChunkRows);
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(full);
      }
    }
    if (lane == 0) {
      const int first = g - kStages > 0 ? g - kStages : 0;
      for (int gg = first; gg < g; ++gg)
        drain_bar(is_v ? L.v_full(gg % kStages) : L.k_full(gg % kStages), (gg / kStages) & 1, prm.err);
    }
  } else if (warp == kQWarp) {
    // ------------------------------------------------------------- Q loader
    // Query tile of item n: row n' = (block row n' / G, head kvh*G + n' % G), rows
    // past the item's nq are zero.  Buffer n % Q_BUFS is refilled once QK^T of the
    // item that used it is complete.
    bool ok = true;
    int n_it = 0;
    for (int it = it_begin; it < it_end && ok; ++it, ++n_it) {
      const AttnItem item = fetch_item(s_items, prm.items, it, it_begin);
      const int qb = n_it % C::Q_BUFS;
      if (n_it >= C::Q_BUFS) {
        ok = wait_warp(L.q_empty(qb), ((n_it / C::Q_BUFS) - 1) & 1, cx);
        if (!ok) break;
      }
      const int nq = item.ni * G;
      const long long row0 = item.c0 + item.i0;
      const uint32_t qd = L.q(qb);
      constexpr int kPer = NT * 16 / 32;   // 16-byte pieces per lane
      constexpr int kBatch = kPer < 16 ? kPer : 16;
#pragma unroll 1
      for (int b0 = 0; b0 < kPer; b0 += kBatch) {
        uint4 v[kBatch];
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int idx = (b0 + i) * 32 + lane, row = idx >> 4, q = idx & 15;
          v[i] = make_uint4(0, 0, 0, 0);
          if (row < nq)
            v[i] = ldg_nc_v4(prm.q + ((row0 + row / G) * prm.Hq + item.kvh * G + row % G) * kD + q * 8);
        }
#pragma unroll
        for (int i = 0; i < kBatch; ++i) {
          const int idx = (b0 + i) * 32 + lane, row = idx >> 4, q = idx & 15;
          st_shared_v4(qd + (q >> 3) * C::Q_CB + sw128_off(row, q & 7), v[i]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(L.q_full(qb));
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    // The whole warp runs the loop (lane 0 issues); before the PV product of a
    // tile whose visible keys end inside a 16-key chunk, the warp zeroes that
    // chunk's V rows past them (TMA copied the whole chunk), so that no stale or
    // foreign value meets a zero probability.
    constexpr uint32_t IDESC_QK = idesc_bf16_f32(kKT, NT, 0, 0);
    constexpr uint32_t IDESC_PV = idesc_bf16_f32(kD, NT / C::PH, 1, 1);
    int g = 0, n_it = 0, last_pv = -1;
    int nh1 = 0;  // products of the second P^T half issued (tiles whose item has rows there)
    bool ok = true;
    // PV of tile gp (local index `local` in its item) into O^T buffer ob, over the
    // 16-key chunks that hold visible keys only; one product per half of P^T as its
    // warpgroup releases it (a half without query rows of the item is released but not
    // multiplied)
    auto issue_pv = [&](int gp, int local, int vis, int ob, int nq) -> bool {
      const int pb = gp % C::P_BUFS;
      if (!wait_warp(L.p_full(pb, 0), (gp / C::P_BUFS) & 1, cx)) return false;
      const int s = gp % kStages;
      if (!wait_warp(L.v_full(s), (gp / kStages) & 1, cx)) return false;
      const uint32_t vb = L.stage(s) + kKVBytes;
      const int nch = ceil_div(vis, 16);
      if (vis & 15) {
        // rows vis .. 16*nch - 1: (rows) x 2 column blocks x 8 16-byte pieces
        const int r0 = vis, nz = (16 * nch - vis) * 16;
        for (int idx = lane; idx < nz; idx += 32) {
          const int row = r0 + (idx >> 4), cb = (idx >> 3) & 1, c = idx & 7;
          st_shared_v4(vb + cb * kTileHalf + sw128_off(row, c), make_uint4(0, 0, 0, 0));
        }
        fence_proxy_async_smem();
      }
      __syncwarp();
      for (int h = 0; h < C::PH; ++h) {
        // the second half exists only for items with rows in it (128-column tile, one P
        // buffer): its barriers count those tiles alone
        if (h > 0 && h * (NT / C::PH) >= nq) continue;
        if (h > 0 && !wait_warp(L.p_full(pb, h), nh1 & 1, cx)) return false;
        if (lane == 0) {
          tc_fence_after();
          const uint32_t d_o = tmem + C::TMEM_O + ob * NT + h * (NT / C::PH);
          for (int kk = 0; kk < nch; ++kk) {
            // A = V^T (M = d, MN-major), B = P^T (N = query rows, MN-major); K = 16 keys
            const uint64_t a = smem_desc(vb + kk * 2048, kTileHalf, 1024, SW_128B);
            const uint64_t b = smem_desc(L.pbuf(pb) + h * (kKT * 128) + kk * 16 * C::P_ROW, kKT * 128,
                                         8 * C::P_ROW, C::P_SW);
            umma_bf16(d_o, a, b, IDESC_PV, (local > 0 || kk > 0) ? 1u : 0u);
          }
          umma_commit(L.p_empty(pb, h));
        }
        __syncwarp();
        if (h > 0) ++nh1;
      }
      if (lane == 0) umma_commit(L.v_empty(s));
      __syncwarp();
      last_pv = gp;
      return true;
    };
    for (int it = it_begin; it < it_end && ok; ++it, ++n_it) {
      const AttnItem item = fetch_item(s_items, prm.items, it, it_begin);
      const int qb = n_it % C::Q_BUFS, ob = n_it & 1;
      const int ctx = item.ctx;
      const int n_r = item.n_r;
      const int ct = ceil_div(ctx, kKT);
      if (!wait_warp(L.q_full(qb), (n_it / C::Q_BUFS) & 1, cx)) { ok = false; break; }
      // O^T buffer ob was last read by the epilogue of item n_it - 2
      if (n_it >= 2 && !wait_warp(L.o_free(ob), ((n_it >> 1) - 1) & 1, cx)) { ok = false; break; }
      const uint32_t qa = L.q(qb);
      const int ntiles = item.te - item.tb;
      int prev_vis = 0;
      for (int l = 0; l < ntiles; ++l, ++g) {
        const int s = g % kStages;
        const int sb = g & 1;
        if (!wait_warp(L.k_full(s), (g / kStages) & 1, cx)) { ok = false; break; }
        if (g >= 2 && !wait_warp(L.s_free(sb), ((g >> 1) - 1) & 1, cx)) { ok = false; break; }
        if (lane == 0) {
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < kD / 16; ++kk) {
            // A = K tile (M = 128 keys, K-major), B = Q (N = query rows, K-major); K = 16 dims
            const uint64_t a = smem_desc(L.stage(s) + (kk >> 2) * kTileHalf + (kk & 3) * 32, 16, 1024, SW_128B);
            const uint64_t b = smem_desc(qa + (kk >> 2) * C::Q_CB + (kk & 3) * 32, 16, 1024, SW_128B);
            umma_bf16(tmem + C::TMEM_S + sb * NT, a, b, IDESC_QK, kk > 0 ? 1u : 0u);
          }
          umma_commit(L.s_full(sb));
          umma_commit(L.k_empty(s));
          if (l == ntiles - 1) umma_commit(L.q_empty(qb));
        }
        __syncwarp();
        if (l >= 1 && !issue_pv(g - 1, l - 1, prev_vis, ob, item.ni * G)) { ok = false; break; }
        prev_vis = visible_keys(item.tb + l, ct, ctx, n_r);
      }
      if (!ok) break;
      if (!issue_pv(g - 1, ntiles - 1, prev_vis, ob, item.ni * G)) { ok = false; break; }
    }
    if (lane == 0 && last_pv >= 0)
      drain_bar(L.p_empty(last_pv % C::P_BUFS, 0), (last_pv / C::P_BUFS) & 1, prm.err);
    if (lane == 0 && nh1 > 0) drain_bar(L.p_empty(0, 1), (nh1 - 1) & 1, prm.err);
  } else if (warp >= kSoftmaxWarp0) {
    // ------------------------------------------------------------- softmax / epilogue
    const int sw = warp & 3;                          // TMEM lane quadrant
    const int wg = (warp - kSoftmaxWarp0) >> 2;       // softmax warpgroup: rows of its own
    const int kl = sw * 32 + lane;                    // key of this thread within a tile (= d in O^T)
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(sw * 32) << 16);
    const float sl2 = prm.scale_log2;
    float* my_mref = s_mref + sw * NT;
    float* my_alpha = s_alpha + sw * NT;
    float* my_mtrue = reinterpret_cast<float*>(bp + C::OFF_MT) + sw * NT;
    // [2][WGS][4]: this warpgroup's flags
    int* s_over = reinterpret_cast<int*>(bp + C::OFF_OVER) + wg * 4;
    // exchange counters of this warpgroup (xw: one per tile it holds rows in; ep: one
    // per item it holds rows in)
    // na: tiles this warpgroup wrote its half of P^T for (the 128-column tile's P
    // barriers of a half count those tiles)
    int g = 0, n_it = 0, n_stg = 0, n_sf = 0, n_ov = 0, n_xw = 0, n_ep = 0, na = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it, ++n_it) {
      const AttnItem item = fetch_item(s_items, prm.items, it, it_begin);
      const int ctx = item.ctx;
      const int c0 = item.c0;
      const int n_r = item.n_r;
      const int ct = ceil_div(ctx, kKT);
      const int nq = item.ni * G;                     // valid query rows (columns)
      const int ng = (nq + 31) >> 5;                  // 32-row groups holding valid rows
      const int nc8 = (nq + 7) >> 3;                  // 8-row chunks holding valid rows
      const int gbeg = wg * C::G32_WG;                // this warpgroup's 32-row groups
      const int gend = min(ng, gbeg + C::G32_WG);     // (none when gend <= gbeg)
      const uint32_t t_o = t_lane + C::TMEM_O + (n_it & 1) * NT;  // this item's O^T
      // per-row state, lane-distributed: row = gi*32 + lane
      // per-row sums of the bf16 P the PV product multiplies, so that the weights
      // applied to V are exactly the normalised rounded P (a rounding of a dominant
      // P cancels in O / l; the lse then carries it, |error| <= ln(1 + 2^-8))
      float mref[C::G32], lacc[C::G32];
#pragma unroll
      for (int gi = 0; gi < C::G32; ++gi) { mref[gi] = -INFINITY; lacc[gi] = 0.f; }
      const int ntiles = item.te - item.tb;
      for (int l = 0; l < ntiles; ++l, ++g) {
        const int t = item.tb + l;
        const int sb = g & 1;
        if (!wait_warp(L.s_full(sb), (g >> 1) & 1, cx)) { ok = false; break; }
        tc_fence_after();
        if constexpr (NT == 128) {
        // NT = 128: passes over the 32-column groups of S^T in rolled loops (the fully
        // unrolled 128-column code outgrows the instruction cache next to the other
        // roles' loops).
        // Keys of this tile visible to column (query row) n: cache tile -> key < ctx;
        // block tile -> block row b visible to n iff b < n_r and n >= (b - i0) * G.
        const bool cache_tile = t < ct;
        const bool key_dead = cache_tile && (t * kKT + kl >= ctx);
        int nmin = 0;
        if (!cache_tile) {
          const int b = (t - ct) * kKT + kl;          // block row of this key
          nmin = b < n_r ? (b - item.i0) * G : 0x7fffffff;
        }
        const uint32_t s_col = t_lane + C::TMEM_S + sb * NT;
        const int pb = g % C::P_BUFS;
        const uint32_t prow = L.pbuf(pb);
        if (gend <= gbeg) {
          // no query row of the item in this warpgroup: release S^T of the tile (its
          // half of P^T takes no part in this item's products)
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(L.s_free(sb));
          continue;
        }
        const int xslot = n_xw & 1;
        float* wmax = s_wmax + xslot * 4 * NT;
        // ---- fast path (items with at most 32 query rows -- warpgroup 0 alone --, every
        // tile but the first): the references rarely move once a tile has set them, so P
        // is computed in one pass against the current references; the 2^8 test that
        // would move a reference is taken per key (a key above its row's reference + 8
        // is exactly a tile maximum above it), and only if some key of some warp passes
        // it does the tile take the full path below, overwriting this P -- so P, the
        // sums and the references are those of the full path bit for bit.  P is formed
        // in registers while the last product of this half may still read the single P
        // buffer; only the stores wait.  (The epilogue's staging reads of the P buffer
        // were waited for at the first tile's exchange.)  Items with more rows keep the
        // two passes: there the max pass is what overlaps the previous product.
        bool full = l == 0 || ng > 1;
        const bool tried_fast = !full;  // the fast pass used this tile's xw exchange
        if (!full) {
          float lnew0 = lacc[0];
          bool over = false;
          uint32_t pk[16];
          {
            float v[32];
            tmem_ld32(s_col, v);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              v[k] = (key_dead || k < nmin) ? -INFINITY : v[k];
              over = over || (v[k] * sl2 > my_mtrue[k] + 8.0f);
            }
#pragma unroll
            for (int h = 0; h < 16; ++h) {
              const int k = 2 * h;
              const float p0 = fast_exp2(fmaf(v[k], sl2, -my_mref[k]));
              const float p1 = fast_exp2(fmaf(v[k + 1], sl2, -my_mref[k + 1]));
              __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
              v[k] = __low2float(b2);
              v[k + 1] = __high2float(b2);
              pk[h] = *reinterpret_cast<uint32_t*>(&b2);
            }
            lnew0 += transpose_reduce<false>(v, lane);
          }
          // the single P buffer: the last product of this half must be done with it
          if (na >= 1 && !wait_warp(L.p_empty(0, wg), (na - 1) & 1, cx)) {
            ok = false;
            break;
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            if (q < nc8) {
              const uint32_t off = sw128_off(kl, q);
              st_shared_v4(prow + off, make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2],
                                                  pk[4 * q + 3]));
            }
          }
          // one flag per warp, exchanged once: does any reference move?
          over = __any_sync(0xffffffffu, over);
          if (lane == 0) s_over[xslot * 4 * C::WGS + sw] = over ? 1 : 0;
          __syncwarp();
          if (lane == 0) mbar_arrive(L.xw(wg, xslot));
          if (!wait_warp(L.xw(wg, xslot), (n_xw >> 1) & 1, cx)) { ok = false; break; }
          ++n_xw;
          const int* ov = s_over + xslot * 4 * C::WGS;
          full = (ov[0] | ov[1] | ov[2] | ov[3]) != 0;
          if (!full) {
            lacc[0] = lnew0;
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(L.s_free(sb));
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) mbar_arrive(L.p_full(pb, wg));
            ++na;
            continue;  // next tile
          }
        }
        // ---- full path, pass 1: tile max per row of this warpgroup's groups (warp
        // transpose-reduce), then across its 4 warps (on xw, or on xs when a fast pass
        // already used xw for this tile)
#pragma unroll 1
        for (int gi = gbeg; gi < gend; ++gi) {
          float v[32];
          tmem_ld32(s_col + gi * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k)
            v[k] = (key_dead || gi * 32 + k < nmin) ? -INFINITY : v[k];
          wmax[sw * NT + gi * 32 + lane] = transpose_reduce<true>(v, lane) * sl2;
        }
        __syncwarp();
        // this warpgroup's share of the P buffer doubles as its epilogue's staging area:
        // those bulk reads must be done before any of its warps passes this exchange and
        // writes P
        if (sw == 0 && lane == 0) bulk_wait_read_all();
        if (!tried_fast) {
          if (lane == 0) mbar_arrive(L.xw(wg, xslot));
          if (!wait_warp(L.xw(wg, xslot), (n_xw >> 1) & 1, cx)) { ok = false; break; }
          ++n_xw;
        } else {
          if (lane == 0) mbar_arrive(L.xs(wg, n_ov & 1));
          if (!wait_warp(L.xs(wg, n_ov & 1), (n_ov >> 1) & 1, cx)) { ok = false; break; }
          ++n_ov;
        }
        bool need_any = false;
#pragma unroll
        for (int gi = 0; gi < C::G32; ++gi) {
          if (gi < gbeg) continue;
          if (gi >= gend) break;
          const int n = gi * 32 + lane;
          const float tm = fmaxf(fmaxf(wmax[n], wmax[NT + n]), fmaxf(wmax[2 * NT + n], wmax[3 * NT + n]));
          float alpha = 1.f;
          if (tm > mref[gi] + 8.0f) {        // lazy: move the reference only on a 2^8 jump
            alpha = (mref[gi] == -INFINITY) ? 0.f : fast_exp2(mref[gi] - tm);
            mref[gi] = tm;
            lacc[gi] *= alpha;
            need_any = true;
          }
          my_mref[n] = mref[gi] == -INFINITY ? 0.f : mref[gi];
          my_mtrue[n] = mref[gi];
          my_alpha[n] = alpha;
        }
        const bool rescale = __any_sync(0xffffffffu, need_any) && l > 0;
        __syncwarp();
        // the single P buffer, and with it this half's O^T columns: the half's last
        // product must be done
        if (na >= 1 && !wait_warp(L.p_empty(0, wg), (na - 1) & 1, cx)) {
          ok = false;
          break;
        }
        if (rescale) {
          tc_fence_after();
#pragma unroll 1
          for (int c = gbeg; c < gend; ++c) {
            float o[32];
            tmem_ld32(t_o + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= my_alpha[c * 32 + k];
            tmem_st32(t_o + c * 32, o);
          }
          tmem_wait_st();
        }
        // ---- pass 2: P^T row of this key, exp2(s * scale - mref[n]) in bf16, and the
        // per-row partial sums over this warp's 32 keys.  Only the 8-column chunks
        // holding valid rows are written: padding columns of P^T are left as they are
        // -- they only reach their own columns of O^T, which are never stored.
#pragma unroll 1
        for (int gi = gbeg; gi < gend; ++gi) {
          float v[32];
          tmem_ld32(s_col + gi * 32, v);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k)
            v[k] = (key_dead || gi * 32 + k < nmin) ? -INFINITY : v[k];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const int n8 = gi * 4 + q;
            if (n8 >= nc8) break;
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const int k = q * 8 + 2 * h;
              const int n = gi * 32 + k;
              const float p0 = fast_exp2(fmaf(v[k], sl2, -my_mref[n]));
              const float p1 = fast_exp2(fmaf(v[k + 1], sl2, -my_mref[n + 1]));
              __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
              v[k] = __low2float(b2);
              v[k + 1] = __high2float(b2);
              w[h] = *reinterpret_cast<uint32_t*>(&b2);
            }
            const uint32_t off = (n8 >> 3) * (kKT * 128) + sw128_off(kl, n8 & 7);
            st_shared_v4(prow + off, make_uint4(w[0], w[1], w[2], w[3]));
          }
          const float rs = transpose_reduce<false>(v, lane);
#pragma unroll
          for (int i = 0; i < C::G32; ++i)
            if (i == gi) lacc[i] += rs;
        }
        // S^T of this tile is read: its TMEM columns may take tile g + 2
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(L.s_free(sb));
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(L.p_full(pb, wg));
        ++na;
        } else {
        float s[NT];
#pragma unroll
        for (int c = 0; c < NT / 32; ++c) {
          float tmp[32];
          tmem_ld32(t_lane + C::TMEM_S + sb * NT + c * 32, tmp);
#pragma unroll
          for (int k = 0; k < 32; ++k) s[c * 32 + k] = tmp[k];
        }
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(L.s_free(sb));
        // ---- visibility: cache tile -> key < ctx; block tile -> block row b <= bi(row)
        if (t < ct) {
          if (t * kKT + kl >= ctx) {
#pragma unroll
            for (int n = 0; n < NT; ++n) s[n] = -INFINITY;
          }
        } else {
          const int b = (t - ct) * kKT + kl;          // block row of this key
          // row n sees key b iff b < n_r and b <= i0 + n / G  <=>  n >= (b - i0) * G
          const int nmin = b < n_r ? (b - item.i0) * G : 0x7fffffff;
#pragma unroll
          for (int n = 0; n < NT; ++n) s[n] = (n >= nmin) ? s[n] : -INFINITY;
        }
        // ---- tile max per row: warp transpose-reduce, then across the 4 warps
        float* wmax = s_wmax + (g & 1) * 4 * NT;
#pragma unroll
        for (int gi = 0; gi < C::G32; ++gi) {
          if (gi >= ng) break;                        // groups of padding rows only
          float v[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = s[gi * 32 + k];
          wmax[sw * NT + gi * 32 + lane] = transpose_reduce<true>(v, lane) * sl2;
        }
        __syncwarp();
        // P buffers double as the epilogue's staging area: its bulk reads must be done
        // before any warp passes this exchange and writes P
        if (warp == kSoftmaxWarp0 && lane == 0) bulk_wait_read_all();
        if (lane == 0) mbar_arrive(L.xw(0, g & 1));
        if (!wait_warp(L.xw(0, g & 1), (g >> 1) & 1, cx)) { ok = false; break; }
        bool need_any = false;
#pragma unroll
        for (int gi = 0; gi < C::G32; ++gi) {
          if (gi >= ng) break;
          const int n = gi * 32 + lane;
          const float tm = fmaxf(fmaxf(wmax[n], wmax[NT + n]), fmaxf(wmax[2 * NT + n], wmax[3 * NT + n]));
          float alpha = 1.f;
          if (tm > mref[gi] + 8.0f) {        // lazy: move the reference only on a 2^8 jump
            alpha = (mref[gi] == -INFINITY) ? 0.f : fast_exp2(mref[gi] - tm);
            mref[gi] = tm;
            lacc[gi] *= alpha;
            need_any = true;
          }
          my_mref[n] = mref[gi] == -INFINITY ? 0.f : mref[gi];
          my_alpha[n] = alpha;
        }
        const bool rescale = __any_sync(0xffffffffu, need_any) && l > 0;
        __syncwarp();
        // P buffer of this tile must be free: PV(g - P_BUFS) done
        const int pb = g % C::P_BUFS;
        if (g >= C::P_BUFS &&
            !wait_warp(L.p_empty((g - C::P_BUFS) % C::P_BUFS, 0), ((g - C::P_BUFS) / C::P_BUFS) & 1, cx)) {
          ok = false;
          break;
        }
        if (rescale) {
          // O^T must hold PV(g-1) before its columns are rescaled
          if (C::P_BUFS > 1 &&
              !wait_warp(L.p_empty((g - 1) % C::P_BUFS, 0), ((g - 1) / C::P_BUFS) & 1, cx)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll 1
          for (int c = 0; c < NT / 32; ++c) {
            float o[32];
            tmem_ld32(t_o + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= my_alpha[c * 32 + k];
            tmem_st32(t_o + c * 32, o);
          }
          tmem_wait_st();
        }
        // ---- P^T row of this key: exp2(s * scale - mref[n]) in bf16
        const uint32_t prow = L.pbuf(pb);
        // only the chunks holding valid rows: padding columns of P^T are left as they
        // are -- they only reach their own columns of O^T, which are never stored
#pragma unroll
        for (int n8 = 0; n8 < NT / 8; ++n8) {
          if (n8 >= nc8) break;
          uint32_t w[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const int n = n8 * 8 + 2 * h;
            const float p0 = fast_exp2(fmaf(s[n], sl2, -my_mref[n]));
            const float p1 = fast_exp2(fmaf(s[n + 1], sl2, -my_mref[n + 1]));
            __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
            s[n] = __low2float(b2);
            s[n + 1] = __high2float(b2);
            w[h] = *reinterpret_cast<uint32_t*>(&b2);
          }
          uint32_t off;
          if (NT == 32) off = sw64_off(kl, n8);
          else off = (n8 >> 3) * (kKT * 128) + sw128_off(kl, n8 & 7);
          st_shared_v4(prow + off, make_uint4(w[0], w[1], w[2], w[3]));
        }
        tc_fence_before();
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(L.p_full(pb, 0));
        // ---- per-row partial sums over this warp's 32 keys
#pragma unroll
        for (int gi = 0; gi < C::G32; ++gi) {
          if (gi >= ng) break;
          float v[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) v[k] = s[gi * 32 + k];
          lacc[gi] += transpose_reduce<false>(v, lane);
        }
        }
      }
      if (!ok) break;
      // ---- epilogue of this warpgroup's rows: l across its warps, then O^T / l
      if (gend > gbeg) {
        float* lsum = s_lsum;
#pragma unroll
        for (int gi = 0; gi < C::G32; ++gi)
          if (gi >= gbeg && gi < gend) lsum[sw * NT + gi * 32 + lane] = lacc[gi];
        __syncwarp();
        if (lane == 0) mbar_arrive(L.ep(wg, n_ep & 1));
        if (!wait_warp(L.ep(wg, n_ep & 1), (n_ep >> 1) & 1, cx)) { ok = false; break; }
        ++n_ep;
        // the item's last product of this warpgroup's rows is complete
        if constexpr (NT == 128) {
          if (!wait_warp(L.p_empty(0, wg), (na - 1) & 1, cx)) { ok = false; break; }
        } else {
          const int gl = g - 1;
          if (!wait_warp(L.p_empty(gl % C::P_BUFS, 0), (gl / C::P_BUFS) & 1, cx)) { ok = false; break; }
        }
        tc_fence_after();
        const bool split = item.nsplit > 1;
        // Row n = gi*32 + lane: 1/l, computed once per row and broadcast below.
        float inv_l[C::G32];
#pragma unroll
        for (int gi = 0; gi < C::G32; ++gi) {
          const int n = gi * 32 + lane;
          inv_l[gi] = 0.f;
          if (gi >= gbeg && gi < gend && n < nq) {
            const float lt = lsum[n] + lsum[NT + n] + lsum[2 * NT + n] + lsum[3 * NT + n];
            inv_l[gi] = lt > 0.f ? 1.f / lt : 0.f;
            if (sw == 0) {  // warp 0 of the warpgroup writes the lse
              const float lse_v = (mref[gi] + log2f(lt)) * 0.69314718055994530942f;
              if (split)
                prm.ws_lse[(long long)item.slot * kKT + n] = lse_v;  // this piece's slot
              else
                prm.lse[((long long)c0 + item.i0 + n / G) * prm.Hq + item.kvh * G + n % G] = lse_v;
            }
          }
        }
        // O^T / l -> row-major rows in this warpgroup's share of the (now idle) P
        // buffers, STG_ROWS rows per pass; one thread then writes each pass out with bulk
        // copies: a slot of ws_o is one contiguous run, an output block row is G
        // consecutive heads.
        float* stg = reinterpret_cast<float*>(bp + C::OFF_P + wg * C::STG_BYTES_WG);
        const int rb = gbeg * 32, re = min(nq, gend * 32);
        for (int p0 = rb; p0 < re; p0 += C::STG_ROWS) {
          const int p1 = min(re, p0 + C::STG_ROWS);
          if (p0 > rb) {  // the previous pass must have been read out of the buffers
            if (!wait_warp(L.stg_free(wg), n_sf & 1, cx)) { ok = false; break; }
            ++n_sf;
          }
#pragma unroll
          for (int c = 0; c < C::G32; ++c) {
            if (c * 32 >= p1 || c * 32 < p0) continue;   // chunk outside this pass (uniform)
            float o[32];
            tmem_ld32(t_o + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) {
              const float il = __shfl_sync(0xffffffffu, inv_l[c], k);
              if (c * 32 + k < p1) stg[(c * 32 + k - p0) * kD + kl] = o[k] * il;
            }
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(L.stg_full(wg));
          if (sw == 0 && lane == 0) {
            if (!wait_bar(L.stg_full(wg), n_stg & 1, cx)) {
              ok = false;
            } else {
              const uint32_t src = L.pbuf(0) + wg * C::STG_BYTES_WG;
              if (split) {
                bulk_store_s2g(prm.ws_o + ((long long)item.slot * kKT + p0) * kD, src,
                               (uint32_t)(p1 - p0) * kD * 4);
              } else {
                for (int n = p0; n < p1;) {
                  const int b = n / G, h0 = n % G;
                  const int run = min(p1 - n, G - h0);
                  bulk_store_s2g(prm.out + (((long long)c0 + item.i0 + b) * prm.Hq + item.kvh * G + h0) * kD,
                                 src + (uint32_t)(n - p0) * kD * 4, (uint32_t)run * kD * 4);
                  n += run;
                }
              }
              bulk_commit();
              if (p1 < re) {
                bulk_wait_read_all();
                mbar_arrive(L.stg_free(wg));
              }
            }
          }
          ++n_stg;
          if (!__all_sync(0xffffffffu, ok)) break;
        }
        if (!ok) break;
        // lsum is rewritten by the next item only after every warp of the warpgroup
        // passed its ep barrier and the next tile's cross-warp barrier; the latter
        // orders it.
      }
      // O^T of this item is read: its TMEM columns may take item n_it + 2
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(L.o_free(n_it & 1));
    }
    if (sw == 0 && lane == 0) bulk_wait_all();  // output writes complete
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------- host side
namespace {

using EncodeFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                              const cuuint64_t*, const cuuint32_t*, const cuuint32_t*,
                              CUtensorMapInterleave, CUtensorMapSwizzle, CUtensorMapL2promotion,
                              CUtensorMapFloatOOBfill);

EncodeFn get_encode() {
  // the driver entry point is the same for every device: looked up once per process
  static const EncodeFn fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      return reinterpret_cast<EncodeFn>(p);
    return static_cast<EncodeFn>(nullptr);
  }();
  return fn;
}

// 4-D map over a [n_pages, P, Hkv, 128] bf16 cache; box = 64 dims x 1 head x box_rows tokens.
bool make_cache_map(CUtensorMap* m, const void* base, int n_pages, int P, int Hkv, int box_rows) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)kD, (cuuint64_t)Hkv, (cuuint64_t)P, (cuuint64_t)n_pages};
  cuuint64_t str[3] = {(cuuint64_t)kD * 2, (cuuint64_t)Hkv * kD * 2, (cuuint64_t)P * Hkv * kD * 2};
  cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, str, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D map over packed block rows [max_rows, Hkv, 128] bf16; box = 64 dims x 1 head x
// kChunkRows rows (rows past max_rows read as zero).
bool make_rows_map(CUtensorMap* m, const void* base, int max_rows, int Hkv) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t dims[3] = {(cuuint64_t)kD, (cuuint64_t)Hkv, (cuuint64_t)max_rows};
  cuuint64_t str[2] = {(cuuint64_t)kD * 2, (cuuint64_t)Hkv * kD * 2};
  cuuint32_t box[3] = {64, 1, (cuuint32_t)kChunkRows};
  cuuint32_t estr[3] = {1, 1, 1};
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, str, box, estr,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

// bf16 tiled map with 128-byte swizzle: rank dims (innermost first), byte strides of
// dims 1..rank-1, box extents.
bool encode_bf16_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, rank, const_cast<void*>(base), d, st, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool encode_f32_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box) {
  EncodeFn enc = get_encode();
  if (!enc) return false;
  cuuint64_t d[5], st[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
    if (i + 1 < rank) st[i] = strides[i];
  }
  return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, rank, const_cast<void*>(base), d, st, bx, es,
             CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

namespace {

template <int NT>
bool configure() {
  static PerDevice<bool> done;
  return once_per_device(done, false, [] {
    return cudaFuncSetAttribute(verify_attn_gqa_kernel<NT>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                Cfg<NT>::SMEM_BYTES) == cudaSuccess;
  });
}

}  // namespace

int query_tile(int Hq, int Hkv, int max_block_rows) {
  const int G = Hq / Hkv;
  const long long rows = (long long)G * (max_block_rows > 0 ? max_block_rows : 1);
  if (rows <= 32) return 32;
  if (rows <= 64) return 64;
  return 128;
}

int launch_kernel(int nt, const void* q, const void* k_new, const void* v_new, const void* k_cache,
                  const void* v_cache, int n_pages, const int32_t* page_table, int max_pages,
                  const int32_t* ctx_len, const int32_t* cu_seqlens, int B, int max_rows, int Hq,
                  int Hkv, int page_size, float scale, const AttnItem* items,
                  const int* item_begin, int grid, float* out, float* lse, float* ws_o,
                  float* ws_lse, cudaStream_t stream) {
  Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.k_new = static_cast<const __nv_bfloat16*>(k_new);
  prm.v_new = static_cast<const __nv_bfloat16*>(v_new);
  prm.k_cache = static_cast<const __nv_bfloat16*>(k_cache);
  prm.v_cache = static_cast<const __nv_bfloat16*>(v_cache);
  prm.page_table = page_table;
  prm.ctx_len = ctx_len;
  prm.cu_seqlens = cu_seqlens;
  prm.items = items;
  prm.item_begin = item_begin;
  prm.out = out;
  prm.lse = lse;
  prm.ws_o = ws_o;
  prm.ws_lse = ws_lse;
  prm.err = device_error_word();
  prm.max_pages = max_pages;
  prm.B = B;
  prm.Hq = Hq;
  prm.Hkv = Hkv;
  prm.page_size = page_size;
  prm.log2_page = 0;
  while ((1 << prm.log2_page) < page_size) ++prm.log2_page;
  prm.max_rows = max_rows;
  prm.n_pages = n_pages;
  prm.scale_log2 = scale * 1.4426950408889634f;
  CUtensorMap tk, tv, tkn, tvn;
  if (!make_cache_map(&tk, k_cache, n_pages, page_size, Hkv, page_size < kKT ? page_size : kKT))
    return DSPARK_ECUDA;
  if (!make_cache_map(&tv, v_cache, n_pages, page_size, Hkv, kChunkRows)) return DSPARK_ECUDA;
  if (!make_rows_map(&tkn, k_new, max_rows, Hkv)) return DSPARK_ECUDA;
  if (!make_rows_map(&tvn, v_new, max_rows, Hkv)) return DSPARK_ECUDA;
  switch (nt) {
    case 32:
      if (!configure<32>()) return DSPARK_ECUDA;
      if (launch_pdl(verify_attn_gqa_kernel<32>, dim3(grid), dim3(Cfg<32>::THREADS), Cfg<32>::SMEM_BYTES,
                     stream, tk, tv, tkn, tvn, prm) != cudaSuccess)
        return DSPARK_ECUDA;
      break;
    case 64:
      if (!configure<64>()) return DSPARK_ECUDA;
      if (launch_pdl(verify_attn_gqa_kernel<64>, dim3(grid), dim3(Cfg<64>::THREADS), Cfg<64>::SMEM_BYTES,
                     stream, tk, tv, tkn, tvn, prm) != cudaSuccess)
        return DSPARK_ECUDA;
      break;
    default:
      if (!configure<128>()) return DSPARK_ECUDA;
      if (launch_pdl(verify_attn_gqa_kernel<128>, dim3(grid), dim3(Cfg<128>::THREADS), Cfg<128>::SMEM_BYTES,
                     stream, tk, tv, tkn, tvn, prm) != cudaSuccess)
        return DSPARK_ECUDA;
      break;
  }
  return DSPARK_OK;
}

}  // namespace gqa
}  // namespace attn
}  // namespace dspark
