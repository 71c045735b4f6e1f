// Varlen verify attention, latent-KV shape: 128 query heads share one 576-dim
// latent key per token, whose first 512 dims are also its value.
//
// What it computes ("DFlash 到 DSpark in SGLang", section "Ragged verify under
// full CUDA graphs": each packed verify token attends only to its own request's
// KV, causal inside the block): packed row cu_seqlens[r] + i, head h attends to the
// ctx_len[r] committed latent keys of request r (paged) and to block rows 0..i of
// its own segment; o = softmax(scale q.K^T) K[:, :512], lse = log-sum-exp.
//
// Why a two-CTA cluster: 128 rows x 512 fp32 of O fill the whole 512-column TMEM of
// one SM, leaving nothing for the scores.  So one work item (one block row of one
// request = its 128 heads, against a range of 64-key tiles) runs on a cluster of two
// CTAs, and CTA rho owns value dims 256 rho .. 256 rho + 255:
//   * the QK^T reduction is split the same way: CTA rho multiplies dims
//     256 rho .. +255 (its own value columns) and rope dims 512 + 32 rho .. +31.
//     It loads only those 5 of the 9 64-wide column blocks of a key tile;
//   * the two partial score tiles, scaled to the log2 domain, are swapped through
//     distributed shared memory in fp32 and added; fp32 addition commutes, so both
//     CTAs hold bit-identical scores and run the identical softmax (same P, max and
//     sum), and the exchange adds no rounding to the scores.  (fp16 partials erred
//     by 2^-11 of the partial's magnitude, up to 2^-6 log2 units at peaked scores,
//     beyond the output tolerance; 24-bit fixed-point ones were exact enough but
//     their packing on the exchange warps' serial path cost more than the bytes it
//     saved);
//   * Q (this CTA's 288 dims) and P sit in TMEM and are the A operand of the MMAs,
//     so each product reads only the key tile (B) from shared memory.
//
//   S_rho [128 heads x 64 keys] = Q_rho . K_rho^T                 (tcgen05, TMEM)
//   x = scale' S_0 + scale' S_1 (exchanged, fp32); P = exp2(x - m)      (SFU)
//   O_rho [128 x 256] += P . K[:, 256 rho .. 256 rho + 255]       (tcgen05, TMEM)
//
// The swap is the narrow point: with both CTAs sending at once and the key tiles
// streaming in, the SM-to-SM network moves only about 7-14 bytes per clock each way.
// Dedicated exchange warps read S from TMEM (releasing it for the next tile's QK^T at
// once), keep their own scaled partial in registers, send it with st.async, whose
// bytes complete on the receiver's mbarrier (no thread waits on a cluster-scope
// fence), wait for the peer's partial, and write the fp32 sum in place of it in the
// exchange slot; the softmax reads the sums from shared memory.
//
// TMEM columns: O [0, 256), S [256, 320), P [320, 352), Q [352, 496).
// Shared memory: a 4-stage ring of key tiles (5 blocks x 64 keys, 40 KB) and two
// exchange slots of 32 KB (the peer's fp32 partials, then the sums in their place).
// Warp roles: 0 TMA producer (a 4-stage ring of key tiles), 1 MMA issuer (one lane)
// that first zeroes the key rows past the visible range of a partial tile (value
// rows met by a zero probability must be finite), 2-5 softmax and epilogue, 6-9
// score exchange; in both groups thread = query head = TMEM lane.  Every wait is
// bounded in time; on expiry the CTA raises DSPARK_DEVERR_WAIT_TIMEOUT and leaves
// its loops, and the peer's waits then expire as well.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"
#include "common.cuh"
#include "ptx.cuh"

namespace dspark {
namespace attn {
namespace mla {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kRows = 128;       // query heads = UMMA M = TMEM lanes
constexpr int kNK = kKeyTile;    // keys per tile
constexpr int kDqk = 576;
constexpr int kDv = 512;
constexpr int kHalf = 256;       // value dims of one CTA
constexpr int kCBs = 5;          // 64-wide column blocks one CTA loads per key tile
constexpr int kCBBytes = kNK * 128;
constexpr int kStageBytes = kCBs * kCBBytes;
constexpr int kStages = 4;
constexpr int kQKSteps = 18;     // 288 dims / 16
// Partial score exchange: a row is 64 fp32 values (256 B); 16-byte piece c of row m
// sits at piece (c & 8) | ((c ^ m) & 7), which keeps 8 consecutive rows on distinct
// banks.
constexpr int kXRow = 256;
constexpr int kXBytes = kRows * kXRow;
constexpr int kChunkRows = 16;   // block-row box
constexpr int kProdWarp = 0;
constexpr int kMmaWarp = 1;
constexpr int kSoftmaxWarp0 = 2;
constexpr int kExchWarp0 = 6;
constexpr int kThreads = 10 * 32;
constexpr int OFF_STAGE = 0;
constexpr int OFF_X = OFF_STAGE + kStages * kStageBytes;
// two exchange slots: the peer's partials arrive there, the sums replace them
constexpr int OFF_BAR = OFF_X + 2 * kXBytes;
// kv_full[S], kv_empty[S], s_full, s_free, p_full, p_empty, q_full, x_full[2], xc,
// sum_full[2]
constexpr int N_BARS = 2 * kStages + 10;
constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
constexpr uint32_t TMEM_O = 0, TMEM_S = 256, TMEM_P = 320, TMEM_Q = 352;
constexpr uint32_t TMEM_COLS = 512;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(TMEM_Q + kQKSteps * 8 <= TMEM_COLS, "tensor memory budget");
static_assert(kStageBytes % 1024 == 0 && kXBytes % 16 == 0, "alignment");

struct Ctx {
  volatile int* abort_flag;
  unsigned int* err;
};

template <bool CLUSTER>
__device__ __forceinline__ bool try_wait(uint32_t bar, uint32_t parity) {
  return CLUSTER ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity);
}

// Bounded wait; false if this CTA is aborting.  CLUSTER: the phase was completed by
// arrivals of the peer CTA, whose stores must be visible afterwards.
template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctx& cx) {
  if (try_wait<CLUSTER>(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (try_wait<CLUSTER>(bar, parity)) return true;
    if ((++n & 31u) == 0) {
      if (*cx.abort_flag) return false;
      if (globaltimer_ns() - t0 > kWaitLimitNs) {
        *cx.abort_flag = 1;
        raise_error(cx.err, DSPARK_DEVERR_WAIT_TIMEOUT);
        return false;
      }
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

template <bool CLUSTER = false>
__device__ __forceinline__ bool wait_warp(uint32_t bar, uint32_t parity, const Ctx& cx) {
  const bool ok = wait_bar<CLUSTER>(bar, parity, cx);
  return __all_sync(0xffffffffu, ok);
}

__device__ __forceinline__ uint32_t sw128_off(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// Byte offset of 16-byte piece c (0..15) of an exchange row of head m.
__device__ __forceinline__ uint32_t x_piece(int c, int m) {
  return static_cast<uint32_t>(((c & 8) | ((c ^ m) & 7)) << 4);
}


__device__ __forceinline__ void st_shared_v4(uint32_t addr, uint4 v) {
  asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w)
               : "memory");
}
__device__ __forceinline__ float4 ld_shared_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
               : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ uint4 ldg_nc_v4(const void* p) {
  uint4 v;
  asm volatile("ld.global.nc.v4.b32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
               : "l"(p));
  return v;
}
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

struct Layout {
  uint32_t base;
  __device__ uint32_t stage(int s) const { return base + OFF_STAGE + s * kStageBytes; }
  __device__ uint32_t x(int b) const { return base + OFF_X + b * kXBytes; }
  __device__ uint32_t bar(int i) const { return base + OFF_BAR + 8 * i; }
  __device__ uint32_t kv_full(int s) const { return bar(s); }
  __device__ uint32_t kv_empty(int s) const { return bar(kStages + s); }
  __device__ uint32_t s_full() const { return bar(2 * kStages); }
  __device__ uint32_t s_free() const { return bar(2 * kStages + 1); }
  __device__ uint32_t p_full() const { return bar(2 * kStages + 2); }
  __device__ uint32_t p_empty() const { return bar(2 * kStages + 3); }
  __device__ uint32_t q_full() const { return bar(2 * kStages + 4); }
  __device__ uint32_t x_full(int b) const { return bar(2 * kStages + 5 + b); }
  __device__ uint32_t xc() const { return bar(2 * kStages + 7); }
  __device__ uint32_t sum_full(int b) const { return bar(2 * kStages + 8 + b); }
};

// Keys of tile t of a request that a query row can see at all: the cache tile's
// keys below ctx, or the block tile's rows below n_r.
__device__ __forceinline__ int visible_keys(int t, int ct, int ctx, int n_r) {
  const int v = t < ct ? ctx - t * kNK : n_r - (t - ct) * kNK;
  return v < kNK ? v : kNK;
}

// Global 64-wide column block of local block j (0..4) for CTA rho.
__device__ __forceinline__ int global_cb(int j, uint32_t rho) {
  return j < 4 ? static_cast<int>(4 * rho) + j : 8;
}

struct Params {
  const __nv_bfloat16* q;
  const int32_t* page_table;
  const AttnItem* items;
  const int* item_begin;  // [clusters + 1]: cluster c runs items [item_begin[c], item_begin[c+1])
  float* out;
  float* lse;
  float* ws_o;
  float* ws_lse;
  unsigned int* err;
  int max_pages, n_pages, page_size, log2_page;
  float scale_log2;
};

__global__ void __launch_bounds__(kThreads, 1)
    verify_attn_mla_kernel(const __grid_constant__ CUtensorMap tm_c,
                           const __grid_constant__ CUtensorMap tm_n, const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* bp = smem_raw + (base - raw);
  const Layout L{base};
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bp + OFF_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bp + OFF_MISC + 16);
  const Ctx cx{abort_flag, prm.err};
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rho = cluster_ctarank();
  const uint32_t peer = rho ^ 1u;
  const int pair = blockIdx.x >> 1;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kStages; ++s) {
      mbar_init(L.kv_full(s), 1);
      mbar_init(L.kv_empty(s), 1);
    }
    mbar_init(L.s_full(), 1);
    mbar_init(L.s_free(), 4);   // the exchange warps read S
    mbar_init(L.p_full(), 4);
    mbar_init(L.p_empty(), 1);
    mbar_init(L.q_full(), 4);
    // armed (expect_tx) by this CTA's exchange warps, completed by the peer's
    // asynchronous stores
    for (int b = 0; b < 2; ++b) mbar_init(L.x_full(b), 1);
    mbar_init(L.xc(), 4);
    for (int b = 0; b < 2; ++b) mbar_init(L.sum_full(b), 4);  // sums in place
    fence_mbar_init();
  }
  if (warp == kProdWarp && lane == 0) {
    prefetch_tensormap(&tm_c);
    prefetch_tensormap(&tm_n);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // both CTAs' barriers exist before any remote arrive
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_release();
  pdl_wait();  // the work list and the step's inputs come from earlier kernels
  const int it_begin = prm.item_begin[pair];
  const int it_end = prm.item_begin[pair + 1];

  if (warp == kProdWarp) {
    // ------------------------------------------------------------- TMA producer
    // Lane j holds page-table slot win_base + j of the current request.  A tile's
    // copies: lane = (box, local column block); cache boxes follow the page (up to a
    // tile), block-row boxes are 16 rows of the packed buffer.
    const int P = prm.page_size;
    const int lp = prm.log2_page;
    const int box_rows = P < kNK ? P : kNK;
    int g = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it) {
      const AttnItem item = prm.items[it];
      const int ctx = item.ctx;
      const int ct = ceil_div(ctx, kNK);
      const int32_t* ptab = prm.page_table + (long long)item.r * prm.max_pages;
      const int nt = ct + ceil_div(item.n_r, kNK);  // the item's tile range wraps at nt
      int win_base = -1, win_page = 0;
      for (int tt = item.tb; tt < item.te; ++tt, ++g) {
        const int t = tt < nt ? tt : tt - nt;
        const int s = g % kStages;
        if (g >= kStages) {
          ok = wait_warp(L.kv_empty(s), ((g / kStages) - 1) & 1, cx);
          if (!ok) break;
        }
        const uint32_t dst0 = L.stage(s);
        const int vis = visible_keys(t, ct, ctx, item.n_r);  // >= 1
        const int rows_box = t < ct ? box_rows : kChunkRows;
        const int nb = ceil_div(vis, rows_box);
        if (lane == 0) mbar_expect_tx(L.kv_full(s), nb * kCBs * rows_box * 128);
        __syncwarp();
        const int bx = lane / kCBs, j = lane % kCBs;
        if (t < ct) {
          const int slot0 = (t * kNK) >> lp;
          const int nslot = ceil_div(kNK, P);
          if (win_base < 0 || slot0 < win_base || slot0 + nslot > win_base + 32) {
            win_base = slot0;
            const int sl = win_base + lane;
            const bool used = (sl << lp) < ctx;
            int pg = 0;
            if (used) {
              pg = sl < prm.max_pages ? ptab[sl] : -1;
              if (pg < 0 || pg >= prm.n_pages) {
                raise_error(prm.err, DSPARK_DEVERR_BAD_INPUT);
                pg = -1;  // the box lies outside the map: read as zeros
              }
            }
            win_page = pg;
          }
          const int kg = t * kNK + bx * rows_box;
          const int src_lane = bx < nb ? ((kg >> lp) - win_base) & 31 : 0;
          const int page = __shfl_sync(0xffffffffu, win_page, src_lane);
          if (bx < nb)
            tma_load_3d(dst0 + j * kCBBytes + bx * rows_box * 128, &tm_c, L.kv_full(s),
                        global_cb(j, rho) * 64, kg & (P - 1), page);
        } else {
          const int b0 = (t - ct) * kNK;
          if (bx < nb)
            tma_load_2d(dst0 + j * kCBBytes + bx * kChunkRows * 128, &tm_n, L.kv_full(s),
                        global_cb(j, rho) * 64, item.c0 + b0 + bx * kChunkRows);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(L.kv_full(s));
      }
    }
    // never leave copies in flight
    if (lane == 0) {
      const int first = g - kStages > 0 ? g - kStages : 0;
      for (int gg = first; gg < g; ++gg) drain_bar(L.kv_full(gg % kStages), (gg / kStages) & 1, prm.err);
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    constexpr uint32_t IDESC_QK = idesc_bf16_f32(kRows, kNK, 0, 0);
    constexpr uint32_t IDESC_PV = idesc_bf16_f32(kRows, kHalf, 0, 1);
    int g = 0, n_it = 0, last_pv = -1, last_qk = -1;
    bool ok = true;
    // O += P V for tile gp (local index `local` in its item)
    auto issue_pv = [&](int gp, int local) -> bool {
      if (!wait_warp(L.p_full(), gp & 1, cx)) return false;
      if (lane == 0) {
        tc_fence_after();
        const uint32_t vb = L.stage(gp % kStages);
#pragma unroll
        for (int kk = 0; kk < kNK / 16; ++kk) {
          // A = P (TMEM, 16 keys per step), B = V (N = 256 value dims, MN-major)
          const uint64_t b = smem_desc(vb + kk * 2048, kCBBytes, 1024, SW_128B);
          umma_bf16_ts(tmem + TMEM_O, tmem + TMEM_P + kk * 8, b, IDESC_PV,
                       (local > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(L.p_empty());
        umma_commit(L.kv_empty(gp % kStages));
      }
      __syncwarp();
      last_pv = gp;
      return true;
    };
    for (int it = it_begin; it < it_end && ok; ++it, ++n_it) {
      const AttnItem item = prm.items[it];
      const int ct = ceil_div(item.ctx, kNK);
      const int nt = ct + ceil_div(item.n_r, kNK);  // the item's tile range wraps at nt
      if (!wait_warp(L.q_full(), n_it & 1, cx)) { ok = false; break; }
      const int ntiles = item.te - item.tb;
      for (int l = 0; l < ntiles; ++l, ++g) {
        const int s = g % kStages;
        const uint32_t st = L.stage(s);
        if (!wait_warp(L.kv_full(s), (g / kStages) & 1, cx)) { ok = false; break; }
        const int tt = item.tb + l;
        const int vis = visible_keys(tt < nt ? tt : tt - nt, ct, item.ctx, item.n_r);
        if (vis < kNK) {
          // rows vis..63 of the 5 column blocks, 8 16-byte pieces per row
          const int nz = (kNK - vis) * kCBs * 8;
          for (int idx = lane; idx < nz; idx += 32) {
            const int row = vis + idx / (kCBs * 8), rem = idx % (kCBs * 8);
            st_shared_v4(st + (rem >> 3) * kCBBytes + sw128_off(row, rem & 7), make_uint4(0, 0, 0, 0));
          }
          fence_proxy_async_smem();
        }
        __syncwarp();
        // the single S buffer: the softmax has read S of the previous tile
        if (g >= 1 && !wait_warp(L.s_free(), (g - 1) & 1, cx)) { ok = false; break; }
        if (lane == 0) {
          tc_fence_after();
#pragma unroll
          for (int k = 0; k < kQKSteps; ++k) {
            // A = Q (TMEM), B = key tile (N = 64 keys, K-major); K = 16 dims
            const int lc = k < 16 ? (k >> 2) : 4;
            const int kq = k < 16 ? (k & 3) : static_cast<int>(2 * rho) + (k - 16);
            const uint64_t b = smem_desc(st + lc * kCBBytes + kq * 32, 16, 1024, SW_128B);
            umma_bf16_ts(tmem + TMEM_S, tmem + TMEM_Q + k * 8, b, IDESC_QK, k > 0 ? 1u : 0u);
          }
          umma_commit(L.s_full());
        }
        __syncwarp();
        last_qk = g;
        if (l >= 1 && !issue_pv(g - 1, l - 1)) { ok = false; break; }
      }
      if (!ok) break;
      if (!issue_pv(g - 1, ntiles - 1)) { ok = false; break; }
    }
    // all issued MMAs must finish before TMEM is released (after an abort the last
    // product issued may be a QK^T)
    if (lane == 0 && last_pv >= 0) drain_bar(L.p_empty(), last_pv & 1, prm.err);
    if (lane == 0 && last_qk > last_pv) drain_bar(L.s_full(), last_qk & 1, prm.err);
  } else if (warp >= kSoftmaxWarp0 && warp < kExchWarp0) {
    // ------------------------------------------------------------- softmax / epilogue
    const int sw = warp & 3;                 // TMEM lane quadrant of this warp
    const int m = sw * 32 + lane;            // query head of this thread
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(sw * 32) << 16);
    const uint32_t x_row = static_cast<uint32_t>(m * kXRow);
    int g = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it) {
      const AttnItem item = prm.items[it];
      const int ctx = item.ctx;
      const int n_r = item.n_r;
      const int ct = ceil_div(ctx, kNK);
      const int bi = item.i0;                // the item's block row
      const int row_g = item.c0 + bi;
      // ---- Q: this CTA's 288 dims of head m into TMEM (two bf16 per column)
      {
        const __nv_bfloat16* qrow = prm.q + ((long long)row_g * kRows + m) * kDqk;
        const uint4* qa = reinterpret_cast<const uint4*>(qrow + rho * kHalf);
        const uint4* qr = reinterpret_cast<const uint4*>(qrow + kDv + rho * 32);
#pragma unroll
        for (int b = 0; b < 2; ++b) {
          uint4 v[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) v[i] = ldg_nc_v4(qa + b * 16 + i);
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            float w[32];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              w[4 * i] = __uint_as_float(v[h * 8 + i].x);
              w[4 * i + 1] = __uint_as_float(v[h * 8 + i].y);
              w[4 * i + 2] = __uint_as_float(v[h * 8 + i].z);
              w[4 * i + 3] = __uint_as_float(v[h * 8 + i].w);
            }
            tmem_st32(t_lane + TMEM_Q + b * 64 + h * 32, w);
          }
        }
        uint32_t w16[16];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint4 v = ldg_nc_v4(qr + i);
          w16[4 * i] = v.x; w16[4 * i + 1] = v.y; w16[4 * i + 2] = v.z; w16[4 * i + 3] = v.w;
        }
        tmem_st16u(t_lane + TMEM_Q + 128, w16);
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(L.q_full());
        // warm L2 with the next item's query row
        if (it + 1 < it_end) {
          const AttnItem nx = prm.items[it + 1];
          const char* nq = reinterpret_cast<const char*>(
              prm.q + ((long long)(nx.c0 + nx.i0) * kRows + m) * kDqk);
#pragma unroll
          for (int i = 0; i < 9; ++i) prefetch_l2(nq + i * 128);
        }
      }
      // m_used: reference max of x; l_sum: sum of exp2(x - m_used) (for the lse);
      // l_sumr: the same sum of the bf16 P the PV product multiplies (for O / l, so
      // that the weights applied to V are exactly the normalised rounded P)
      float m_used = -INFINITY, l_sum = 0.f, l_sumr = 0.f;
      const int ntiles = item.te - item.tb;
      const int nt = ct + ceil_div(n_r, kNK);  // the item's tile range wraps at nt
      for (int l = 0; l < ntiles; ++l, ++g) {
        const int t = item.tb + l < nt ? item.tb + l : item.tb + l - nt;
        const int xb = g & 1;
        // ---- x = S * scale * log2(e) = x_0 + x_1, summed in fp32 by the exchange
        // warps (the sum commutes, so both CTAs hold identical bits)
        if (!wait_warp(L.sum_full(xb), (g >> 1) & 1, cx)) { ok = false; break; }
        float s[kNK];
        {
          const uint32_t rp = L.x(xb) + x_row;
#pragma unroll
          for (int c = 0; c < 16; ++c) {
            const float4 v = ld_shared_f4(rp + x_piece(c, m));
            s[4 * c] = v.x;
            s[4 * c + 1] = v.y;
            s[4 * c + 2] = v.z;
            s[4 * c + 3] = v.w;
          }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(L.xc());  // tile g's exchange buffers are read
        // ---- mask: keys [0, lim) of this tile are visible to the block row (the
        // same for every head, so the branch is uniform)
        const int lim = t >= ct ? min(bi + 1, n_r) - (t - ct) * kNK : ctx - t * kNK;
        if (lim < kNK) {
#pragma unroll
          for (int k = 0; k < kNK; ++k) s[k] = (k < lim) ? s[k] : -INFINITY;
        }
        float mx[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) mx[j] = s[j];
#pragma unroll
        for (int k = 8; k < kNK; ++k) mx[k & 7] = fmaxf(mx[k & 7], s[k]);
        const float mt = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
        // lazy rescale: move the reference only when the max grows by more than 2^8
        const bool need = mt > m_used + 8.0f;
        const float m_new = need ? mt : m_used;
        const float mref = (m_new == -INFINITY) ? 0.f : m_new;
        uint32_t pw[32];
        float psum[4] = {0.f, 0.f, 0.f, 0.f}, psumr[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int k = 0; k < 32; ++k) {
          const float p0 = fast_exp2(s[2 * k] - mref);
          const float p1 = fast_exp2(s[2 * k + 1] - mref);
          psum[k & 3] += p0 + p1;
          __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
          psumr[k & 3] += __low2float(b2) + __high2float(b2);
          pw[k] = *reinterpret_cast<uint32_t*>(&b2);
        }
        // ---- P's TMEM columns are free and O is current once PV of the previous tile is done
        if (g >= 1 && !wait_warp(L.p_empty(), (g - 1) & 1, cx)) { ok = false; break; }
        tc_fence_after();
        if (__any_sync(0xffffffffu, need) && l > 0) {
          const float alpha = need ? fast_exp2(m_used - mt) : 1.0f;
#pragma unroll 1
          for (int c = 0; c < kHalf / 32; ++c) {
            float o[32];
            tmem_ld32(t_lane + TMEM_O + c * 32, o);
            tmem_wait_ld();
#pragma unroll
            for (int k = 0; k < 32; ++k) o[k] *= alpha;
            tmem_st32(t_lane + TMEM_O + c * 32, o);
          }
        }
        if (need) {
          const float a = (l > 0) ? fast_exp2(m_used - mt) : 0.f;
          l_sum *= a;
          l_sumr *= a;
          m_used = mt;
        }
        l_sum += (psum[0] + psum[1]) + (psum[2] + psum[3]);
        l_sumr += (psumr[0] + psumr[1]) + (psumr[2] + psumr[3]);
        {
          float pf[32];
#pragma unroll
          for (int k = 0; k < 32; ++k) pf[k] = __uint_as_float(pw[k]);
          tmem_st32(t_lane + TMEM_P, pf);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(L.p_full());
      }
      if (!ok) break;
      // ---- epilogue: O / l for this CTA's value half (a split piece writes its partial)
      {
        const int gl = g - 1;
        if (!wait_warp(L.p_empty(), gl & 1, cx)) { ok = false; break; }
        tc_fence_after();
        const float inv_l = l_sumr > 0.f ? 1.f / l_sumr : 0.f;
        const bool split = item.nsplit > 1;
        float* obase = split ? prm.ws_o + ((long long)item.slot * kRows + m) * kDv + rho * kHalf
                             : prm.out + ((long long)row_g * kRows + m) * kDv + rho * kHalf;
#pragma unroll 1
        for (int c = 0; c < kHalf / 32; ++c) {
          float o[32];
          tmem_ld32(t_lane + TMEM_O + c * 32, o);
          tmem_wait_ld();
          float4* dst = reinterpret_cast<float4*>(obase + c * 32);
#pragma unroll
          for (int k = 0; k < 8; ++k)
            dst[k] = make_float4(o[4 * k] * inv_l, o[4 * k + 1] * inv_l, o[4 * k + 2] * inv_l,
                                 o[4 * k + 3] * inv_l);
        }
        if (rho == 0) {
          const float lse_v = (m_used + log2f(l_sum)) * 0.69314718055994530942f;
          if (split)
            prm.ws_lse[(long long)item.slot * kRows + m] = lse_v;
          else
            prm.lse[(long long)row_g * kRows + m] = lse_v;
        }
        tc_fence_before();
        __syncwarp();
      }
    }
  }

  if (warp >= kExchWarp0) {
    // ------------------------------------------------------------- score exchange
    // Per tile: S_rho from TMEM (released as soon as it is in registers), scaled to
    // the log2 domain, sent in fp32 to the peer's exchange slot; then, once the peer's
    // partial has arrived in this CTA's slot, the sum x = own + peer replaces it there
    // for the softmax.  The send of tile g waits until this CTA's softmax has read
    // the sums of tile g - 1: the peer's slot of tile g (used for g - 2 before) is
    // then free, because the peer sent tile g - 1 only after its own softmax had read
    // the sums of tile g - 2.
    const int sw = warp & 3;
    const int m = sw * 32 + lane;
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(sw * 32) << 16);
    const uint32_t x_row = static_cast<uint32_t>(m * kXRow);
    const float sl2 = prm.scale_log2;
    const uint32_t x_peer = mapa_shared(L.x(0), peer) + x_row;
    const uint32_t xf_peer = mapa_shared(L.x_full(0), peer);
    int g = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it) {
      const AttnItem item = prm.items[it];
      const int ntiles = item.te - item.tb;
      for (int l = 0; l < ntiles; ++l, ++g) {
        const int xb = g & 1;
        if (!wait_warp(L.s_full(), g & 1, cx)) { ok = false; break; }
        tc_fence_after();
        float x[kNK];
        {
          float a[32], b[32];
          tmem_ld32(t_lane + TMEM_S, a);
          tmem_ld32(t_lane + TMEM_S + 32, b);
          tmem_wait_ld();
#pragma unroll
          for (int k = 0; k < 32; ++k) { x[k] = a[k] * sl2; x[32 + k] = b[k] * sl2; }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(L.s_free());
        if (g >= 1 && !wait_warp(L.xc(), (g - 1) & 1, cx)) { ok = false; break; }
        // this CTA's slot xb receives the peer's partial of tile g
        if (m == 0) mbar_arrive_expect_tx(L.x_full(xb), kXBytes);
        const uint32_t dst = x_peer + xb * kXBytes;
        const uint32_t bar = xf_peer + 8 * xb;
#pragma unroll
        for (int c = 0; c < 16; ++c)
          st_async_v4(dst + x_piece(c, m),
                      make_uint4(__float_as_uint(x[4 * c]), __float_as_uint(x[4 * c + 1]),
                                 __float_as_uint(x[4 * c + 2]), __float_as_uint(x[4 * c + 3])),
                      bar);
        if (!wait_warp<true>(L.x_full(xb), (g >> 1) & 1, cx)) { ok = false; break; }
        // x = own + peer: fp32 addition commutes, so both CTAs get identical bits
        const uint32_t row = L.x(xb) + x_row;
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          const float4 p = ld_shared_f4(row + x_piece(c, m));
          st_shared_v4(row + x_piece(c, m),
                       make_uint4(__float_as_uint(x[4 * c] + p.x), __float_as_uint(x[4 * c + 1] + p.y),
                                  __float_as_uint(x[4 * c + 2] + p.z),
                                  __float_as_uint(x[4 * c + 3] + p.w)));
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(L.sum_full(xb));  // sums of tile g in place
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, TMEM_COLS);
  // the peer may still write into this CTA's exchange buffers and barriers until
  // it arrives here
  cluster_sync();
}

// ---------------------------------------------------------------- host side
namespace {

bool configure() {
  static PerDevice<bool> done;
  return once_per_device(done, false, [] {
    return cudaFuncSetAttribute(verify_attn_mla_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SMEM_BYTES) == cudaSuccess;
  });
}

}  // namespace

int clusters() {
  static PerDevice<int> clus;
  return once_per_device(clus, 1, [] {
    const int sms = num_sms_cached();
    int n = sms / 2 > 0 ? sms / 2 : 1;
    if (configure()) {
      cudaLaunchConfig_t cfg = {};
      cfg.gridDim = dim3(2 * n);
      cfg.blockDim = dim3(kThreads);
      cfg.dynamicSmemBytes = SMEM_BYTES;
      cudaLaunchAttribute attr[1];
      attr[0].id = cudaLaunchAttributeClusterDimension;
      attr[0].val.clusterDim.x = 2;
      attr[0].val.clusterDim.y = 1;
      attr[0].val.clusterDim.z = 1;
      cfg.attrs = attr;
      cfg.numAttrs = 1;
      int c = 0;
      if (cudaOccupancyMaxActiveClusters(&c, verify_attn_mla_kernel, &cfg) == cudaSuccess && c > 0 &&
          c < n)
        n = c;
      else
        cudaGetLastError();
    }
    return n;
  });
}

int launch_kernel(const void* q, const void* k_new, const void* k_cache, int n_pages,
                  const int32_t* page_table, int max_pages, int max_rows, int page_size,
                  float scale, const AttnItem* items, const int* item_begin, int n_clusters,
                  float* out, float* lse, float* ws_o, float* ws_lse, cudaStream_t stream) {
  Params prm;
  prm.q = static_cast<const __nv_bfloat16*>(q);
  prm.page_table = page_table;
  prm.items = items;
  prm.item_begin = item_begin;
  prm.out = out;
  prm.lse = lse;
  prm.ws_o = ws_o;
  prm.ws_lse = ws_lse;
  prm.err = device_error_word();
  prm.max_pages = max_pages;
  prm.n_pages = n_pages;
  prm.page_size = page_size;
  prm.log2_page = 0;
  while ((1 << prm.log2_page) < page_size) ++prm.log2_page;
  prm.scale_log2 = scale * 1.4426950408889634f;
  // cache [n_pages, P, 576]: box 64 dims x min(P, 64) tokens x 1 page
  CUtensorMap tc, tn;
  {
    const uint64_t dims[3] = {(uint64_t)kDqk, (uint64_t)page_size, (uint64_t)n_pages};
    const uint64_t str[2] = {(uint64_t)kDqk * 2, (uint64_t)page_size * kDqk * 2};
    const uint32_t box[3] = {64, (uint32_t)(page_size < kNK ? page_size : kNK), 1};
    if (!gqa::encode_bf16_map(&tc, k_cache, 3, dims, str, box)) return DSPARK_ECUDA;
  }
  // block rows [max_rows, 576]: box 64 dims x 16 rows (rows past max_rows read as zero)
  {
    const uint64_t dims[2] = {(uint64_t)kDqk, (uint64_t)max_rows};
    const uint64_t str[1] = {(uint64_t)kDqk * 2};
    const uint32_t box[2] = {64, (uint32_t)kChunkRows};
    if (!gqa::encode_bf16_map(&tn, k_new, 2, dims, str, box)) return DSPARK_ECUDA;
  }
  if (!configure()) return DSPARK_ECUDA;
  if (launch_pdl_cluster(verify_attn_mla_kernel, dim3(2 * n_clusters), dim3(kThreads), SMEM_BYTES,
                         stream, 2, tc, tn, prm) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}

}  // namespace mla
}  // namespace attn
}  // namespace dspark
