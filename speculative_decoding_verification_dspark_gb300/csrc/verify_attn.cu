// Varlen verify attention over a paged KV cache, causal inside the draft block.
//
// What it computes ("DFlash 到 DSpark in SGLang", section "Ragged verify under
// full CUDA graphs": the packed verify tokens each attend only to their own
// request's KV): packed row cu_seqlens[r] + i, query head h, attends to the
// ctx_len[r] committed keys of request r (read through its page table) and to
// block rows 0..i of its own segment; o = softmax(scale q.K^T) V, lse = log-sum-exp.
//
// How (sm_103a):
//   * one work item = (request, KV head, block-row tile, value-column part, KV split);
//     its query rows (block rows x the query heads of one KV head, or the 128 heads
//     of one block row for the latent-KV shape) form one 128-row UMMA tile;
//   * a persistent grid (one CTA per SM) walks the item list;
//   * warps 0-3 stream K/V tiles into a shared-memory ring with 16-byte cp.async
//     copies written straight into the 128-byte-swizzled K-major layout the tensor
//     cores read (masked rows are zero-filled by the copy itself).  With 16-token
//     pages a TMA box holds at most 2 KB, and the TMA unit's per-box cost caps it
//     below the HBM rate; 128 threads of cp.async keep enough bytes in flight;
//   * warp 4 (one lane) issues tcgen05.mma: S = Q K^T into a double-buffered TMEM
//     tile, then O += P V into a TMEM accumulator;
//   * warps 5-8 own one query row per thread: read S from TMEM, mask, online
//     softmax in fp32 (exp2 domain, lazy rescale of O when the running max grows
//     by more than 2^8), write P (bf16) to shared memory, and finally normalise O;
//   * long contexts split across items; a log-sum-exp combine merges the pieces.
// Every mbarrier wait is bounded in time; a wait that runs out raises
// DSPARK_DEVERR_WAIT_TIMEOUT, the CTA waits for its own copies, frees TMEM and exits.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"
#include "common.cuh"
#include "ptx.cuh"

namespace dspark {
namespace attn {

using namespace ptx;

constexpr uint64_t kWaitLimitNs = 2000000000ull;  // 2 s
constexpr int kProducerWarps = 4;
constexpr int kMmaWarp = 4;
constexpr int kSoftmaxWarp0 = 5;
constexpr int kThreads = 9 * 32;
constexpr int kProducerThreads = kProducerWarps * 32;
constexpr int kRows = 128;                         // UMMA M

template <int D_QK_, int DV_, int NK_, int STAGES_, bool MLA_>
struct Cfg {
  static constexpr int D_QK = D_QK_;
  static constexpr int DV = DV_;          // value columns handled by one item
  static constexpr int NK = NK_;          // keys per tile
  static constexpr int STAGES = STAGES_;
  static constexpr bool MLA = MLA_;
  static constexpr int QK_CB = D_QK / 64;                 // 64-wide swizzle column blocks
  static constexpr int Q_CB_BYTES = kRows * 128;          // one column block of Q
  static constexpr int Q_BYTES = QK_CB * Q_CB_BYTES;
  static constexpr int KV_CB_BYTES = NK * 128;            // one column block of a K/V tile
  static constexpr int K_BYTES = QK_CB * KV_CB_BYTES;
  static constexpr int V_BYTES = MLA ? 0 : (DV / 64) * KV_CB_BYTES;
  static constexpr int STAGE_BYTES = K_BYTES + V_BYTES;
  static constexpr int K_CHUNKS = NK * (D_QK / 8);        // 16-byte chunks of K per tile
  static constexpr int V_CHUNKS = MLA ? 0 : NK * (DV / 8);
  static constexpr int CHUNKS_PER_THREAD = (K_CHUNKS + V_CHUNKS) / kProducerThreads;
  static constexpr int P_ROW_BYTES = NK * 2;              // 128 (NK=64) or 64 (NK=32)
  static constexpr int P_BYTES = kRows * P_ROW_BYTES;
  static constexpr int P_BUFS = MLA ? 1 : 2;
  static constexpr SwizzleMode P_SW = (NK == 64) ? SW_128B : SW_64B;
  static constexpr int OFF_Q = 0;
  static constexpr int OFF_STAGE = OFF_Q + Q_BYTES;
  static constexpr int OFF_P = OFF_STAGE + STAGES * STAGE_BYTES;
  static constexpr int OFF_BAR = OFF_P + P_BUFS * P_BYTES;
  // barriers: kv_full[S], kv_empty[S], s_full[2], s_free[2], p_full[PB], p_empty[PB], q_full
  static constexpr int N_BARS = 2 * STAGES + 4 + 2 * P_BUFS + 1;
  static constexpr int OFF_MISC = OFF_BAR + N_BARS * 8;
  static constexpr int SMEM_BYTES = OFF_MISC + 64 + 1024;  // + alignment slack
  static constexpr int TMEM_S = 0;                         // two S tiles of NK columns
  static constexpr int TMEM_O = 2 * NK;
  static constexpr int TMEM_COLS_USED = 2 * NK + DV;
  static constexpr int TMEM_COLS = TMEM_COLS_USED <= 256 ? 256 : 512;
  static_assert(SMEM_BYTES <= 232448, "shared memory budget");
  static_assert(TMEM_COLS_USED <= 512, "tensor memory budget");
  static_assert(NK == 64 || NK == 32, "tile width");
  static_assert((K_CHUNKS + V_CHUNKS) % kProducerThreads == 0, "copy split");
  // Copy groups a producer thread keeps in flight before publishing a tile.
  // Publishing tile g needs tile g+LAG issued, hence PV(g+LAG-STAGES) done, which
  // the MMA warp issues only once tile g+LAG-STAGES+1 is published: LAG <= STAGES-2.
  static constexpr int LAG = STAGES - 2;
  static_assert(LAG >= 0, "pipeline depth");
  static_assert(STAGE_BYTES % 1024 == 0 && Q_BYTES % 1024 == 0 && P_BYTES % 1024 == 0, "align");
};

using CfgMLA = Cfg<576, 256, 32, 2, true>;

struct Ctx {
  volatile int* abort_flag;
  unsigned int* err;
};

// Wait for the phase of `bar` with the given parity; bounded.  Returns false if
// the CTA is aborting.
__device__ __forceinline__ bool wait_bar(uint32_t bar, uint32_t parity, const Ctx& cx) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  uint32_t n = 0;
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
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

// Used only on the way out: wait regardless of the abort flag, bounded.
__device__ __forceinline__ void drain_bar(uint32_t bar, uint32_t parity, unsigned int* err) {
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > kWaitLimitNs) {
      raise_error(err, DSPARK_DEVERR_WAIT_TIMEOUT);
      return;
    }
  }
}

// 16-byte chunk q (0-based, 8 per 128-byte row) of row `row` in a 128B-swizzled
// K-major tile: chunk index XOR (row mod 8).
__device__ __forceinline__ uint32_t sw128_off(int row, int chunk) {
  return static_cast<uint32_t>(row * 128 + ((chunk ^ (row & 7)) << 4));
}
// 64B swizzle, 64-byte rows: chunk (0..3) XOR ((row / 2) mod 4).
__device__ __forceinline__ uint32_t sw64_off(int row, int chunk) {
  return static_cast<uint32_t>(row * 64 + ((chunk ^ ((row >> 1) & 3)) << 4));
}

// 2^x on the SFU (ex2.approx.ftz: -inf -> +0).  The softmax weights are rounded
// to bf16 right after, so the approximation error is far below that rounding.
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

// 16-byte global -> shared copy; src_bytes = 0 writes zeros without reading.
__device__ __forceinline__ void cp_async16(uint32_t dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() {
  asm volatile("cp.async.commit_group;" ::: "memory");
}
template <int N>
__device__ __forceinline__ void cp_async_wait() {
  asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory");
}

template <class C>
struct Layout {
  uint32_t q, stage0, p0, bar0;
  __device__ uint32_t stage(int s) const { return stage0 + s * C::STAGE_BYTES; }
  __device__ uint32_t pbuf(int b) const { return p0 + b * C::P_BYTES; }
  __device__ uint32_t kv_full(int s) const { return bar0 + 8 * s; }
  __device__ uint32_t kv_empty(int s) const { return bar0 + 8 * (C::STAGES + s); }
  __device__ uint32_t s_full(int b) const { return bar0 + 8 * (2 * C::STAGES + b); }
  __device__ uint32_t s_free(int b) const { return bar0 + 8 * (2 * C::STAGES + 2 + b); }
  __device__ uint32_t p_full(int b) const { return bar0 + 8 * (2 * C::STAGES + 4 + b); }
  __device__ uint32_t p_empty(int b) const {
    return bar0 + 8 * (2 * C::STAGES + 4 + C::P_BUFS + b);
  }
  __device__ uint32_t q_full() const { return bar0 + 8 * (2 * C::STAGES + 4 + 2 * C::P_BUFS); }
};

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
  int max_pages, B, Hq, Hkv, page_size, log2_page, max_rows, d_v_total, n_pages;
  float scale_log2;
};

// Page indices of the (at most NK/16) pages cache tile t touches, -1 for a
// corrupt entry (read as zeros, reported).  Issued one tile ahead so that the
// page-table latency overlaps the previous tile's copies.
template <class C>
__device__ __forceinline__ void load_tile_pages(const Params& prm, const int32_t* ptab, int t,
                                                int ct, int ctx, int (&pg)[C::NK / 16]) {
  const int slot0 = (t * C::NK) >> prm.log2_page;
#pragma unroll
  for (int j = 0; j < C::NK / 16; ++j) {
    const int sl = slot0 + j;
    const bool in = t < ct && (sl << prm.log2_page) < ctx;
    int p = in ? ptab[sl] : 0;
    if (in && (p < 0 || p >= prm.n_pages)) {
      raise_error(prm.err, DSPARK_DEVERR_BAD_INPUT);
      p = -1;
    }
    pg[j] = p;
  }
}

// One K/V tile into the stage at `kdst`: cache tile t < ct (keys t*NK ..) or a
// block tile (the request's own packed rows).  Each producer thread issues
// CHUNKS_PER_THREAD 16-byte copies; consecutive threads take consecutive chunks
// of a row, so every warp-wide copy reads whole 256-byte (or 1152-byte) rows.
template <class C>
__device__ __forceinline__ void produce_tile(const Params& prm, const AttnItem& item, int t, int ct,
                                             int ctx, int c0, int n_r, const int (&pg)[C::NK / 16],
                                             uint32_t kdst, int pt) {
  constexpr int KCH = C::D_QK / 8;   // chunks per K row
  constexpr int VCH = C::DV / 8;     // chunks per V row (GQA)
  const long long rs = C::MLA ? C::D_QK : (long long)prm.Hkv * C::D_QK;  // row stride (elements)
  const int lp = prm.log2_page;
  const bool cache = t < ct;
  const __nv_bfloat16* kbase;
  const __nv_bfloat16* vbase;
  int valid;                         // rows [0, valid) of this tile exist
  if (cache) {
    kbase = prm.k_cache + (C::MLA ? 0 : (long long)item.kvh * C::D_QK);
    vbase = C::MLA ? nullptr : prm.v_cache + (long long)item.kvh * C::D_QK;
    valid = ctx - t * C::NK;
  } else {
    const int b0 = (t - ct) * C::NK;
    const long long off = (long long)(c0 + b0) * rs + (C::MLA ? 0 : (long long)item.kvh * C::D_QK);
    kbase = prm.k_new + off;
    vbase = C::MLA ? nullptr : prm.v_new + off;
    valid = n_r - b0;
  }
  const int slot0 = (t * C::NK) >> lp;
  const uint32_t vdst = kdst + C::K_BYTES;
#pragma unroll
  for (int k = 0; k < C::CHUNKS_PER_THREAD; ++k) {
    const int c = pt + k * kProducerThreads;
    const bool is_v = !C::MLA && c >= C::K_CHUNKS;
    const int cc = is_v ? c - C::K_CHUNKS : c;
    const int row = is_v ? cc / VCH : cc / KCH;
    const int q = is_v ? cc % VCH : cc % KCH;
    const __nv_bfloat16* base = is_v ? vbase : kbase;
    bool ok = row < valid;
    long long src_row = row;
    if (cache) {
      const int key = t * C::NK + row;
      const int j = (key >> lp) - slot0;
      int p = pg[0];
#pragma unroll
      for (int jj = 1; jj < C::NK / 16; ++jj) p = (j == jj) ? pg[jj] : p;
      ok = ok && p >= 0;
      src_row = ((long long)(ok ? p : 0) << lp) + (key & ((1 << lp) - 1));
    }
    const __nv_bfloat16* src = ok ? base + src_row * rs + q * 8 : prm.k_cache;
    const uint32_t dst = (is_v ? vdst : kdst) + (q >> 3) * C::KV_CB_BYTES + sw128_off(row, q & 7);
    cp_async16(dst, src, ok ? 16u : 0u);
  }
}

template <class C>
__global__ void __launch_bounds__(kThreads, 1) verify_attn_kernel(const Params prm) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_addr(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint8_t* base_ptr = smem_raw + (base - raw);
  Layout<C> L{base + C::OFF_Q, base + C::OFF_STAGE, base + C::OFF_P, base + C::OFF_BAR};
  volatile int* abort_flag = reinterpret_cast<volatile int*>(base_ptr + C::OFF_MISC);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(base_ptr + C::OFF_MISC + 16);
  const Ctx cx{abort_flag, prm.err};

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < C::STAGES; ++s) {
      mbar_init(L.kv_full(s), kProducerWarps);
      mbar_init(L.kv_empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(L.s_full(b), 1);
      mbar_init(L.s_free(b), 4);
    }
    for (int b = 0; b < C::P_BUFS; ++b) {
      mbar_init(L.p_full(b), 4);
      mbar_init(L.p_empty(b), 1);
    }
    mbar_init(L.q_full(), 1);
    fence_mbar_init();
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_addr(tmem_slot), C::TMEM_COLS);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  pdl_release();
  pdl_wait();  // the work list and the step's inputs come from earlier kernels
  const int it_begin = prm.item_begin[blockIdx.x];
  const int it_end = prm.item_begin[blockIdx.x + 1];
  const int G = C::MLA ? kRows : prm.Hq / prm.Hkv;  // query rows per block row

  if (warp < kProducerWarps) {
    // ------------------------------------------------------------- producers
    const int pt = threadIdx.x;  // 0..127
    int g = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it) {
      const AttnItem item = prm.items[it];
      const int r = item.r;
      const int ctx = item.ctx;
      const int c0 = item.c0;
      const int n_r = item.n_r;
      const int ct = ceil_div(ctx, C::NK);
      const int32_t* ptab = prm.page_table + (long long)r * prm.max_pages;
      int pg[C::NK / 16];
      load_tile_pages<C>(prm, ptab, item.tb, ct, ctx, pg);
      for (int t = item.tb; t < item.te; ++t, ++g) {
        const int s = g % C::STAGES;
        if (g >= C::STAGES) {
          ok = wait_bar(L.kv_empty(s), ((g / C::STAGES) - 1) & 1, cx);
          ok = __all_sync(0xffffffffu, ok);
          if (!ok) break;
        }
        produce_tile<C>(prm, item, t, ct, ctx, c0, n_r, pg, L.stage(s), pt);
        cp_async_commit();
        if (t + 1 < item.te) load_tile_pages<C>(prm, ptab, t + 1, ct, ctx, pg);
        if (g >= C::LAG) {
          // tile g - LAG has landed for this thread: publish it to the tensor cores
          cp_async_wait<C::LAG>();
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(L.kv_full((g - C::LAG) % C::STAGES));
        }
      }
    }
    // publish the last tiles (and never leave copies in flight)
    cp_async_wait<0>();
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      const int first = g - C::LAG > 0 ? g - C::LAG : 0;
      for (int gg = first; gg < g; ++gg) mbar_arrive(L.kv_full(gg % C::STAGES));
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      constexpr uint32_t IDESC_QK = idesc_bf16_f32(kRows, C::NK, 0, 0);
      constexpr uint32_t IDESC_PV = idesc_bf16_f32(kRows, C::DV, 0, 1);
      int g = 0, n_it = 0, last_pv = -1;
      bool ok = true;
      auto issue_pv = [&](int gp, int local, int part) -> bool {
        const int pb = gp % C::P_BUFS;
        if (!wait_bar(L.p_full(pb), (gp / C::P_BUFS) & 1, cx)) return false;
        tc_fence_after();
        const int s = gp % C::STAGES;
        const uint32_t vbase =
            C::MLA ? L.stage(s) + part * 4 * C::KV_CB_BYTES : L.stage(s) + C::K_BYTES;
#pragma unroll
        for (int kk = 0; kk < C::NK / 16; ++kk) {
          const uint64_t a = smem_desc(L.pbuf(pb) + kk * 32, 16, 8 * C::P_ROW_BYTES, C::P_SW);
          const uint64_t b = smem_desc(vbase + kk * 2048, C::KV_CB_BYTES, 1024, SW_128B);
          umma_bf16(tmem + C::TMEM_O, a, b, IDESC_PV, (local > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(L.p_empty(pb));
        umma_commit(L.kv_empty(s));
        last_pv = gp;
        return true;
      };
      for (int it = it_begin; it < it_end && ok; ++it, ++n_it) {
        const AttnItem item = prm.items[it];
        if (!wait_bar(L.q_full(), n_it & 1, cx)) { ok = false; break; }
        const int ntiles = item.te - item.tb;
        for (int l = 0; l < ntiles; ++l, ++g) {
          const int s = g % C::STAGES;
          const int sb = g & 1;
          if (!wait_bar(L.kv_full(s), (g / C::STAGES) & 1, cx)) { ok = false; break; }
          if (g >= 2 && !wait_bar(L.s_free(sb), ((g >> 1) - 1) & 1, cx)) { ok = false; break; }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < C::D_QK / 16; ++kk) {
            const uint64_t a = smem_desc(L.q + (kk >> 2) * C::Q_CB_BYTES + (kk & 3) * 32, 16, 1024, SW_128B);
            const uint64_t b = smem_desc(L.stage(s) + (kk >> 2) * C::KV_CB_BYTES + (kk & 3) * 32, 16, 1024, SW_128B);
            umma_bf16(tmem + C::TMEM_S + sb * C::NK, a, b, IDESC_QK, kk > 0 ? 1u : 0u);
          }
          umma_commit(L.s_full(sb));
          if (l >= 1 && !issue_pv(g - 1, l - 1, item.part)) { ok = false; break; }
        }
        if (!ok) break;
        if (!issue_pv(g - 1, ntiles - 1, item.part)) { ok = false; break; }
      }
      // all issued MMAs must finish before TMEM is released
      if (last_pv >= 0) drain_bar(L.p_empty(last_pv % C::P_BUFS), (last_pv / C::P_BUFS) & 1, prm.err);
    }
  } else {
    // ------------------------------------------------------------- softmax / epilogue
    const int sw = warp & 3;                 // TMEM lane quadrant of this warp
    const int m = sw * 32 + lane;            // query row of this thread
    const uint32_t t_lane = tmem + (static_cast<uint32_t>(sw * 32) << 16);
    const int stid = threadIdx.x - kSoftmaxWarp0 * 32;  // 0..127
    const float sl2 = prm.scale_log2;
    int g = 0;
    bool ok = true;
    for (int it = it_begin; it < it_end && ok; ++it) {
      const AttnItem item = prm.items[it];
      const int ctx = item.ctx;
      const int c0 = item.c0;
      const int n_r = item.n_r;
      const int ct = ceil_div(ctx, C::NK);
      const int rows_valid = C::MLA ? kRows : item.ni * G;
      // ---- Q tile (rows beyond rows_valid are zero)
      {
        constexpr int CH = C::D_QK / 8;
        for (int idx = stid; idx < kRows * CH; idx += 128) {
          const int row = idx / CH, q = idx % CH;
          uint4 v = make_uint4(0, 0, 0, 0);
          if (row < rows_valid) {
            long long src;
            if (C::MLA)
              src = ((long long)(c0 + item.i0) * prm.Hq + row) * C::D_QK;
            else
              src = ((long long)(c0 + item.i0 + row / G) * prm.Hq + item.kvh * G + row % G) * C::D_QK;
            v = ldg_nc_v4(prm.q + src + q * 8);
          }
          st_shared_v4(L.q + (q >> 3) * C::Q_CB_BYTES + sw128_off(row, q & 7), v);
        }
        fence_proxy_async_smem();
        asm volatile("bar.sync 1, 128;" ::: "memory");
        if (stid == 0) mbar_arrive(L.q_full());
      }
      const bool row_ok = m < rows_valid;
      const bool warp_active = __any_sync(0xffffffffu, row_ok);
      const int bi = C::MLA ? item.i0 : item.i0 + m / G;   // block index of this row
      // m_used: reference max (log2 domain, scaled); l_sum: sum of exp2(s*sl2 - m_used)
      float m_used = -INFINITY, l_sum = 0.f;
      const int ntiles = item.te - item.tb;
      for (int l = 0; l < ntiles; ++l, ++g) {
        const int t = item.tb + l;
        const int sb = g & 1;
        bool w_ok = wait_bar(L.s_full(sb), (g >> 1) & 1, cx);
        w_ok = __all_sync(0xffffffffu, w_ok);
        if (!w_ok) { ok = false; break; }
        tc_fence_after();
        float s[C::NK];
        if (warp_active) {
#pragma unroll
          for (int c = 0; c < C::NK / 32; ++c) {
            float tmp[32];
            tmem_ld32(t_lane + C::TMEM_S + sb * C::NK + c * 32, tmp);
#pragma unroll
            for (int k = 0; k < 32; ++k) s[c * 32 + k] = tmp[k];
          }
          tmem_wait_ld();
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(L.s_free(sb));
        // P buffer of this tile must be free: PV(g - P_BUFS) done
        const int pb = g % C::P_BUFS;
        if (g >= C::P_BUFS) {
          const int gp = g - C::P_BUFS;
          w_ok = wait_bar(L.p_empty(gp % C::P_BUFS), (gp / C::P_BUFS) & 1, cx);
          w_ok = __all_sync(0xffffffffu, w_ok);
          if (!w_ok) { ok = false; break; }
        }
        if (warp_active) {
          // ---- mask (only the last cache tile and the block tile need it) + tile max
          // Keys [0, lim) of this tile are visible to this row: the committed
          // context for a cache tile, block rows 0..bi for the block tile.
          const bool block_tile = t >= ct;
          const int lim = block_tile ? min(bi + 1, n_r) - (t - ct) * C::NK : ctx - t * C::NK;
          if (__any_sync(0xffffffffu, lim < C::NK)) {
#pragma unroll
            for (int k = 0; k < C::NK; ++k) s[k] = (k < lim) ? s[k] : -INFINITY;
          }
          float mx[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) mx[j] = s[j];
#pragma unroll
          for (int k = 8; k < C::NK; ++k) mx[k & 7] = fmaxf(mx[k & 7], s[k]);
          const float mt =
              fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                    fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7]))) * sl2;
          // ---- lazy rescale of O when the running max grows by more than 2^8
          const bool need = row_ok && (mt > m_used + 8.0f);
          if (__any_sync(0xffffffffu, need) && l > 0) {
            // O must hold PV(g-1): wait for it (its P buffer's barrier)
            const int gq = g - 1;
            if (C::P_BUFS > 1) {
              w_ok = wait_bar(L.p_empty(gq % C::P_BUFS), (gq / C::P_BUFS) & 1, cx);
              w_ok = __all_sync(0xffffffffu, w_ok);
              if (!w_ok) { ok = false; break; }
            }
            tc_fence_after();
            const float alpha = need ? fast_exp2(m_used - mt) : 1.0f;
#pragma unroll 1
            for (int c = 0; c < C::DV / 32; ++c) {
              float o[32];
              tmem_ld32(t_lane + C::TMEM_O + c * 32, o);
              tmem_wait_ld();
#pragma unroll
              for (int k = 0; k < 32; ++k) o[k] *= alpha;
              tmem_st32(t_lane + C::TMEM_O + c * 32, o);
            }
            tmem_wait_st();
          }
          if (need) {
            l_sum *= (l > 0) ? fast_exp2(m_used - mt) : 0.f;
            m_used = mt;
          }
          // ---- P = exp2(s*scale - m_used), bf16, swizzled K-major row m.  Rows
          // past rows_valid compute harmless values: they only feed their own O
          // rows, which are never stored.
          const uint32_t prow = L.pbuf(pb);
          const float mref = (m_used == -INFINITY) ? 0.f : m_used;
          float psum[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int q = 0; q < C::NK / 8; ++q) {
            uint32_t w[4];
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              const float p0 = fast_exp2(fmaf(s[q * 8 + 2 * h], sl2, -mref));
              const float p1 = fast_exp2(fmaf(s[q * 8 + 2 * h + 1], sl2, -mref));
              psum[h] += p0 + p1;
              __nv_bfloat162 b2 = __floats2bfloat162_rn(p0, p1);
              w[h] = *reinterpret_cast<uint32_t*>(&b2);
            }
            const uint32_t off = (C::NK == 64) ? sw128_off(m, q) : sw64_off(m, q);
            st_shared_v4(prow + off, make_uint4(w[0], w[1], w[2], w[3]));
          }
          l_sum += (psum[0] + psum[1]) + (psum[2] + psum[3]);
          tc_fence_before();
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(L.p_full(pb));
      }
      if (!ok) break;
      // ---- epilogue: O / l  (split items write partials for the combine)
      {
        const int gl = g - 1;
        bool w_ok = wait_bar(L.p_empty(gl % C::P_BUFS), (gl / C::P_BUFS) & 1, cx);
        w_ok = __all_sync(0xffffffffu, w_ok);
        if (!w_ok) { ok = false; break; }
        tc_fence_after();
        if (warp_active) {
          const int row_g = c0 + bi;
          const int head = C::MLA ? m : item.kvh * G + m % G;
          const float inv_l = l_sum > 0.f ? 1.f / l_sum : 0.f;
          const bool split = item.nsplit > 1;
          float* obase;
          // a piece of a split context writes its partial rows into its own slot
          if (split)
            obase = prm.ws_o + ((long long)item.slot * kRows + m) * C::DV;
          else
            obase = prm.out + ((long long)row_g * prm.Hq + head) * prm.d_v_total + item.part * C::DV;
#pragma unroll 1
          for (int c = 0; c < C::DV / 32; ++c) {
            float o[32];
            tmem_ld32(t_lane + C::TMEM_O + c * 32, o);
            tmem_wait_ld();
            if (row_ok) {
              float4* dst = reinterpret_cast<float4*>(obase + c * 32);
#pragma unroll
              for (int k = 0; k < 8; ++k)
                dst[k] = make_float4(o[4 * k] * inv_l, o[4 * k + 1] * inv_l, o[4 * k + 2] * inv_l,
                                     o[4 * k + 3] * inv_l);
            }
          }
          if (row_ok) {
            const float lse_v = (m_used + log2f(l_sum)) * 0.69314718055994530942f;
            if (split)
              prm.ws_lse[(long long)item.slot * kRows + m] = lse_v;
            else if (item.part == 0)
              prm.lse[(long long)row_g * prm.Hq + head] = lse_v;
          }
        }
        tc_fence_before();
        __syncwarp();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, C::TMEM_COLS);
}

// ---------------------------------------------------------------- work list
// One CTA.  Stream-K style split: the key tiles of every (request, row tile, value
// part, KV head) group are laid end to end (U units) and CTA c of the persistent
// grid receives units [c*U/n, (c+1)*U/n) -- the same number of tiles for every
// CTA, whatever the context-length mix.  A group cut by CTA boundaries becomes
// pieces, one per CTA it meets; such a piece is always the first or the last piece
// of its CTA and writes partial (o, lse) rows into slot 2c or 2c + 1.  The CTA that
// runs the last piece of a split group records the group for the combine.
__device__ __forceinline__ int cta_of_unit(long long x, long long U, int n) {
  return static_cast<int>(((x + 1) * n - 1) / U);  // largest c with c*U/n <= x
}

template <class T>
__device__ __forceinline__ T warp_incl_scan(T v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const T u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

// Exclusive block scan (blockDim.x = 1024); *total receives the sum.
template <class T>
__device__ __forceinline__ T block_excl_scan(T v, T* s_w, T* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const T incl = warp_incl_scan(v, lane);
  if (lane == 31) s_w[wid] = incl;
  __syncthreads();
  if (wid == 0) s_w[lane] = warp_incl_scan(s_w[lane], lane);
  __syncthreads();
  const T ex = (wid > 0 ? s_w[wid - 1] : T(0)) + incl - v;
  *total = s_w[31];
  __syncthreads();  // s_w may be reused by the caller's next scan
  return ex;
}

__global__ void __launch_bounds__(1024)
    worklist_kernel(const int32_t* __restrict__ ctx_len, const int32_t* __restrict__ cu_seqlens,
                    int B, int max_rows, int Hkv, int parts, int rows_per_tile, int NK, int ncta,
                    int max_splits, int max_items, AttnItem* __restrict__ items,
                    int* __restrict__ item_begin, SplitGroup* __restrict__ groups,
                    unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  __shared__ long long s_off[DSPARK_MAX_B + 1];
  __shared__ int s_tt[DSPARK_MAX_B];
  __shared__ int s_n[DSPARK_MAX_B];
  __shared__ int s_ctx[DSPARK_MAX_B];
  __shared__ int s_c0[DSPARK_MAX_B];
  __shared__ long long s_w64[32];
  __shared__ int s_w32[32];
  const int tid = threadIdx.x, lane = tid & 31;
  const int ng_per_tile = parts * Hkv;
  const bool rows_ok = cu_seqlens[B] <= max_rows;  // else: report and run nothing
  long long units = 0;
  int tt = 0;
  if (tid < B) {
    const int c0 = cu_seqlens[tid];
    const int n = cu_seqlens[tid + 1] - c0;
    const int ctx = ctx_len[tid];
    tt = ceil_div(ctx, NK) + ceil_div(n, NK);
    units = (long long)tt * ceil_div(n, rows_per_tile) * ng_per_tile;
    s_tt[tid] = tt;
    s_n[tid] = n;
    s_ctx[tid] = ctx;
    s_c0[tid] = c0;
  }
  // largest group, in tiles
  int tmax = tt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
  if (lane == 0) s_w32[tid >> 5] = tmax;
  __syncthreads();
  tmax = s_w32[lane];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, o));
  __syncthreads();
  long long U;
  const long long ex = block_excl_scan(units, s_w64, &U);
  if (tid < B) s_off[tid] = ex;
  if (tid == 0) s_off[B] = U;
  // No group may be cut into more than max_splits pieces.  Every CTA range holds at
  // least L = floor(U/n) units, and a group of T units meets at most
  // ceil((T-1)/L) + 1 ranges, so L >= ceil((T_max-1)/(max_splits-1)) suffices:
  // n <= U / that.  Then n <= U too, so no CTA range is empty and the pieces of a
  // group sit in consecutive CTAs.
  int n_eff = ncta;
  {
    long long l_req = tmax > 1 ? ((long long)tmax - 1 + max_splits - 2) / (max_splits - 1) : 1;
    if (l_req < 1) l_req = 1;
    const long long cap = U / l_req;
    if (cap < n_eff) n_eff = cap > 0 ? static_cast<int>(cap) : 1;
  }
  __syncthreads();
  const int c = tid;
  const bool active = c < ncta && c < n_eff && U > 0;
  const long long lo = active ? (long long)c * U / n_eff : 0;
  const long long hi = active ? (long long)(c + 1) * U / n_eff : 0;
  // walk CTA c's unit range: count (emit = false) or write its pieces
  auto walk = [&](bool emit, int base) -> int {
    long long u = lo;
    int k = 0;
    bool wrote_group = false;
    while (u < hi) {
      int a = 0, b = B;  // request: s_off[a] <= u < s_off[a + 1]
      while (b - a > 1) {
        const int mid = (a + b) >> 1;
        if (s_off[mid] <= u) a = mid; else b = mid;
      }
      const int r = a;
      const int t_r = s_tt[r];
      const long long lu = u - s_off[r];
      const int lg = static_cast<int>(lu / t_r);          // group within the request
      const long long gstart = s_off[r] + (long long)lg * t_r;
      const long long gend = gstart + t_r;
      const long long next = gend < hi ? gend : hi;
      if (emit) {
        const int c_first = cta_of_unit(gstart, U, n_eff);
        const int c_last = cta_of_unit(gend - 1, U, n_eff);
        const int t = lg / ng_per_tile, p = (lg / Hkv) % parts, h = lg % Hkv;
        const int i0 = t * rows_per_tile;
        const int ni = min(rows_per_tile, s_n[r] - i0);
        AttnItem it;
        it.r = r; it.kvh = h; it.i0 = i0; it.ni = ni;
        it.part = p; it.split = c - c_first;
        it.tb = static_cast<int>(lu - (long long)lg * t_r);
        it.te = it.tb + static_cast<int>(next - u);
        it.nsplit = c_last - c_first + 1;
        it.slot = u == lo ? 2 * c : 2 * c + 1;
        it.pad0 = 0; it.pad1 = 0;
        it.ctx = s_ctx[r]; it.c0 = s_c0[r]; it.n_r = s_n[r]; it.pad2 = 0;
        items[base + k] = it;
        if (it.nsplit > 1 && c == c_last) {
          SplitGroup sg;
          sg.r = r; sg.kvh = h; sg.part = p; sg.i0 = i0;
          sg.ni = ni; sg.c_first = c_first; sg.nsplit = it.nsplit;
          sg.slot0_last = gstart != (long long)c_first * U / n_eff;
          groups[c] = sg;
          wrote_group = true;
        }
      }
      ++k;
      u = next;
    }
    if (emit && !wrote_group) {
      SplitGroup sg{};
      groups[c] = sg;  // nsplit = 0: no group ends here
    }
    return k;
  };
  const int cnt = walk(false, 0);
  int total;
  const int base = block_excl_scan(cnt, s_w32, &total);
  const bool fits = rows_ok && total <= max_items;
  if (tid == 0 && !fits)
    raise_error(err, rows_ok ? DSPARK_DEVERR_WORK_OVERFLOW : DSPARK_DEVERR_ROWS_OVERFLOW);
  if (c < ncta) item_begin[c] = fits ? base : 0;
  if (tid == 0) item_begin[ncta] = fits ? total : 0;
  if (c < ncta) {
    if (fits) {
      walk(true, base);
    } else {
      SplitGroup sg{};
      groups[c] = sg;
    }
  }
}

// ---------------------------------------------------------------- split combine
// Block (c, y): the split group recorded by CTA c, query rows 8y..8y+7, one warp per
// row, lanes over 4-wide value columns:
//   lse = log sum_s e^{lse_s},  o = sum_s e^{lse_s - lse} o_s
// over the group's pieces' partial slots.
__global__ void __launch_bounds__(256)
    combine_kernel(const int32_t* __restrict__ cu_seqlens, const SplitGroup* __restrict__ groups,
                   int G, int Hq, int rows_per_slot, int d_part, int d_v_total,
                   const float* __restrict__ ws_o, const float* __restrict__ ws_lse,
                   float* __restrict__ out, float* __restrict__ lse, int mla) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  const int lane = threadIdx.x & 31;
  const SplitGroup sg = groups[blockIdx.x];
  const int ns = sg.nsplit;
  if (ns <= 1) return;
  const int nq = mla ? Hq : sg.ni * G;
  const int n = blockIdx.y * (blockDim.x >> 5) + (threadIdx.x >> 5);
  if (n >= nq) return;
  int slot = 0;
  float my = -INFINITY;
  if (lane < ns) {
    slot = (lane == 0 && sg.slot0_last) ? 2 * sg.c_first + 1 : 2 * (sg.c_first + lane);
    my = ws_lse[(long long)slot * rows_per_slot + n];
  }
  float mx = my;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, o));
  const float wgt = lane < ns ? expf(my - mx) : 0.f;
  float sum = wgt;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  const float inv = 1.f / sum;
  int row_g, head;
  const int c0 = cu_seqlens[sg.r];
  if (mla) { row_g = c0 + sg.i0; head = n; }
  else { row_g = c0 + sg.i0 + n / G; head = sg.kvh * G + n % G; }
  float4* dst = reinterpret_cast<float4*>(out + ((long long)row_g * Hq + head) * d_v_total +
                                          sg.part * d_part);
  for (int d4 = lane; d4 < (d_part >> 2); d4 += 32) {
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int sp = 0; sp < ns; ++sp) {
      const float ws = __shfl_sync(0xffffffffu, wgt, sp);
      const int sl = __shfl_sync(0xffffffffu, slot, sp);
      const float4 v =
          reinterpret_cast<const float4*>(ws_o + ((long long)sl * rows_per_slot + n) * d_part)[d4];
      acc.x += ws * v.x; acc.y += ws * v.y; acc.z += ws * v.z; acc.w += ws * v.w;
    }
    dst[d4] = make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
  }
  if (lane == 0 && sg.part == 0) lse[(long long)row_g * Hq + head] = mx + logf(sum);
}

// ---------------------------------------------------------------- host side
namespace {

template <class C>
bool configure_smem() {
  static bool done = false, okv = false;
  if (!done) {
    done = true;
    okv = cudaFuncSetAttribute(verify_attn_kernel<C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               C::SMEM_BYTES) == cudaSuccess;
  }
  return okv;
}

}  // namespace

Plan plan(int B, int max_rows, int Hq, int Hkv, int d_qk, int d_v, int max_splits,
          int max_block_rows) {
  Plan p{};
  p.mla = (d_qk == 576);
  const int G = p.mla ? Hq : Hq / Hkv;
  p.parts = p.mla ? 2 : 1;
  p.nt = p.mla ? kRows : gqa::query_tile(Hq, Hkv, max_block_rows);
  p.rows_per_tile = p.mla ? 1 : (p.nt / G);
  p.nk = p.mla ? CfgMLA::NK : gqa::kKeyTile;
  p.d_part = p.mla ? CfgMLA::DV : d_v;
  p.ncta = num_sms_cached();
  if (p.ncta > 1024) p.ncta = 1024;  // the work list keeps one counter per CTA in shared memory
  const long long groups = (long long)Hkv * p.parts * ((long long)max_rows / p.rows_per_tile + B);
  p.max_items = groups + p.ncta;
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (bytes + 255) & ~size_t(255);
    return o;
  };
  p.off_items = take(sizeof(AttnItem) * (size_t)p.max_items);
  p.off_begin = take(sizeof(int) * (size_t)(p.ncta + 1));
  p.off_groups = take(sizeof(SplitGroup) * (size_t)p.ncta);
  p.off_o = take(sizeof(float) * (size_t)2 * p.ncta * kRows * p.d_part);   // slots 2c, 2c + 1
  p.off_lse = take(sizeof(float) * (size_t)2 * p.ncta * kRows);
  p.bytes = off;
  (void)max_splits;
  return p;
}

int launch(const void* q, const void* k_new, const void* v_new, const void* k_cache,
           const void* v_cache, int n_pages, const int32_t* page_table, int max_pages,
           const int32_t* ctx_len, const int32_t* cu_seqlens, int B, int max_rows, int Hq, int Hkv,
           int d_qk, int d_v, int page_size, float scale, int max_splits, float* out, float* lse,
           void* ws, const Plan& pl, cudaStream_t stream) {
  uint8_t* w = static_cast<uint8_t*>(ws);
  AttnItem* items = reinterpret_cast<AttnItem*>(w + pl.off_items);
  int* item_begin = reinterpret_cast<int*>(w + pl.off_begin);
  SplitGroup* groups = reinterpret_cast<SplitGroup*>(w + pl.off_groups);
  float* ws_o = reinterpret_cast<float*>(w + pl.off_o);
  float* ws_lse = reinterpret_cast<float*>(w + pl.off_lse);
  unsigned int* err = device_error_word();
  const int ncta = pl.ncta;
  const int max_items = pl.max_items > 0x7fffffff ? 0x7fffffff : (int)pl.max_items;
  const int splits = max_splits < 2 ? 2 : (max_splits > 32 ? 32 : max_splits);

  if (launch_pdl(worklist_kernel, dim3(1), dim3(1024), 0, stream, ctx_len, cu_seqlens, B, max_rows,
                 Hkv, pl.parts, pl.rows_per_tile, pl.nk, ncta, splits, max_items, items, item_begin,
                 groups, err) != cudaSuccess)
    return DSPARK_ECUDA;

  if (pl.mla) {
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
    prm.err = err;
    prm.max_pages = max_pages;
    prm.B = B;
    prm.Hq = Hq;
    prm.Hkv = Hkv;
    prm.page_size = page_size;
    prm.log2_page = 0;
    while ((1 << prm.log2_page) < page_size) ++prm.log2_page;
    prm.max_rows = max_rows;
    prm.d_v_total = d_v;
    prm.n_pages = n_pages;
    prm.scale_log2 = scale * 1.4426950408889634f;
    if (!configure_smem<CfgMLA>()) return DSPARK_ECUDA;
    if (launch_pdl(verify_attn_kernel<CfgMLA>, dim3(ncta), dim3(kThreads), CfgMLA::SMEM_BYTES, stream,
                   prm) != cudaSuccess)
      return DSPARK_ECUDA;
  } else {
    const int rc = gqa::launch_kernel(pl.nt, q, k_new, v_new, k_cache, v_cache, n_pages, page_table,
                                      max_pages, ctx_len, cu_seqlens, B, max_rows, Hq, Hkv,
                                      page_size, scale, items, item_begin, ncta, out, lse, ws_o,
                                      ws_lse, stream);
    if (rc != DSPARK_OK) return rc;
  }
  const int G = pl.mla ? Hq : Hq / Hkv;
  if (launch_pdl(combine_kernel, dim3(ncta, kRows / 8), dim3(256), 0, stream, cu_seqlens, groups, G,
                 Hq, kRows, pl.d_part, d_v, ws_o, ws_lse, out, lse, pl.mla ? 1 : 0) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}

}  // namespace attn
}  // namespace dspark
