// Varlen verify attention over a paged KV cache, causal inside the draft block.
//
// What it computes ("DFlash 到 DSpark in SGLang", section "Ragged verify under
// full CUDA graphs": the packed verify tokens each attend only to their own
// request's KV): packed row cu_seqlens[r] + i, query head h, attends to the
// ctx_len[r] committed keys of request r (read through its page table) and to
// block rows 0..i of its own segment; o = softmax(scale q.K^T) V, lse = log-sum-exp.
//
// This file holds what both head shapes share: the work list, the split combine
// and the host planner.  The kernels themselves:
//   * GQA (head dim 128): verify_attn_gqa.cu, keys on the MMA's M side, one CTA
//     per SM persistent over its range of the work list;
//   * latent KV (576/512): verify_attn_mla.cu, one block row's 128 heads on a
//     cluster of two CTAs that split the value dims and the QK^T reduction.
// A work item = (request, KV head, block-row tile, value-column part, KV split);
// long contexts split across items, and a log-sum-exp combine merges the pieces.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "attn.h"
#include "common.cuh"
#include "ptx.cuh"

namespace dspark {
namespace attn {

using namespace ptx;

constexpr int kRows = 128;  // query rows of one work item (UMMA M / N side)

// ---------------------------------------------------------------- work list
// One CTA.  Stream-K style split: the key tiles of every (request, row tile, value
// part, KV head) group are laid end to end (U units) and CTA c of the persistent
// grid receives units [c*U/n, (c+1)*U/n) -- the same number of tiles for every
// CTA, whatever the context-length mix.  A group cut by CTA boundaries becomes
// pieces, one per CTA it meets; such a piece is always the first or the last piece
// of its CTA and writes partial (o, lse) rows into slot 2c or 2c + 1.  The CTA that
// runs the last piece of a split group records the group for the combine.
//
// Latent-KV items take their group's tiles in a rotated order (see the group loop):
// a request's block rows run as separate groups, and rotating each by the time it
// starts makes the rows that run at the same time on different clusters read the
// same key tile, which the L2 then serves once.
//
// Built in parallel: a thread per CTA counts the groups its range meets (they are
// consecutive, so the count is the difference of two group indices) and a block scan
// gives each CTA's first item; then a thread per group writes the group's pieces
// straight to their places (piece of group g in CTA c: item base_c + g - first_c).
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

// Largest r in [0, n) with off[r] <= x (off non-decreasing, off[0] = 0 <= x).
template <class T>
__device__ __forceinline__ int last_at_or_below(const T* off, int n, T x) {
  int a = 0, b = n;
  while (b - a > 1) {
    const int mid = (a + b) >> 1;
    if (off[mid] <= x) a = mid; else b = mid;
  }
  return a;
}

__global__ void __launch_bounds__(1024)
    worklist_kernel(const int32_t* __restrict__ ctx_len, const int32_t* __restrict__ cu_seqlens,
                    int B, int max_rows, int Hkv, int parts, int rows_per_tile, int NK, int ncta,
                    int max_splits, int rotate, int max_items, AttnItem* __restrict__ items,
                    int* __restrict__ item_begin, SplitGroup* __restrict__ groups,
                    unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  __shared__ long long s_off[DSPARK_MAX_B + 1];  // first unit of request r
  __shared__ int s_goff[DSPARK_MAX_B + 1];       // first group of request r
  __shared__ int s_tt[DSPARK_MAX_B];             // tiles per group of request r
  __shared__ int s_n[DSPARK_MAX_B];
  __shared__ int s_ctx[DSPARK_MAX_B];
  __shared__ int s_c0[DSPARK_MAX_B];
  __shared__ int s_base[1024];                   // first item of CTA c
  __shared__ int s_gfirst[1024];                 // first group CTA c meets
  __shared__ long long s_lo[1025];               // first unit of CTA c: c*U/n
  __shared__ long long s_w64[32];
  __shared__ int s_w32[32];
  const int tid = threadIdx.x, lane = tid & 31;
  const int ng_per_tile = parts * Hkv;
  const bool rows_ok = cu_seqlens[B] <= max_rows;  // else: report and run nothing
  long long units = 0;
  int tt = 0, ngr = 0;
  if (tid < B) {
    const int c0 = cu_seqlens[tid];
    const int n = cu_seqlens[tid + 1] - c0;
    const int ctx = ctx_len[tid];
    tt = ceil_div(ctx, NK) + ceil_div(n, NK);
    ngr = ceil_div(n, rows_per_tile) * ng_per_tile;
    units = (long long)tt * ngr;
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
  int NG;
  const int gex = block_excl_scan(ngr, s_w32, &NG);
  if (tid < B) {
    s_off[tid] = ex;
    s_goff[tid] = gex;
  }
  if (tid == 0) {
    s_off[B] = U;
    s_goff[B] = NG;
  }
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
  // The CTA boundaries, once: the CTA of a unit is then a search over them (the
  // 64-bit divisions were the kernel's longest dependency chains).  U >= n_eff, so
  // the boundaries strictly increase.
  for (int cc = tid; cc <= n_eff; cc += blockDim.x) s_lo[cc] = (long long)cc * U / n_eff;
  const bool small = U < (1ll << 31);  // unit offsets fit 32-bit division
  __syncthreads();
  // ---- per CTA: the groups its range meets
  const int c = tid;
  const bool active = c < ncta && c < n_eff && U > 0;
  int gfirst = 0, cnt = 0;
  if (active) {
    const long long lo = s_lo[c];
    const long long hi = s_lo[c + 1];
    const int r0 = last_at_or_below(s_off, B, lo);
    const int r1 = last_at_or_below(s_off, B, hi - 1);
    const long long d0 = lo - s_off[r0], d1 = hi - 1 - s_off[r1];
    gfirst = s_goff[r0] + (small ? static_cast<int>(d0) / s_tt[r0] : static_cast<int>(d0 / s_tt[r0]));
    const int glast =
        s_goff[r1] + (small ? static_cast<int>(d1) / s_tt[r1] : static_cast<int>(d1 / s_tt[r1]));
    cnt = glast - gfirst + 1;
  }
  int total;
  const int base = block_excl_scan(cnt, s_w32, &total);
  const bool fits = rows_ok && total <= max_items;
  if (tid == 0 && !fits)
    raise_error(err, rows_ok ? DSPARK_DEVERR_WORK_OVERFLOW : DSPARK_DEVERR_ROWS_OVERFLOW);
  if (c < ncta) {
    item_begin[c] = fits ? base : 0;
    s_base[c] = base;
    s_gfirst[c] = gfirst;
    SplitGroup sg{};
    groups[c] = sg;  // nsplit = 0 unless a split group ends in CTA c (written below)
  }
  if (tid == 0) item_begin[ncta] = fits ? total : 0;
  __syncthreads();
  if (!fits || U == 0) return;
  // ---- per group: its pieces
  for (int g = tid; g < NG; g += blockDim.x) {
    const int r = last_at_or_below(s_goff, B, g);
    const int lg = g - s_goff[r];                  // group within the request
    const int t_r = s_tt[r];
    const long long gstart = s_off[r] + (long long)lg * t_r;
    const long long gend = gstart + t_r;
    const int c_first = last_at_or_below(s_lo, n_eff, gstart);  // largest c: c*U/n <= x
    const int c_last = last_at_or_below(s_lo, n_eff, gend - 1);
    const int t = lg / ng_per_tile, p = (lg / Hkv) % parts, h = lg % Hkv;
    const int i0 = t * rows_per_tile;
    const int ni = min(rows_per_tile, s_n[r] - i0);
    const int nsplit = c_last - c_first + 1;
    // rotate: the group's tiles are taken in the order rot, rot + 1, ... (mod t_r),
    // rot = the time (in units) at which the group starts on its first CTA; every
    // group started this way reads tile (time mod t_r) at a given time, so the rows
    // of one request that run at the same time on different CTAs read the same tile
    const long long since = gstart - s_lo[c_first];
    const int rot = !rotate ? 0
                    : small ? static_cast<int>(since) % t_r
                            : static_cast<int>(since % t_r);
    for (int cc = c_first; cc <= c_last; ++cc) {
      const long long lo = s_lo[cc];
      const long long hi = s_lo[cc + 1];
      const long long u0 = gstart > lo ? gstart : lo;
      const long long u1 = gend < hi ? gend : hi;
      AttnItem it;
      it.r = r; it.kvh = h; it.i0 = i0; it.ni = ni;
      it.part = p; it.split = cc - c_first;
      it.tb = static_cast<int>(u0 - gstart) + rot;
      if (it.tb >= t_r) it.tb -= t_r;
      it.te = it.tb + static_cast<int>(u1 - u0);  // may pass t_r: the tile index wraps
      it.nsplit = nsplit;
      it.slot = u0 == lo ? 2 * cc : 2 * cc + 1;
      it.pad0 = 0; it.pad1 = 0;
      it.ctx = s_ctx[r]; it.c0 = s_c0[r]; it.n_r = s_n[r]; it.pad2 = 0;
      items[s_base[cc] + (g - s_gfirst[cc])] = it;
    }
    if (nsplit > 1) {
      SplitGroup sg;
      sg.r = r; sg.kvh = h; sg.part = p; sg.i0 = i0;
      sg.ni = ni; sg.c_first = c_first; sg.nsplit = nsplit;
      sg.slot0_last = gstart != s_lo[c_first];
      groups[c_last] = sg;
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

Plan plan(int B, int max_rows, int Hq, int Hkv, int d_qk, int d_v, int max_splits,
          int max_block_rows) {
  Plan p{};
  p.mla = (d_qk == 576);
  const int G = p.mla ? Hq : Hq / Hkv;
  p.parts = 1;
  p.nt = p.mla ? kRows : gqa::query_tile(Hq, Hkv, max_block_rows);
  p.rows_per_tile = p.mla ? 1 : (p.nt / G);
  p.nk = p.mla ? mla::kKeyTile : gqa::kKeyTile;
  p.d_part = d_v;
  // one work-list slot per CTA (GQA) or per two-CTA cluster (latent KV)
  p.ncta = p.mla ? mla::clusters() : num_sms_cached();
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
                 Hkv, pl.parts, pl.rows_per_tile, pl.nk, ncta, splits, pl.mla ? 1 : 0, max_items,
                 items, item_begin,
                 groups, err) != cudaSuccess)
    return DSPARK_ECUDA;

  if (pl.mla) {
    const int rc = mla::launch_kernel(q, k_new, k_cache, n_pages, page_table, max_pages, max_rows,
                                      page_size, scale, items, item_begin, ncta, out, lse, ws_o,
                                      ws_lse, stream);
    if (rc != DSPARK_OK) return rc;
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
