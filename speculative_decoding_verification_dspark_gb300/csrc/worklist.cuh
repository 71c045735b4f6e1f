// Attention work list: built by its own kernel before the attention call, or by the
// pack kernel in the same launch (dspark_pack_plan).  One CTA of 1024 threads.
#pragma once

#include <stdint.h>

#include "attn.h"
#include "common.cuh"

namespace dspark {
namespace attn {

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

// Shared memory of build_work_list (about 45 KB).
struct WorkListSmem {
  long long off[DSPARK_MAX_B + 1];
  int goff[DSPARK_MAX_B + 1];
  int tt[DSPARK_MAX_B];
  int n[DSPARK_MAX_B];
  int ctx[DSPARK_MAX_B];
  int c0[DSPARK_MAX_B];
  int base[1024];
  int gfirst[1024];
  long long lo[1025];
  long long w64[32];
  int w32[32];
};

// Called by every thread of a 1024-thread CTA, after the inputs are visible to it.
// cu_seqlens is not __restrict__: in the pack kernel this CTA has just written it, so
// its loads must not take the read-only (non-coherent) path.
__device__ inline void build_work_list(WorkListSmem& S, const int32_t* __restrict__ ctx_len,
                                       const int32_t* cu_seqlens, int B, int max_rows,
                                       int Hkv, int parts, int rows_per_tile, int NK, int ncta,
                                       int max_splits, int rotate, int max_items,
                                       AttnItem* __restrict__ items, int* __restrict__ item_begin,
                                       SplitGroup* __restrict__ groups,
                                       unsigned int* __restrict__ err) {
  long long* s_off = S.off;    // first unit of request r
  int* s_goff = S.goff;         // first group of request r
  int* s_tt = S.tt;             // tiles per group of request r
  int* s_n = S.n;
  int* s_ctx = S.ctx;
  int* s_c0 = S.c0;
  int* s_base = S.base;         // first item of CTA c
  int* s_gfirst = S.gfirst;     // first group CTA c meets
  long long* s_lo = S.lo;       // first unit of CTA c: c*U/n
  long long* s_w64 = S.w64;
  int* s_w32 = S.w32;
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

}  // namespace attn
}  // namespace dspark
