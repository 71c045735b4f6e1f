// The attention work list, built by every attention CTA for itself in its prologue.
//
// Stream-K style split: the key tiles of every (request, row tile, value part, KV
// head) group are laid end to end (U units) and work-list slot c (a CTA, or a
// cluster of two) receives units [c*U/n, (c+1)*U/n) -- the same number of tiles for
// every slot, whatever the context-length mix.  A group cut by slot boundaries
// becomes pieces, one per slot it meets; such a piece is always the first or the
// last piece of its slot and writes partial (o, lse) rows into partial slot 2c or
// 2c + 1.  The slot that runs the last piece of a split group records the group for
// the combine.
//
// Every CTA reads the request table (ctx_len, cu_seqlens), scans it, counts the
// groups each slot's range meets (they are consecutive: the difference of two group
// indices), scans the counts for its own first item, and writes its own items: piece
// k of slot c is a piece of group first_c + k.  So there is no separate work-list
// launch between the packer and the attention.
#pragma once

#include <stdint.h>

#include "attn.h"
#include "common.cuh"
#include "ptx.cuh"

namespace dspark {
namespace attn {

// Shared-memory scratch of build_items (a region the kernel uses only later).
struct WorkScratch {
  long long off[DSPARK_MAX_B + 1];  // first unit of request r
  int goff[DSPARK_MAX_B + 1];       // first group of request r
  int tt[DSPARK_MAX_B];             // tiles per group of request r
  int n[DSPARK_MAX_B];
  int ctx[DSPARK_MAX_B];
  int c0[DSPARK_MAX_B];
  int cnt[1024];                    // items of slot c
  long long w64[32];
  int w32[32];
  int res[4];
};

namespace work {

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

// Exclusive scan over the block (blockDim.x a multiple of 32); *total = the sum.
template <class T>
__device__ __forceinline__ T block_excl_scan(T v, T* s_w, T* total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
  const T incl = warp_incl_scan(v, lane);
  if (lane == 31) s_w[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    T x = lane < nw ? s_w[lane] : T(0);
    x = warp_incl_scan(x, lane);
    s_w[lane] = x;
  }
  __syncthreads();
  const T ex = (wid > 0 ? s_w[wid - 1] : T(0)) + incl - v;
  *total = s_w[nw - 1];
  __syncthreads();  // s_w may be reused by the next scan
  return ex;
}

__device__ __forceinline__ int block_max(int v, int* s_w) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  if (lane == 0) s_w[wid] = v;
  __syncthreads();
  v = lane < nw ? s_w[lane] : 0;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
  __syncthreads();
  return v;
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

// Two exclusive scans over the block in one pass (one barrier round); blockDim.x a
// multiple of 32.
template <class T1, class T2>
__device__ __forceinline__ void block_excl_scan2(T1 v1, T2 v2, T1* s1, T2* s2, T1* ex1, T2* ex2,
                                                 T1* tot1, T2* tot2) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int nw = static_cast<int>(blockDim.x >> 5);
  const T1 i1 = warp_incl_scan(v1, lane);
  const T2 i2 = warp_incl_scan(v2, lane);
  if (lane == 31) {
    s1[wid] = i1;
    s2[wid] = i2;
  }
  __syncthreads();
  if (wid == 0) {
    T1 x1 = lane < nw ? s1[lane] : T1(0);
    T2 x2 = lane < nw ? s2[lane] : T2(0);
    x1 = warp_incl_scan(x1, lane);
    x2 = warp_incl_scan(x2, lane);
    s1[lane] = x1;
    s2[lane] = x2;
  }
  __syncthreads();
  *ex1 = (wid > 0 ? s1[wid - 1] : T1(0)) + i1 - v1;
  *ex2 = (wid > 0 ? s2[wid - 1] : T2(0)) + i2 - v2;
  *tot1 = s1[nw - 1];
  *tot2 = s2[nw - 1];
}

}  // namespace work

// Items of work-list slot `cs` into s_items[0 .. min(count, n_smem)) and, when
// write_global, into a.items[base .. base + count) (with groups[cs]).  Call from every
// thread of the CTA after the inputs are visible (after pdl_wait); it ends with a
// barrier.  Returns the count; *base_out the slot's first global index.  A request
// table that does not fit (cu_seqlens[B] > max_rows, or more pieces than max_items)
// raises the matching device error and yields no items.
//
// Unit arithmetic runs in 32 bits when n_slots * U < 2^32 (every realistic step), in
// 64 bits otherwise: the result is the same, the 64-bit divisions are only slower.
template <class UT>
__device__ __forceinline__ int build_items_t(const WorkArgs& a, int cs, WorkScratch* w,
                                             AttnItem* s_items, int n_smem, bool write_global,
                                             int* base_out, long long U64, int n_eff,
                                             bool fits_rows) {
  using namespace work;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int ngpt = a.parts * a.Hkv;
  const UT U = static_cast<UT>(U64);
  const UT ne = static_cast<UT>(n_eff);
  // ---- slots: the groups each range meets
  const int cper = (a.n_slots + nthr - 1) / nthr;
  const int c_lo = min(a.n_slots, tid * cper), c_hi = min(a.n_slots, c_lo + cper);
  int c_sum = 0;
  for (int c = c_lo; c < c_hi; ++c) {
    int cnt = 0;
    if (c < n_eff && U > 0) {
      const UT lo = static_cast<UT>(c) * U / ne;
      const UT hi = static_cast<UT>(c + 1) * U / ne;
      const int r0 = last_at_or_below(w->off, a.B, static_cast<long long>(lo));
      const int r1 = last_at_or_below(w->off, a.B, static_cast<long long>(hi - 1));
      const int gf = w->goff[r0] + static_cast<int>((lo - static_cast<UT>(w->off[r0])) /
                                                    static_cast<UT>(w->tt[r0]));
      const int gl = w->goff[r1] + static_cast<int>((hi - 1 - static_cast<UT>(w->off[r1])) /
                                                    static_cast<UT>(w->tt[r1]));
      cnt = gl - gf + 1;
    }
    w->cnt[c] = cnt;
    c_sum += cnt;
  }
  int total;
  const int c_ex = block_excl_scan(c_sum, w->w32, &total);
  if (cs >= c_lo && cs < c_hi) {
    int b = c_ex;
    for (int c = c_lo; c < cs; ++c) b += w->cnt[c];
    w->res[0] = b;
  }
  __syncthreads();
  const int base = w->res[0];
  const bool fits = fits_rows && total <= a.max_items;
  const int cnt = fits ? w->cnt[cs] : 0;
  if (!fits && tid == 0 && cs == 0 && write_global)
    raise_error(a.err, fits_rows ? DSPARK_DEVERR_WORK_OVERFLOW : DSPARK_DEVERR_ROWS_OVERFLOW);
  // ---- this slot's items
  UT lo = 0, hi = 0;
  int gfirst = 0;
  if (cnt > 0) {
    lo = static_cast<UT>(cs) * U / ne;
    hi = static_cast<UT>(cs + 1) * U / ne;
    const int r0 = last_at_or_below(w->off, a.B, static_cast<long long>(lo));
    gfirst = w->goff[r0] + static_cast<int>((lo - static_cast<UT>(w->off[r0])) /
                                            static_cast<UT>(w->tt[r0]));
  }
  auto cta_of = [&](UT x) { return static_cast<int>(((x + 1) * ne - 1) / U); };
  for (int k = tid; k < cnt; k += nthr) {
    const int g = gfirst + k;
    const int r = last_at_or_below(w->goff, a.B, g);
    const int lg = g - w->goff[r];                  // group within the request
    const int t_r = w->tt[r];
    const UT gstart = static_cast<UT>(w->off[r]) + static_cast<UT>(lg) * static_cast<UT>(t_r);
    const UT gend = gstart + static_cast<UT>(t_r);
    const int c_first = cta_of(gstart);
    const int c_last = cta_of(gend - 1);
    const int t = lg / ngpt, p = (lg / a.Hkv) % a.parts, h = lg % a.Hkv;
    const int i0 = t * a.rows_per_tile;
    const UT u0 = gstart > lo ? gstart : lo;
    const UT u1 = gend < hi ? gend : hi;
    AttnItem it;
    it.r = r; it.kvh = h; it.i0 = i0; it.ni = min(a.rows_per_tile, w->n[r] - i0);
    it.part = p; it.split = cs - c_first;
    it.tb = static_cast<int>(u0 - gstart);
    it.te = static_cast<int>(u1 - gstart);
    it.nsplit = c_last - c_first + 1;
    it.slot = u0 == lo ? 2 * cs : 2 * cs + 1;
    it.pad0 = 0; it.pad1 = 0;
    it.ctx = w->ctx[r]; it.c0 = w->c0[r]; it.n_r = w->n[r]; it.pad2 = 0;
    if (k < n_smem) s_items[k] = it;
    if (write_global) a.items[base + k] = it;
  }
  // the split group whose last piece runs here: only the slot's first group can have
  // started before the range
  if (tid == 0 && write_global) {
    SplitGroup sg{};
    if (cnt > 0) {
      const int r = last_at_or_below(w->goff, a.B, gfirst);
      const int lg = gfirst - w->goff[r];
      const int t_r = w->tt[r];
      const UT gstart = static_cast<UT>(w->off[r]) + static_cast<UT>(lg) * static_cast<UT>(t_r);
      const UT gend = gstart + static_cast<UT>(t_r);
      if (gstart < lo && gend <= hi) {
        const int c_first = cta_of(gstart);
        sg.r = r;
        sg.kvh = lg % a.Hkv;
        sg.part = (lg / a.Hkv) % a.parts;
        sg.i0 = (lg / ngpt) * a.rows_per_tile;
        sg.ni = min(a.rows_per_tile, w->n[r] - sg.i0);
        sg.c_first = c_first;
        sg.nsplit = cs - c_first + 1;
        sg.slot0_last = gstart != static_cast<UT>(c_first) * U / ne;
      }
    }
    a.groups[cs] = sg;
  }
  *base_out = base;
  ptx::fence_proxy_async_smem();  // the scratch is reused by TMA (async proxy) later
  __syncthreads();
  return cnt;
}

__device__ __forceinline__ int build_items(const WorkArgs& a, int cs, WorkScratch* w,
                                           AttnItem* s_items, int n_smem, bool write_global,
                                           int* base_out) {
  using namespace work;
  const int tid = threadIdx.x, nthr = blockDim.x;
  const int ngpt = a.parts * a.Hkv;
  // ---- requests: a contiguous chunk per thread; every load issued before any use
  const int per = (a.B + nthr - 1) / nthr;
  const int r_lo = min(a.B, tid * per), r_hi = min(a.B, r_lo + per);
  const int m_total = a.cu_seqlens[a.B];
  long long u_sum = 0;
  int g_sum = 0, tmax = 0;
  for (int r = r_lo; r < r_hi; ++r) {
    const int c0 = a.cu_seqlens[r];
    const int c1 = a.cu_seqlens[r + 1];
    const int ctx = a.ctx_len[r];
    const int n = c1 - c0;
    const int tt = ceil_div(ctx, a.NK) + ceil_div(n, a.NK);
    const int ngr = ceil_div(n, a.rows_per_tile) * ngpt;
    w->tt[r] = tt;
    w->n[r] = n;
    w->ctx[r] = ctx;
    w->c0[r] = c0;
    u_sum += (long long)tt * ngr;
    g_sum += ngr;
    tmax = max(tmax, tt);
  }
  const bool fits_rows = m_total <= a.max_rows;
  tmax = block_max(tmax, w->w32);
  long long U, u_ex;
  int NG, g_ex;
  block_excl_scan2(u_sum, g_sum, w->w64, w->w32, &u_ex, &g_ex, &U, &NG);
  {
    long long uo = u_ex;
    int go = g_ex;
    for (int r = r_lo; r < r_hi; ++r) {
      const int ngr = ceil_div(w->n[r], a.rows_per_tile) * ngpt;
      w->off[r] = uo;
      w->goff[r] = go;
      uo += (long long)w->tt[r] * ngr;
      go += ngr;
    }
  }
  if (tid == 0) {
    w->off[a.B] = U;
    w->goff[a.B] = NG;
  }
  // No group may be cut into more than max_splits pieces.  Every slot range holds at
  // least L = floor(U/n) units, and a group of T units meets at most
  // ceil((T-1)/L) + 1 ranges, so L >= ceil((T_max-1)/(max_splits-1)) suffices:
  // n <= U / that.  Then n <= U too, so no slot range is empty and the pieces of a
  // group sit in consecutive slots.
  int n_eff = a.n_slots;
  {
    long long l_req = tmax > 1 ? ((long long)tmax - 1 + a.max_splits - 2) / (a.max_splits - 1) : 1;
    if (l_req < 1) l_req = 1;
    const long long cap = U / l_req;
    if (cap < n_eff) n_eff = cap > 0 ? static_cast<int>(cap) : 1;
  }
  __syncthreads();
  if ((unsigned long long)U * (unsigned long long)(a.n_slots + 1) < (1ull << 32))
    return build_items_t<uint32_t>(a, cs, w, s_items, n_smem, write_global, base_out, U, n_eff,
                                   fits_rows);
  return build_items_t<unsigned long long>(a, cs, w, s_items, n_smem, write_global, base_out, U,
                                           n_eff, fits_rows);
}

}  // namespace attn
}  // namespace dspark
