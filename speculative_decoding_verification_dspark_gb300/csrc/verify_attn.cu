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
#include "worklist.cuh"

namespace dspark {
namespace attn {

using namespace ptx;

constexpr int kRows = 128;  // query rows of one work item (UMMA M / N side)

// ---------------------------------------------------------------- work list
// (build_work_list in worklist.cuh)
__global__ void __launch_bounds__(1024)
    worklist_kernel(const int32_t* __restrict__ ctx_len, const int32_t* __restrict__ cu_seqlens,
                    int B, int max_rows, int Hkv, int parts, int rows_per_tile, int NK, int ncta,
                    int max_splits, int rotate, int max_items, AttnItem* __restrict__ items,
                    int* __restrict__ item_begin, SplitGroup* __restrict__ groups,
                    unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  __shared__ WorkListSmem S;
  build_work_list(S, ctx_len, cu_seqlens, B, max_rows, Hkv, parts, rows_per_tile, NK, ncta,
                  max_splits, rotate, max_items, items, item_begin, groups, err);
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
                   float* __restrict__ out, float* __restrict__ lse, int mla, int B, int max_rows,
                   unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  // packed rows beyond the call's buffers: the work list ran nothing; say so here too,
  // for the call whose work list was built by the pack call
  if (blockIdx.x == 0 && blockIdx.y == 0 && threadIdx.x == 0 && cu_seqlens[B] > max_rows)
    raise_error(err, DSPARK_DEVERR_ROWS_OVERFLOW);
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
           void* ws, const Plan& pl, cudaStream_t stream, bool planned) {
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

  // planned: the pack call already wrote the work list (same plan) into ws
  if (!planned &&
      launch_pdl(worklist_kernel, dim3(1), dim3(1024), 0, stream, ctx_len, cu_seqlens, B, max_rows,
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
                 Hq, kRows, pl.d_part, d_v, ws_o, ws_lse, out, lse, pl.mla ? 1 : 0, B, max_rows,
                 err) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}

}  // namespace attn
}  // namespace dspark
