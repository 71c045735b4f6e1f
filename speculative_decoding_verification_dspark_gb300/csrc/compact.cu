// Commit of the verification step: compact scatter of the accepted KV rows and
// page-table append ("DFlash 到 DSpark in SGLang", section "Zero-overhead
// scheduling 与 kernel": a fused compact-scatter kernel and a device-resident page
// table, so the step needs no host synchronisation).
//
//   compact_alloc_kernel  one CTA, one thread per request: new-page counts, an
//                         exclusive scan that assigns pages from the top of the
//                         free stack in request order, page-table append,
//                         ctx_len / anchor / committed-token updates.  If the stack
//                         or a page-table row is too short nothing is changed.
//   compact_copy_kernel   one CTA per (request, kept row): 16-byte copies of the
//                         K (and V) row into its cache slot.

#include <cuda_runtime.h>
#include <stdint.h>

#include "common.cuh"
#include "kernels.h"

namespace dspark {

namespace {

struct CompactWs {
  int ok;
  int pad[63];
};

__device__ __forceinline__ int warp_incl_scan(int v) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int u = __shfl_up_sync(0xffffffffu, v, o);
    if (lane >= o) v += u;
  }
  return v;
}

}  // namespace

__global__ void __launch_bounds__(1024)
    compact_alloc_kernel(const int32_t* __restrict__ cu, int max_rows,
                         const int32_t* __restrict__ accept_len, const int32_t* __restrict__ out_tok,
                         const int32_t* __restrict__ draft_tok, int B, int gamma, int page_size,
                         int max_pages, int n_pages, int32_t* __restrict__ page_table,
                         int32_t* __restrict__ ctx_len, int32_t* __restrict__ anchor,
                         const int32_t* __restrict__ free_pages, int32_t* __restrict__ free_top,
                         int32_t* __restrict__ committed, int32_t* __restrict__ n_committed,
                         CompactWs* __restrict__ cws, int* __restrict__ old_ctx,
                         unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  __shared__ int s_warp[32];
  __shared__ int s_flags;
  __shared__ int s_top;
  const int tid = threadIdx.x;
  if (tid == 0) {
    cws->ok = 0;
    s_flags = cu[B] > max_rows ? DSPARK_DEVERR_ROWS_OVERFLOW : 0;
    s_top = *free_top;
  }
  __syncthreads();
  int L = 0, c0 = 0, keep = 0, have = 0, need = 0, nn = 0;
  if (tid < B) {
    L = accept_len[tid];
    if (L < 0 || L > gamma) {
      atomicOr(&s_flags, DSPARK_DEVERR_BAD_INPUT);
      L = L < 0 ? 0 : gamma;
    }
    keep = L + 1;
    if (keep > cu[tid + 1] - cu[tid]) atomicOr(&s_flags, DSPARK_DEVERR_BAD_INPUT);  // unverified rows
    c0 = ctx_len[tid];
    have = ceil_div(c0, page_size);
    need = ceil_div(c0 + keep, page_size);
    nn = need - have;
    if (need > max_pages) atomicOr(&s_flags, DSPARK_DEVERR_PAGE_ROW_FULL);
  }
  const int incl = warp_incl_scan(nn);
  if ((tid & 31) == 31) s_warp[tid >> 5] = incl;
  __syncthreads();
  if (tid < 32) {
    int w = s_warp[tid];
    w = warp_incl_scan(w);
    s_warp[tid] = w;
  }
  __syncthreads();
  const int off = ((tid >> 5) ? s_warp[(tid >> 5) - 1] : 0) + incl - nn;
  const int total = s_warp[31];
  if (tid == 0 && total > s_top) atomicOr(&s_flags, DSPARK_DEVERR_NO_FREE_PAGE);
  __syncthreads();
  if (s_flags) {
    if (tid == 0) raise_error(err, s_flags);
    return;
  }
  if (tid < B) {
    for (int k = 0; k < nn; ++k) {
      int page = free_pages[s_top - 1 - off - k];
      if (page < 0 || page >= n_pages) {
        raise_error(err, DSPARK_DEVERR_BAD_INPUT);
        page = 0;
      }
      page_table[(long long)tid * max_pages + have + k] = page;
    }
    old_ctx[tid] = c0;
    ctx_len[tid] = c0 + keep;
    const int tok = out_tok[tid];
    anchor[tid] = tok;
    for (int i = 0; i <= gamma; ++i)
      committed[tid * (gamma + 1) + i] = (i < L) ? draft_tok[tid * gamma + i] : (i == L ? tok : -1);
    n_committed[tid] = keep;
  }
  __syncthreads();
  if (tid == 0) {
    *free_top = s_top - total;
    cws->ok = 1;
  }
}

__global__ void __launch_bounds__(128)
    compact_copy_kernel(const uint8_t* __restrict__ k_new, const uint8_t* __restrict__ v_new,
                        int row_bytes, const int32_t* __restrict__ cu,
                        const int32_t* __restrict__ accept_len, int gamma, int page_size,
                        int max_pages, int n_pages, const int32_t* __restrict__ page_table,
                        const int* __restrict__ old_ctx, const CompactWs* __restrict__ cws,
                        uint8_t* __restrict__ k_cache, uint8_t* __restrict__ v_cache,
                        unsigned int* __restrict__ err) {
  pdl_release();
  pdl_wait();  // inputs come from the kernels before this one
  const int r = blockIdx.x;
  const int i = blockIdx.y;
  if (!cws->ok) return;
  int L = accept_len[r];
  L = L < 0 ? 0 : (L > gamma ? gamma : L);
  if (i > L) return;
  const int pos = old_ctx[r] + i;
  const int page = page_table[(long long)r * max_pages + pos / page_size];
  if (page < 0 || page >= n_pages) {
    if (threadIdx.x == 0) raise_error(err, DSPARK_DEVERR_BAD_INPUT);
    return;
  }
  const long long dst = ((long long)page * page_size + pos % page_size) * row_bytes;
  const long long src = (long long)(cu[r] + i) * row_bytes;
  for (int b = threadIdx.x * 16; b < row_bytes; b += blockDim.x * 16) {
    *reinterpret_cast<uint4*>(k_cache + dst + b) =
        *reinterpret_cast<const uint4*>(k_new + src + b);
    if (v_new)
      *reinterpret_cast<uint4*>(v_cache + dst + b) =
          *reinterpret_cast<const uint4*>(v_new + src + b);
  }
}

size_t compact_workspace(int B) { return sizeof(CompactWs) + (((size_t)B * sizeof(int) + 255) & ~size_t(255)); }

int launch_compact(const void* k_new, const void* v_new, int row_bytes, int max_rows,
                   const int32_t* cu,
                   const int32_t* accept_len, const int32_t* out_tok, const int32_t* draft_tok,
                   int B, int gamma, int page_size, int max_pages, int n_pages, int32_t* page_table,
                   int32_t* ctx_len, int32_t* anchor, const int32_t* free_pages, int32_t* free_top,
                   void* k_cache, void* v_cache, int32_t* committed, int32_t* n_committed, void* ws,
                   cudaStream_t stream) {
  CompactWs* cws = static_cast<CompactWs*>(ws);
  int* old_ctx = reinterpret_cast<int*>(static_cast<uint8_t*>(ws) + sizeof(CompactWs));
  if (launch_pdl(compact_alloc_kernel, dim3(1), dim3(1024), 0, stream, cu, max_rows, accept_len,
                 out_tok, draft_tok, B, gamma, page_size, max_pages, n_pages, page_table, ctx_len,
                 anchor, free_pages, free_top, committed, n_committed, cws, old_ctx,
                 device_error_word()) != cudaSuccess)
    return DSPARK_ECUDA;
  dim3 grid(B, gamma + 1);
  if (launch_pdl(compact_copy_kernel, grid, dim3(128), 0, stream, static_cast<const uint8_t*>(k_new),
                 static_cast<const uint8_t*>(v_new), row_bytes, cu, accept_len, gamma, page_size,
                 max_pages, n_pages, page_table, old_ctx, cws, static_cast<uint8_t*>(k_cache),
                 static_cast<uint8_t*>(v_cache), device_error_word()) != cudaSuccess)
    return DSPARK_ECUDA;
  return DSPARK_OK;
}

}  // namespace dspark
