// Internal interface of the verify-attention launchers (host side).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

namespace dspark {
namespace attn {

// One unit of work: a tile of query rows of one request against a range of its key tiles
// (tiles tb .. te-1 of the request's ceil(ctx/nk) cache tiles followed by its block
// tiles; in the latent-KV work list the range may pass the tile count T and then
// wraps: tile t >= T means t - T); nsplit = the group's piece count (1: not split); a
// piece of a split group writes
// partial rows into partial slot `slot`: 2c for the first piece of CTA c, 2c + 1 for
// its last (a split piece is always one of the two).
struct __align__(16) AttnItem {
  int r, kvh, i0, ni;        // request, KV head, first block row, block rows in the tile
  int part, split, tb, te;   // value-column part, split index, key-tile range [tb, te)
  int nsplit, slot, pad0, pad1;
  int ctx, c0, n_r, pad2;    // request r: ctx_len, cu_seqlens[r], segment rows
};

// A (request, row tile, part, KV head) group whose key range was cut into pieces,
// recorded at the index of the CTA that runs its last piece (nsplit = 0: none).
// Piece s runs on CTA c_first + s; its partial slot is 2 (c_first + s), except for
// piece 0 when it is the last but not the first piece of CTA c_first (slot0_last):
// then 2 c_first + 1.
struct __align__(16) SplitGroup {
  int r, kvh, part, i0;
  int ni, c_first, nsplit, slot0_last;
};

struct Plan {
  bool mla;
  int parts, rows_per_tile, nk, nt, d_part, ncta;
  long long max_items;
  size_t off_items, off_begin, off_groups, off_o, off_lse, bytes;
};

Plan plan(int B, int max_rows, int Hq, int Hkv, int d_qk, int d_v, int max_splits,
          int max_block_rows);

int launch(const void* q, const void* k_new, const void* v_new, const void* k_cache,
           const void* v_cache, int n_pages, const int32_t* page_table, int max_pages,
           const int32_t* ctx_len, const int32_t* cu_seqlens, int B, int max_rows, int Hq, int Hkv,
           int d_qk, int d_v, int page_size, float scale, int max_splits, float* out, float* lse,
           void* ws, const Plan& pl, cudaStream_t stream, bool planned = false);

namespace gqa {
// Query-row tile (32, 64 or 128) for G = Hq/Hkv heads per KV head and
// max_block_rows rows per request segment (<= 0 counts as 1); a longer segment
// runs as several row tiles.
int query_tile(int Hq, int Hkv, int max_block_rows);
int launch_kernel(int nt, const void* q, const void* k_new, const void* v_new, const void* k_cache,
                  const void* v_cache, int n_pages, const int32_t* page_table, int max_pages,
                  const int32_t* ctx_len, const int32_t* cu_seqlens, int B, int max_rows, int Hq,
                  int Hkv, int page_size, float scale, const AttnItem* items,
                  const int* item_begin, int grid, float* out, float* lse, float* ws_o,
                  float* ws_lse, cudaStream_t stream);
constexpr int kKeyTile = 128;
// bf16 tiled tensor map, 128-byte swizzle (rank <= 5; strides in bytes of dims 1..).
bool encode_bf16_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                     const uint64_t* strides, const uint32_t* box);
// The same for fp32 data without swizzle (rows land in shared memory packed).
bool encode_f32_map(CUtensorMap* m, const void* base, int rank, const uint64_t* dims,
                    const uint64_t* strides, const uint32_t* box);
}  // namespace gqa

namespace mla {
constexpr int kKeyTile = 64;
// Two-CTA clusters that can be resident at once (the kernel's grid, in clusters).
int clusters();
int launch_kernel(const void* q, const void* k_new, const void* k_cache, int n_pages,
                  const int32_t* page_table, int max_pages, int max_rows, int page_size,
                  float scale, const AttnItem* items, const int* item_begin, int n_clusters,
                  float* out, float* lse, float* ws_o, float* ws_lse, cudaStream_t stream);
}  // namespace mla

}  // namespace attn
}  // namespace dspark
