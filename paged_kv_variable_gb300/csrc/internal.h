// Internal layout shared by the host plan and the device kernels.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/pkv.h"

namespace pkv {

constexpr int kKvTile = 128;        // keys per K/V tile (one pipeline stage)
constexpr int kDecodeRows = 16;     // rows (query tokens x G) of a decode tile
constexpr int kPrefillRowsTc = 128;  // rows of a prefill tile (tcgen05, one TMEM lane per row)
constexpr int kBoxRows = 8;         // smallest TMA box (cache rows, 1 KB at 128 B a row, so every box
                                    // starts on a 128-byte-swizzle atom); every page size is a multiple

// Keys per K/V tile of the attention kernel: 128, or 64 at head_dim 256.
inline int kv_tile_keys(int head_dim) { return head_dim == 256 ? 64 : kKvTile; }

// Query rows a decode (warp-MMA) tile holds: 16, or 8 at head_dim 256.
inline int decode_rows(int head_dim) { return head_dim == 256 ? 8 : kDecodeRows; }

// Rows per TMA box for a cache: for a contiguous cache the largest power of
// two (8..tile) not above its capacity, else the largest power of two
// (8..tile) dividing the page size, so a box never crosses a page or a tile.
inline int cache_box_rows(int page_size, int capacity, int tile) {
  int r = tile;
  if (page_size <= 0) {
    while (r > kBoxRows && r > capacity) r >>= 1;
  } else {
    while (page_size % r != 0) r >>= 1;
  }
  return r;
}

enum ItemKind : int32_t { kDecode = 0, kPrefill = 1 };

// Heads of one query-head group that a tensor-core tile holds: the whole
// group up to 128 heads; larger groups are cut into sub-groups of 128.
#ifdef __CUDACC__
#define PKV_HOST_DEVICE __host__ __device__
#else
#define PKV_HOST_DEVICE
#endif
PKV_HOST_DEVICE inline int tc_group_heads(int G) { return G < kPrefillRowsTc ? G : kPrefillRowsTc; }

// Query tiles of 128 rows a tensor-core prefill item may hold: two over an
// fp8 cache at head_dim <= 128, whose K/V tiles (converted to f16 once) then
// serve both, each with its own S and O in tensor memory and its own softmax
// warpgroup; one otherwise (a bf16 cache measured slower with two).  The plan
// pairs tiles only in plans without decode tiles.
PKV_HOST_DEVICE constexpr int prefill_q_tiles(int head_dim, bool fp8) { return fp8 && head_dim <= 128 ? 2 : 1; }

// One tile of work for one persistent CTA.  Rows of the tile are
// (query token, head of the tile's head sub-group) pairs: row r = token * nh + g,
// query head = hk * G + h0 + g.
struct WorkItem {
  int32_t b;         // sequence
  int32_t hk;        // kv head
  int32_t q_row0;    // packed-q index of the tile's first query token (prefix sums of the plan's
                     // lengths; with rows placed by the caller, cu_seqlens_q[b] + q_i0 instead)
  int32_t q_i0;      // index of that token within its sequence
  int32_t n_q;       // query tokens in the tile
  int32_t lq;        // query length of the sequence
  int32_t lk;        // attended keys of the sequence (cache + new)
  int32_t kv_begin;  // key range of this item, kv_begin a multiple of kKvTile
  int32_t kv_end;
  int32_t kind;      // ItemKind
  int32_t partial;   // -1: write the final output; else the first partial slot (16 rows each)
  int32_t h0;        // first query head of the group in this tile
  int32_t nh;        // heads of the group in this tile (rows = n_q * nh)
  int32_t pad[3];
};
static_assert(sizeof(WorkItem) == 64, "WorkItem layout");

// A unit split into KV chunks, merged by the combine kernel: chunk s wrote
// rows [0, n_q * nh) starting at partial slot slot0 + s * slot_stride.
struct CombineItem {
  int32_t b;            // sequence
  int32_t q_row0;       // its first query row when rows are packed (else cu_seqlens_q[b])
  int32_t n_q;
  int32_t hk;
  int32_t nsplit;
  int32_t slot0;
  int32_t slot_stride;  // 16-row slots per chunk: ceil(n_q * nh / 16)
  int32_t h0;
  int32_t nh;
  int32_t pad[3];
};
static_assert(sizeof(CombineItem) == 48, "CombineItem layout");

// Byte offsets of the sections of the caller's workspace.
struct WorkspaceLayout {
  size_t status;        // int32[4]: code, info0, info1, info2
  size_t items;         // WorkItem[num_items], grouped by CTA
  size_t cta_begin;     // int32[num_ctas + 1]
  size_t combine;       // CombineItem[num_combine]
  size_t plan_lc;       // int32[B] cache lengths the plan was made for
  size_t partial_o;     // float[num_slots * kDecodeRows * D]
  size_t partial_lse;   // float[num_slots * kDecodeRows] (log2 domain)
  size_t total;
};

}  // namespace pkv

// Host plan object (opaque to callers).
struct pkv_plan_s {
  pkv_problem problem;
  int32_t num_ctas;
  int32_t num_slots;
  int32_t total_q;
  int32_t total_new;
  int32_t max_items_per_cta;
  int32_t num_decode_items, num_prefill_items, num_split_units;
  double max_cta_cost, mean_cta_cost;
  pkv::WorkspaceLayout layout;
  // host staging image of the workspace head (everything except partials)
  unsigned char* image;
  size_t image_bytes;
  int32_t num_items;
  int32_t num_combine;
  int32_t dynamic;  // cache lengths read on the device; plan_lc holds their bounds
  double* item_cost;  // [num_items] model cost of each item, in work-list order
};

namespace pkv {
// thread-local error message helpers (api.cu)
pkv_status fail(pkv_status st, const char* fmt, ...);
// host checks of an attention call other than its workspace (api.cu)
pkv_status validate_call(const pkv_problem* problem, const pkv_fwd_args* args, pkv_plan_t plan);
}  // namespace pkv
