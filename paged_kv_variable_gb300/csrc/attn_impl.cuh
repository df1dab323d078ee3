// Persistent attention kernel over a paged or contiguous KV cache.
//
// One CTA per SM walks its host-assigned list of work items (flashinfer PR
// "[Refactor] Uniform PoDAttention API with Horizontal Fusion SMs Schedule",
// Key Changes 2: prefill and decode work share one persistent launch).
//
// Warp roles (224 threads without prefill tiles; 256 with them, 384 for an
// fp8 cache):
//   warps 0, 6  TMA producers (K and Q; V): tiles of 128 keys, boxes of up to
//               128 rows per (page, 128-byte column chunk), page numbers read from
//               block_table or a ragged page list (vLLM PR "[Kernel][Triton][FP8]
//               ...", review: block_table support; TransformerEngine PR "Add KV
//               cache for paged/non-paged attention": one table for K and V, bshd
//               pages; the kv_indptr / kv_indices form asked for in the review of
//               the cutlass-sycl PR "Extend FlashAttention Prefill with KV cache")
//               into rings of shared-memory stages (that PR's cached-KV
//               prefetch); plus the 128-row Q tile of a prefill item.  Pages of
//               1, 2 or 4 tokens are gathered row by row with cp.async.
//   warp 1      owns tensor memory and issues S = Q K^T of prefill tiles into
//               TMEM (three buffers).
//   last warp   (with prefill tiles) issues O += P V into TMEM, P read from
//               TMEM where the softmax wrote it over S.
//   warps 2..5  consumers.  Prefill tile: one query row per thread, masked
//               online softmax on S read from TMEM, P written back to TMEM for
//               the next MMA, O rescaled in TMEM, epilogue.  Decode tile
//               (<= 16 rows): warp-level MMAs, the four warps split the keys
//               of each tile and merge at the end of the item.
//   warps 7..10 (fp8 cache with prefill tiles) convert e4m3 K/V tiles and the
//               bf16 Q tile into f16 MMA operands in shared memory (with
//               q_scale: Q into e4m3 for kind::f8f6f4 MMAs on the raw K
//               tiles, and V alone into f16).
//
// fp8 caches (vLLM PR, 8-bit KV cache): decode tiles convert e4m3 to f16 in
// registers, straight into MMA fragments (exact); k_scale is folded into the
// logit scale and v_scale applied to the normalised output.
#pragma once

#include <cuda_bf16.h>

#include <atomic>

#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kConsumerWarps = 4;                  // warp-MMA consumers (decode, fp8 prefill): warps 2..5
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr float kLn2 = 0.693147180559945309f;
// Tensor memory: at D <= 128 (two query tiles per prefill item) query tile q
// has one S buffer of a tile's keys (fp32) at 256q and its O (D fp32 columns)
// at 256q + 128; at D = 256 three S buffers [0,64), [64,128), [128,192) of the
// 64-key tiles, then O [192, 448).  P of a tile (bf16 or f16 pairs: a tile's
// keys in half as many columns) overwrites the first columns of its own S
// buffer once the softmax has read S, so a buffer is free again when P V of
// its tile has completed.
constexpr uint32_t kTmemCols = 512;
constexpr int kSBufsMax = 3;          // S buffers (barrier slots); S of tile T+kSBufs waits only for P V of tile T

template <int D, bool FP8, bool PF>
struct Layout {
  // Warp roles with prefill tiles (tcgen05) at D = 256 over a bf16 cache: 0
  // K/Q producer, 1 S = Q K^T issuer, 2..5 consumers (softmax of prefill
  // tiles, warp-MMA decode tiles), 6 V producer, 7 O += P V issuer.
  // Decode-only plans: 0 K producer, 1 V producer, 2.. decode consumers.
  // Otherwise (prefill tiles at D <= 128, or an fp8 cache) the roles are
  // grouped by warpgroup so that setmaxnreg can move registers between them:
  // softmax warps first (one warpgroup per query tile of an item), then the
  // four converters of an fp8 cache (e4m3 K/V tiles and the bf16 Q tiles to
  // f16 MMA operands), then K/Q producer, S issuer, V producer, P V issuer.
  static constexpr int kD = D;
  static constexpr bool kTc = PF;                           // prefill tiles (on tcgen05) in the plan
  // query tiles of a prefill item: two over an fp8 cache at D <= 128, sharing
  // every K/V tile (each with one S buffer and its O in tensor memory, and a
  // softmax warpgroup of its own: the two tiles' MMAs run while the other's
  // softmax does, and each converted K/V tile serves both); one otherwise
  static constexpr int kQTiles = PF ? prefill_q_tiles(D, FP8) : 1;
  static constexpr bool kQQ = kQTiles == 2;
  static constexpr int kSoftmaxWarps = kConsumerWarps * kQTiles;  // one per TMEM lane quarter and query tile
  // Decode-only plans over an fp8 cache, whose tiles carry half the bytes of a
  // bf16 tile for the same arithmetic: each consumer warp copies its share of
  // a K and a V tile into registers and releases both stages at once (a stage
  // is held for a few shared-memory loads, not the tile's arithmetic).  One
  // group of consumer warps: two groups taking alternate tiles measured slower.
  static constexpr bool kStageRegs = FP8 && !PF && D <= 128;
  static constexpr int kDecGroups = 1;
  static constexpr int kDecWarps = kConsumerWarps * kDecGroups;  // decode consumer warps
  static constexpr bool kSplitRegs = PF && (FP8 || kQQ);
  static constexpr int kConvWarps = (FP8 && PF) ? 4 : 0;
  static constexpr int kCons0 = kSplitRegs ? 0 : 2;  // first consumer (softmax / decode) warp
  static constexpr int kSingle0 = kSoftmaxWarps + kConvWarps;  // (split) first single-role warp
  static constexpr int kKProdWarp = kSplitRegs ? kSingle0 : 0;
  static constexpr int kSWarp = kSplitRegs ? kSingle0 + 1 : 1;
  static constexpr int kVProducerWarp = kSplitRegs ? kSingle0 + 2 : (PF ? 2 + kSoftmaxWarps : 1);
  static constexpr int kConvWarp0 = kSplitRegs ? kSoftmaxWarps : 2 + kSoftmaxWarps + 1;
  static constexpr int kPvWarp = kSplitRegs ? kSingle0 + 3 : kConvWarp0 + kConvWarps;
  static constexpr int kThreads = PF ? 32 * (3 + kSoftmaxWarps + kConvWarps + 1) : 32 * (2 + kDecWarps);
  // registers a thread at launch (one block per SM) and, with the split, after
  // each warpgroup's setmaxnreg: softmax, converters, single-role warps
  static constexpr int kLaunchRegs = kThreads > 384 ? 128 : 168;
  static constexpr int kRegsSoftmax = kThreads > 384 ? 144 : (kQQ ? 216 : 240);
  static constexpr int kRegsConv = 152;
  static constexpr int kRegsSingle = kQQ ? 72 : 112;
  static constexpr int kEsize = FP8 ? 1 : 2;
  // keys per K/V tile (one pipeline stage): 128, or 64 at D = 256 (stages of
  // 32 KB, and TMEM for three 64-column S buffers beside a 256-column O)
  static constexpr int kTile = D == 256 ? 64 : kKvTile;
  // S buffers (per query tile); tensor memory of query tile q starts at
  // q * kQCols: its S buffers, then its O
  static constexpr int kSBufs = kQQ ? 1 : 3;
  static constexpr uint32_t kQCols = kQQ ? 256 : 0;
  static constexpr uint32_t kTmemO = kSBufs * kTile;
  static_assert((kQQ ? kQCols * kQTiles : kTmemO + D) <= kTmemCols && (!kQQ || kTmemO + D <= kQCols),
                "tensor memory budget");
  // decode-only plans give all shared memory to the rings; over an fp8 cache
  // at D <= 128 and a bf16 one at D = 64 (tiles of 128-byte rows) two CTAs
  // share an SM (each with 3 + 3 stages of 16 KB, the same bytes in flight as
  // one CTA with 6 + 6): twice the decode warps to hide the per-tile chain of
  // conversions, warp MMAs and softmax (bf16 at D = 64: 61.3 -> 55.0 us on the
  // decode batch)
  static constexpr int kCtasPerSm = (!PF && (FP8 ? D <= 128 : D == 64)) ? 2 : 1;
  static constexpr int kStagesK =
      PF ? (FP8 ? 2 : (D == 64 ? 4 : kQQ ? 2 : 3)) : (kCtasPerSm == 2 ? 3 : (FP8 || D == 64 ? 6 : 4));
  static constexpr int kStagesV =
      PF ? (FP8 ? 2 : (D == 64 ? 4 : D == 256 || kQQ ? 2 : 3)) : (kCtasPerSm == 2 ? 3 : (FP8 || D == 64 ? 6 : 3));
  static constexpr int kTileBytes = kTile * D * kEsize;     // one raw K (or V) tile
  // A raw tile is [column chunks][128 rows][kRowBytes]: 128-byte chunks with
  // the 128-byte swizzle, or (an fp8 cache at D = 64) one chunk of 64-byte
  // rows with the 64-byte swizzle.
  static constexpr int kRowBytes = D * kEsize < 128 ? D * kEsize : 128;
  static constexpr int kChunks = D * kEsize / kRowBytes;      // column chunks per cache row
  static constexpr int kKOff = 0;                             // K ring
  static constexpr int kVOff = kStagesK * kTileBytes;         // V ring
  static constexpr int kQOff = kVOff + kStagesV * kTileBytes; // Q tiles (128 x D, bf16; f16 after conversion)
  static constexpr int kQBytes = kPrefillRowsTc * D * 2;      // one Q tile
  static constexpr int kConvTile = kTile * D * 2;             // one converted (f16) K or V tile
  // converted K and V tiles: two each, or one each at D = 256 and (two query
  // tiles per item, D = 128) where shared memory is short (one more converted
  // K or V tile there measured slower)
  static constexpr int kConvBufsK = (D == 256 || (kQQ && D == 128)) ? 1 : 2;
  static constexpr int kConvBufsV = kConvBufsK;
  static constexpr int kKcOff = kQOff + (PF ? kQTiles * kQBytes : 0);  // fp8: converted K tiles
  static constexpr int kVcOff = kKcOff + (kConvWarps ? kConvBufsK * kConvTile : 0);  // fp8: converted V tiles
  // decode merge scratch: the item's last V stage, borrowed before it is
  // released, or (tiles staged in registers, every stage released at once)
  // its own area
  static constexpr int kMergeOff = kVcOff + (kConvWarps ? kConvBufsV * kConvTile : 0);
  // (tiles staged in registers: every warp's O^T of one 8-column tile, or the
  // tree's slots of two column tiles)
  static constexpr int kMergeBytes = kStageRegs ? kDecWarps * (D / 16) * 32 * 16 : 0;
  static constexpr int kMlOff = kMergeOff + kMergeBytes;     // float[kDecWarps][16][2] (m, l), int[kDecWarps]
  static constexpr int kBarOff = kMlOff + kDecWarps * kDecodeRows * 2 * 4 + kDecWarps * 4;  // + failed-wait flags
  static constexpr int kNumBars = 2 * kStagesK + 2 * kStagesV + 3 + 3 * kSBufsMax + 9 + 1 + 3;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;     // tmem base, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes;                       // base is 1024-aligned (checked in the kernel)
};

struct Bars {
  uint64_t* full_k;
  uint64_t* empty_k;
  uint64_t* full_v;
  uint64_t* empty_v;
  uint64_t* q_full;
  uint64_t* q_empty;
  // per S buffer (tile T uses T % kSBufs)
  uint64_t* s_full;   // S of the tile is in TMEM
  uint64_t* p_full;   // P of the tile is in TMEM (and O rescaled, V rows past the sequence zeroed)
  uint64_t* o_done;   // P V of the tile has completed: the buffer is free
  uint64_t* drain;    // MMA completion before tensor memory is freed after an abort
  // fp8 cache only
  uint64_t* qc_full;   // the Q tile is f16
  uint64_t* kc_full;   // [2] converted K tile ready
  uint64_t* kc_empty;  // [2] S of the tile using it has completed
  uint64_t* vc_full;   // [2] converted V tile ready
  uint64_t* vc_empty;  // [2] P V of the tile using it has completed
  uint64_t* drain_pv;  // P V MMA completion before tensor memory is freed after an abort
  // the second query tile of an item (two query tiles per item)
  uint64_t* q_full_b;
  uint64_t* q_empty_b;
  uint64_t* qc_full_b;
  __device__ __forceinline__ uint64_t* qfull(int q) const { return q ? q_full_b : q_full; }
  __device__ __forceinline__ uint64_t* qempty(int q) const { return q ? q_empty_b : q_empty; }
  __device__ __forceinline__ uint64_t* qcfull(int q) const { return q ? qc_full_b : qc_full; }
};

// Byte offset of 16-byte chunk c of row r in a tile of ROWS rows stored as
// [128-byte column chunks][ROWS rows][128 B] with the 128-byte TMA swizzle
// (bf16 K / V tiles, the Q tile, converted f16 tiles).
template <int ROWS>
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * (ROWS * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

// Byte offset of 16-byte chunk c of row r in a raw cache tile of ROWS rows
// whose column chunks are RB bytes wide: 128-byte chunks with the 128-byte TMA
// swizzle (the chunk index XOR row % 8), or (an fp8 cache at D = 64) one
// 64-byte chunk with the 64-byte swizzle (XOR (row / 2) % 4, the pattern
// repeating every 512 bytes).
template <int RB, int ROWS>
__device__ __forceinline__ uint32_t raw_off(int r, int c) {
  static_assert(RB == 128 || RB == 64, "raw tile rows");
  if constexpr (RB == 128) return tile_off<ROWS>(r, c);
  return (uint32_t)(r * 64 + ((c ^ ((r >> 1) & 3)) << 4));
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// Work item `it` as this call runs it.  Its query rows start at q_row0 of
// the plan, or (rows placed by the caller) at cu_seqlens_q[b] + q_i0.  A
// dynamic plan was made for bounds on
// the cache lengths: the sequence's current length (cache_seqlens, clamped to
// its bound) cuts the item's key range.  Every role of the kernel reads items
// through here, so they all see the same tiles.
__device__ __forceinline__ WorkItem load_item(const AttnParams& p, int it) {
  WorkItem w = p.items[it];
  // rows placed by the caller: the sequence's query rows start where
  // cu_seqlens_q says (packed rows keep the plan's prefix sums, no load)
  if (p.q_offsets != nullptr) w.q_row0 = __ldg(p.q_offsets + w.b) + w.q_i0;
  if (p.dynamic) {
    const int bound = __ldg(p.plan_lc + w.b);
    const int lc = min(max(__ldg(p.cache_seqlens + w.b), 0), bound);
    w.lk = w.lk - bound + lc;  // the plan's key count holds bound + new tokens
    w.kv_end = min(w.kv_end, w.lk);
    w.kv_begin = min(w.kv_begin, w.kv_end);
  }
  return w;
}

template <int TILE>
__device__ __forceinline__ int num_tiles(const WorkItem& w) {
  return w.kv_end > w.kv_begin ? (w.kv_end - w.kv_begin + TILE - 1) / TILE : 0;
}

// Query tile q (0 or 1) of a prefill item as an item of its own: its tokens
// (none if the item has fewer) and, causal, the keys up to its last token's.
// Every role derives the tiles of each query tile through here.
__device__ __forceinline__ WorkItem q_tile(const WorkItem& w, int q, bool causal) {
  WorkItem v = w;
  const int tq = kPrefillRowsTc / w.nh;  // query tokens of a tile
  v.q_i0 = w.q_i0 + q * tq;
  v.q_row0 = w.q_row0 + q * tq;
  v.n_q = max(0, min(tq, w.n_q - q * tq));
  if (v.n_q == 0)
    v.kv_end = v.kv_begin;
  else if (causal)
    v.kv_end = max(v.kv_begin, min(w.kv_end, v.q_i0 + v.n_q + w.lk - w.lq));
  return v;
}

struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  template <int NS>
  __device__ __forceinline__ void advance(int n = 1) {
    for (int i = 0; i < n; ++i) {
      if (++stage == NS) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
};

// Row gather of one tile (pages of P = 1, 2 or 4 tokens): lane l copies rows
// l, l+32, l+64, l+96 in 16-byte cp.async pieces into the swizzled layout
// (rows past the key range become zeros).  Row r's page is entry r / P of the
// tile, held by lane (r / P) % 32 in ent[(r / P) / 32] = ent[i / P]; pages of
// one token: each lane loads its rows' entries itself (those loads are
// coalesced already; the shuffled form measured slower).  Decode-only
// instances: the producers of instances with prefill tiles run on few
// registers and keep a simpler form.
template <int N>
struct PageEntries {
  int v[N];
};
template <class L, bool kIsV, int P>
__device__ __forceinline__ void gather_rows(const AttnParams& p, const WorkItem& w, int t0, uint8_t* stage,
                                            PageEntries<L::kTile / 32> ent) {
  constexpr int kTile = L::kTile;
  constexpr int kPieces = L::kD * L::kEsize / 16;  // 16-byte pieces of a cache row
  const int lane = threadIdx.x & 31;
  const uint8_t* base = static_cast<const uint8_t*>(kIsV ? p.vc : p.kc);
#pragma unroll
  for (int i = 0; i < kTile / 32; ++i) {
    const int r = lane + 32 * i, j = t0 + r;
    int pg;
    if constexpr (P == 1) {
      int npages;
      const int32_t* pages = seq_pages(p.block_table, p.bt_stride, p.page_indptr, w.b, &npages);
      pg = (j >= w.kv_end || (npages >= 0 && j >= npages)) ? -1 : __ldg(pages + j);
    } else {
      pg = __shfl_sync(0xffffffffu, ent.v[i / P], (r / P) & 31);
    }
    const uint8_t* src = base;
    uint32_t bytes = 0;
    if (j < w.kv_end) {
      if (pg < 0 || pg >= p.num_pages) {
        if (!kIsV) record_status(p.status, PKV_ERR_DEVICE_BOUNDS, w.b, pg);
      } else {
        src = base + ((int64_t)pg * p.c_stride_page + (int64_t)(j % P) * p.c_stride_tok +
                      (int64_t)w.hk * p.c_stride_head) * L::kEsize;
        bytes = 16;
      }
    }
#pragma unroll
    for (int c = 0; c < kPieces; ++c)
      cp_async_16(stage + raw_off<L::kRowBytes, kTile>(r, c), src + (bytes ? c * 16 : 0), bytes);
  }
  cp_async_commit();
}

// ------------------------------------------------------------------ producers
// Two producer warps, one per ring: warp 0 loads Q tiles and K tiles, the V
// producer warp loads V tiles, each as soon as a stage of its own ring is
// free.  The whole warp issues: lane l owns box (l % boxes) of 128-byte column
// chunk (l / boxes) of every tile, where a tile of 128 keys is `boxes` boxes
// of box_rows cache rows (128 for a contiguous cache, the largest power of two
// dividing the page size for a paged one).
//
// Within an item no global load sits between a free stage and its copy:
// block_table entries are read one warp-wide load per group of 32 / boxes
// tiles (lane l: box l % boxes of tile l / boxes of the group), a group ahead
// of its use.  (Loading the next item's descriptor ahead as well measured
// slower on prefill plans.)
template <int D, bool FP8, bool PF, bool kIsV>
__device__ void producer(const AttnParams& p, const CUtensorMap* tm_kv, const CUtensorMap* tm_q, uint8_t* smem,
                         const Bars& B, volatile int* abort_flag, int it0, int it1) {
  using L = Layout<D, FP8, PF>;
  constexpr int kStages = kIsV ? L::kStagesV : L::kStagesK;
  uint64_t* full = kIsV ? B.full_v : B.full_k;
  uint64_t* empty = kIsV ? B.empty_v : B.empty_k;
  uint8_t* ring_base = smem + (kIsV ? L::kVOff : L::kKOff);
  const int lane = threadIdx.x & 31;
  constexpr int kTile = L::kTile;
  const int boxes = kTile / p.box_rows;
  const int grp = lane % boxes, chunk = lane / boxes;
  const bool active = chunk < L::kChunks;
  const int box_off = chunk * (kTile * L::kRowBytes) + grp * (p.box_rows * L::kRowBytes);
  const bool paged = p.page_size > 0;
  const bool rows = p.row_gather != 0;          // pages of 1, 2 or 4 tokens
  const int per = boxes <= 32 ? 32 / boxes : 1;  // tiles whose page numbers one warp-wide load covers
  if (lane == 0) tma_prefetch_desc(tm_kv);

  // block_table entry of box (lane % boxes) of tile (lane / boxes) of the group
  // of tiles starting at key t0g of item w (-1 past the sequence's page list)
  auto load_pages = [&](const WorkItem& w, int t0g) -> int {
    if (!paged || rows) return 0;
    const int j = t0g + (lane / boxes) * kTile + (lane % boxes) * p.box_rows;
    if (j >= w.kv_end) return 0;
    int npages;
    const int32_t* pages = seq_pages(p.block_table, p.bt_stride, p.page_indptr, w.b, &npages);
    const int pgi = j / p.page_size;
    return (npages >= 0 && pgi >= npages) ? -1 : __ldg(pages + pgi);
  };

  // (decode-only instances; instances with prefill tiles, whose producers run
  // on few registers, look the pages up row by row)
  constexpr bool kEnt = !PF;
  // Row gather (pages of 1, 2 or 4 tokens): the tile's page numbers, one a
  // page (kTile / page_size of them), come from one coalesced load, lane e
  // holding entries e, e + 32, ... (-1 past the sequence's page list), taken
  // a tile ahead of the copies that use them (pages of 2 and 4 tokens: 0.25 ->
  // 0.20 ms on the decode batch, where each lane had loaded its rows' entries
  // as it copied them).
  auto load_entries = [&](const WorkItem& w, int t0) {
    PageEntries<kTile / 32> ent;
    int npages;
    const int32_t* pages = seq_pages(p.block_table, p.bt_stride, p.page_indptr, w.b, &npages);
    const int E = kTile / p.page_size;
#pragma unroll
    for (int k = 0; k < kTile / 32; ++k) {
      const int e = lane + 32 * k;
      const int pgi = t0 / p.page_size + e;
      ent.v[k] = (e < E && pgi * p.page_size < w.kv_end && !(npages >= 0 && pgi >= npages)) ? __ldg(pages + pgi) : -1;
    }
    return ent;
  };
  // Row gather in instances with prefill tiles: lane l copies rows l, l+32,
  // l+64, l+96 of a tile in 16-byte cp.async pieces into the swizzled layout
  // (rows past the key range become zeros), looking each row's page up as it
  // goes.  A gathered tile is marked full once its copies have landed, which
  // is checked when the next tile has been issued (or at the end).
  auto gather_tile = [&](const WorkItem& w, int t0, uint8_t* stage) {
    const uint8_t* base = static_cast<const uint8_t*>(kIsV ? p.vc : p.kc);
    constexpr int kPieces = D * L::kEsize / 16;  // 16-byte pieces of a cache row
#pragma unroll
    for (int i = 0; i < kTile / 32; ++i) {
      const int r = lane + 32 * i, j = t0 + r;
      const uint8_t* src = base;
      uint32_t bytes = 0;
      if (j < w.kv_end) {
        int npages;
        const int32_t* pages = seq_pages(p.block_table, p.bt_stride, p.page_indptr, w.b, &npages);
        const int pgi = j / p.page_size;
        const int pg = (npages >= 0 && pgi >= npages) ? -1 : __ldg(pages + pgi);
        if (pg < 0 || pg >= p.num_pages) {
          if (!kIsV) record_status(p.status, PKV_ERR_DEVICE_BOUNDS, w.b, pg);
        } else {
          src = base + ((int64_t)pg * p.c_stride_page + (int64_t)(j % p.page_size) * p.c_stride_tok +
                        (int64_t)w.hk * p.c_stride_head) * L::kEsize;
          bytes = 16;
        }
      }
#pragma unroll
      for (int c = 0; c < kPieces; ++c)
        cp_async_16(stage + raw_off<L::kRowBytes, kTile>(r, c), src + (bytes ? c * 16 : 0), bytes);
    }
    cp_async_commit();
  };
  int pend = -1;  // row gather: stage whose copies are in flight, not yet marked full
  auto mark_full = [&](int stage) {
    fence_proxy_async_smem();  // the copies (generic proxy) before tensor-core reads of the stage
    mbar_arrive(&full[stage]);
  };

  Ring ring;
  int issued = 0;
  uint32_t pi[2] = {0, 0};  // Q tiles loaded, per query tile of an item
  bool ok = true;
  bool dep_done = false;  // waited for the append kernel (rows at or past the old cache length)

  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = load_item(p, it);
    if (!kIsV && !PF && w.kind == kDecode) {
      // the decode consumers read the item's query rows from global memory
      // when they reach it: bring the rows into this SM's L1 now, while they
      // still work on the tiles this warp has loaded ahead (decode-only
      // plans: 97.6 -> 95.6 us on the bf16 decode batch; the mixed batch did
      // not gain)
      constexpr int kLines = D * 2 / 128;  // 128-byte lines of a bf16 query row
      const int R = w.n_q * p.G;
      for (int i = lane; i < R * kLines; i += 32) {
        const int r = i / kLines, c = i % kLines;
        prefetch_l1(p.q + (int64_t)(w.q_row0 + r / p.G) * p.q_stride_tok +
                    (int64_t)(w.hk * p.G + r % p.G) * p.q_stride_head + c * 64);
      }
    }
    // cache length before this call's append
    const int lc_old = p.dynamic ? min(max(__ldg(p.cache_seqlens + w.b), 0), __ldg(p.plan_lc + w.b))
                                 : __ldg(p.plan_lc + w.b);
    int gcur = load_pages(w, w.kv_begin);
    int t0g = w.kv_begin;
    int gnext = load_pages(w, t0g + per * kTile);
    PageEntries<kTile / 32> ent{};  // row gather: the page numbers of the next tile to copy
    if (kEnt && rows && p.page_size > 1) ent = load_entries(w, w.kv_begin);
    if (!kIsV && L::kTc && w.kind == kPrefill && num_tiles<L::kTile>(w) > 0) {
      // Row gather: the last tile of the previous item is still unmarked (a
      // tile is marked once the next one has been issued), and the Q buffer
      // frees only when that tile's S MMAs have run: mark it now, or the two
      // would wait on each other.
      if (rows && pend >= 0) {
        cp_async_wait_group<0>();
        mark_full(pend);
        pend = -1;
      }
      // each query tile of the item that has keys to attend, into its own buffer
      for (int q = 0; q < L::kQTiles; ++q) {
        const WorkItem wq = L::kQQ ? q_tile(w, q, p.causal) : w;
        if (num_tiles<L::kTile>(wq) == 0) continue;
        if (!warp_wait(B.qempty(q), (pi[q] & 1) ^ 1, abort_flag)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          if (pi[0] + pi[1] == 0) tma_prefetch_desc(tm_q);
          // the box: nh_tc heads x (128 / nh_tc) tokens, every byte credited (zero fill included)
          const int nh_tc = tc_group_heads(p.G);
          mbar_arrive_expect_tx(B.qfull(q), (uint32_t)((D / 64) * nh_tc * (kPrefillRowsTc / nh_tc) * 128));
        }
        __syncwarp();
        if (lane < D / 64)
          tma_load_3d(smem + L::kQOff + q * L::kQBytes + lane * (kPrefillRowsTc * 128), tm_q, B.qfull(q), lane * 64,
                      w.hk * p.G + w.h0, wq.q_row0);
        ++pi[q];
      }
      if (!ok) break;
    }
    int q = 0;  // tile of the current page group
    for (int t0 = w.kv_begin; t0 < w.kv_end; t0 += kTile) {
      if (q == per) {
        gcur = gnext;
        t0g += per * kTile;
        q = 0;
        gnext = load_pages(w, t0g + per * kTile);
      }
      const int pg = rows ? 0 : __shfl_sync(0xffffffffu, gcur, q * boxes + grp);
      ++q;
      // this lane's box: page and slot (an out-of-range page fills zeros)
      const int j0 = t0 + grp * p.box_rows;
      int page = p.num_pages, slot = 0;
      if (j0 < w.kv_end) {
        if (paged) {
          if (pg < 0 || pg >= p.num_pages) {
            if (active && !kIsV) record_status(p.status, PKV_ERR_DEVICE_BOUNDS, w.b, pg);
          } else {
            page = pg;
            slot = j0 % p.page_size;
          }
        } else {
          page = w.b;
          slot = j0;
        }
      }
      if (!dep_done && t0 + kTile > lc_old && lc_old < w.lk) {
        grid_dep_wait();
        dep_done = true;
      }
      if (!warp_wait(&empty[ring.stage], ring.phase ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      if (rows) {
        uint8_t* stage = ring_base + ring.stage * L::kTileBytes;
        if constexpr (!kEnt) gather_tile(w, t0, stage);
        else if (p.page_size == 1) gather_rows<L, kIsV, 1>(p, w, t0, stage, ent);
        else if (p.page_size == 2) gather_rows<L, kIsV, 2>(p, w, t0, stage, ent);
        else gather_rows<L, kIsV, 4>(p, w, t0, stage, ent);
        if (kEnt && p.page_size > 1 && t0 + kTile < w.kv_end)
          ent = load_entries(w, t0 + kTile);  // in flight during the wait below
        if (pend >= 0) {
          cp_async_wait_group<1>();  // all but the tile just issued have landed
          mark_full(pend);
        }
        pend = ring.stage;
      } else {
        if (lane == 0) mbar_arrive_expect_tx(&full[ring.stage], L::kTileBytes);
        __syncwarp();
        if (active)
          tma_load_4d(ring_base + ring.stage * L::kTileBytes + box_off, tm_kv, &full[ring.stage],
                      chunk * (128 / L::kEsize), w.hk, slot, page);
      }
      ++issued;
      ring.advance<kStages>();
    }
  }
  if (rows) {
    // the last tile's copies land before it is marked full (and before the CTA can exit)
    cp_async_wait_group<0>();
    if (ok && pend >= 0) mark_full(pend);
  }
  if (!ok) {
    if (lane == 0) record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, kIsV ? 2 : 1);
    *abort_flag = 1;
    // let the copies already issued land before the CTA can exit (bounded)
    if (lane == 0 && !rows) {
      int zero = 0;
      const int n = issued < kStages ? issued : kStages;
      for (int k = issued - n; k < issued; ++k) mbar_wait(&full[k % kStages], (uint32_t)((k / kStages) & 1), &zero);
    }
    __syncwarp();
  }
  // this CTA ends only after the append kernel has: work issued after this
  // launch on the stream then also follows the append
  if (!dep_done) grid_dep_wait();
}

// ------------------------------------------------------------------ MMA issuers (prefill tiles)
// Two threads issue the tcgen05 MMAs of prefill tiles, each queue in order:
// warp 1 S_j = Q K_j^T (needs K_j, and S buffer j % 3 free: P V of tile j-3
// completed), the P V warp O += P_j V_j (needs P_j, written by the softmax
// into S buffer j % 3, and V_j).  An MMA issue does not return while the
// tensor pipe is busy with the ones before it, so with one thread per queue
// the waits and bookkeeping of one overlap the other's MMAs.  With an fp8
// cache the K and V operands are the converted f16 tiles (buffer T % 2) and Q
// is f16 too.
// QF8 (fp8 cache with q_scale): the converter warps quantise Q to e4m3 (into
// the first converted-K buffer) and S = Q K^T runs as kind::f8f6f4 MMAs on the
// raw e4m3 K stage, which this thread releases when the MMAs have completed;
// the converters then turn only V into f16.
template <int D, bool FP8, bool PF, bool QF8>
__device__ bool s_issuer(const AttnParams& p, uint8_t* smem, const Bars& B, volatile int* abort_flag, uint32_t tmem,
                         int it0, int it1) {
  using L = Layout<D, FP8, PF>;
  constexpr int kAB = FP8 ? 0 : 1;  // operand type: f16 or bf16 (e4m3 for QF8: the same code)
  constexpr int kTile = L::kTile;
  constexpr uint32_t kIdescQK = idesc_f16(kAB, 0, 128, kTile);
  const uint32_t q_base = smem_u32(smem + (QF8 ? L::kKcOff : L::kQOff));
  Ring rk;
  uint32_t pt = 0, pi = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = load_item(p, it);
    const int n = num_tiles<L::kTile>(w);
    if (w.kind != kPrefill) {
      rk.advance<L::kStagesK>(n);
      continue;
    }
    if (n == 0) continue;
    if (!mbar_wait(FP8 ? B.qc_full : B.q_full, pi & 1, abort_flag)) return false;
    for (int j = 0; j < n; ++j) {
      const uint32_t T = pt + j, b = T % L::kSBufs, use = T / L::kSBufs;
      uint32_t k_base;
      if constexpr (FP8 && !QF8) {
        constexpr int NB = L::kConvBufsK;
        if (!mbar_wait(&B.kc_full[T % NB], (T / NB) & 1, abort_flag)) return false;
        k_base = smem_u32(smem + L::kKcOff + (T % NB) * L::kConvTile);
      } else {
        if (!mbar_wait(&B.full_k[rk.stage], rk.phase, abort_flag)) return false;
        k_base = smem_u32(smem + L::kKOff + rk.stage * L::kTileBytes);
      }
      // the buffer last held S and P of tile T - kSBufs: P V of that tile has completed
      if (use >= 1 && !mbar_wait(&B.o_done[b], (use - 1) & 1, abort_flag)) return false;
      tc_fence_after();
      if constexpr (QF8) {
        // e4m3 rows in 128-byte column chunks (128-byte swizzle; one 64-byte
        // chunk with the 64-byte swizzle at D = 64): K=32 per MMA, 32 bytes apart
#pragma unroll
        for (int k = 0; k < D / 32; ++k) {
          if constexpr (D >= 128)
            umma_ss_e4m3(tmem + b * kTile,
                         sdesc_sw128(q_base + (k >> 2) * (kPrefillRowsTc * 128) + (k & 3) * 32, 16, 1024),
                         sdesc_sw128(k_base + (k >> 2) * (kTile * 128) + (k & 3) * 32, 16, 1024), kIdescQK,
                         k > 0 ? 1u : 0u);
          else
            umma_ss_e4m3(tmem + b * kTile, sdesc_sw64(q_base + k * 32, 16, 512), sdesc_sw64(k_base + k * 32, 16, 512),
                         kIdescQK, k > 0 ? 1u : 0u);
        }
      } else {
#pragma unroll
        for (int k = 0; k < D / 16; ++k) {
          const uint32_t qoff = (k >> 2) * (kPrefillRowsTc * 128) + (k & 3) * 32;
          const uint32_t koff = (k >> 2) * (kTile * 128) + (k & 3) * 32;
          umma_ss(tmem + b * kTile, sdesc_sw128(q_base + qoff, 16, 1024), sdesc_sw128(k_base + koff, 16, 1024),
                  kIdescQK, k > 0 ? 1u : 0u);
        }
      }
      umma_commit(&B.s_full[b]);  // bf16: the softmax warps release the K stage once they have seen S complete
      if constexpr (QF8) {
        // the raw K stage barrier expects one arrival per consumer warp: all but
        // one now, the last when these MMAs complete
        mbar_arrive_cnt(&B.empty_k[rk.stage], kConsumerWarps - 1);
        umma_commit(&B.empty_k[rk.stage]);
      } else if constexpr (FP8) {
        umma_commit(&B.kc_empty[T % L::kConvBufsK]);
      }
      rk.advance<L::kStagesK>();
    }
    umma_commit(B.q_empty);
    pt += n;
    ++pi;
  }
  return true;
}

template <int D, bool FP8, bool PF>
__device__ bool pv_issuer(const AttnParams& p, uint8_t* smem, const Bars& B, volatile int* abort_flag, uint32_t tmem,
                          int it0, int it1) {
  using L = Layout<D, FP8, PF>;
  constexpr int kAB = FP8 ? 0 : 1;
  constexpr int kTile = L::kTile;
  constexpr uint32_t kIdescPV = idesc_f16(kAB, 1, 128, D);
  Ring rv;
  uint32_t pt = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = load_item(p, it);
    const int n = num_tiles<L::kTile>(w);
    if (w.kind != kPrefill) {
      rv.advance<L::kStagesV>(n);
      continue;
    }
    for (int j = 0; j < n; ++j) {
      const uint32_t T = pt + j, b = T % L::kSBufs;
      if (!mbar_wait(&B.p_full[b], (T / L::kSBufs) & 1, abort_flag)) return false;
      uint32_t v_base;
      if constexpr (FP8) {
        constexpr int NB = L::kConvBufsV;
        if (!mbar_wait(&B.vc_full[T % NB], (T / NB) & 1, abort_flag)) return false;
        v_base = smem_u32(smem + L::kVcOff + (T % NB) * L::kConvTile);
      } else {
        if (!mbar_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) return false;
        v_base = smem_u32(smem + L::kVOff + rv.stage * L::kTileBytes);
      }
      tc_fence_after();
      const uint32_t p_tmem = tmem + b * kTile;  // P over the first columns of the tile's S buffer
#pragma unroll
      for (int k = 0; k < kTile / 16; ++k) {
        const uint64_t bd = sdesc_sw128(v_base + k * 16 * 128, kTile * 128, 1024);
        umma_ts(tmem + L::kTmemO, p_tmem + k * 8, bd, kIdescPV, (j == 0 && k == 0) ? 0u : 1u);
      }
      umma_commit(&B.o_done[b]);
      if constexpr (FP8) {
        umma_commit(&B.vc_empty[T % L::kConvBufsV]);
      } else {
        // the V stage barrier expects one arrival per consumer warp (as the decode
        // warps give): all but one now, the last when these MMAs complete
        mbar_arrive_cnt(&B.empty_v[rv.stage], kConsumerWarps - 1);
        umma_commit(&B.empty_v[rv.stage]);
      }
      rv.advance<L::kStagesV>();
    }
    pt += n;
  }
  return true;
}

// The same two queues with two query tiles per item (D <= 128): query tile q
// has one S buffer (at q * 256 in tensor memory) and its O, and barriers
// s_full / p_full / o_done [q].  For K tile j the S issuer runs S_q = Q_q K_j^T
// for each query tile whose keys reach tile j (once P V of that tile's
// previous K/V tile has freed its S buffer) and then releases the K tile; the
// P V issuer runs O_q += P_q V_j as each tile's P is written, except that on a
// tile whose V rows past the sequence a softmax warpgroup zeroes (bf16 cache;
// the second tile's, which always reaches the item's last K/V tile) both P
// are waited for first.  So one query tile's MMAs run while the other's
// softmax does.
template <int D, bool FP8, bool PF, bool QF8>
__device__ bool s_issuer_qq(const AttnParams& p, uint8_t* smem, const Bars& B, volatile int* abort_flag, uint32_t tmem,
                            int it0, int it1) {
  using L = Layout<D, FP8, PF>;
  constexpr int kAB = FP8 ? 0 : 1;
  constexpr int kTile = L::kTile;
  constexpr uint32_t kIdescQK = idesc_f16(kAB, 0, 128, kTile);
  constexpr int NB = L::kConvBufsK;
  Ring rk;
  uint32_t pt[2] = {0, 0}, pi[2] = {0, 0}, ck = 0;  // S tiles and items per query tile; K tiles (converted)
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = load_item(p, it);
    const int n = num_tiles<kTile>(w);
    if (w.kind != kPrefill) {
      rk.advance<L::kStagesK>(n);
      continue;
    }
    if (n == 0) continue;
    int nq[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) nq[q] = num_tiles<kTile>(q_tile(w, q, p.causal));
    // the item's Q tiles first (the producer loads them after every K tile
    // of the items before)
#pragma unroll
    for (int q = 0; q < 2; ++q)
      if (nq[q] > 0 && !mbar_wait(FP8 ? B.qcfull(q) : B.qfull(q), pi[q] & 1, abort_flag)) return false;
    for (int j = 0; j < n; ++j) {
      uint32_t k_base;
      if constexpr (FP8 && !QF8) {
        if (!mbar_wait(&B.kc_full[ck % NB], (ck / NB) & 1, abort_flag)) return false;
        k_base = smem_u32(smem + L::kKcOff + (ck % NB) * L::kConvTile);
      } else {
        if (!mbar_wait(&B.full_k[rk.stage], rk.phase, abort_flag)) return false;
        k_base = smem_u32(smem + L::kKOff + rk.stage * L::kTileBytes);
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (j >= nq[q]) continue;
        // the S buffer last held S and P of this query tile's previous tile
        if (pt[q] >= 1 && !mbar_wait(&B.o_done[q], (pt[q] - 1) & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t s_tmem = tmem + q * L::kQCols;
        if constexpr (QF8) {
          const uint32_t q_base = smem_u32(smem + L::kKcOff + q * (kPrefillRowsTc * D));
#pragma unroll
          for (int k = 0; k < D / 32; ++k) {
            if constexpr (D >= 128)
              umma_ss_e4m3(s_tmem, sdesc_sw128(q_base + (k >> 2) * (kPrefillRowsTc * 128) + (k & 3) * 32, 16, 1024),
                           sdesc_sw128(k_base + (k >> 2) * (kTile * 128) + (k & 3) * 32, 16, 1024), kIdescQK,
                           k > 0 ? 1u : 0u);
            else
              umma_ss_e4m3(s_tmem, sdesc_sw64(q_base + k * 32, 16, 512), sdesc_sw64(k_base + k * 32, 16, 512),
                           kIdescQK, k > 0 ? 1u : 0u);
          }
        } else {
          const uint32_t q_base = smem_u32(smem + L::kQOff + q * L::kQBytes);
#pragma unroll
          for (int k = 0; k < D / 16; ++k) {
            const uint32_t qoff = (k >> 2) * (kPrefillRowsTc * 128) + (k & 3) * 32;
            const uint32_t koff = (k >> 2) * (kTile * 128) + (k & 3) * 32;
            umma_ss(s_tmem, sdesc_sw128(q_base + qoff, 16, 1024), sdesc_sw128(k_base + koff, 16, 1024), kIdescQK,
                    k > 0 ? 1u : 0u);
          }
        }
        umma_commit(&B.s_full[q]);
        ++pt[q];
      }
      // the K tile is free once these MMAs have completed (the raw-stage
      // barrier expects one arrival per consumer warp: all but one now)
      if constexpr (FP8 && !QF8) {
        umma_commit(&B.kc_empty[ck % NB]);
        ++ck;
      } else {
        mbar_arrive_cnt(&B.empty_k[rk.stage], kConsumerWarps - 1);
        umma_commit(&B.empty_k[rk.stage]);
      }
      rk.advance<L::kStagesK>();
    }
#pragma unroll
    for (int q = 0; q < 2; ++q) {
      if (nq[q] == 0) continue;
      umma_commit(B.qempty(q));
      ++pi[q];
    }
  }
  return true;
}

template <int D, bool FP8, bool PF>
__device__ bool pv_issuer_qq(const AttnParams& p, uint8_t* smem, const Bars& B, volatile int* abort_flag,
                             uint32_t tmem, int it0, int it1) {
  using L = Layout<D, FP8, PF>;
  constexpr int kAB = FP8 ? 0 : 1;
  constexpr int kTile = L::kTile;
  constexpr uint32_t kIdescPV = idesc_f16(kAB, 1, 128, D);
  constexpr int NB = L::kConvBufsV;
  Ring rv;
  uint32_t pt[2] = {0, 0}, cv = 0;  // P V tiles per query tile; V tiles (converted)
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = load_item(p, it);
    const int n = num_tiles<kTile>(w);
    if (w.kind != kPrefill) {
      rv.advance<L::kStagesV>(n);
      continue;
    }
    int nq[2];
#pragma unroll
    for (int q = 0; q < 2; ++q) nq[q] = num_tiles<kTile>(q_tile(w, q, p.causal));
    for (int j = 0; j < n; ++j) {
      // bf16: V rows past the sequence are zeroed by the second query tile's
      // warps when both reach this tile: the first tile's P V waits for them
      const bool both = !FP8 && w.kv_begin + (j + 1) * kTile > w.lk && j < nq[0] && j < nq[1];
      // P of the first query tile reaching this tile before its V (the
      // softmax has then seen S of the tile, so every fill before it is in)
      const int q0 = j < nq[0] ? 0 : 1;
      if (!mbar_wait(&B.p_full[q0], pt[q0] & 1, abort_flag)) return false;
      if (both && !mbar_wait(&B.p_full[1], pt[1] & 1, abort_flag)) return false;
      uint32_t v_base;
      if constexpr (FP8) {
        if (!mbar_wait(&B.vc_full[cv % NB], (cv / NB) & 1, abort_flag)) return false;
        v_base = smem_u32(smem + L::kVcOff + (cv % NB) * L::kConvTile);
      } else {
        if (!mbar_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) return false;
        v_base = smem_u32(smem + L::kVOff + rv.stage * L::kTileBytes);
      }
#pragma unroll
      for (int q = 0; q < 2; ++q) {
        if (j >= nq[q]) continue;
        if (q != q0 && !(both && q == 1) && !mbar_wait(&B.p_full[q], pt[q] & 1, abort_flag)) return false;
        tc_fence_after();
        const uint32_t p_tmem = tmem + q * L::kQCols;  // P over the first columns of the S buffer
#pragma unroll
        for (int k = 0; k < kTile / 16; ++k) {
          const uint64_t bd = sdesc_sw128(v_base + k * 16 * 128, kTile * 128, 1024);
          umma_ts(p_tmem + L::kTmemO, p_tmem + k * 8, bd, kIdescPV, (j == 0 && k == 0) ? 0u : 1u);
        }
        umma_commit(&B.o_done[q]);
        ++pt[q];
      }
      if constexpr (FP8) {
        umma_commit(&B.vc_empty[cv % NB]);
        ++cv;
      } else {
        mbar_arrive_cnt(&B.empty_v[rv.stage], kConsumerWarps - 1);
        umma_commit(&B.empty_v[rv.stage]);
      }
      rv.advance<L::kStagesV>();
    }
  }
  return true;
}

// ------------------------------------------------------------------ converters (fp8 cache, prefill tiles)
// Four warps turn each raw e4m3 K / V tile (128 rows x 128 B, swizzled) into
// an f16 tile in the layout the MMA reads (2 x [128 rows][128 B], swizzled),
// exactly (every e4m3 value is an f16 value), zeroing V rows past the
// sequence; and the bf16 Q tile of each item into f16 in place.  Converted
// tiles are double-buffered (T % 2); raw stages are released after conversion.
//
// Unit u of the 16-byte raw chunks (ct + 128 k) maps to row (u % 8) + 8 m and
// chunk column (u / 8) % kCpr, m = u / (8 kCpr): the eight threads of a
// quarter-warp (which one 16-byte shared access serves at a time) take eight
// consecutive rows at one column, so under either swizzle (chunk XOR row % 8,
// or the 64-byte one) their loads and each of their two stores fall on eight
// distinct 16-byte bank groups.  (Eight chunks of one row would put chunks
// 2c and 2c + 8 of the f16 row on the same group.)
template <int kCpr>
__device__ __forceinline__ void conv_unit(int u, int& r, int& c) {
  c = (u >> 3) % kCpr;
  r = (u & 7) + 8 * ((u >> 3) / kCpr);
}

template <int D, int TILE>
__device__ __forceinline__ void convert_tile(const uint8_t* raw, uint8_t* conv, int ct, int zero_from) {
  constexpr int kCpr = D / 16;       // raw 16-byte chunks per row (e4m3 rows of D bytes)
  constexpr int RB = D < 128 ? D : 128;
#pragma unroll
  for (int k = 0; k < TILE * kCpr / 128; ++k) {
    int r, c;  // raw 16-byte chunk c of row r: d = 16c .. 16c+15
    conv_unit<kCpr>(ct + 128 * k, r, c);
    // every row is read and converted (the loads are not behind a branch, so
    // they can all be in flight at once); rows at or past zero_from then
    // become zeros by select
    uint4 lo, hi;
    const uint4 w = *reinterpret_cast<const uint4*>(raw + raw_off<RB, TILE>(r, c));
    e4m3x4_to_f16x4(w.x, lo.x, lo.y);
    e4m3x4_to_f16x4(w.y, lo.z, lo.w);
    e4m3x4_to_f16x4(w.z, hi.x, hi.y);
    e4m3x4_to_f16x4(w.w, hi.z, hi.w);
    if (r >= zero_from) lo = hi = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(conv + tile_off<TILE>(r, 2 * c)) = lo;
    *reinterpret_cast<uint4*>(conv + tile_off<TILE>(r, 2 * c + 1)) = hi;
  }
}

template <int D, bool PF, bool QF8>
__device__ bool converter(const AttnParams& p, uint8_t* smem, const Bars& B, volatile int* abort_flag, int it0,
                          int it1) {
  using L = Layout<D, true, PF>;
  const int lane = threadIdx.x & 31;
  const int ct = threadIdx.x - 32 * L::kConvWarp0;  // 0..127
  Ring rk, rv;
  uint32_t pt = 0, pi[2] = {0, 0};
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = load_item(p, it);
    const int n = num_tiles<L::kTile>(w);
    if (w.kind != kPrefill) {
      rk.advance<L::kStagesK>(n);
      rv.advance<L::kStagesV>(n);
      continue;
    }
    if (n == 0) continue;
    // each query tile of the item that has keys to attend
    for (int qt = 0; qt < L::kQTiles; ++qt) {
      if (L::kQQ && num_tiles<L::kTile>(q_tile(w, qt, p.causal)) == 0) continue;
      if (!warp_wait(B.qfull(qt), pi[qt] & 1, abort_flag)) return false;
      if constexpr (QF8) {
        // Q: bf16 -> e4m3 with the cache's encode (one IEEE reciprocal of
        // q_scale, an RN multiply per value, RN satfinite), into the converted-K
        // area (query tile q at q x 128 x D bytes) as [128 rows][128 B]
        // swizzled: the 16 values of e4m3 chunk c of row r come from bf16
        // chunks 2c and 2c+1 of that row
        const float inv_q = __frcp_rn(__ldg(p.q_scale));
        auto quant4 = [&](uint32_t w0, uint32_t w1) -> uint32_t {
          auto lo = [](uint32_t v) { return __uint_as_float(v << 16); };
          auto hi = [](uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); };
          const uint32_t a = f32x2_to_e4m3x2(__fmul_rn(lo(w0), inv_q), __fmul_rn(hi(w0), inv_q));
          const uint32_t b = f32x2_to_e4m3x2(__fmul_rn(lo(w1), inv_q), __fmul_rn(hi(w1), inv_q));
          return a | (b << 16);
        };
        const uint8_t* qb = smem + L::kQOff + qt * L::kQBytes;
        uint8_t* q8 = smem + L::kKcOff + qt * (kPrefillRowsTc * D);
        constexpr int kCpr = D / 16;  // e4m3 16-byte chunks per row
#pragma unroll 2
        for (int k = 0; k < kCpr; ++k) {
          int r, c;
          conv_unit<kCpr>(ct + 128 * k, r, c);
          const uint4 a = *reinterpret_cast<const uint4*>(qb + tile_off<kPrefillRowsTc>(r, 2 * c));
          const uint4 b = *reinterpret_cast<const uint4*>(qb + tile_off<kPrefillRowsTc>(r, 2 * c + 1));
          *reinterpret_cast<uint4*>(q8 + raw_off<L::kRowBytes, kPrefillRowsTc>(r, c)) =
              make_uint4(quant4(a.x, a.y), quant4(a.z, a.w), quant4(b.x, b.y), quant4(b.z, b.w));
        }
      } else {
        // Q: bf16 -> f16 in place (elementwise, so the swizzle does not matter)
        uint4* q = reinterpret_cast<uint4*>(smem + L::kQOff + qt * L::kQBytes);
#pragma unroll 4
        for (int k = 0; k < kPrefillRowsTc * D * 2 / 16 / 128; ++k) {
          uint4 v = q[ct + 128 * k];
          v = make_uint4(bf16x2_to_f16x2(v.x), bf16x2_to_f16x2(v.y), bf16x2_to_f16x2(v.z), bf16x2_to_f16x2(v.w));
          q[ct + 128 * k] = v;
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(B.qcfull(qt));
      ++pi[qt];
    }
    constexpr int NB = L::kConvBufsK, NV = L::kConvBufsV;
    for (int j = 0; j < n; ++j) {
      const uint32_t T = pt + j;
      const int t0 = w.kv_begin + j * L::kTile;
      if constexpr (!QF8) {
        if (!warp_wait(&B.full_k[rk.stage], rk.phase, abort_flag)) return false;
        if (T >= NB && !warp_wait(&B.kc_empty[T % NB], ((T / NB) - 1) & 1, abort_flag)) return false;
        convert_tile<D, L::kTile>(smem + L::kKOff + rk.stage * L::kTileBytes, smem + L::kKcOff + (T % NB) * L::kConvTile,
                                  ct, L::kTile);
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&B.kc_full[T % NB]);
          mbar_arrive(&B.empty_k[rk.stage]);
        }
      }
      if (!warp_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) return false;
      if (T >= NV && !warp_wait(&B.vc_empty[T % NV], ((T / NV) - 1) & 1, abort_flag)) return false;
      // rows past the sequence may hold anything (even NaN): they become zeros
      convert_tile<D, L::kTile>(smem + L::kVOff + rv.stage * L::kTileBytes, smem + L::kVcOff + (T % NV) * L::kConvTile,
                                ct, w.lk - t0);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&B.vc_full[T % NV]);
        mbar_arrive(&B.empty_v[rv.stage]);
      }
      rk.advance<L::kStagesK>();
      rv.advance<L::kStagesV>();
    }
    pt += n;
  }
  return true;
}

// ------------------------------------------------------------------ prefill epilogue
// The epilogue of a prefill item (O / l to bf16 rows, the LSE) is deferred:
// it runs inside the next prefill item's first tile, once that tile's P is in
// tensor memory and before the softmax lets P V of the tile (which starts O
// afresh) be issued, or at the end of the CTA's work.  So the softmax warps do
// not wait for the item's last P V to complete: by then it has, and the S of
// the next item's tiles are already in tensor memory.
struct PendingEpi {
  bool has = false;                // warp-uniform
  uint32_t T = 0;                  // the item's last tile: O is final once its P V has completed
  float inv = 0.f;                 // scale of the output (v_scale / l, or 0)
  float lse = 0.f;                 // natural-log LSE of the row
  __nv_bfloat16* dst = nullptr;    // this thread's output row (null: none)
  float* lse_dst = nullptr;
};

// Writes the pending item's rows (waits for its last P V), 32 columns at a time
// (query tile qt of the item: its O and its P V barrier)
template <class L>
__device__ __forceinline__ bool epi_run(const AttnParams& p, const Bars& B, const PendingEpi& e, uint32_t t_lane,
                                        int qt, volatile int* abort_flag) {
  constexpr int D = L::kD;
  if (!warp_wait(&B.o_done[L::kQQ ? qt : e.T % L::kSBufs], (e.T / L::kSBufs) & 1, abort_flag)) return false;
  tc_fence_after();
  const uint32_t o_col = qt * L::kQCols + L::kTmemO;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(t_lane + o_col + c * 32, o);
    tmem_wait_ld();
    if (e.dst != nullptr) {
      uint4 v[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        v[q].x = pack_bf16(__uint_as_float(o[8 * q + 0]) * e.inv, __uint_as_float(o[8 * q + 1]) * e.inv);
        v[q].y = pack_bf16(__uint_as_float(o[8 * q + 2]) * e.inv, __uint_as_float(o[8 * q + 3]) * e.inv);
        v[q].z = pack_bf16(__uint_as_float(o[8 * q + 4]) * e.inv, __uint_as_float(o[8 * q + 5]) * e.inv);
        v[q].w = pack_bf16(__uint_as_float(o[8 * q + 6]) * e.inv, __uint_as_float(o[8 * q + 7]) * e.inv);
      }
      // a row is written in 32-byte pieces where it is aligned for them (whole
      // sectors, half the store instructions), else in 16-byte ones
      if (p.out_v8) {
        st_global_v8(e.dst + c * 32, v[0], v[1]);
        st_global_v8(e.dst + c * 32 + 16, v[2], v[3]);
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) *reinterpret_cast<uint4*>(e.dst + c * 32 + q * 8) = v[q];
      }
    }
  }
  if (e.lse_dst != nullptr) *e.lse_dst = e.lse;
  return true;
}

// The epilogue of a split-KV chunk of a tensor-core item (rare: a unit whose
// queries fit one tile, cut along the keys), run at once at the end of its
// item: waits for its last P V, then writes the normalised fp32 row and the
// log2 LSE into the item's partial slots, so that the deferred epilogue of
// the common case carries no state for it.
template <class L>
__device__ __forceinline__ bool epi_partial(const Bars& B, uint32_t T, int qt, float inv, float lse2, float* pdst,
                                            float* lse_dst, uint32_t t_lane, volatile int* abort_flag) {
  constexpr int D = L::kD;
  if (!warp_wait(&B.o_done[L::kQQ ? qt : T % L::kSBufs], (T / L::kSBufs) & 1, abort_flag)) return false;
  tc_fence_after();
  const uint32_t o_col = qt * L::kQCols + L::kTmemO;
#pragma unroll
  for (int c = 0; c < D / 32; ++c) {
    uint32_t o[32];
    tmem_ld32(t_lane + o_col + c * 32, o);
    tmem_wait_ld();
    if (pdst != nullptr) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        float f[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) f[k] = __uint_as_float(o[8 * q + k]) * inv;
        st_global_v8(pdst + c * 32 + q * 8,
                     make_uint4(__float_as_uint(f[0]), __float_as_uint(f[1]), __float_as_uint(f[2]), __float_as_uint(f[3])),
                     make_uint4(__float_as_uint(f[4]), __float_as_uint(f[5]), __float_as_uint(f[6]), __float_as_uint(f[7])));
      }
    }
  }
  if (lse_dst != nullptr) *lse_dst = lse2;
  tc_fence_before();
  return true;
}

// ------------------------------------------------------------------ prefill tile softmax (tcgen05 path)
// Four warps, one query row per thread (TMEM lane), all 128 keys of a tile.
// P of tile T overwrites the S it was computed from (its S buffer is only
// reused once P V of the tile has completed), so the softmax never waits for
// a P buffer; O is rescaled (which needs P V of tile T-1 done) only when a
// row's running max moves.  bf16 cache: P is bf16, this warp releases the K stage
// and zeroes V rows past the sequence.  fp8 cache: P is f16 (the MMA runs on
// f16), the converter warps own the raw stages and the zeroing, S is read in
// two 64-column passes (fewer live registers in the larger block), and the
// output carries v_scale.
template <int D, bool FP8, bool PF>
__device__ bool softmax_item(const AttnParams& p, const WorkItem& w, uint8_t* smem, const Bars& B,
                             volatile int* abort_flag, uint32_t tmem, Ring& rk, Ring& rv, uint32_t& pt, float sl2,
                             float vscale, PendingEpi& pend, int qt_, int n_ring, bool zero_owner) {
  using L = Layout<D, FP8, PF>;
  constexpr int kTile = L::kTile;
  const int qt = L::kQQ ? qt_ : 0;  // (compile-time 0 with one query tile per item)
  // (two query tiles per item: w is query tile qt of the item, whose K/V tiles
  // number n_ring; its S buffer, O and barriers are its own)
  const uint32_t o_col = qt * L::kQCols + L::kTmemO;
  // S columns held in registers at a time (all of a tile's but in the fp8
  // block without its register split)
  constexpr int kPass = (FP8 && !L::kSplitRegs ? 64 : 128) < kTile ? (FP8 && !L::kSplitRegs ? 64 : 128) : kTile;
  constexpr bool kTwoPass = kPass < kTile;  // S read twice (max, then probabilities)
  // fp8 cache: S is read from tensor memory twice, the max pass at once (or,
  // on tiles that need the mask, 32 columns at a time) and the probability
  // pass 32 columns at a time in a loop that is not unrolled: the warps share
  // their SM sub-partitions with the converters, and the smaller instruction
  // footprint measured faster than the unrolled one-pass form (and than
  // 64-column steps, or a second register buffer loading ahead); the bf16
  // tile, without the converters, measured faster unrolled
  constexpr bool kRolled = FP8 && L::kSplitRegs;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qw = warp & 3;                   // TMEM lane quarter this warp may access
  const int r = qw * 32 + lane;              // tile row == TMEM lane
  const uint32_t t_lane = tmem + ((uint32_t)(qw * 32) << 16);
  // rows: token r / nh of the tile, head h0 + r % nh of the group
  const int R = w.n_q * w.nh;
  const bool valid = r < R;
  const int tok = w.q_row0 + r / w.nh;
  const int head = w.hk * p.G + w.h0 + r % w.nh;
  int lim = 0;
  if (valid) {
    lim = w.kv_end;
    if (p.causal) lim = min(lim, w.q_i0 + r / w.nh + w.lk - w.lq + 1);
  }
  const int n = num_tiles<L::kTile>(w);
  float m = -INFINITY, l = 0.f;

  for (int j = 0; j < n; ++j) {
    const uint32_t T = pt + j;
    const int t0 = w.kv_begin + j * kTile;
    const uint32_t sb = L::kQQ ? qt : T % L::kSBufs;
    const uint32_t s_col = L::kQQ ? qt * L::kQCols : sb * kTile;
    if (!warp_wait(&B.s_full[sb], (T / L::kSBufs) & 1, abort_flag)) return false;
    tc_fence_after();
    const bool need_mask = __any_sync(0xffffffffu, t0 + kTile > lim);
    uint32_t s[kPass];  // (unused when rolled)

    // row max as a tree, masked by select (rows past the sequence see nothing)
    float mx8[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) mx8[e] = -INFINITY;
    if constexpr (kRolled) {
      if (!need_mask) {
        // the whole tile at once: every load in flight, one wait
        uint32_t st[kTile];
#pragma unroll
        for (int c = 0; c < kTile / 32; ++c) tmem_ld32(t_lane + s_col + c * 32, st + c * 32);
        tmem_wait_ld();
#pragma unroll
        for (int c = 0; c < kTile; c += 2)
          mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], __uint_as_float(st[c]), __uint_as_float(st[c + 1]));
      } else {
#pragma unroll 1
        for (int h = 0; h < kTile / 32; ++h) {
          uint32_t c32[32];
          tmem_ld32(t_lane + s_col + h * 32, c32);
          tmem_wait_ld();
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (t0 + h * 32 + c >= lim) c32[c] = __float_as_uint(-INFINITY);
#pragma unroll
          for (int c = 0; c < 32; c += 2)
            mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], __uint_as_float(c32[c]), __uint_as_float(c32[c + 1]));
        }
      }
    }
#pragma unroll
    for (int h = 0; h < (kRolled ? 0 : kTile / kPass); ++h) {
#pragma unroll
      for (int c = 0; c < kPass / 32; ++c) tmem_ld32(t_lane + s_col + h * kPass + c * 32, s + c * 32);
      tmem_wait_ld();
      if constexpr (!FP8 && !L::kQQ) {
        // S of this tile is complete: its K stage is free (with two query
        // tiles the S issuer releases it)
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.empty_k[rk.stage]);
      }
      if (need_mask) {
#pragma unroll
        for (int c = 0; c < kPass; ++c) {
          const float v = (t0 + h * kPass + c < lim) ? __uint_as_float(s[c]) : -INFINITY;
          s[c] = __float_as_uint(v);
        }
      }
#pragma unroll
      for (int c = 0; c < kPass; c += 2)
        mx8[(c >> 1) & 7] = fmax3(mx8[(c >> 1) & 7], __uint_as_float(s[c]), __uint_as_float(s[c + 1]));
    }
    const float mx = fmaxf(fmaxf(fmaxf(mx8[0], mx8[1]), fmaxf(mx8[2], mx8[3])),
                           fmaxf(fmaxf(mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])));
    // The running max m only moves when the tile's max exceeds it by more than
    // 2^8: probabilities then stay below 256, and l and O, both accumulated
    // against the same m, still give the exact O / l and LSE = m + log2 l.
    const float mx2 = mx * sl2;
    const bool bump = mx2 > m + 8.f;
    const float m_new = bump ? mx2 : m;
    const float mu = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = bump ? ex2(m - mu) : 1.f;
    m = m_new;

    // probabilities two at a time: one packed FMA for the scaled logits, one
    // packed add into the row sum
    const uint64_t sl2x2 = f32x2(sl2, sl2), nmu2 = f32x2(-mu, -mu);
    uint64_t sum2[2] = {0ull, 0ull};
    if constexpr (kRolled) {
      // P of columns 32h .. 32h+31 goes to packed columns 16h .. 16h+15, whose
      // S has been read already
#pragma unroll 1
      for (int h = 0; h < kTile / 32; ++h) {
        uint32_t c32[32];
        tmem_ld32(t_lane + s_col + h * 32, c32);
        tmem_wait_ld();
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < 32; ++c)
            if (t0 + h * 32 + c >= lim) c32[c] = __float_as_uint(-INFINITY);
        }
        uint32_t pk[16];
#pragma unroll
        for (int c = 0; c < 16; ++c) {
          float y0, y1;
          f32x2_split(fma_f32x2(f32x2(__uint_as_float(c32[2 * c]), __uint_as_float(c32[2 * c + 1])), sl2x2, nmu2), y0,
                      y1);
          const float p0 = ex2(y0), p1 = ex2(y1);
          sum2[c & 1] = add_f32x2(sum2[c & 1], f32x2(p0, p1));
          pk[c] = pack_f16(p0, p1);
        }
        tmem_st16(t_lane + s_col + h * 16, pk);
      }
    }
#pragma unroll
    for (int h = 0; h < (kRolled ? 0 : kTile / kPass); ++h) {
      if constexpr (kTwoPass) {
        // second pass: read this part of S again
#pragma unroll
        for (int c = 0; c < kPass / 32; ++c) tmem_ld32(t_lane + s_col + h * kPass + c * 32, s + c * 32);
        tmem_wait_ld();
        if (need_mask) {
#pragma unroll
          for (int c = 0; c < kPass; ++c)
            if (t0 + h * kPass + c >= lim) s[c] = __float_as_uint(-INFINITY);
        }
      }
      uint32_t pk[kPass / 2];
#pragma unroll
      for (int c = 0; c < kPass / 2; ++c) {
        float y0, y1;
        f32x2_split(fma_f32x2(f32x2(__uint_as_float(s[2 * c]), __uint_as_float(s[2 * c + 1])), sl2x2, nmu2), y0, y1);
        const float p0 = ex2(y0), p1 = ex2(y1);
        sum2[c & 1] = add_f32x2(sum2[c & 1], f32x2(p0, p1));
        pk[c] = FP8 ? pack_f16(p0, p1) : pack_bf16(p0, p1);
      }
#pragma unroll
      for (int c = 0; c < kPass / 64; ++c)
        tmem_st32(t_lane + s_col + h * (kPass / 2) + c * 32, pk + c * 32);
    }
    float q0, q1, q2, q3;
    f32x2_split(sum2[0], q0, q1);
    f32x2_split(sum2[1], q2, q3);
    l = l * alpha + ((q0 + q2) + (q1 + q3));

    const bool zero_v = !FP8 && (!L::kQQ || zero_owner) && t0 + kTile > w.lk;
    if (zero_v) {
      // rows past the sequence may hold anything (even NaN): zero them in V
      if (!warp_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) return false;
      if (r < kTile && t0 + r >= w.lk) {
        uint8_t* vrow = smem + L::kVOff + rv.stage * L::kTileBytes + r * 128;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
#pragma unroll
          for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vrow + c * (kTile * 128) + q * 16) = make_uint4(0, 0, 0, 0);
      }
    }
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
      // O must hold P V of tile T-1 before it is rescaled
      if (!warp_wait(&B.o_done[L::kQQ ? qt : (T - 1) % L::kSBufs], ((T - 1) / L::kSBufs) & 1, abort_flag))
        return false;
      tc_fence_after();
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_lane + o_col + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(t_lane + o_col + c * 32, o);
      }
    }
    // the previous item's O is written out before P V of this item's first tile
    // may replace it
    if (j == 0 && pend.has) {
      if (!epi_run<L>(p, B, pend, t_lane, qt, abort_flag)) return false;
      pend.has = false;
    }
    tmem_wait_st();
    if (zero_v) fence_proxy_async_smem();  // the zeroed V rows (generic stores) before the MMA reads them
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.p_full[sb]);
    rk.advance<L::kStagesK>();
    rv.advance<L::kStagesV>();
  }
  // (the item's K/V tiles past this query tile's keys)
  if (L::kQQ && n_ring > n) {
    rk.advance<L::kStagesK>(n_ring - n);
    rv.advance<L::kStagesV>(n_ring - n);
  }

  // epilogue: O / l -> bf16 rows and the natural-log LSE (or, for a split-KV
  // chunk, fp32 partial rows and log2 LSEs), deferred to the next prefill
  // item's first tile (or the end of the CTA's work)
  const bool part = w.partial >= 0;
  __nv_bfloat16* dst = p.out + (int64_t)tok * p.o_stride_tok + (int64_t)head * p.o_stride_head;
  float* pdst = p.partial_o + ((int64_t)w.partial * kDecodeRows + r) * D;
  float* lse_dst = !valid ? nullptr
                   : part ? p.partial_lse + (int64_t)w.partial * kDecodeRows + r
                          : (p.lse != nullptr ? p.lse + (int64_t)head * p.total_q + tok : nullptr);
  const float lse = l > 0.f ? (part ? m + __log2f(l) : (m + __log2f(l)) * kLn2) : -INFINITY;
  if (n > 0 && part) {
    // a split-KV chunk: its partial rows at once (the previous item's deferred
    // epilogue ran in this item's first tile)
    if (!epi_partial<L>(B, pt + n - 1, qt, l > 0.f ? vscale / l : 0.f, lse, valid ? pdst : nullptr, lse_dst, t_lane,
                        abort_flag))
      return false;
  } else if (n > 0) {
    pend.has = true;
    pend.T = pt + n - 1;
    pend.inv = l > 0.f ? vscale / l : 0.f;
    pend.lse = lse;
    pend.dst = valid ? dst : nullptr;
    pend.lse_dst = lse_dst;
  } else {
    if (valid && part) {
#pragma unroll
      for (int c = 0; c < D / 4; ++c) *reinterpret_cast<float4*>(pdst + c * 4) = make_float4(0.f, 0.f, 0.f, 0.f);
    } else if (valid) {
#pragma unroll
      for (int c = 0; c < D / 8; ++c) *reinterpret_cast<uint4*>(dst + c * 8) = make_uint4(0, 0, 0, 0);
    }
    if (lse_dst != nullptr) *lse_dst = lse;
  }
  pt += n;
  return true;
}

// ------------------------------------------------------------------ decode tiles (warp MMAs)
// A decode unit has R = n_q * G <= 16 query rows.  The four consumer warps
// split each 128-key tile (32 keys each) and compute it transposed: keys and
// head dims fill the 16-row M side of m16n8k16 MMAs and the unit's query rows
// the 8-column N side (NQ column tiles of 8), S^T = K Q^T, then O^T += V^T P^T,
// P^T handed from the S^T accumulators to the B operand by 8x8 transposes
// (movmatrix).  With G = 4 query rows this takes half the MMAs of the
// untransposed form, whose 16-row M was three quarters padding; the legacy
// warp-MMA path is what bounded these tiles.
//
// fp8 cache: e4m3 K and V become f16 in registers (exact).  A dot product does
// not depend on the order of d, so the k slots of k-step 4c+u of a thread with
// column index t map to d = 64c + 16t + 4u + {0,1 | 2,3} for both K and Q: one
// 16-byte read of a key row serves four k-steps.  For V an ldmatrix.trans on
// byte pairs gives a thread keys (2t, 2t+1) x d (2g, 2g+1) of a 16-byte chunk;
// a byte permute splits that into the A rows g (d = 2g) and g+8 (d = 2g+1), so
// the O^T rows of chunk c are d = 16c + 2g and 16c + 2g + 1.  With q_scale
// (QF8) S^T runs as m16n8k32 e4m3 MMAs on the raw K bytes (k-step 2c+h: words
// 2h, 2h+1 of chunk 4c+t).
//
// Decode-only plans over an fp8 cache (kStageRegs) copy each warp's share of
// the K and V tiles into registers and release both stages before any
// arithmetic; otherwise K is released after S and V after P V, the item's
// last V stage serving as the merge scratch.
template <int D, bool FP8, bool PF, bool QF8, int NQ>
__device__ bool run_decode(const AttnParams& p, const WorkItem& w, uint8_t* smem, const Bars& B,
                           volatile int* abort_flag, Ring& rk, Ring& rv, float sl2, float vscale, uint32_t& dtc) {
  using L = Layout<D, FP8, PF>;
  constexpr bool kArea = L::kStageRegs;          // the merge area exists (else: the borrowed V stage)
  constexpr bool kRegs = L::kStageRegs && NQ == 1;  // tiles staged in registers (no room at NQ = 2)
  constexpr int W = L::kDecWarps;                // consumer warps merged at the end of the item
  constexpr int kThreadsW = 32 * W;
  constexpr int kTile = L::kTile;
  constexpr int KPW = kTile / kConsumerWarps;    // keys of each tile per warp
  constexpr int MT = KPW / 16;                   // key m-tiles per warp
  constexpr int DT = D / 16;                     // head-dim m-tiles of O^T
  constexpr int KS = QF8 ? D / 32 : D / 16;      // k-steps of S^T
  constexpr int RB = L::kRowBytes;
  constexpr int kFin = D + 4;                    // row stride (floats) of the merged O in shared memory
  const int lane = threadIdx.x & 31;
  const int cw = (threadIdx.x >> 5) - L::kCons0;  // 0 .. W-1
  const int gi = cw / kConsumerWarps;            // consumer group: it runs the tiles with dtc % groups == gi
  const int ctid = threadIdx.x - 32 * L::kCons0;
  const int g = lane >> 2, t = lane & 3;
  const int mi = lane >> 3;                      // ldmatrix: the 8x8 matrix this lane addresses
  const int kw0 = (cw % kConsumerWarps) * KPW;   // this warp's keys of each of its group's tiles
  // Key of row x (0..7, and x + 8) of a 16-key m-tile: x, or (fp8 cache with
  // 128-byte rows, swizzled chunk XOR row % 8) the interleaving 0 4 1 5 2 6 3 7,
  // so that the two key rows a quarter-warp's 16-byte K reads span (rows of g
  // and g + 1, four chunks each) fall on different bank groups; V and the
  // masks follow the same order.
  constexpr bool kPerm = FP8 && RB == 128;
  auto krow = [](int x) { return kPerm ? (((x & 1) << 2) | (x >> 1)) : x; };
  const int R = w.n_q * p.G;

  // this thread's query rows (N columns of S^T and O^T): 8j + 2t + e
  int lim[NQ][2];
#pragma unroll
  for (int j = 0; j < NQ; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      const int r = 8 * j + 2 * t + e;
      int l = w.kv_begin;
      if (r < R) {
        l = w.kv_end;
        if (p.causal) l = min(l, w.q_i0 + r / p.G + w.lk - w.lq + 1);
      }
      lim[j][e] = l;
    }

  // Q^T (B operand): query row 8j + g of the tile
  uint32_t qb[NQ][KS][2];
#pragma unroll
  for (int j = 0; j < NQ; ++j) {
    const int r = 8 * j + g;
    const __nv_bfloat16* qr =
        r < R ? p.q + (int64_t)(w.q_row0 + r / p.G) * p.q_stride_tok + (int64_t)(w.hk * p.G + r % p.G) * p.q_stride_head
              : nullptr;
    if constexpr (QF8) {
      // the cache's encode: one IEEE reciprocal, an RN multiply per value, RN satfinite to e4m3
      const float inv_q = __frcp_rn(__ldg(p.q_scale));
      auto quant4 = [&](uint32_t w0, uint32_t w1) -> uint32_t {
        auto lo = [](uint32_t v) { return __uint_as_float(v << 16); };
        auto hi = [](uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); };
        const uint32_t a = f32x2_to_e4m3x2(__fmul_rn(lo(w0), inv_q), __fmul_rn(hi(w0), inv_q));
        const uint32_t b = f32x2_to_e4m3x2(__fmul_rn(lo(w1), inv_q), __fmul_rn(hi(w1), inv_q));
        return a | (b << 16);
      };
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int d0 = 16 * (4 * (ks >> 1) + t) + 8 * (ks & 1);
        const uint4 v = qr ? __ldg(reinterpret_cast<const uint4*>(qr + d0)) : make_uint4(0, 0, 0, 0);
        qb[j][ks][0] = quant4(v.x, v.y);
        qb[j][ks][1] = quant4(v.z, v.w);
      }
    } else if constexpr (FP8) {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int d0 = 64 * (ks >> 2) + 16 * t + 4 * (ks & 3);
        qb[j][ks][0] = qr ? bf16x2_to_f16x2(ld_u32(qr + d0)) : 0u;
        qb[j][ks][1] = qr ? bf16x2_to_f16x2(ld_u32(qr + d0 + 2)) : 0u;
      }
    } else {
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        qb[j][ks][0] = qr ? ld_u32(qr + 16 * ks + 2 * t) : 0u;
        qb[j][ks][1] = qr ? ld_u32(qr + 16 * ks + 8 + 2 * t) : 0u;
      }
    }
  }

  float o[NQ][DT][4];
#pragma unroll
  for (int j = 0; j < NQ; ++j)
#pragma unroll
    for (int dt = 0; dt < DT; ++dt) o[j][dt][0] = o[j][dt][1] = o[j][dt][2] = o[j][dt][3] = 0.f;
  float m[NQ][2], l[NQ][2];
#pragma unroll
  for (int j = 0; j < NQ; ++j) m[j][0] = m[j][1] = -INFINITY, l[j][0] = l[j][1] = 0.f;
  int merge_stage = -1;
  // A failed (timed-out or aborted) wait ends this warp's tiles, but the warp
  // still passes every barrier of the merge below, so that no other consumer
  // warp can be left waiting there.
  bool failed = false;

  for (int t0 = w.kv_begin; t0 < w.kv_end; t0 += kTile) {
    const bool mine = L::kDecGroups == 1 || (int)(dtc % L::kDecGroups) == gi;
    ++dtc;
    if (!mine) {  // the other group's tile: every warp advances the rings over all tiles
      rk.advance<L::kStagesK>();
      rv.advance<L::kStagesV>();
      continue;
    }
    if (!warp_wait(&B.full_k[rk.stage], rk.phase, abort_flag)) {
      failed = true;
      break;
    }
    const uint32_t kb = smem_u32(smem + L::kKOff + rk.stage * L::kTileBytes);
    const uint32_t vb = smem_u32(smem + L::kVOff + rv.stage * L::kTileBytes);
    // fp8: this warp's K rows (16 bytes of each per lane) and, staged, its V fragments
    uint4 kreg[kRegs ? MT : 1][2][kRegs ? D / 64 : 1];
    uint32_t vreg[kRegs ? MT : 1][kRegs ? D / 32 : 1][4];
    if constexpr (kRegs) {
#pragma unroll
      for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int h = 0; h < 2; ++h)
#pragma unroll
          for (int c = 0; c < D / 64; ++c)
            kreg[i][h][c] = lds_u128(kb + raw_off<RB, kTile>(kw0 + 16 * i + 8 * h + krow(g), 4 * c + t));
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.empty_k[rk.stage]);
      if (!warp_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) {
        failed = true;
        break;
      }
#pragma unroll
      for (int i = 0; i < MT; ++i)
#pragma unroll
        for (int cp = 0; cp < D / 32; ++cp)
          ldsm_x4_t(vb + raw_off<RB, kTile>(kw0 + 16 * i + (mi & 1) * 8 + krow(lane & 7), 2 * cp + (mi >> 1)), vreg[i][cp][0],
                    vreg[i][cp][1], vreg[i][cp][2], vreg[i][cp][3]);
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.empty_v[rv.stage]);
    }

    // S^T = K Q^T: key m-tile i, query column tile j
    float s[NQ][MT][4];
#pragma unroll
    for (int j = 0; j < NQ; ++j)
#pragma unroll
      for (int i = 0; i < MT; ++i) s[j][i][0] = s[j][i][1] = s[j][i][2] = s[j][i][3] = 0.f;
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      if constexpr (FP8) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint4 ka, kc;
          if constexpr (kRegs) {
            ka = kreg[i][0][c];
            kc = kreg[i][1][c];
          } else {
            ka = lds_u128(kb + raw_off<RB, kTile>(kw0 + 16 * i + krow(g), 4 * c + t));
            kc = lds_u128(kb + raw_off<RB, kTile>(kw0 + 16 * i + 8 + krow(g), 4 * c + t));
          }
          const uint32_t wa[4] = {ka.x, ka.y, ka.z, ka.w}, wc[4] = {kc.x, kc.y, kc.z, kc.w};
          if constexpr (QF8) {
#pragma unroll
            for (int h = 0; h < 2; ++h)
#pragma unroll
              for (int j = 0; j < NQ; ++j)
                mma_e4m3(s[j][i], wa[2 * h], wc[2 * h], wa[2 * h + 1], wc[2 * h + 1], qb[j][2 * c + h][0],
                         qb[j][2 * c + h][1]);
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint32_t a0, a1, a2, a3;
              e4m3x4_to_f16x4(wa[u], a0, a2);
              e4m3x4_to_f16x4(wc[u], a1, a3);
#pragma unroll
              for (int j = 0; j < NQ; ++j) mma_f16(s[j][i], a0, a1, a2, a3, qb[j][4 * c + u][0], qb[j][4 * c + u][1]);
            }
          }
        }
      } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4(kb + tile_off<kTile>(kw0 + 16 * i + (mi & 1) * 8 + (lane & 7), 2 * ks + (mi >> 1)), a0, a1, a2, a3);
#pragma unroll
          for (int j = 0; j < NQ; ++j) mma_bf16(s[j][i], a0, a1, a2, a3, qb[j][ks][0], qb[j][ks][1]);
        }
      }
    }
    if constexpr (!kRegs) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.empty_k[rk.stage]);
    }

    // mask (select, never add) and online softmax in the log2 domain; a
    // query row's keys are spread over the 8 lanes of its column (g)
    float al[NQ][2];
#pragma unroll
    for (int j = 0; j < NQ; ++j) {
      float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        const int ka = t0 + kw0 + 16 * i + krow(g), kc = ka + 8;
        s[j][i][0] = ka < lim[j][0] ? s[j][i][0] * sl2 : -INFINITY;
        s[j][i][1] = ka < lim[j][1] ? s[j][i][1] * sl2 : -INFINITY;
        s[j][i][2] = kc < lim[j][0] ? s[j][i][2] * sl2 : -INFINITY;
        s[j][i][3] = kc < lim[j][1] ? s[j][i][3] * sl2 : -INFINITY;
        mx[0] = fmax3(mx[0], s[j][i][0], s[j][i][2]);
        mx[1] = fmax3(mx[1], s[j][i][1], s[j][i][3]);
      }
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 4));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 8));
        mx[e] = fmaxf(mx[e], __shfl_xor_sync(0xffffffffu, mx[e], 16));
        const float mn = fmaxf(m[j][e], mx[e]);
        const float mu = mn == -INFINITY ? 0.f : mn;
        al[j][e] = ex2(m[j][e] - mu);
        m[j][e] = mn;
        mx[e] = mu;
      }
      float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
      for (int i = 0; i < MT; ++i) {
        s[j][i][0] = ex2(s[j][i][0] - mx[0]);
        s[j][i][1] = ex2(s[j][i][1] - mx[1]);
        s[j][i][2] = ex2(s[j][i][2] - mx[0]);
        s[j][i][3] = ex2(s[j][i][3] - mx[1]);
        ls0 += s[j][i][0] + s[j][i][2];
        ls1 += s[j][i][1] + s[j][i][3];
      }
      l[j][0] = l[j][0] * al[j][0] + ls0;
      l[j][1] = l[j][1] * al[j][1] + ls1;
#pragma unroll
      for (int dt = 0; dt < DT; ++dt) {
        o[j][dt][0] *= al[j][0];
        o[j][dt][1] *= al[j][1];
        o[j][dt][2] *= al[j][0];
        o[j][dt][3] *= al[j][1];
      }
    }

    if (!kRegs && !warp_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) {
      failed = true;
      break;
    }
    // O^T += V^T P^T, one key m-tile of P^T (16 keys) per k-step
    const bool vmask = t0 + kTile > w.lk;  // rows past the sequence may hold anything: zero them
#pragma unroll
    for (int i = 0; i < MT; ++i) {
      uint32_t pb[NQ][2];
#pragma unroll
      for (int j = 0; j < NQ; ++j) {
        pb[j][0] = movm_t(FP8 ? pack_f16(s[j][i][0], s[j][i][1]) : pack_bf16(s[j][i][0], s[j][i][1]));
        pb[j][1] = movm_t(FP8 ? pack_f16(s[j][i][2], s[j][i][3]) : pack_bf16(s[j][i][2], s[j][i][3]));
      }
      const int k0 = t0 + kw0 + 16 * i + krow(2 * t), k1 = t0 + kw0 + 16 * i + krow(2 * t + 1);
      const uint32_t mlo = (k0 < w.lk ? 0x0000FFFFu : 0u) | (k1 < w.lk ? 0xFFFF0000u : 0u);
      const uint32_t mhi = (k0 + 8 < w.lk ? 0x0000FFFFu : 0u) | (k1 + 8 < w.lk ? 0xFFFF0000u : 0u);
      if constexpr (FP8) {
#pragma unroll
        for (int cp = 0; cp < D / 32; ++cp) {
          uint32_t v[4];
          if constexpr (kRegs) {
            v[0] = vreg[i][cp][0], v[1] = vreg[i][cp][1], v[2] = vreg[i][cp][2], v[3] = vreg[i][cp][3];
          } else {
            ldsm_x4_t(vb + raw_off<RB, kTile>(kw0 + 16 * i + (mi & 1) * 8 + krow(lane & 7), 2 * cp + (mi >> 1)), v[0], v[1],
                      v[2], v[3]);
          }
#pragma unroll
          for (int h = 0; h < 2; ++h) {  // chunk 2cp + h: O^T m-tile 2cp + h
            // bytes (0, 2) and (1, 3) of each word: one permute, then its halves
            uint32_t a0, a1, a2, a3;
            e4m3x4_to_f16x4(prmt(v[2 * h], 0u, 0x3120u), a0, a1);
            e4m3x4_to_f16x4(prmt(v[2 * h + 1], 0u, 0x3120u), a2, a3);
            if (vmask) {
              a0 &= mlo;
              a1 &= mlo;
              a2 &= mhi;
              a3 &= mhi;
            }
#pragma unroll
            for (int j = 0; j < NQ; ++j) mma_f16(o[j][2 * cp + h], a0, a1, a2, a3, pb[j][0], pb[j][1]);
          }
        }
      } else {
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          uint32_t a0, a1, a2, a3;
          ldsm_x4_t(vb + tile_off<kTile>(kw0 + 16 * i + (mi >> 1) * 8 + (lane & 7), 2 * dt + (mi & 1)), a0, a1, a2, a3);
          if (vmask) {
            a0 &= mlo;
            a1 &= mlo;
            a2 &= mhi;
            a3 &= mhi;
          }
#pragma unroll
          for (int j = 0; j < NQ; ++j) mma_bf16(o[j][dt], a0, a1, a2, a3, pb[j][0], pb[j][1]);
        }
      }
    }
    if constexpr (!kRegs) {
      if (!kArea && t0 + kTile >= w.kv_end) {
        merge_stage = rv.stage;  // released after the merge below, which uses it as scratch
      } else {
        __syncwarp();
        if (lane == 0) mbar_arrive(&B.empty_v[rv.stage]);
      }
    }
    rk.advance<L::kStagesK>();
    rv.advance<L::kStagesV>();
  }

  // ---------------------------------------------------------------- epilogue
  // the row sums were accumulated per lane over its own keys
#pragma unroll
  for (int j = 0; j < NQ; ++j)
#pragma unroll
    for (int e = 0; e < 2; ++e) {
      l[j][e] += __shfl_xor_sync(0xffffffffu, l[j][e], 4);
      l[j][e] += __shfl_xor_sync(0xffffffffu, l[j][e], 8);
      l[j][e] += __shfl_xor_sync(0xffffffffu, l[j][e], 16);
    }
  if (num_tiles<L::kTile>(w) == 0) {
    // no key at all: every row is 0 with LSE -inf (a split-KV chunk that a
    // dynamic plan's current length left empty gives such a partial)
    for (int idx = ctid; idx < R * D; idx += kThreadsW) {
      const int row = idx / D, d = idx % D;
      if (w.partial >= 0) {
        p.partial_o[((int64_t)w.partial * kDecodeRows + row) * D + d] = 0.f;
        if (d == 0) p.partial_lse[w.partial * kDecodeRows + row] = -INFINITY;
        continue;
      }
      const int tok = w.q_row0 + row / p.G;
      const int head = w.hk * p.G + row % p.G;
      p.out[(int64_t)tok * p.o_stride_tok + (int64_t)head * p.o_stride_head + d] = __float2bfloat16_rn(0.f);
      if (d == 0 && p.lse != nullptr) p.lse[(int64_t)head * p.total_q + tok] = -INFINITY;
    }
    return true;
  }
  // Merge of the W warps' partial results.  The warps write their (m, l) per
  // row; then either (one column tile, merge area) every warp writes its O^T
  // fragments and every consumer thread sums the W warps' values of the
  // output columns it writes, or the fragments are added in fragment order in
  // a tree (the upper half of the remaining warps putting, the lower half
  // adding) until warp 0 holds the sum and stores O / l as a [16][D] matrix
  // over the slots it has read, and every consumer thread writes whole output
  // rows from it.  Scratch: the borrowed V stage or the merge area.
  constexpr bool kFlat = kArea && NQ == 1;
  constexpr int kSlot = NQ * DT * 32;  // float4 per slot
  constexpr int kScratch = kArea ? L::kMergeBytes : L::kTileBytes;
  static_assert((kFlat ? W : W / 2) * kSlot * 16 <= kScratch, "merge slots fit the scratch");
  static_assert(kFlat || 8 * NQ * kFin * 4 <= kScratch, "merged rows fit the scratch");
  float* ml = reinterpret_cast<float*>(smem + L::kMlOff);
  uint8_t* scratch = smem + (kArea ? L::kMergeOff : L::kVOff + merge_stage * L::kTileBytes);
  float4* buf = reinterpret_cast<float4*>(scratch);  // [slots][NQ][DT][32] float4
  float* fin = reinterpret_cast<float*>(scratch);    // [8 * NQ][kFin], after the tree
  int* bad = reinterpret_cast<int*>(ml + W * kDecodeRows * 2);  // [warp]: its waits failed
  if (g == 0) {
#pragma unroll
    for (int j = 0; j < NQ; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int row = 8 * j + 2 * t + e;
        ml[(cw * 16 + row) * 2 + 0] = m[j][e];
        ml[(cw * 16 + row) * 2 + 1] = l[j][e];
      }
  }
  if (lane == 0) bad[cw] = failed ? 1 : 0;
  if (failed && lane == 0) *abort_flag = 1;
  auto put = [&](int slot) {
#pragma unroll
    for (int j = 0; j < NQ; ++j)
#pragma unroll
      for (int dt = 0; dt < DT; ++dt)
        buf[(slot * NQ * DT + j * DT + dt) * 32 + lane] = make_float4(o[j][dt][0], o[j][dt][1], o[j][dt][2], o[j][dt][3]);
  };
  if constexpr (kFlat) {
    if (!failed) put(cw);
  }
  named_bar_sync(1, kThreadsW);
  bool any_bad = false;
#pragma unroll
  for (int ww = 0; ww < W; ++ww) any_bad |= bad[ww] != 0;
  // row statistics over the W warps: the common max, the sum, and the log2 LSE
  auto row_stats = [&](int row, float& mu, float& Lsum) {
    float M = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < W; ++ww) M = fmaxf(M, ml[(ww * 16 + row) * 2]);
    mu = M == -INFINITY ? 0.f : M;
    Lsum = 0.f;
#pragma unroll
    for (int ww = 0; ww < W; ++ww) Lsum += ml[(ww * 16 + row) * 2 + 1] * ex2(ml[(ww * 16 + row) * 2] - mu);
  };
  auto write_lse = [&](int row, float mu, float Lsum) {
    const float lse2 = Lsum > 0.f ? mu + __log2f(Lsum) : -INFINITY;
    if (w.partial >= 0) {
      p.partial_lse[w.partial * kDecodeRows + row] = lse2;
    } else if (p.lse != nullptr) {
      const int tok = w.q_row0 + row / p.G;
      const int head = w.hk * p.G + row % p.G;
      p.lse[(int64_t)head * p.total_q + tok] = lse2 * kLn2;
    }
  };
  auto write_row8 = [&](int row, int d, const float* v) {
    if (w.partial >= 0) {
      float* dst = p.partial_o + ((int64_t)w.partial * kDecodeRows + row) * D + d;
      *reinterpret_cast<float4*>(dst) = make_float4(v[0], v[1], v[2], v[3]);
      *reinterpret_cast<float4*>(dst + 4) = make_float4(v[4], v[5], v[6], v[7]);
    } else {
      const int tok = w.q_row0 + row / p.G;
      const int head = w.hk * p.G + row % p.G;
      *reinterpret_cast<uint4*>(p.out + (int64_t)tok * p.o_stride_tok + (int64_t)head * p.o_stride_head + d) =
          make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
    }
  };
  if constexpr (kFlat) {
    // thread: row r, columns d .. d+7.  Row r = 2t + e of the fragments; column
    // d of m-tile dt sits at (g, component) = bf16 V: (d % 8, e + 2 * (d % 16 >= 8)),
    // fp8 V: ((d % 16) / 2, e + 2 * (d % 2))
    for (int idx = ctid; idx < R * (D / 8) && !any_bad; idx += kThreadsW) {
      const int row = idx / (D / 8), d0 = (idx % (D / 8)) * 8;
      const int rt = row >> 1, re = row & 1, dt = d0 >> 4;
      float mu, Lsum;
      row_stats(row, mu, Lsum);
      const float inv = Lsum > 0.f ? vscale / Lsum : 0.f;
      float v[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
      for (int ww = 0; ww < W; ++ww) {
        const float f = ex2(ml[(ww * 16 + row) * 2] - mu) * inv;
        const float* sl = reinterpret_cast<const float*>(buf + (ww * DT + dt) * 32);
#pragma unroll
        for (int k = 0; k < 8; ++k) {
          const int dd = (d0 & 15) + k;
          const int gg = FP8 ? dd >> 1 : dd & 7;
          const int cc = FP8 ? re + 2 * (dd & 1) : re + 2 * (dd >> 3);
          v[k] += f * sl[(4 * gg + rt) * 4 + cc];
        }
      }
      write_row8(row, d0, v);
      if (d0 == 0) write_lse(row, mu, Lsum);
    }
  } else {
    float Mu[NQ][2], Ls[NQ][2];
#pragma unroll
    for (int j = 0; j < NQ; ++j)
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        row_stats(8 * j + 2 * t + e, Mu[j][e], Ls[j][e]);
        const float f = ex2(m[j][e] - Mu[j][e]);
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          o[j][dt][e] *= f;
          o[j][dt][2 + e] *= f;
        }
      }
    auto add = [&](int slot) {
#pragma unroll
      for (int j = 0; j < NQ; ++j)
#pragma unroll
        for (int dt = 0; dt < DT; ++dt) {
          const float4 v = buf[(slot * NQ * DT + j * DT + dt) * 32 + lane];
          o[j][dt][0] += v.x;
          o[j][dt][1] += v.y;
          o[j][dt][2] += v.z;
          o[j][dt][3] += v.w;
        }
    };
#pragma unroll
    for (int half = W / 2; half >= 1; half >>= 1) {
      if (!any_bad && cw >= half && cw < 2 * half) put(cw - half);
      named_bar_sync(1, kThreadsW);
      if (!any_bad && cw < half) add(cw);
      if (half > 1) named_bar_sync(1, kThreadsW);
    }
    if (!any_bad && cw == 0) {
      __syncwarp();  // every lane has read slot 0 before it is overwritten
#pragma unroll
      for (int j = 0; j < NQ; ++j)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int row = 8 * j + 2 * t + e;
          const float inv = Ls[j][e] > 0.f ? vscale / Ls[j][e] : 0.f;
#pragma unroll
          for (int dt = 0; dt < DT; ++dt) {
            // O^T rows g and g+8 of m-tile dt: d = 16dt + g, 16dt + 8 + g (bf16 V), or 16dt + 2g, 16dt + 2g + 1 (fp8 V)
            const int da = FP8 ? 16 * dt + 2 * g : 16 * dt + g;
            const int dc = FP8 ? da + 1 : da + 8;
            fin[row * kFin + da] = o[j][dt][e] * inv;
            fin[row * kFin + dc] = o[j][dt][2 + e] * inv;
          }
          if (g == 0 && row < R) write_lse(row, Mu[j][e], Ls[j][e]);
        }
    }
    named_bar_sync(1, kThreadsW);
    // every consumer thread writes 8 consecutive columns of a row at a time
    for (int idx = ctid; idx < R * (D / 8) && !any_bad; idx += kThreadsW) {
      const int row = idx / (D / 8), d = (idx % (D / 8)) * 8;
      float v[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) v[k] = fin[row * kFin + d + k];
      write_row8(row, d, v);
    }
  }
  named_bar_sync(1, kThreadsW);
  if (merge_stage >= 0) {
    // the borrowed V stage goes back to the producer (generic writes before the next async copy)
    fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.empty_v[merge_stage]);
  }
  return !any_bad;
}

template <int D, bool FP8, bool PF, bool QF8, bool DEC>
__device__ bool consumer(const AttnParams& p, uint8_t* smem, const Bars& B, volatile int* abort_flag, uint32_t tmem,
                         int it0, int it1) {
  using L = Layout<D, FP8, PF>;
  const int ctid = threadIdx.x - 32 * L::kCons0;
  const bool mma_consumer = ctid < 32 * L::kDecWarps;  // the decode consumer warps
  if (blockIdx.x == 0 && mma_consumer) {
    for (int b = ctid; b < p.batch; b += 32 * L::kDecWarps) {
      const int lc = __ldg(p.cache_seqlens + b), planned = __ldg(p.plan_lc + b);
      if (p.dynamic ? (lc < 0 || lc > planned) : lc != planned) record_status(p.status, PKV_ERR_PLAN_MISMATCH, b, lc);
    }
  }
  const float kscale = FP8 ? __ldg(p.k_scale) : 1.f;
  const float vscale = FP8 ? __ldg(p.v_scale) : 1.f;
  const float sl2 = p.scale_log2 * kscale;
  // quantised queries: S = codes(Q) . codes(K), times q_scale and k_scale
  const float sl2q = (FP8 && p.q_scale) ? sl2 * __ldg(p.q_scale) : sl2;
  Ring rk, rv;
  uint32_t pt = 0;
  uint32_t dtc = 0;  // decode tiles seen (consumer groups take alternate ones)
  PendingEpi pend;
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = load_item(p, it);
    if (it + 1 < it1) {
      // the next descriptor is in L1 when this item ends
      prefetch_l1(p.items + it + 1);
      prefetch_l1(reinterpret_cast<const char*>(p.items + it + 2) - 1);
    }
    bool ok = true;
    if (w.kind == kDecode) {
      if (mma_consumer) {
        // one or two 8-column query tiles (decode units hold at most 16 rows)
        // (at D = 256 the plan gives decode tiles at most 8 rows)
        // (a kernel built without decode tiles never receives them)
        if constexpr (DEC) {
          if (D > 128 || w.n_q * p.G <= 8)
            ok = run_decode<D, FP8, PF, QF8, 1>(p, w, smem, B, abort_flag, rk, rv, QF8 ? sl2q : sl2, vscale, dtc);
          else if constexpr (D <= 128)
            ok = run_decode<D, FP8, PF, QF8, 2>(p, w, smem, B, abort_flag, rk, rv, QF8 ? sl2q : sl2, vscale, dtc);
        } else {
          ok = false;
        }
      } else {
        rk.advance<L::kStagesK>(num_tiles<L::kTile>(w));
        rv.advance<L::kStagesV>(num_tiles<L::kTile>(w));
      }
    } else if constexpr (PF) {
      // (two query tiles per item: warpgroup qt takes tile qt; the second
      // tile's warps zero V rows past the sequence whenever it has keys)
      const int qt = L::kQQ ? ((threadIdx.x >> 5) - L::kCons0) >> 2 : 0;
      const WorkItem wq = L::kQQ ? q_tile(w, qt, p.causal) : w;
      const bool zero_owner = !L::kQQ || qt == 1 || num_tiles<L::kTile>(q_tile(w, 1, p.causal)) == 0;
      ok = softmax_item<D, FP8, PF>(p, wq, smem, B, abort_flag, tmem, rk, rv, pt, QF8 ? sl2q : sl2, vscale, pend, qt,
                                    num_tiles<L::kTile>(w), zero_owner);
    } else {
      ok = false;  // a decode-only launch never receives prefill tiles
    }
    if (!ok) {
      record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, it);
      *abort_flag = 1;
      return false;
    }
  }
  if constexpr (PF) {
    if (pend.has) {
      // the last prefill item's epilogue
      const int qw = (threadIdx.x >> 5) & 3;
      const int qt = L::kQQ ? ((threadIdx.x >> 5) - L::kCons0) >> 2 : 0;
      if (!epi_run<L>(p, B, pend, tmem + ((uint32_t)(qw * 32) << 16), qt, abort_flag)) {
        record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, it1);
        *abort_flag = 1;
        return false;
      }
      tc_fence_before();
    }
  }
  return true;
}

// DEC: the plan has decode tiles.  Plans with prefill tiles only run an
// instance without the decode tile's code, whose register demand would
// otherwise weigh on the softmax path (measured: 133 -> 123 us on the
// cached-prefix prefill batch).
template <int D, bool FP8, bool PF, bool QF8, bool DEC>
__global__ void __launch_bounds__(Layout<D, FP8, PF>::kThreads, Layout<D, FP8, PF>::kCtasPerSm)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q) {
  using L = Layout<D, FP8, PF>;
  extern __shared__ __align__(1024) uint8_t smem_raw[];
  if ((smem_u32(smem_raw) & 1023) != 0) {
    // the swizzled TMA / MMA layouts need a 1024-byte aligned base: refuse, never overrun
    if (threadIdx.x == 0) record_status(p.status, PKV_ERR_UNSUPPORTED, blockIdx.x, (int)(smem_u32(smem_raw) & 1023));
    return;
  }
  uint8_t* smem = smem_raw;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  Bars B;
  B.full_k = bars;
  B.empty_k = bars + L::kStagesK;
  B.full_v = bars + 2 * L::kStagesK;
  B.empty_v = bars + 2 * L::kStagesK + L::kStagesV;
  B.q_full = bars + 2 * L::kStagesK + 2 * L::kStagesV;
  B.q_empty = B.q_full + 1;
  B.drain = B.q_full + 2;
  B.s_full = B.q_full + 3;
  B.p_full = B.s_full + kSBufsMax;
  B.o_done = B.p_full + kSBufsMax;
  B.qc_full = B.o_done + kSBufsMax;
  B.kc_full = B.qc_full + 1;
  B.kc_empty = B.kc_full + 2;
  B.vc_full = B.kc_empty + 2;
  B.vc_empty = B.vc_full + 2;
  B.drain_pv = B.vc_empty + 2;
  B.q_full_b = B.drain_pv + 1;
  B.q_empty_b = B.drain_pv + 2;
  B.qc_full_b = B.drain_pv + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    // a full barrier takes the producer's arrival (with the copies' bytes), or
    // one arrival per producer lane when rows are gathered
    const uint32_t full_count = p.row_gather ? 32u : 1u;
    for (int s = 0; s < L::kStagesK; ++s) {
      mbar_init(&B.full_k[s], full_count);
      mbar_init(&B.empty_k[s], kConsumerWarps);
    }
    for (int s = 0; s < L::kStagesV; ++s) {
      mbar_init(&B.full_v[s], full_count);
      mbar_init(&B.empty_v[s], kConsumerWarps);
    }
    mbar_init(B.q_full, 1);
    mbar_init(B.q_empty, 1);
    mbar_init(B.q_full_b, 1);
    mbar_init(B.q_empty_b, 1);
    for (int i = 0; i < kSBufsMax; ++i) {
      mbar_init(&B.s_full[i], 1);
      // one arrival per softmax warp of the query tile the buffer serves
      mbar_init(&B.p_full[i], L::kQQ ? kConsumerWarps : L::kSoftmaxWarps);
      mbar_init(&B.o_done[i], 1);
    }
    if (L::kConvWarps > 0) {
      mbar_init(B.qc_full, L::kConvWarps);
      mbar_init(B.qc_full_b, L::kConvWarps);
      for (int i = 0; i < 2; ++i) {
        mbar_init(&B.kc_full[i], L::kConvWarps);
        mbar_init(&B.kc_empty[i], 1);
        mbar_init(&B.vc_full[i], L::kConvWarps);
        mbar_init(&B.vc_empty[i], 1);
      }
    }
    mbar_init(B.drain, 1);
    mbar_init(B.drain_pv, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (L::kTc && warp == L::kSWarp) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = L::kTc ? *tmem_slot : 0u;
  grid_dep_launch();  // the combine kernel may be scheduled; it waits for this grid to finish
  const int it0 = p.cta_begin[blockIdx.x], it1 = p.cta_begin[blockIdx.x + 1];
  if constexpr (L::kSplitRegs) {
    // softmax (one warpgroup per query tile), converters (fp8 cache),
    // producers and issuers: the registers of the warpgroups add up to exactly
    // what the block was launched with (fp8, two query tiles: 2 x 144 + 152 +
    // 72 of 4 x 128; bf16, two query tiles: 2 x 216 + 72 of 3 x 168; fp8 at
    // D = 256: 240 + 152 + 112 of 3 x 168).  Each warpgroup runs one setmaxnreg
    // at the head of its branch.
    static_assert((L::kSoftmaxWarps * L::kRegsSoftmax + L::kConvWarps * L::kRegsConv + 4 * L::kRegsSingle) * 32 ==
                      L::kLaunchRegs * L::kThreads,
                  "register split");
    if (warp >= L::kSingle0) {
      reg_dealloc<L::kRegsSingle>();
      if (warp == L::kKProdWarp) {
        producer<D, FP8, PF, false>(p, &tm_k, &tm_q, smem, B, abort_flag, it0, it1);
        return;
      }
      if (warp == L::kVProducerWarp) {
        producer<D, FP8, PF, true>(p, &tm_v, &tm_q, smem, B, abort_flag, it0, it1);
        return;
      }
      if (lane == 0) {
        const bool pv = warp == L::kPvWarp;
        bool ok;
        if constexpr (L::kQQ)
          ok = pv ? pv_issuer_qq<D, FP8, PF>(p, smem, B, abort_flag, tmem, it0, it1)
                  : s_issuer_qq<D, FP8, PF, QF8>(p, smem, B, abort_flag, tmem, it0, it1);
        else
          ok = pv ? pv_issuer<D, FP8, PF>(p, smem, B, abort_flag, tmem, it0, it1)
                  : s_issuer<D, FP8, PF, QF8>(p, smem, B, abort_flag, tmem, it0, it1);
        if (!ok) {
          record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, pv ? -3 : -1);
          *abort_flag = 1;
          int zero = 0;
          umma_commit(pv ? B.drain_pv : B.drain);
          mbar_wait(pv ? B.drain_pv : B.drain, 0, &zero);
        }
      }
      __syncwarp();
    } else if (L::kConvWarps > 0 && warp >= L::kConvWarp0) {
      if constexpr (L::kConvWarps > 0) {
        if constexpr (L::kRegsConv > L::kLaunchRegs) reg_alloc<L::kRegsConv>();
        else reg_dealloc<L::kRegsConv>();
        if (!converter<D, PF, QF8>(p, smem, B, abort_flag, it0, it1)) {
          if (lane == 0) record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, -2);
          *abort_flag = 1;
        }
      }
      return;
    } else {
      reg_alloc<L::kRegsSoftmax>();
      consumer<D, FP8, PF, QF8, DEC>(p, smem, B, abort_flag, tmem, it0, it1);
    }
    // the S issuer, the consumers and the P V warp: every tensor-memory access
    // is done before the S issuer's warp frees it
    tc_fence_before();
    named_bar_sync(2, 32 * (2 + L::kSoftmaxWarps));
    tc_fence_after();
    if (warp == L::kSWarp) tmem_dealloc(tmem, kTmemCols);
    return;
  }
  if (warp == L::kKProdWarp) {
    producer<D, FP8, PF, false>(p, &tm_k, &tm_q, smem, B, abort_flag, it0, it1);
    return;
  }
  if (warp == L::kVProducerWarp) {
    producer<D, FP8, PF, true>(p, &tm_v, &tm_q, smem, B, abort_flag, it0, it1);
    return;
  }
  if constexpr (L::kConvWarps > 0) {
    if (warp >= L::kConvWarp0 && warp < L::kConvWarp0 + L::kConvWarps) {
      if (!converter<D, PF, QF8>(p, smem, B, abort_flag, it0, it1)) {
        if (lane == 0) record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, -2);
        *abort_flag = 1;
      }
      return;
    }
  }
  if (L::kTc && (warp == L::kSWarp || warp == L::kPvWarp)) {
    if constexpr (L::kTc) {
      if (lane == 0) {
        const bool pv = warp == L::kPvWarp;
        if (!(pv ? pv_issuer<D, FP8, PF>(p, smem, B, abort_flag, tmem, it0, it1)
                 : s_issuer<D, FP8, PF, QF8>(p, smem, B, abort_flag, tmem, it0, it1))) {
          record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, pv ? -3 : -1);
          *abort_flag = 1;
          // wait (bounded) for this thread's MMAs already issued before the memory is freed
          int zero = 0;
          umma_commit(pv ? B.drain_pv : B.drain);
          mbar_wait(pv ? B.drain_pv : B.drain, 0, &zero);
        }
      }
      __syncwarp();
    }
  } else {
    consumer<D, FP8, PF, QF8, DEC>(p, smem, B, abort_flag, tmem, it0, it1);
  }
  if constexpr (L::kTc) {
    // the S issuer, the consumers and the P V warp: every tensor-memory access
    // is done before the S issuer's warp frees it
    tc_fence_before();
    named_bar_sync(2, 32 * (2 + L::kSoftmaxWarps));
    tc_fence_after();
    if (warp == L::kSWarp) tmem_dealloc(tmem, kTmemCols);
  }
}

template <int D, bool FP8, bool PF, bool QF8, bool DEC>
cudaError_t launch_t(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                     int num_ctas, bool overlap_prev, cudaStream_t s) {
  using L = Layout<D, FP8, PF>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  // (two CTAs an SM: both fit the SM's 228 KB with the 1 KB each reserves)
  static_assert(L::kCtasPerSm == 1 || L::kCtasPerSm * (L::kAlloc + 1024) <= 233472, "two CTAs an SM");
  // once per device (kept out of the launch path, so the call can be captured in a graph)
  static std::atomic<uint64_t> configured{0};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  const uint64_t bit = 1ull << (dev & 63);
  if (!(configured.load() & bit)) {
    e = cudaFuncSetAttribute(attn_kernel<D, FP8, PF, QF8, DEC>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             L::kAlloc);
    if (e != cudaSuccess) return e;
    if constexpr (L::kSplitRegs) {
      // the register split adds up to exactly the registers a thread has at
      // launch: a build with any other count could leave a warpgroup's increase
      // waiting, so it is refused before it runs
      cudaFuncAttributes fa{};
      e = cudaFuncGetAttributes(&fa, attn_kernel<D, FP8, PF, QF8, DEC>);
      if (e != cudaSuccess) return e;
      if (fa.numRegs != L::kLaunchRegs) return cudaErrorInvalidConfiguration;
    }
    configured.fetch_or(bit);
  }
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)num_ctas);
  cfg.blockDim = dim3(L::kThreads);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_prev ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, attn_kernel<D, FP8, PF, QF8, DEC>, p, tk, tv, tq);
}

// The instance for a plan: decode-only, prefill-only or mixed; quantised
// queries (fp8 caches) in instances of their own.
template <int D, bool FP8, bool QF8>
cudaError_t launch_kind(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                        int num_ctas, bool has_prefill, bool has_decode, bool o, cudaStream_t s) {
  if (!has_prefill) return launch_t<D, FP8, false, QF8, true>(p, tk, tv, tq, num_ctas, o, s);
  if (!has_decode) return launch_t<D, FP8, true, QF8, false>(p, tk, tv, tq, num_ctas, o, s);
  return launch_t<D, FP8, true, QF8, true>(p, tk, tv, tq, num_ctas, o, s);
}

template <int D>
cudaError_t launch_dim(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                       int num_ctas, bool fp8, bool has_prefill, bool has_decode, bool o, cudaStream_t s) {
  if (!fp8) return launch_kind<D, false, false>(p, tk, tv, tq, num_ctas, has_prefill, has_decode, o, s);
  if (p.q_scale) return launch_kind<D, true, true>(p, tk, tv, tq, num_ctas, has_prefill, has_decode, o, s);
  return launch_kind<D, true, false>(p, tk, tv, tq, num_ctas, has_prefill, has_decode, o, s);
}

}  // namespace

}  // namespace pkv
