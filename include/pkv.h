/*
 * pkv.h -- C ABI of the GB300 (sm_103a) library for forward attention over a
 * batched, variable-length KV cache (paged or contiguous).
 *
 * What the library computes, per sequence b, query head h (kv head h / G,
 * G = Hq / Hkv) and query row i:
 *     out[i,h] = softmax_j( scale * q[i,h] . K_b[j] + mask(i,j) ) V_b[j]
 * over the keys of the cache after the new tokens of this call are appended.
 * Sources (the pages this library follows):
 *  - flash-attention PR "Add flash_attn_varlen_func_with_kvcache", Usage:
 *    packed q with cu_seqlens_q / max_seqlen_q, optional new k/v appended into
 *    the cache in place, cache-only attention when k/v are absent, contiguous
 *    cache (batch_size_cache, seqlen_cache, n_heads, head_dim); Minor Changes:
 *    per-sequence cache lengths apart from cu_seqlens_knew; Limitation:
 *    num_splits fixed to 1 hurts decode (this library splits the KV instead).
 *  - TransformerEngine PR "Add KV cache for paged/non-paged attention",
 *    backend table and notes: paged and non-paged bshd caches, one page table
 *    for K and V, pure prefill / pure decode / mixed phases in one call.
 *  - vLLM PR "[Kernel][Triton][FP8] Adding fp8 and variable length sequence
 *    support to Triton FAv2 kernel", feature list: causal masking, GQA/MQA,
 *    8-bit KV cache; review: block_table support and mixed prefill/decode.
 *  - flashinfer PR "[Refactor] Uniform PoDAttention API with Horizontal Fusion
 *    SMs Schedule", Key Changes 2 and Limitations: one persistent launch for
 *    prefill and decode work, partitioned by KV load; a host classifier of
 *    prefill vs decode by query length (pkv_plan below).
 *
 * Conventions
 *  - Pointers are DEVICE pointers unless the name starts with h_.  Every
 *    device buffer is owned by the caller; the library never allocates or frees
 *    device memory.  The plan (pkv_plan_t) is a host object owned by the
 *    library until pkv_plan_destroy.
 *  - bf16 tensors: q, out, k_new, v_new, and a bf16 cache.  fp8 caches hold OCP
 *    e4m3 ("fn") codes with per-tensor fp32 scales: value = code * scale.
 *  - Strides are in ELEMENTS (of the tensor's own type).  The innermost
 *    (head_dim) stride is 1.  All base pointers must be 16-byte aligned and all
 *    strides multiples of 16 bytes.
 *  - Causal masking is bottom-right aligned: query i of a sequence with Lq
 *    queries and Lk keys sees keys j <= i + Lk - Lq.  A query row that sees no
 *    key gets out = 0 and lse = -inf.
 *  - Head mapping: query head h reads kv head h / (Hq / Hkv).
 *  - stream arguments are cudaStream_t passed as void* (NULL = legacy stream).
 *  - Errors: every entry point returns a pkv_status.  Problems detectable on
 *    the host are reported before anything is launched.  Problems found on the
 *    device (a block_table entry out of range, an append past the capacity, a
 *    bounded wait that ran out, lengths that differ from the plan's) never trap:
 *    the kernel skips the access, and records the first such code in a device
 *    status word that pkv_get_status reads.  pkv_last_error() returns a
 *    thread-local message for the last failing call.
 */
#ifndef PKV_H_
#define PKV_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  PKV_OK = 0,
  PKV_ERR_INVALID_ARG = 1,          /* bad pointer, shape, stride or length      */
  PKV_ERR_UNSUPPORTED = 2,          /* valid but outside the supported set        */
  PKV_ERR_WORKSPACE_TOO_SMALL = 3,  /* workspace smaller than the plan requires  */
  PKV_ERR_CUDA = 4,                 /* a CUDA runtime/driver call failed          */
  PKV_ERR_DEVICE_TIMEOUT = 5,       /* device: a bounded wait gave up             */
  PKV_ERR_DEVICE_BOUNDS = 6,        /* device: block_table entry / slot out of range */
  PKV_ERR_PLAN_MISMATCH = 7         /* device: cache_seqlens differ from the plan */
} pkv_status;

typedef enum { PKV_BF16 = 0, PKV_FP8_E4M3 = 1 } pkv_dtype;

/* Problem shape shared by the plan, the append and the attention call. */
typedef struct {
  int32_t batch;          /* number of sequences B                                   */
  int32_t num_heads_q;    /* Hq                                                      */
  int32_t num_heads_kv;   /* Hkv; Hq % Hkv == 0 (MQA: Hkv = 1)                       */
  int32_t head_dim;       /* D: 64, 128 or 256, either cache dtype                   */
  int32_t page_size;      /* 0 = contiguous cache; else 1, 2, 4 or a multiple of 8,
                             <= 256 (pages under 8 tokens are gathered row by row) */
  int32_t cache_capacity; /* tokens one sequence can hold: contiguous seqlen_cache,
                             paged max_pages_per_seq * page_size                     */
  int32_t num_pages;      /* paged: pages in the pool; contiguous: batch_size_cache  */
  int32_t cache_dtype;    /* pkv_dtype                                               */
  int32_t causal;         /* 0 / 1                                                   */
  float softmax_scale;    /* e.g. 1/sqrt(D)                                          */
} pkv_problem;

/* Device tensors of one call. */
typedef struct {
  const void* q;                 /* (total_q, Hq, D) bf16                            */
  int64_t q_stride_tok, q_stride_head;
  void* out;                     /* (total_q, Hq, D) bf16, written                   */
  int64_t o_stride_tok, o_stride_head;
  float* lse;                    /* nullable; (Hq, q_rows) fp32 natural-log LSE      */
  const int32_t* cu_seqlens_q;   /* [B+1] query row offsets: sequence b's Lq[b] query
                                    (and output) rows start at row cu_seqlens_q[b],
                                    Lq[b] being the plan's query length.  With q_rows
                                    = 0 the rows are packed (the prefix sums of the
                                    plan's lengths, which cu_seqlens_q must hold).
                                    With q_rows > 0 any start offsets (gaps, any
                                    order: the non-contiguous Q/O layout of the
                                    flashinfer PR "Uniform PoDAttention API", Key
                                    Changes 1, q_indptr with q_lenptr) are read on
                                    the device.                                      */
  int32_t max_seqlen_q;          /* upper bound of the query lengths                 */
  const void* k_new;             /* nullable; (total_new, Hkv, D) bf16               */
  const void* v_new;             /* nullable iff k_new is                            */
  int64_t knew_stride_tok, knew_stride_head;
  const int32_t* cu_seqlens_knew;/* [B+1]; required iff k_new is given               */
  void* k_cache;                 /* paged (pages, P, Hkv, D) | contiguous (Bc, S, Hkv, D) */
  void* v_cache;                 /* same shape and strides as k_cache                */
  int64_t kc_stride_page;        /* paged: elements between pages; contiguous: between
                                    batch rows                                       */
  int64_t kc_stride_tok, kc_stride_head;
  const int32_t* cache_seqlens;  /* [B] cache length BEFORE this call's append       */
  const int32_t* block_table;    /* [B, block_table_stride]; NULL for contiguous     */
  int32_t block_table_stride;
  const float* k_scale;          /* fp8 cache only: device fp32 scalar               */
  const float* v_scale;          /* fp8 cache only: device fp32 scalar               */
  const int32_t* page_indptr;    /* nullable.  Ragged page list (the kv_indptr /
                                    kv_indices form of the cutlass-sycl and flashinfer
                                    pages): sequence b's pages are block_table[
                                    page_indptr[b] + i], i < page_indptr[b+1] -
                                    page_indptr[b]; block_table_stride is ignored.  */
  const float* q_scale;          /* nullable; fp8 cache only.  Q is quantised to e4m3
                                    with this per-tensor scale (the cache's encode:
                                    code = e4m3_rn_satfinite(q * fp32(1/scale))) and
                                    Q.K^T runs on fp8 tensor cores, as for the fp8
                                    "QKV" models of the vLLM PR "[Kernel][Triton][FP8]
                                    ..." (feature list, lm-eval notes); P.V stays f16.
                                    Decode tiles use warp-level e4m3 MMAs, prefill
                                    tiles tcgen05 kind::f8f6f4 on the raw cache tile.
                                    A bf16 cache returns PKV_ERR_UNSUPPORTED.        */
  int32_t q_rows;                /* 0: packed rows (the plan's total query count);
                                    > 0: rows placed by cu_seqlens_q, and the row
                                    count of q, out and lse (>= every cu_seqlens_q[b]
                                    + Lq[b]).                                        */
} pkv_fwd_args;

typedef struct pkv_plan_s* pkv_plan_t;

/* Plan statistics (tests and benchmarks). */
typedef struct {
  int32_t num_items;         /* CTA work items (tiles)                      */
  int32_t num_decode_items;  /* of which decode tiles                       */
  int32_t num_prefill_items; /* of which prefill tiles                      */
  int32_t num_split_units;   /* decode units cut into several KV chunks     */
  int32_t num_ctas;          /* persistent grid size                        */
  int32_t total_q;           /* sum of query lengths                        */
  int32_t total_new;         /* sum of appended tokens                      */
  int32_t max_items_per_cta;
  double max_cta_cost;       /* LPT makespan, model units                   */
  double mean_cta_cost;
  int64_t upload_bytes;      /* bytes pkv_plan_upload copies to the device  */
  int64_t workspace_bytes;   /* device workspace the plan needs             */
} pkv_plan_stats;

/*
 * pkv_plan -- host scheduling step (flashinfer PR "Uniform PoDAttention API",
 * Key Changes 2: partition by KV-cache load; Limitations: classifier on the
 * query length).  Validates the shape, classifies every (sequence, kv head)
 * as decode work (Lq*G <= 16 rows: warp-MMA tiles) or tensor-core work
 * (tiles of 128 rows = 128/G query tokens x the G heads of the group; a group
 * of more than 128 heads is cut into sub-groups of 128, so any G >= 1 is
 * served), cuts long units whose queries fit one tile (decode steps, short
 * query runs) into KV chunks (split-KV, flash-attention PR, Limitation), and
 * assigns all tiles to persistent CTAs longest first: num_sms of them (the
 * GPU's SM count), or 2 * num_sms for a plan of decode tiles only over an fp8
 * cache at head_dim <= 128 or a bf16 cache at head_dim 64, whose kernel runs
 * two CTAs an SM (the plan's stats report the count).
 * h_q_lens / h_cache_lens / h_new_lens: host int32 [B]; h_new_lens may be NULL
 * when the call appends nothing.  Zero lengths are accepted.  On success
 * *out_plan owns a host work list and *out_workspace_bytes is the device
 * workspace size that pkv_plan_upload and pkv_attn_varlen_kvcache_fwd need.
 * Pure host code: no CUDA call.
 */
pkv_status pkv_plan(const pkv_problem* problem, const int32_t* h_q_lens,
                    const int32_t* h_cache_lens, const int32_t* h_new_lens,
                    int32_t num_sms, pkv_plan_t* out_plan, size_t* out_workspace_bytes);

/*
 * pkv_plan_decode_dynamic -- a plan for decode steps whose cache lengths are
 * read on the device at every call, so that a serving loop can capture
 * pkv_attn_varlen_kvcache_fwd once in a CUDA graph and replay it while
 * cache_seqlens grows (flashinfer PR "[Refactor] Uniform PoDAttention API ...",
 * Limitations: a host plan per step keeps the scheduler out of CUDA graphs;
 * TransformerEngine PR "Add KV cache for paged/non-paged attention": its
 * backends support graphs).  h_max_cache_lens[b] bounds cache_seqlens[b] of
 * every call made with the plan; q lengths and new-token lengths are fixed by
 * it.  Work is split and scheduled for the bounds; at run time each work
 * item's key range is cut at the sequence's current key count (split-KV
 * chunks past it contribute nothing).  Every request's queries must fit one
 * tile (q_len * Hq/Hkv <= 16, or q_len <= 128 / min(Hq/Hkv, 128)), else
 * PKV_ERR_UNSUPPORTED.  A call whose
 * cache_seqlens[b] exceeds its bound records PKV_ERR_PLAN_MISMATCH in the
 * device status and attends at most the bound.  Pure host code.
 */
pkv_status pkv_plan_decode_dynamic(const pkv_problem* problem, const int32_t* h_q_lens,
                                   const int32_t* h_max_cache_lens, const int32_t* h_new_lens,
                                   int32_t num_sms, pkv_plan_t* out_plan, size_t* out_workspace_bytes);

/* Copies the plan's work list into the caller's device workspace on `stream`
 * (asynchronously; the host copy stays valid until pkv_plan_destroy) and clears
 * the device status word.  Must precede pkv_attn_varlen_kvcache_fwd with this
 * workspace. */
pkv_status pkv_plan_upload(pkv_plan_t plan, void* workspace, size_t workspace_bytes,
                           void* stream);

/* Statistics of a plan (host only). */
pkv_status pkv_plan_get_stats(pkv_plan_t plan, pkv_plan_stats* stats);

/* One scheduled tile as the plan made it (diagnostics and tests).  Rows of a
 * tile are (query token, head of the tile's heads) pairs, row = token *
 * num_heads + g, query head = kv_head * G + head0 + g. */
typedef struct {
  int32_t seq;          /* sequence b                                        */
  int32_t kv_head;      /* kv head                                           */
  int32_t q_row0;       /* packed-q index of the first query token           */
  int32_t q_index0;     /* index of that token within the sequence           */
  int32_t n_q;          /* query tokens in the tile                          */
  int32_t q_len;        /* Lq of the sequence                                */
  int32_t kv_len;       /* Lk = cache_len + new_len                          */
  int32_t kv_begin;     /* keys [kv_begin, kv_end) handled by this tile      */
  int32_t kv_end;
  int32_t kind;         /* 0 decode tile, 1 prefill tile                     */
  int32_t partial_slot; /* -1: writes the output; else its first split-KV
                           partial slot (16 rows per slot)                   */
  int32_t cta;          /* persistent CTA that runs it                       */
  int32_t head0;        /* first query head of the group in the tile         */
  int32_t num_heads;    /* query heads of the group in the tile              */
  double cost;          /* the plan's cost model of the tile (model units): the
                           longest-first assignment sorts and balances by it */
} pkv_work_item;

/* Copies up to `capacity` tiles, in CTA order, into h_items (host memory);
 * *count receives the number of tiles in the plan. */
pkv_status pkv_plan_get_items(pkv_plan_t plan, pkv_work_item* h_items, int32_t capacity, int32_t* count);

/*
 * pkv_attn_varlen_kvcache_fwd -- the whole call (flash-attention PR "Add
 * flash_attn_varlen_func_with_kvcache", Usage): if args->k_new is given, the
 * new tokens are first written into the cache at positions cache_seqlens[b] ..
 * cache_seqlens[b] + new_len[b] - 1 (as pkv_kv_append), then every query
 * attends the first cache_seqlens[b] + new_len[b] keys of its sequence.
 * cache_seqlens itself is NOT advanced (the caller does that).  Launches the
 * append (if any), one persistent attention kernel and, when a unit was
 * split, one combine kernel; no host synchronisation and no allocation.
 * The plan must have been made from the same lengths and uploaded into
 * `workspace`.
 */
pkv_status pkv_attn_varlen_kvcache_fwd(const pkv_problem* problem, const pkv_fwd_args* args,
                                       pkv_plan_t plan, void* workspace,
                                       size_t workspace_bytes, void* stream);

/*
 * pkv_attn_varlen_kvcache_fwd_noalloc -- the same call as
 * pkv_attn_varlen_kvcache_fwd for callers that cannot provide a device
 * workspace: hosts whose device memory is owned by their own pool and may not
 * be allocated from, latency-critical loops that must not call cudaMalloc
 * (it synchronises the device), or bindings without an allocator.  (The pages
 * have no counterpart; this is an interface convenience of this library.)
 * The work list, split-KV partials and status word live in a fixed 32 MiB
 * device array that every GPU loading the library reserves until the process
 * exits; the entry point allocates nothing and frees nothing.  It uploads the
 * plan into that array and then runs the call on `stream`.
 *  - The first call on a device resolves the array's device address
 *    (cudaGetSymbolAddress, checked) with that device current, once.
 *  - A plan needing more than 32 MiB of workspace is rejected with
 *    PKV_ERR_WORKSPACE_TOO_SMALL before anything is launched.
 *  - Every host-side check (problem, plan, cache, q / out, new tokens, size)
 *    runs before the array is touched: a rejected call copies nothing.
 *  - Every call on a device shares the one array: calls that overlap on the
 *    GPU (other streams, other host threads) race and must be serialised by
 *    the caller.  Each call rewrites what it reads, including the status word,
 *    which it clears; pkv_get_status_noalloc reads it.
 */
pkv_status pkv_attn_varlen_kvcache_fwd_noalloc(const pkv_problem* problem, const pkv_fwd_args* args,
                                               pkv_plan_t plan, void* stream);

/*
 * pkv_get_status_noalloc -- pkv_get_status for the calls above: synchronises
 * `stream`, reads the device status word that the last
 * pkv_attn_varlen_kvcache_fwd_noalloc on the current device left in the fixed
 * array into *device_status (a pkv_status; a bad block_table entry gives
 * PKV_ERR_DEVICE_BOUNDS, a length past a dynamic plan's bound
 * PKV_ERR_PLAN_MISMATCH) and resets it to PKV_OK.  Allocates nothing.  (No
 * counterpart on the pages, like the entry point it reads for.)
 */
pkv_status pkv_get_status_noalloc(void* stream, int32_t* device_status);

/*
 * pkv_kv_append -- in-place append alone (flash-attention PR, Usage: "kv cache
 * will be updated in-place"; TE PR: paged / non-paged bshd caches).  Writes
 * token t of sequence b (t < new_len[b], new_len from cu_seqlens_knew) to
 * logical position cache_seqlens[b] + t: page block_table[b][pos / P], slot
 * pos % P (or row pos of batch b for a contiguous cache).  bf16 caches get the
 * bits unchanged; fp8 caches get e4m3_rn_satfinite(fp32(x) * fp32(1/scale)),
 * bit-exact.  total_new = sum of new lengths (host int).  device_status:
 * nullable device int32 that receives the first device error code.
 */
pkv_status pkv_kv_append(const pkv_problem* problem, const pkv_fwd_args* args,
                         int32_t total_new, int32_t* device_status, void* stream);

/* Synchronises `stream`, reads the device status word of `workspace` into
 * *device_status (a pkv_status) and resets it to PKV_OK. */
pkv_status pkv_get_status(void* workspace, void* stream, int32_t* device_status);

void pkv_plan_destroy(pkv_plan_t plan);

/* Thread-local message describing the last failing call ("" if none). */
const char* pkv_last_error(void);

/* Timing hook for benchmarks: when start/stop are non-NULL (cudaEvent_t
 * passed as void*), every later pkv_attn_varlen_kvcache_fwd on this host
 * thread records `start` immediately before and `stop` immediately after the
 * persistent attention kernel, on the call's stream.  NULL, NULL turns it off.
 * A call captured into a CUDA graph records them as event-record nodes, so each
 * replay of the graph re-records them.  The events stay owned by the caller. */
pkv_status pkv_set_profile_events(void* start_event, void* stop_event);

/* Library version string. */
const char* pkv_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PKV_H_ */
