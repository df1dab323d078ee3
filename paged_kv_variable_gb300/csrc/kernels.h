// Kernel parameter blocks and launchers (internal).
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace pkv {

struct AppendParams {
  const __nv_bfloat16* k_new;
  const __nv_bfloat16* v_new;
  int64_t n_stride_tok, n_stride_head;
  const int32_t* cu_knew;
  const int32_t* cache_seqlens;
  void* k_cache;
  void* v_cache;
  int64_t c_stride_page, c_stride_tok, c_stride_head;
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* page_indptr;  // nullable: ragged page list offsets
  int32_t page_size;
  int32_t num_pages;
  int32_t capacity;
  int32_t batch;
  int32_t hkv;
  int32_t total_new;
  const float* k_scale;
  const float* v_scale;
  int* status;
};

struct CombineParams {
  const CombineItem* items;
  const int32_t* q_offsets;  // nullable: query row offsets of the sequences (rows placed by the caller)
  const float* partial_o;
  const float* partial_lse;
  __nv_bfloat16* out;
  int64_t o_stride_tok, o_stride_head;
  float* lse;
  int32_t total_q;
  int32_t G;
};

struct AttnParams {
  const __nv_bfloat16* q;
  int64_t q_stride_tok, q_stride_head;
  __nv_bfloat16* out;
  int64_t o_stride_tok, o_stride_head;
  int32_t out_v8;      // every output row starts on 32 bytes: prefill rows are written 32 bytes per store
  float* lse;
  int32_t total_q;     // rows of q / out / lse
  const int32_t* q_offsets;  // nullable: query row offsets of the sequences (rows placed by the caller)
  const int32_t* block_table;
  int32_t bt_stride;
  const int32_t* page_indptr;  // nullable: ragged page list offsets
  int32_t page_size;   // 0 = contiguous
  int32_t box_rows;    // cache rows per TMA box (divides 128 and the page size)
  int32_t row_gather;  // pages of 1, 2 or 4 tokens: rows gathered with cp.async instead of TMA boxes
  const void* kc;      // caches and their element strides (row gather)
  const void* vc;
  int64_t c_stride_page, c_stride_tok, c_stride_head;
  int32_t num_pages;   // page pool size (contiguous: batch rows of the cache)
  int32_t G;
  int32_t causal;
  float scale_log2;    // softmax_scale * log2(e)
  const float* k_scale;
  const float* v_scale;
  const float* q_scale;  // nullable (fp8 cache, decode tiles): Q quantised to e4m3 for Q K^T
  const WorkItem* items;
  const int32_t* cta_begin;
  float* partial_o;
  float* partial_lse;
  int* status;
  const int32_t* cache_seqlens;
  const int32_t* plan_lc;
  int32_t batch;
  int32_t dynamic;     // plan_lc holds bounds; the cache lengths come from cache_seqlens
};

// Start of sequence b's page list, and how many pages it has (-1: unchecked).
__device__ __forceinline__ const int32_t* seq_pages(const int32_t* bt, int32_t stride, const int32_t* indptr, int b,
                                                    int* count) {
  if (indptr != nullptr) {
    const int a = __ldg(indptr + b);
    *count = __ldg(indptr + b + 1) - a;
    return bt + a;
  }
  *count = -1;
  return bt + (int64_t)b * stride;
}

cudaError_t launch_kv_append(const AppendParams& p, int head_dim, bool fp8, cudaStream_t stream);
// overlap_prev: launch with programmatic stream serialization, so that the
// kernel's start overlaps the end of the kernel issued just before it on the
// stream (the append kernel for the attention, the attention for the combine);
// the kernel waits for that one before reading what it wrote.
cudaError_t launch_combine(const CombineParams& p, int num_items, int head_dim, bool overlap_prev,
                           cudaStream_t stream);
cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const CUtensorMap& tm_q, int num_ctas, int head_dim, bool fp8, bool has_prefill,
                             bool has_decode, bool overlap_prev, cudaStream_t stream);

}  // namespace pkv
