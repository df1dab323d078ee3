// KV append scatter and split-KV combine kernels.
//
// Append: flash-attention PR "Add flash_attn_varlen_func_with_kvcache", Usage
// ("kv cache will be updated in-place"; new k/v packed with cu_seqlens_k) and
// Minor Changes (cache lengths kept apart from cu_seqlens_knew);
// TransformerEngine PR "Add KV cache for paged/non-paged attention" (paged and
// non-paged bshd caches, one page table for K and V); vLLM PR "[Kernel][Triton]
// [FP8] ..." (8-bit KV cache).
//
// Combine: merge of the normalised partial outputs of KV chunks of one decode
// unit by their log-sum-exp (the split-KV decode named in the flash-attention
// PR's Limitation and review).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace pkv {

constexpr int kCombineThreads = 256;

// One warp per (new token, kv head) row; lane l moves elements [l*E, l*E+E).
template <int D, bool FP8>
__global__ void __launch_bounds__(256) kv_append_kernel(const AppendParams p) {
  constexpr int E = D / 32;  // elements per lane: 8 (D=256), 4 (D=128) or 2 (D=64)
  grid_dep_launch();         // the attention kernel may start; it waits before reading appended rows
  const int64_t row = ((int64_t)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const int lane = threadIdx.x & 31;
  if (row >= (int64_t)p.total_new * p.hkv) return;
  const int t = (int)(row / p.hkv);
  const int h = (int)(row % p.hkv);
  // sequence of token t: the largest b with cu_knew[b] <= t
  int lo = 0, hi = p.batch;
  while (hi - lo > 1) {
    int mid = (lo + hi) >> 1;
    if (__ldg(p.cu_knew + mid) <= t) lo = mid; else hi = mid;
  }
  const int b = lo;
  const int pos = __ldg(p.cache_seqlens + b) + (t - __ldg(p.cu_knew + b));
  if (pos < 0 || pos >= p.capacity) {
    if (lane == 0) record_status(p.status, PKV_ERR_DEVICE_BOUNDS, b, pos);
    return;
  }
  int64_t dst;
  if (p.page_size > 0) {
    int npages;
    const int32_t* pages = seq_pages(p.block_table, p.bt_stride, p.page_indptr, b, &npages);
    const int pi = pos / p.page_size;
    const int page = (npages >= 0 && pi >= npages) ? -1 : __ldg(pages + pi);
    if (page < 0 || page >= p.num_pages) {
      if (lane == 0) record_status(p.status, PKV_ERR_DEVICE_BOUNDS, b, page);
      return;
    }
    dst = (int64_t)page * p.c_stride_page + (int64_t)(pos % p.page_size) * p.c_stride_tok;
  } else {
    dst = (int64_t)b * p.c_stride_page + (int64_t)pos * p.c_stride_tok;
  }
  dst += (int64_t)h * p.c_stride_head + lane * E;
  const int64_t src = (int64_t)t * p.n_stride_tok + (int64_t)h * p.n_stride_head + lane * E;
  const __nv_bfloat16* kin = p.k_new + src;
  const __nv_bfloat16* vin = p.v_new + src;
  if constexpr (!FP8) {
    __nv_bfloat16* kc = reinterpret_cast<__nv_bfloat16*>(p.k_cache) + dst;
    __nv_bfloat16* vc = reinterpret_cast<__nv_bfloat16*>(p.v_cache) + dst;
    if constexpr (E == 8) {
      *reinterpret_cast<uint4*>(kc) = __ldg(reinterpret_cast<const uint4*>(kin));
      *reinterpret_cast<uint4*>(vc) = __ldg(reinterpret_cast<const uint4*>(vin));
    } else if constexpr (E == 4) {
      *reinterpret_cast<uint2*>(kc) = __ldg(reinterpret_cast<const uint2*>(kin));
      *reinterpret_cast<uint2*>(vc) = __ldg(reinterpret_cast<const uint2*>(vin));
    } else {
      *reinterpret_cast<uint32_t*>(kc) = __ldg(reinterpret_cast<const uint32_t*>(kin));
      *reinterpret_cast<uint32_t*>(vc) = __ldg(reinterpret_cast<const uint32_t*>(vin));
    }
  } else {
    // one IEEE reciprocal per call, then an RN multiply per element (no FMA)
    const float inv_k = __frcp_rn(__ldg(p.k_scale));
    const float inv_v = __frcp_rn(__ldg(p.v_scale));
    auto lo_f = [](uint32_t w) { return __uint_as_float(w << 16); };
    auto hi_f = [](uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); };
    auto enc2 = [&](uint32_t w, float inv) -> uint32_t {
      return f32x2_to_e4m3x2(__fmul_rn(lo_f(w), inv), __fmul_rn(hi_f(w), inv));
    };
    uint8_t* kc = reinterpret_cast<uint8_t*>(p.k_cache) + dst;
    uint8_t* vc = reinterpret_cast<uint8_t*>(p.v_cache) + dst;
    if constexpr (E == 8) {
      const uint4 kr = __ldg(reinterpret_cast<const uint4*>(kin));
      const uint4 vr = __ldg(reinterpret_cast<const uint4*>(vin));
      *reinterpret_cast<uint2*>(kc) = make_uint2(enc2(kr.x, inv_k) | (enc2(kr.y, inv_k) << 16),
                                                 enc2(kr.z, inv_k) | (enc2(kr.w, inv_k) << 16));
      *reinterpret_cast<uint2*>(vc) = make_uint2(enc2(vr.x, inv_v) | (enc2(vr.y, inv_v) << 16),
                                                 enc2(vr.z, inv_v) | (enc2(vr.w, inv_v) << 16));
    } else if constexpr (E == 4) {
      const uint2 kr = __ldg(reinterpret_cast<const uint2*>(kin));
      const uint2 vr = __ldg(reinterpret_cast<const uint2*>(vin));
      *reinterpret_cast<uint32_t*>(kc) = enc2(kr.x, inv_k) | (enc2(kr.y, inv_k) << 16);
      *reinterpret_cast<uint32_t*>(vc) = enc2(vr.x, inv_v) | (enc2(vr.y, inv_v) << 16);
    } else {
      // D = 64: two elements a lane, one 2-byte store each
      *reinterpret_cast<uint16_t*>(kc) = (uint16_t)enc2(__ldg(reinterpret_cast<const uint32_t*>(kin)), inv_k);
      *reinterpret_cast<uint16_t*>(vc) = (uint16_t)enc2(__ldg(reinterpret_cast<const uint32_t*>(vin)), inv_v);
    }
  }
}

// One block per split unit; a thread owns 8 consecutive columns of a row and
// walks the unit's rows (up to 128: a tensor-core tile of a wide head group).
// Partials are normalised outputs with log2-domain LSEs; chunk s of the unit
// wrote slot0 + s * slot_stride; the merge order over chunks is fixed
// (deterministic).
template <int D>
__global__ void __launch_bounds__(kCombineThreads) combine_kernel(const CombineParams p) {
  const CombineItem ci = p.items[blockIdx.x];
  constexpr int kPerRow = D / 8;
  const int d0 = (threadIdx.x % kPerRow) * 8;
  const int rows = ci.n_q * ci.nh;
  grid_dep_wait();  // the partials come from the attention kernel launched just before
  constexpr float kLn2 = 0.693147180559945309f;
  const int64_t chunk_rows = (int64_t)ci.slot_stride * kDecodeRows;
  for (int row = threadIdx.x / kPerRow; row < rows; row += kCombineThreads / kPerRow) {
    const float* lse = p.partial_lse + (int64_t)ci.slot0 * kDecodeRows + row;
    float m = -INFINITY;
    for (int s = 0; s < ci.nsplit; ++s) m = fmaxf(m, __ldg(lse + s * chunk_rows));
    const float m_use = m == -INFINITY ? 0.f : m;
    float wsum = 0.f;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    const float* po = p.partial_o + ((int64_t)ci.slot0 * kDecodeRows + row) * D + d0;
    for (int s = 0; s < ci.nsplit; ++s) {
      const float w = ex2(__ldg(lse + s * chunk_rows) - m_use);
      const float4 a = __ldg(reinterpret_cast<const float4*>(po + s * chunk_rows * D));
      const float4 b = __ldg(reinterpret_cast<const float4*>(po + s * chunk_rows * D + 4));
      wsum += w;
      acc[0] += w * a.x; acc[1] += w * a.y; acc[2] += w * a.z; acc[3] += w * a.w;
      acc[4] += w * b.x; acc[5] += w * b.y; acc[6] += w * b.z; acc[7] += w * b.w;
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    const int tok = (p.q_offsets != nullptr ? __ldg(p.q_offsets + ci.b) : ci.q_row0) + row / ci.nh;
    const int head = ci.hk * p.G + ci.h0 + row % ci.nh;
    uint4 v;
    v.x = pack_bf16(acc[0] * inv, acc[1] * inv);
    v.y = pack_bf16(acc[2] * inv, acc[3] * inv);
    v.z = pack_bf16(acc[4] * inv, acc[5] * inv);
    v.w = pack_bf16(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4*>(p.out + (int64_t)tok * p.o_stride_tok + (int64_t)head * p.o_stride_head + d0) = v;
    if (p.lse != nullptr && d0 == 0)
      p.lse[(int64_t)head * p.total_q + tok] = wsum > 0.f ? (m_use + __log2f(wsum)) * kLn2 : -INFINITY;
  }
}

cudaError_t launch_kv_append(const AppendParams& p, int head_dim, bool fp8, cudaStream_t stream) {
  const int64_t rows = (int64_t)p.total_new * p.hkv;
  if (rows == 0) return cudaSuccess;
  const int threads = 256;
  const int64_t blocks = (rows * 32 + threads - 1) / threads;
  if (blocks > INT32_MAX) return cudaErrorInvalidValue;
  if (fp8 && head_dim == 256) {
    kv_append_kernel<256, true><<<(unsigned)blocks, threads, 0, stream>>>(p);
  } else if (fp8 && head_dim == 128) {
    kv_append_kernel<128, true><<<(unsigned)blocks, threads, 0, stream>>>(p);
  } else if (fp8) {
    kv_append_kernel<64, true><<<(unsigned)blocks, threads, 0, stream>>>(p);
  } else if (head_dim == 256) {
    kv_append_kernel<256, false><<<(unsigned)blocks, threads, 0, stream>>>(p);
  } else if (head_dim == 128) {
    kv_append_kernel<128, false><<<(unsigned)blocks, threads, 0, stream>>>(p);
  } else {
    kv_append_kernel<64, false><<<(unsigned)blocks, threads, 0, stream>>>(p);
  }
  return cudaGetLastError();
}

cudaError_t launch_combine(const CombineParams& p, int num_items, int head_dim, bool overlap_prev,
                           cudaStream_t stream) {
  if (num_items == 0) return cudaSuccess;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3((unsigned)num_items);
  cfg.blockDim = dim3((unsigned)kCombineThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = overlap_prev ? 1 : 0;
  return head_dim == 256   ? cudaLaunchKernelEx(&cfg, combine_kernel<256>, p)
         : head_dim == 128 ? cudaLaunchKernelEx(&cfg, combine_kernel<128>, p)
                           : cudaLaunchKernelEx(&cfg, combine_kernel<64>, p);
}

}  // namespace pkv
