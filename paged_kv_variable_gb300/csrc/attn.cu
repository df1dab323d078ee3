// Persistent attention kernel over a paged or contiguous KV cache.
//
// One CTA per SM walks its host-assigned list of work items (flashinfer PR
// "[Refactor] Uniform PoDAttention API with Horizontal Fusion SMs Schedule",
// Key Changes 2: prefill and decode work share one persistent launch).  Warp 0
// gathers K/V tiles of 128 keys with TMA: one 16-row box per (page, 128-byte
// column chunk), page numbers read from block_table (vLLM PR "[Kernel][Triton]
// [FP8] ...", review: block_table support; TransformerEngine PR "Add KV cache
// for paged/non-paged attention": one table for K and V, bshd pages), into a
// ring of shared-memory stages guarded by mbarriers (the prefetch of cached KV
// of the cutlass-sycl PR "Extend FlashAttention Prefill with KV cache").
// Warps 1..4 compute S = Q K^T, the masked online softmax and O += P V on the
// tensor cores and write either the final output or a split-KV partial.
//
// Tile kinds:
//   decode  -- up to 16 rows (query tokens x group heads); the 4 warps split
//              the 128 keys of each tile and merge at the end of the item.
//   prefill -- 64 rows; each warp owns 16 rows and all 128 keys of a tile.
// fp8 caches (vLLM PR, 8-bit KV cache) are converted to bf16 in shared memory
// (exact), with k_scale folded into the logit scale and v_scale applied to the
// normalised output.
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"

namespace pkv {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (1 + kConsumerWarps);
constexpr float kLn2 = 0.693147180559945309f;

template <int D, bool FP8>
struct Layout {
  static constexpr int kEsize = FP8 ? 1 : 2;
  static constexpr int kStages = 3;
  static constexpr int kTileBytes = kKvTile * D * kEsize;   // one raw K (or V) tile
  static constexpr int kChunks = D * kEsize / 128;            // 128-byte column chunks per cache row
  static constexpr int kBf16Tile = kKvTile * D * 2;
  static constexpr int kStageOff = 0;                         // [stage][K, V]
  static constexpr int kDeqOff = kStages * 2 * kTileBytes;    // fp8: bf16 copies of K and V
  static constexpr int kMergeOff = kDeqOff + (FP8 ? 2 * kBf16Tile : 0);
  static constexpr int kMergeBytes = kConsumerWarps * kDecodeRows * D * 4;
  static constexpr int kMlOff = kMergeOff + kMergeBytes;      // float[4][16][2]: (m, l)
  static constexpr int kBarOff = kMlOff + kConsumerWarps * kDecodeRows * 2 * 4;
  static constexpr int kAbortOff = kBarOff + 3 * kStages * 8;
  static constexpr int kBytes = kAbortOff + 16;
  static constexpr int kAlloc = kBytes + 1024;                // room to align the base to 1024
};

// Byte offset of 16-byte chunk c of row r in a bf16 tile stored as
// [D/64 column chunks][128 rows][128 B] with the 128-byte TMA swizzle.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * (kKvTile * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

// fp8 K or V tile (128 rows x 128 codes, swizzled) -> bf16 tile in the layout above.
__device__ __forceinline__ void dequant_tile(const uint8_t* raw, uint8_t* dst, int ctid) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int u = ctid + 128 * k;
    const int r = u >> 3, c = u & 7;
    const uint4 w = *reinterpret_cast<const uint4*>(raw + r * 128 + (((c ^ (r & 7))) << 4));
    uint4 lo, hi;
    lo.x = e4m3x2_to_bf16x2((uint16_t)(w.x & 0xFFFF));
    lo.y = e4m3x2_to_bf16x2((uint16_t)(w.x >> 16));
    lo.z = e4m3x2_to_bf16x2((uint16_t)(w.y & 0xFFFF));
    lo.w = e4m3x2_to_bf16x2((uint16_t)(w.y >> 16));
    hi.x = e4m3x2_to_bf16x2((uint16_t)(w.z & 0xFFFF));
    hi.y = e4m3x2_to_bf16x2((uint16_t)(w.z >> 16));
    hi.z = e4m3x2_to_bf16x2((uint16_t)(w.w & 0xFFFF));
    hi.w = e4m3x2_to_bf16x2((uint16_t)(w.w >> 16));
    *reinterpret_cast<uint4*>(dst + tile_off(r, 2 * c)) = lo;
    *reinterpret_cast<uint4*>(dst + tile_off(r, 2 * c + 1)) = hi;
  }
}

struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  template <int NS>
  __device__ __forceinline__ void advance() {
    if (++stage == NS) {
      stage = 0;
      phase ^= 1;
    }
  }
};

// ------------------------------------------------------------------ producer
template <int D, bool FP8>
__device__ void producer(const AttnParams& p, const CUtensorMap* tm_k, const CUtensorMap* tm_v, uint8_t* smem,
                         uint64_t* full_k, uint64_t* full_v, uint64_t* empty, volatile int* abort_flag, int it0,
                         int it1) {
  using L = Layout<D, FP8>;
  tma_prefetch_desc(tm_k);
  tma_prefetch_desc(tm_v);
  Ring ring;
  int issued = 0;
  bool ok = true;
  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = p.items[it];
    const int32_t* bt = p.block_table + (int64_t)w.b * p.bt_stride;
    for (int t0 = w.kv_begin; t0 < w.kv_end; t0 += kKvTile) {
      if (!mbar_wait(&empty[ring.stage], ring.phase ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      uint8_t* kdst = smem + L::kStageOff + ring.stage * 2 * L::kTileBytes;
      uint8_t* vdst = kdst + L::kTileBytes;
      mbar_arrive_expect_tx(&full_k[ring.stage], L::kTileBytes);
      mbar_arrive_expect_tx(&full_v[ring.stage], L::kTileBytes);
#pragma unroll 1
      for (int g = 0; g < kKvTile / kBoxRows; ++g) {
        const int j0 = t0 + g * kBoxRows;
        int page = p.num_pages, slot = 0;  // out of range: the copy fills zeros
        if (j0 < w.kv_end) {
          if (p.page_size > 0) {
            page = __ldg(bt + j0 / p.page_size);
            slot = j0 % p.page_size;
            if (page < 0 || page >= p.num_pages) {
              record_status(p.status, PKV_ERR_DEVICE_BOUNDS, w.b, page);
              page = p.num_pages;
              slot = 0;
            }
          } else {
            page = w.b;
            slot = j0;
          }
        }
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          const int off = c * (kKvTile * 128) + g * (kBoxRows * 128);
          tma_load_4d(kdst + off, tm_k, &full_k[ring.stage], c * (128 / L::kEsize), w.hk, slot, page);
          tma_load_4d(vdst + off, tm_v, &full_v[ring.stage], c * (128 / L::kEsize), w.hk, slot, page);
        }
      }
      ++issued;
      ring.advance<L::kStages>();
    }
  }
  if (!ok) {
    record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, 0);
    *abort_flag = 1;
    // let the copies already issued land before the CTA can exit (bounded)
    int zero = 0;
    const int n = issued < L::kStages ? issued : L::kStages;
    for (int k = issued - n; k < issued; ++k) {
      const int s = k % L::kStages;
      const uint32_t ph = (uint32_t)((k / L::kStages) & 1);
      mbar_wait(&full_k[s], ph, &zero);
      mbar_wait(&full_v[s], ph, &zero);
    }
  }
}

// ------------------------------------------------------------------ consumers
// KPW = keys of each 128-key tile handled by one warp: 32 (decode), 128 (prefill).
template <int D, bool FP8, int KPW>
__device__ bool run_item(const AttnParams& p, const WorkItem& w, uint8_t* smem, uint64_t* full_k, uint64_t* full_v,
                         uint64_t* empty, volatile int* abort_flag, Ring& ring, float sl2, float vscale) {
  using L = Layout<D, FP8>;
  constexpr int NT = KPW / 8;       // S column tiles per warp
  constexpr int KS = D / 16;        // k-steps of Q K^T
  constexpr int NO = D / 8;         // O column tiles
  constexpr bool kDecodeTile = (KPW != kKvTile);
  const int lane = threadIdx.x & 31;
  const int cw = (threadIdx.x >> 5) - 1;  // consumer warp 0..3
  const int ctid = threadIdx.x - 32;
  const int g = lane >> 2, t = lane & 3;
  const int row_blk = kDecodeTile ? 0 : cw;
  const int kw0 = kDecodeTile ? cw * KPW : 0;
  const int R = w.n_q * p.G;
  const int r0 = row_blk * 16 + g, r1 = r0 + 8;

  auto limit_of = [&](int r) {
    if (r >= R) return w.kv_begin;
    int lim = w.kv_end;
    if (p.causal) lim = min(lim, w.q_i0 + r / p.G + w.lk - w.lq + 1);
    return lim;
  };
  const int lim0 = limit_of(r0), lim1 = limit_of(r1);

  // Q fragments (A operand of m16n8k16), rows r0 / r1
  uint32_t qa[KS][4];
  {
    const __nv_bfloat16* q0 = nullptr;
    const __nv_bfloat16* q1 = nullptr;
    if (r0 < R)
      q0 = p.q + (int64_t)(w.q_row0 + r0 / p.G) * p.q_stride_tok + (int64_t)(w.hk * p.G + r0 % p.G) * p.q_stride_head;
    if (r1 < R)
      q1 = p.q + (int64_t)(w.q_row0 + r1 / p.G) * p.q_stride_tok + (int64_t)(w.hk * p.G + r1 % p.G) * p.q_stride_head;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
      const int c = ks * 16 + 2 * t;
      qa[ks][0] = q0 ? ld_u32(q0 + c) : 0u;
      qa[ks][1] = q1 ? ld_u32(q1 + c) : 0u;
      qa[ks][2] = q0 ? ld_u32(q0 + c + 8) : 0u;
      qa[ks][3] = q1 ? ld_u32(q1 + c + 8) : 0u;
    }
  }

  float o[NO][4];
#pragma unroll
  for (int n = 0; n < NO; ++n) o[n][0] = o[n][1] = o[n][2] = o[n][3] = 0.f;
  float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

  for (int t0 = w.kv_begin; t0 < w.kv_end; t0 += kKvTile) {
    if (!mbar_wait(&full_k[ring.stage], ring.phase, abort_flag)) return false;
    uint8_t* stage_k = smem + L::kStageOff + ring.stage * 2 * L::kTileBytes;
    uint8_t* stage_v = stage_k + L::kTileBytes;
    uint32_t kb, vb;
    if constexpr (FP8) {
      uint8_t* dk = smem + L::kDeqOff;
      uint8_t* dv = dk + L::kBf16Tile;
      dequant_tile(stage_k, dk, ctid);
      if (!mbar_wait(&full_v[ring.stage], ring.phase, abort_flag)) return false;
      dequant_tile(stage_v, dv, ctid);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[ring.stage]);
      named_bar_sync(1, 32 * kConsumerWarps);
      kb = smem_u32(dk);
      vb = smem_u32(dv);
    } else {
      kb = smem_u32(stage_k);
      vb = smem_u32(stage_v);
    }

    // S = Q K^T over this warp's keys
    float s[NT][4];
#pragma unroll
    for (int n = 0; n < NT; ++n) s[n][0] = s[n][1] = s[n][2] = s[n][3] = 0.f;
#pragma unroll
    for (int ks = 0; ks < KS; ++ks) {
#pragma unroll
      for (int np = 0; np < NT / 2; ++np) {
        const int r = kw0 + np * 16 + (lane >> 4) * 8 + (lane & 7);
        const int c = 2 * ks + ((lane >> 3) & 1);
        uint32_t b0, b1, b2, b3;
        ldsm_x4(kb + tile_off(r, c), b0, b1, b2, b3);
        mma_bf16(s[2 * np], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
        mma_bf16(s[2 * np + 1], qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
      }
    }

    // mask (select, never add) + online softmax in the log2 domain
    const int jb = t0 + kw0 + 2 * t;
    float mx0 = -INFINITY, mx1 = -INFINITY;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
#pragma unroll
      for (int e = 0; e < 2; ++e) {
        const int j = jb + n * 8 + e;
        s[n][e] = j < lim0 ? s[n][e] * sl2 : -INFINITY;
        s[n][2 + e] = j < lim1 ? s[n][2 + e] * sl2 : -INFINITY;
        mx0 = fmaxf(mx0, s[n][e]);
        mx1 = fmaxf(mx1, s[n][2 + e]);
      }
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    const float mn0 = fmaxf(m0, mx0), mn1 = fmaxf(m1, mx1);
    const float mu0 = mn0 == -INFINITY ? 0.f : mn0;
    const float mu1 = mn1 == -INFINITY ? 0.f : mn1;
    const float al0 = ex2(m0 - mu0), al1 = ex2(m1 - mu1);
    m0 = mn0;
    m1 = mn1;
    float ls0 = 0.f, ls1 = 0.f;
#pragma unroll
    for (int n = 0; n < NT; ++n) {
      s[n][0] = ex2(s[n][0] - mu0);
      s[n][1] = ex2(s[n][1] - mu0);
      s[n][2] = ex2(s[n][2] - mu1);
      s[n][3] = ex2(s[n][3] - mu1);
      ls0 += s[n][0] + s[n][1];
      ls1 += s[n][2] + s[n][3];
    }
    l0 = l0 * al0 + ls0;
    l1 = l1 * al1 + ls1;
#pragma unroll
    for (int n = 0; n < NO; ++n) {
      o[n][0] *= al0;
      o[n][1] *= al0;
      o[n][2] *= al1;
      o[n][3] *= al1;
    }

    // O += P V
    if constexpr (!FP8) {
      if (!mbar_wait(&full_v[ring.stage], ring.phase, abort_flag)) return false;
    }
    const bool vmask = t0 + kKvTile > w.lk;  // rows past the sequence may hold anything: zero them
#pragma unroll
    for (int kk = 0; kk < KPW / 16; ++kk) {
      const uint32_t a0 = pack_bf16(s[2 * kk][0], s[2 * kk][1]);
      const uint32_t a1 = pack_bf16(s[2 * kk][2], s[2 * kk][3]);
      const uint32_t a2 = pack_bf16(s[2 * kk + 1][0], s[2 * kk + 1][1]);
      const uint32_t a3 = pack_bf16(s[2 * kk + 1][2], s[2 * kk + 1][3]);
      const int kbase = t0 + kw0 + kk * 16 + 2 * t;
      const uint32_t mlo0 = (kbase < w.lk ? 0x0000FFFFu : 0u) | (kbase + 1 < w.lk ? 0xFFFF0000u : 0u);
      const uint32_t mlo1 = (kbase + 8 < w.lk ? 0x0000FFFFu : 0u) | (kbase + 9 < w.lk ? 0xFFFF0000u : 0u);
#pragma unroll
      for (int dp = 0; dp < D / 16; ++dp) {
        const int r = kw0 + kk * 16 + ((lane >> 3) & 1) * 8 + (lane & 7);
        const int c = 2 * dp + (lane >> 4);
        uint32_t b0, b1, b2, b3;
        ldsm_x4_t(vb + tile_off(r, c), b0, b1, b2, b3);
        if (vmask) {
          b0 &= mlo0;
          b2 &= mlo0;
          b1 &= mlo1;
          b3 &= mlo1;
        }
        mma_bf16(o[2 * dp], a0, a1, a2, a3, b0, b1);
        mma_bf16(o[2 * dp + 1], a0, a1, a2, a3, b2, b3);
      }
    }
    if constexpr (!FP8) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[ring.stage]);
    } else {
      named_bar_sync(1, 32 * kConsumerWarps);  // bf16 copies free for the next tile
    }
    ring.advance<L::kStages>();
  }

  // ---------------------------------------------------------------- epilogue
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  if constexpr (kDecodeTile) {
    float* ml = reinterpret_cast<float*>(smem + L::kMlOff);
    float* mo = reinterpret_cast<float*>(smem + L::kMergeOff);
    if (t == 0) {
      ml[(cw * 16 + g) * 2 + 0] = m0;
      ml[(cw * 16 + g) * 2 + 1] = l0;
      ml[(cw * 16 + g + 8) * 2 + 0] = m1;
      ml[(cw * 16 + g + 8) * 2 + 1] = l1;
    }
    named_bar_sync(1, 32 * kConsumerWarps);
    float M0 = -INFINITY, M1 = -INFINITY;
#pragma unroll
    for (int ww = 0; ww < kConsumerWarps; ++ww) {
      M0 = fmaxf(M0, ml[(ww * 16 + g) * 2]);
      M1 = fmaxf(M1, ml[(ww * 16 + g + 8) * 2]);
    }
    const float f0 = ex2(m0 - (M0 == -INFINITY ? 0.f : M0));
    const float f1 = ex2(m1 - (M1 == -INFINITY ? 0.f : M1));
#pragma unroll
    for (int n = 0; n < NO; ++n) {
      *reinterpret_cast<float2*>(mo + (cw * 16 + g) * D + n * 8 + 2 * t) = make_float2(o[n][0] * f0, o[n][1] * f0);
      *reinterpret_cast<float2*>(mo + (cw * 16 + g + 8) * D + n * 8 + 2 * t) =
          make_float2(o[n][2] * f1, o[n][3] * f1);
    }
    named_bar_sync(1, 32 * kConsumerWarps);
    for (int idx = ctid; idx < R * D; idx += 32 * kConsumerWarps) {
      const int row = idx / D, d = idx % D;
      float M = -INFINITY;
#pragma unroll
      for (int ww = 0; ww < kConsumerWarps; ++ww) M = fmaxf(M, ml[(ww * 16 + row) * 2]);
      const float Mu = M == -INFINITY ? 0.f : M;
      float Lsum = 0.f, acc = 0.f;
#pragma unroll
      for (int ww = 0; ww < kConsumerWarps; ++ww) {
        Lsum += ml[(ww * 16 + row) * 2 + 1] * ex2(ml[(ww * 16 + row) * 2] - Mu);
        acc += mo[(ww * 16 + row) * D + d];
      }
      const float val = Lsum > 0.f ? acc / Lsum * vscale : 0.f;
      const float lse2 = Lsum > 0.f ? Mu + __log2f(Lsum) : -INFINITY;
      if (w.partial >= 0) {
        p.partial_o[((int64_t)w.partial * kDecodeRows + row) * D + d] = val;
        if (d == 0) p.partial_lse[w.partial * kDecodeRows + row] = lse2;
      } else {
        const int tok = w.q_row0 + row / p.G;
        const int head = w.hk * p.G + row % p.G;
        p.out[(int64_t)tok * p.o_stride_tok + (int64_t)head * p.o_stride_head + d] = __float2bfloat16_rn(val);
        if (d == 0 && p.lse != nullptr) p.lse[(int64_t)head * p.total_q + tok] = lse2 * kLn2;
      }
    }
    named_bar_sync(1, 32 * kConsumerWarps);
  } else {
#pragma unroll
    for (int half = 0; half < 2; ++half) {
      const int r = half ? r1 : r0;
      if (r >= R) continue;
      const float l = half ? l1 : l0;
      const float m = half ? m1 : m0;
      const float inv = l > 0.f ? vscale / l : 0.f;
      const int tok = w.q_row0 + r / p.G;
      const int head = w.hk * p.G + r % p.G;
      __nv_bfloat16* dst = p.out + (int64_t)tok * p.o_stride_tok + (int64_t)head * p.o_stride_head;
#pragma unroll
      for (int n = 0; n < NO; ++n) {
        const float x = o[n][half * 2] * inv, y = o[n][half * 2 + 1] * inv;
        *reinterpret_cast<uint32_t*>(dst + n * 8 + 2 * t) = pack_bf16(x, y);
      }
      if (t == 0 && p.lse != nullptr)
        p.lse[(int64_t)head * p.total_q + tok] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
    }
  }
  return true;
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v) {
  using L = Layout<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* full_k = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  uint64_t* full_v = full_k + L::kStages;
  uint64_t* empty = full_v + L::kStages;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kAbortOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(&full_k[s], 1);
      mbar_init(&full_v[s], 1);
      mbar_init(&empty[s], kConsumerWarps);
    }
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  __syncthreads();
  const int it0 = p.cta_begin[blockIdx.x], it1 = p.cta_begin[blockIdx.x + 1];
  if (warp == 0) {
    if (lane == 0) producer<D, FP8>(p, &tm_k, &tm_v, smem, full_k, full_v, empty, abort_flag, it0, it1);
    return;
  }
  const int ctid = threadIdx.x - 32;
  if (blockIdx.x == 0) {
    for (int b = ctid; b < p.batch; b += 32 * kConsumerWarps)
      if (__ldg(p.cache_seqlens + b) != __ldg(p.plan_lc + b))
        record_status(p.status, PKV_ERR_PLAN_MISMATCH, b, __ldg(p.cache_seqlens + b));
  }
  const float kscale = FP8 ? __ldg(p.k_scale) : 1.f;
  const float vscale = FP8 ? __ldg(p.v_scale) : 1.f;
  const float sl2 = p.scale_log2 * kscale;
  Ring ring;
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = p.items[it];
    bool ok;
    if (w.kind == kDecode)
      ok = run_item<D, FP8, kKvTile / kConsumerWarps>(p, w, smem, full_k, full_v, empty, abort_flag, ring, sl2, vscale);
    else
      ok = run_item<D, FP8, kKvTile>(p, w, smem, full_k, full_v, empty, abort_flag, ring, sl2, vscale);
    if (!ok) {
      record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, it);
      *abort_flag = 1;
      return;
    }
  }
}

template <int D, bool FP8>
cudaError_t launch_t(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, int num_ctas, cudaStream_t s) {
  using L = Layout<D, FP8>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  attn_kernel<D, FP8><<<num_ctas, kThreads, L::kAlloc, s>>>(p, tk, tv);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v, int num_ctas,
                             int head_dim, bool fp8, cudaStream_t stream) {
  if (num_ctas == 0) return cudaSuccess;
  if (fp8) return launch_t<128, true>(p, tm_k, tm_v, num_ctas, stream);
  if (head_dim == 128) return launch_t<128, false>(p, tm_k, tm_v, num_ctas, stream);
  return launch_t<64, false>(p, tm_k, tm_v, num_ctas, stream);
}

}  // namespace pkv
