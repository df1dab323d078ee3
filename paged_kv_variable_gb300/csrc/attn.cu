// Persistent attention kernel over a paged or contiguous KV cache.
//
// One CTA per SM walks its host-assigned list of work items (flashinfer PR
// "[Refactor] Uniform PoDAttention API with Horizontal Fusion SMs Schedule",
// Key Changes 2: prefill and decode work share one persistent launch).
//
// Warp roles (192 threads):
//   warp 0      TMA producer: K/V tiles of 128 keys, one 16-row box per
//               (page, 128-byte column chunk), page numbers read from
//               block_table (vLLM PR "[Kernel][Triton][FP8] ...", review:
//               block_table support; TransformerEngine PR "Add KV cache for
//               paged/non-paged attention": one table for K and V, bshd pages)
//               into a ring of shared-memory stages (the cached-KV prefetch of
//               the cutlass-sycl PR "Extend FlashAttention Prefill with KV
//               cache"); plus the 128-row Q tile of a prefill item.
//   warp 1      owns tensor memory and issues the tcgen05 MMAs of prefill
//               tiles: S = Q K^T into TMEM (two buffers), O += P V into TMEM.
//   warps 2..5  consumers.  Prefill tile: one query row per thread, masked
//               online softmax on S read from TMEM, P written to shared memory
//               for the next MMA, O rescaled in TMEM, epilogue.  Decode tile
//               (<= 16 rows): warp-level MMAs, the four warps split the keys
//               of each tile and merge at the end of the item.
//
// fp8 caches (vLLM PR, 8-bit KV cache) are converted to bf16 in shared memory
// (exact), with k_scale folded into the logit scale and v_scale applied to the
// normalised output; their prefill tiles use the warp-level MMA path (64 rows).
#include <cuda_bf16.h>

#include "kernels.h"
#include "ptx.cuh"
#include "tcgen05.cuh"

namespace pkv {

namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = 32 * (2 + kConsumerWarps);
constexpr int kConsumerThreads = 32 * kConsumerWarps;
constexpr float kLn2 = 0.693147180559945309f;
constexpr uint32_t kTmemCols = 512;   // S0 [0,128), S1 [128,256), O [256, 256+D)
constexpr uint32_t kTmemO = 256;

template <int D, bool FP8>
struct Layout {
  static constexpr bool kTc = !FP8;                        // tensor-core (tcgen05) prefill tiles
  static constexpr int kEsize = FP8 ? 1 : 2;
  static constexpr int kStagesK = (FP8 || D == 128) ? 3 : 4;  // K ring (released after S = Q K^T)
  static constexpr int kStagesV = (FP8 || D == 128) ? (FP8 ? 3 : 2) : 4;  // V ring (released after O += P V)
  static constexpr int kTileBytes = kKvTile * D * kEsize;   // one raw K (or V) tile
  static constexpr int kChunks = D * kEsize / 128;            // 128-byte column chunks per cache row
  static constexpr int kBf16Tile = kKvTile * D * 2;
  static constexpr int kKOff = 0;                             // K ring
  static constexpr int kVOff = kStagesK * kTileBytes;         // V ring
  static constexpr int kQOff = kVOff + kStagesV * kTileBytes; // tcgen05 path: Q tile (128 x D bf16)
  static constexpr int kDeqOff = kQOff + (kTc ? kKvTile * D * 2 : 0);  // fp8: bf16 copies of K and V
  static constexpr int kPOff = kDeqOff + (FP8 ? 2 * kBf16Tile : 0);    // P (128 x 128 bf16) / decode merge
  static constexpr int kMergeBytes = kConsumerWarps * kDecodeRows * D * 4;
  static constexpr int kPBytes = kTc ? (kMergeBytes > 32768 ? kMergeBytes : 32768) : kMergeBytes;
  static constexpr int kMlOff = kPOff + kPBytes;              // float[4][16][2]: (m, l)
  static constexpr int kBarOff = kMlOff + kConsumerWarps * kDecodeRows * 2 * 4;
  static constexpr int kNumBars = 2 * kStagesK + 2 * kStagesV + 9;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;     // tmem base, abort flag
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;                // room to align the base to 1024
};

struct Bars {
  uint64_t* full_k;
  uint64_t* empty_k;
  uint64_t* full_v;
  uint64_t* empty_v;
  uint64_t* q_full;
  uint64_t* q_empty;
  uint64_t* s_full;   // [2]
  uint64_t* s_free;   // [2]
  uint64_t* p_full;
  uint64_t* o_done;
  uint64_t* drain;    // MMA completion before tensor memory is freed after an abort
};

// Byte offset of 16-byte chunk c of row r in a bf16 tile stored as
// [D/64 column chunks][128 rows][128 B] with the 128-byte TMA swizzle.
__device__ __forceinline__ uint32_t tile_off(int r, int c) {
  return (uint32_t)((c >> 3) * (kKvTile * 128) + r * 128 + (((c & 7) ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t ld_u32(const __nv_bfloat16* p) {
  return __ldg(reinterpret_cast<const unsigned int*>(p));
}

__device__ __forceinline__ int num_tiles(const WorkItem& w) {
  return w.kv_end > w.kv_begin ? (w.kv_end - w.kv_begin + kKvTile - 1) / kKvTile : 0;
}

// fp8 K or V tile (128 rows x 128 codes, swizzled) -> bf16 tile in the layout above.
__device__ __forceinline__ void dequant_tile(const uint8_t* raw, uint8_t* dst, int ctid) {
#pragma unroll
  for (int k = 0; k < 8; ++k) {
    const int u = ctid + kConsumerThreads * k;
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
  __device__ __forceinline__ void advance(int n = 1) {
    for (int i = 0; i < n; ++i) {
      if (++stage == NS) {
        stage = 0;
        phase ^= 1;
      }
    }
  }
};

// ------------------------------------------------------------------ producer
// The whole warp issues: lane l owns the 16-row box of group (l % 8) and
// 128-byte column chunk (l / 8) of every tile, so the 8 block_table reads of a
// tile are one coalesced load instead of 8 dependent ones.  K of tile j+1 is
// issued before V of tile j, so that S = Q K^T of the next tile never waits
// behind the V ring.
template <int D, bool FP8>
__device__ void producer(const AttnParams& p, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                         const CUtensorMap* tm_q, uint8_t* smem, const Bars& B, volatile int* abort_flag, int it0,
                         int it1) {
  using L = Layout<D, FP8>;
  constexpr int kGroups = kKvTile / kBoxRows;
  const int lane = threadIdx.x & 31;
  const int grp = lane % kGroups, chunk = lane / kGroups;
  const bool active = chunk < L::kChunks;
  if (lane == 0) {
    tma_prefetch_desc(tm_k);
    tma_prefetch_desc(tm_v);
  }
  Ring rk, rv;
  int issued_k = 0, issued_v = 0;
  uint32_t pi = 0;  // prefill items with at least one tile
  bool ok = true, pending = false;
  int pend_page = 0, pend_slot = 0, pend_hk = 0;

  // this lane's box of a tile: page and slot (an out-of-range page fills zeros)
  auto locate = [&](const WorkItem& w, int t0, int& page, int& slot) {
    const int j0 = t0 + grp * kBoxRows;
    page = p.num_pages;
    slot = 0;
    if (j0 < w.kv_end) {
      if (p.page_size > 0) {
        const int pg = __ldg(p.block_table + (int64_t)w.b * p.bt_stride + j0 / p.page_size);
        if (pg < 0 || pg >= p.num_pages) {
          if (active) record_status(p.status, PKV_ERR_DEVICE_BOUNDS, w.b, pg);
        } else {
          page = pg;
          slot = j0 % p.page_size;
        }
      } else {
        page = w.b;
        slot = j0;
      }
    }
  };
  auto issue_v = [&]() -> bool {
    if (!warp_wait(&B.empty_v[rv.stage], rv.phase ^ 1, abort_flag)) return false;
    if (lane == 0) mbar_arrive_expect_tx(&B.full_v[rv.stage], L::kTileBytes);
    __syncwarp();
    if (active)
      tma_load_4d(smem + L::kVOff + rv.stage * L::kTileBytes + chunk * (kKvTile * 128) + grp * (kBoxRows * 128),
                  tm_v, &B.full_v[rv.stage], chunk * (128 / L::kEsize), pend_hk, pend_slot, pend_page);
    ++issued_v;
    rv.advance<L::kStagesV>();
    return true;
  };

  for (int it = it0; it < it1 && ok; ++it) {
    const WorkItem w = p.items[it];
    if (L::kTc && w.kind == kPrefill && num_tiles(w) > 0) {
      if (!warp_wait(B.q_empty, (pi & 1) ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      if (lane == 0) {
        if (pi == 0) tma_prefetch_desc(tm_q);
        const int tq = kPrefillRowsTc / p.G;
        mbar_arrive_expect_tx(B.q_full, (uint32_t)((D / 64) * p.G * tq * 128));
      }
      __syncwarp();
      if (lane < D / 64)
        tma_load_3d(smem + L::kQOff + lane * (kKvTile * 128), tm_q, B.q_full, lane * 64, w.hk * p.G, w.q_row0);
      ++pi;
    }
    for (int t0 = w.kv_begin; t0 < w.kv_end; t0 += kKvTile) {
      int page, slot;
      locate(w, t0, page, slot);  // block_table read overlaps the wait below
      if (!warp_wait(&B.empty_k[rk.stage], rk.phase ^ 1, abort_flag)) {
        ok = false;
        break;
      }
      if (lane == 0) mbar_arrive_expect_tx(&B.full_k[rk.stage], L::kTileBytes);
      __syncwarp();
      if (active)
        tma_load_4d(smem + L::kKOff + rk.stage * L::kTileBytes + chunk * (kKvTile * 128) + grp * (kBoxRows * 128),
                    tm_k, &B.full_k[rk.stage], chunk * (128 / L::kEsize), w.hk, slot, page);
      ++issued_k;
      rk.advance<L::kStagesK>();
      if (pending && !issue_v()) {
        ok = false;
        break;
      }
      pend_page = page;
      pend_slot = slot;
      pend_hk = w.hk;
      pending = true;
    }
  }
  if (ok && pending) ok = issue_v();
  if (!ok) {
    if (lane == 0) record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, 0);
    *abort_flag = 1;
    // let the copies already issued land before the CTA can exit (bounded)
    if (lane == 0) {
      int zero = 0;
      const int nk = issued_k < L::kStagesK ? issued_k : L::kStagesK;
      for (int k = issued_k - nk; k < issued_k; ++k)
        mbar_wait(&B.full_k[k % L::kStagesK], (uint32_t)((k / L::kStagesK) & 1), &zero);
      const int nv = issued_v < L::kStagesV ? issued_v : L::kStagesV;
      for (int k = issued_v - nv; k < issued_v; ++k)
        mbar_wait(&B.full_v[k % L::kStagesV], (uint32_t)((k / L::kStagesV) & 1), &zero);
    }
    __syncwarp();
  }
}

// ------------------------------------------------------------------ MMA issuer (prefill tiles)
template <int D>
__device__ bool mma_issuer(const AttnParams& p, uint8_t* smem, const Bars& B, volatile int* abort_flag,
                           uint32_t tmem, int it0, int it1) {
  using L = Layout<D, false>;
  constexpr uint32_t kIdescQK = idesc_f16(1, 0, 128, 128);
  constexpr uint32_t kIdescPV = idesc_f16(1, 1, 128, D);
  const uint32_t q_base = smem_u32(smem + L::kQOff);
  const uint32_t p_base = smem_u32(smem + L::kPOff);
  Ring rk, rv;
  uint32_t pt = 0, pi = 0;

  auto do_pv = [&](uint32_t T, bool first) -> bool {
    if (!mbar_wait(B.p_full, T & 1, abort_flag)) return false;
    if (!mbar_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) return false;
    tc_fence_after();
    const uint32_t v_base = smem_u32(smem + L::kVOff + rv.stage * L::kTileBytes);
#pragma unroll
    for (int k = 0; k < kKvTile / 16; ++k) {
      const uint64_t a = sdesc_sw128(p_base + (k >> 2) * (kKvTile * 128) + (k & 3) * 32, 16, 1024);
      const uint64_t b = sdesc_sw128(v_base + k * 16 * 128, kKvTile * 128, 1024);
      umma_ss(tmem + kTmemO, a, b, kIdescPV, (first && k == 0) ? 0u : 1u);
    }
    umma_commit(B.o_done);
#pragma unroll
    for (int i = 0; i < kConsumerWarps; ++i) umma_commit(&B.empty_v[rv.stage]);
    rv.advance<L::kStagesV>();
    return true;
  };

  for (int it = it0; it < it1; ++it) {
    const WorkItem w = p.items[it];
    const int n = num_tiles(w);
    if (w.kind != kPrefill) {
      rk.advance<L::kStagesK>(n);
      rv.advance<L::kStagesV>(n);
      continue;
    }
    if (n == 0) continue;
    if (!mbar_wait(B.q_full, pi & 1, abort_flag)) return false;
    for (int j = 0; j < n; ++j) {
      const uint32_t T = pt + j;
      if (!mbar_wait(&B.full_k[rk.stage], rk.phase, abort_flag)) return false;
      if (T >= 2 && !mbar_wait(&B.s_free[T & 1], ((T >> 1) & 1) ^ 1, abort_flag)) return false;
      tc_fence_after();
      const uint32_t k_base = smem_u32(smem + L::kKOff + rk.stage * L::kTileBytes);
#pragma unroll
      for (int k = 0; k < D / 16; ++k) {
        const uint32_t off = (k >> 2) * (kKvTile * 128) + (k & 3) * 32;
        umma_ss(tmem + (T & 1) * 128, sdesc_sw128(q_base + off, 16, 1024), sdesc_sw128(k_base + off, 16, 1024),
                kIdescQK, k > 0 ? 1u : 0u);
      }
      umma_commit(&B.s_full[T & 1]);
#pragma unroll
      for (int i = 0; i < kConsumerWarps; ++i) umma_commit(&B.empty_k[rk.stage]);
      if (j == n - 1) umma_commit(B.q_empty);
      rk.advance<L::kStagesK>();
      if (j >= 1 && !do_pv(T - 1, j == 1)) return false;
    }
    if (!do_pv(pt + n - 1, n == 1)) return false;
    pt += n;
    ++pi;
  }
  return true;
}

// ------------------------------------------------------------------ prefill tile softmax (tcgen05 path)
template <int D>
__device__ bool softmax_item(const AttnParams& p, const WorkItem& w, uint8_t* smem, const Bars& B,
                             volatile int* abort_flag, uint32_t tmem, Ring& rk, Ring& rv, uint32_t& pt, float sl2) {
  using L = Layout<D, false>;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int qw = warp & 3;                   // TMEM lane quarter this warp may access
  const int r = qw * 32 + lane;              // tile row == TMEM lane
  const uint32_t t_lane = tmem + ((uint32_t)(qw * 32) << 16);
  const int R = w.n_q * p.G;
  const bool valid = r < R;
  const int tok = w.q_row0 + r / p.G;
  const int head = w.hk * p.G + r % p.G;
  int lim = 0;
  if (valid) {
    lim = w.kv_end;
    if (p.causal) lim = min(lim, w.q_i0 + r / p.G + w.lk - w.lq + 1);
  }
  const int n = num_tiles(w);
  float m = -INFINITY, l = 0.f;
  uint8_t* pbuf = smem + L::kPOff;

  for (int j = 0; j < n; ++j) {
    const uint32_t T = pt + j;
    const int t0 = w.kv_begin + j * kKvTile;
    if (!warp_wait(&B.s_full[T & 1], (T >> 1) & 1, abort_flag)) return false;
    tc_fence_after();
    uint32_t s[128];
#pragma unroll
    for (int c = 0; c < 4; ++c) tmem_ld32(t_lane + (T & 1) * 128 + c * 32, s + c * 32);
    tmem_wait_ld();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(&B.s_free[T & 1]);

    // mask by select (rows past the sequence see nothing), row max
    const bool need_mask = t0 + kKvTile > lim;
    float mx = -INFINITY;
    if (__any_sync(0xffffffffu, need_mask)) {
#pragma unroll
      for (int c = 0; c < 128; ++c) {
        const float v = (t0 + c < lim) ? __uint_as_float(s[c]) : -INFINITY;
        s[c] = __float_as_uint(v);
        mx = fmaxf(mx, v);
      }
    } else {
#pragma unroll
      for (int c = 0; c < 128; ++c) mx = fmaxf(mx, __uint_as_float(s[c]));
    }
    const float m_new = fmaxf(m, mx * sl2);
    const float mu = m_new == -INFINITY ? 0.f : m_new;
    const float alpha = ex2(m - mu);
    float sum = 0.f;
    uint32_t pk[64];
#pragma unroll
    for (int c = 0; c < 64; ++c) {
      const float p0 = ex2(fmaf(__uint_as_float(s[2 * c]), sl2, -mu));
      const float p1 = ex2(fmaf(__uint_as_float(s[2 * c + 1]), sl2, -mu));
      sum += p0 + p1;
      pk[c] = pack_bf16(p0, p1);
    }
    l = l * alpha + sum;
    m = m_new;

    // P buffer and O are free once the previous tile's P V has completed
    if (j > 0 && !warp_wait(B.o_done, (T - 1) & 1, abort_flag)) return false;
    tc_fence_after();
    if (t0 + kKvTile > w.lk) {
      // rows past the sequence may hold anything (even NaN): zero them in V
      if (!warp_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) return false;
      if (t0 + r >= w.lk) {
        uint8_t* vrow = smem + L::kVOff + rv.stage * L::kTileBytes + r * 128;
#pragma unroll
        for (int c = 0; c < D / 64; ++c)
#pragma unroll
          for (int q = 0; q < 8; ++q) *reinterpret_cast<uint4*>(vrow + c * (kKvTile * 128) + q * 16) = make_uint4(0, 0, 0, 0);
      }
    }
#pragma unroll
    for (int c = 0; c < 16; ++c)
      *reinterpret_cast<uint4*>(pbuf + tile_off(r, c)) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
    if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld32(t_lane + kTmemO + c * 32, o);
        tmem_wait_ld();
#pragma unroll
        for (int e = 0; e < 32; ++e) o[e] = __float_as_uint(__uint_as_float(o[e]) * alpha);
        tmem_st32(t_lane + kTmemO + c * 32, o);
      }
      tmem_wait_st();
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncwarp();
    if (lane == 0) mbar_arrive(B.p_full);
    rk.advance<L::kStagesK>();
    rv.advance<L::kStagesV>();
  }

  // epilogue: O / l -> bf16 rows, natural-log LSE
  __nv_bfloat16* dst = p.out + (int64_t)tok * p.o_stride_tok + (int64_t)head * p.o_stride_head;
  if (n > 0) {
    if (!warp_wait(B.o_done, (pt + n - 1) & 1, abort_flag)) return false;
    tc_fence_after();
    const float inv = l > 0.f ? 1.f / l : 0.f;
#pragma unroll
    for (int c = 0; c < D / 32; ++c) {
      uint32_t o[32];
      tmem_ld32(t_lane + kTmemO + c * 32, o);
      tmem_wait_ld();
      if (valid) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          uint4 v;
          v.x = pack_bf16(__uint_as_float(o[8 * q + 0]) * inv, __uint_as_float(o[8 * q + 1]) * inv);
          v.y = pack_bf16(__uint_as_float(o[8 * q + 2]) * inv, __uint_as_float(o[8 * q + 3]) * inv);
          v.z = pack_bf16(__uint_as_float(o[8 * q + 4]) * inv, __uint_as_float(o[8 * q + 5]) * inv);
          v.w = pack_bf16(__uint_as_float(o[8 * q + 6]) * inv, __uint_as_float(o[8 * q + 7]) * inv);
          *reinterpret_cast<uint4*>(dst + c * 32 + q * 8) = v;
        }
      }
    }
    tc_fence_before();
  } else if (valid) {
#pragma unroll
    for (int c = 0; c < D / 8; ++c) *reinterpret_cast<uint4*>(dst + c * 8) = make_uint4(0, 0, 0, 0);
  }
  if (valid && p.lse != nullptr)
    p.lse[(int64_t)head * p.total_q + tok] = l > 0.f ? (m + __log2f(l)) * kLn2 : -INFINITY;
  pt += n;
  return true;
}

// ------------------------------------------------------------------ warp-MMA tiles (decode; fp8 prefill)
// KPW = keys of each 128-key tile handled by one warp: 32 (decode), 128 (prefill).
template <int D, bool FP8, int KPW>
__device__ bool run_item(const AttnParams& p, const WorkItem& w, uint8_t* smem, const Bars& B,
                         volatile int* abort_flag, Ring& rk, Ring& rv, float sl2, float vscale) {
  using L = Layout<D, FP8>;
  constexpr int NT = KPW / 8;       // S column tiles per warp
  constexpr int KS = D / 16;        // k-steps of Q K^T
  constexpr int NO = D / 8;         // O column tiles
  constexpr bool kDecodeTile = (KPW != kKvTile);
  const int lane = threadIdx.x & 31;
  const int cw = (threadIdx.x >> 5) - 2;  // consumer warp 0..3
  const int ctid = threadIdx.x - 64;
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
    if (!warp_wait(&B.full_k[rk.stage], rk.phase, abort_flag)) return false;
    uint8_t* stage_k = smem + L::kKOff + rk.stage * L::kTileBytes;
    uint8_t* stage_v = smem + L::kVOff + rv.stage * L::kTileBytes;
    uint32_t kb, vb;
    if constexpr (FP8) {
      uint8_t* dk = smem + L::kDeqOff;
      uint8_t* dv = dk + L::kBf16Tile;
      dequant_tile(stage_k, dk, ctid);
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.empty_k[rk.stage]);
      if (!warp_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) return false;
      dequant_tile(stage_v, dv, ctid);
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.empty_v[rv.stage]);
      named_bar_sync(1, kConsumerThreads);
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

    if constexpr (!FP8) {
      __syncwarp();
      if (lane == 0) mbar_arrive(&B.empty_k[rk.stage]);
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
      if (!warp_wait(&B.full_v[rv.stage], rv.phase, abort_flag)) return false;
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
      if (lane == 0) mbar_arrive(&B.empty_v[rv.stage]);
    } else {
      named_bar_sync(1, kConsumerThreads);  // bf16 copies free for the next tile
    }
    rk.advance<L::kStagesK>();
    rv.advance<L::kStagesV>();
  }

  // ---------------------------------------------------------------- epilogue
  l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
  l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
  l1 += __shfl_xor_sync(0xffffffffu, l1, 2);

  if constexpr (kDecodeTile) {
    float* ml = reinterpret_cast<float*>(smem + L::kMlOff);
    float* mo = reinterpret_cast<float*>(smem + L::kPOff);
    if (t == 0) {
      ml[(cw * 16 + g) * 2 + 0] = m0;
      ml[(cw * 16 + g) * 2 + 1] = l0;
      ml[(cw * 16 + g + 8) * 2 + 0] = m1;
      ml[(cw * 16 + g + 8) * 2 + 1] = l1;
    }
    named_bar_sync(1, kConsumerThreads);
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
    named_bar_sync(1, kConsumerThreads);
    for (int idx = ctid; idx < R * D; idx += kConsumerThreads) {
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
    named_bar_sync(1, kConsumerThreads);
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
__device__ bool consumer(const AttnParams& p, uint8_t* smem, const Bars& B, volatile int* abort_flag, uint32_t tmem,
                         int it0, int it1) {
  using L = Layout<D, FP8>;
  const int ctid = threadIdx.x - 64;
  if (blockIdx.x == 0) {
    for (int b = ctid; b < p.batch; b += kConsumerThreads)
      if (__ldg(p.cache_seqlens + b) != __ldg(p.plan_lc + b))
        record_status(p.status, PKV_ERR_PLAN_MISMATCH, b, __ldg(p.cache_seqlens + b));
  }
  const float kscale = FP8 ? __ldg(p.k_scale) : 1.f;
  const float vscale = FP8 ? __ldg(p.v_scale) : 1.f;
  const float sl2 = p.scale_log2 * kscale;
  Ring rk, rv;
  uint32_t pt = 0;
  for (int it = it0; it < it1; ++it) {
    const WorkItem w = p.items[it];
    bool ok;
    if (w.kind == kDecode) {
      ok = run_item<D, FP8, kKvTile / kConsumerWarps>(p, w, smem, B, abort_flag, rk, rv, sl2, vscale);
    } else if constexpr (L::kTc) {
      ok = softmax_item<D>(p, w, smem, B, abort_flag, tmem, rk, rv, pt, sl2);
    } else {
      ok = run_item<D, FP8, kKvTile>(p, w, smem, B, abort_flag, rk, rv, sl2, vscale);
    }
    if (!ok) {
      record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, it);
      *abort_flag = 1;
      return false;
    }
  }
  return true;
}

template <int D, bool FP8>
__global__ void __launch_bounds__(kThreads, 1)
    attn_kernel(const __grid_constant__ AttnParams p, const __grid_constant__ CUtensorMap tm_k,
                const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_q) {
  using L = Layout<D, FP8>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + L::kBarOff);
  Bars B;
  B.full_k = bars;
  B.empty_k = bars + L::kStagesK;
  B.full_v = bars + 2 * L::kStagesK;
  B.empty_v = bars + 2 * L::kStagesK + L::kStagesV;
  B.q_full = bars + 2 * L::kStagesK + 2 * L::kStagesV;
  B.q_empty = B.q_full + 1;
  B.s_full = B.q_full + 2;
  B.s_free = B.q_full + 4;
  B.p_full = B.q_full + 6;
  B.o_done = B.q_full + 7;
  B.drain = B.q_full + 8;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kMiscOff);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kMiscOff + 4);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < L::kStagesK; ++s) {
      mbar_init(&B.full_k[s], 1);
      mbar_init(&B.empty_k[s], kConsumerWarps);
    }
    for (int s = 0; s < L::kStagesV; ++s) {
      mbar_init(&B.full_v[s], 1);
      mbar_init(&B.empty_v[s], kConsumerWarps);
    }
    mbar_init(B.q_full, 1);
    mbar_init(B.q_empty, 1);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&B.s_full[i], 1);
      mbar_init(&B.s_free[i], kConsumerWarps);
    }
    mbar_init(B.p_full, kConsumerWarps);
    mbar_init(B.o_done, 1);
    mbar_init(B.drain, 1);
    *abort_flag = 0;
    fence_mbarrier_init();
  }
  if (L::kTc && warp == 1) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = L::kTc ? *tmem_slot : 0u;
  const int it0 = p.cta_begin[blockIdx.x], it1 = p.cta_begin[blockIdx.x + 1];
  if (warp == 0) {
    producer<D, FP8>(p, &tm_k, &tm_v, &tm_q, smem, B, abort_flag, it0, it1);
    return;
  }
  if (warp == 1) {
    if constexpr (L::kTc) {
      if (lane == 0) {
        if (!mma_issuer<D>(p, smem, B, abort_flag, tmem, it0, it1)) {
          record_status(p.status, PKV_ERR_DEVICE_TIMEOUT, blockIdx.x, -1);
          *abort_flag = 1;
          // wait (bounded) for the MMAs already issued before the memory is freed
          int zero = 0;
          umma_commit(B.drain);
          mbar_wait(B.drain, 0, &zero);
        }
      }
      __syncwarp();
    }
  } else {
    consumer<D, FP8>(p, smem, B, abort_flag, tmem, it0, it1);
  }
  // warps 1..5: every tensor-memory access is done before warp 1 frees it
  tc_fence_before();
  named_bar_sync(2, 32 * (1 + kConsumerWarps));
  tc_fence_after();
  if (L::kTc && warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int D, bool FP8>
cudaError_t launch_t(const AttnParams& p, const CUtensorMap& tk, const CUtensorMap& tv, const CUtensorMap& tq,
                     int num_ctas, cudaStream_t s) {
  using L = Layout<D, FP8>;
  static_assert(L::kAlloc <= 232448, "shared memory budget");
  cudaError_t e = cudaFuncSetAttribute(attn_kernel<D, FP8>, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  attn_kernel<D, FP8><<<num_ctas, kThreads, L::kAlloc, s>>>(p, tk, tv, tq);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attention(const AttnParams& p, const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                             const CUtensorMap& tm_q, int num_ctas, int head_dim, bool fp8, cudaStream_t stream) {
  if (num_ctas == 0) return cudaSuccess;
  if (fp8) return launch_t<128, true>(p, tm_k, tm_v, tm_q, num_ctas, stream);
  if (head_dim == 128) return launch_t<128, false>(p, tm_k, tm_v, tm_q, num_ctas, stream);
  return launch_t<64, false>(p, tm_k, tm_v, tm_q, num_ctas, stream);
}

}  // namespace pkv
