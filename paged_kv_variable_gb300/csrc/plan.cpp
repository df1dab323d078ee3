// Host scheduling step: validation, prefill/decode classification, split-KV
// chunking and longest-processing-time assignment of tiles to persistent CTAs.
//
// flashinfer PR "[Refactor] Uniform PoDAttention API with Horizontal Fusion SMs
// Schedule": one persistent launch serves prefill and decode requests, the
// partition of SMs follows the KV-cache load (Key Changes 2), requests are
// classified by query length (Limitations: "qo_len > threshold"), and a zero
// KV length must not be rejected (the review's failing test).  flash-attention
// PR "Add flash_attn_varlen_func_with_kvcache", Limitation: a fixed
// num_splits = 1 hurts decode, so decode units are cut into KV chunks here.
#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <functional>
#include <new>
#include <vector>

#include "internal.h"

namespace pkv {

namespace {

size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

struct Tile {
  WorkItem item;
  double cost;
};

// Per-key model costs (relative units): a decode key streams 2*D*esize bytes
// from HBM for one kv head; a prefill key costs one 128-row MMA step.  (The
// weight of a prefill key against a decode key was measured on the mixed
// prefill + decode batch: 0.418 ms at this weight, 0.440 at 0.7 of it, 0.426
// at 1.2 times and 0.442 at twice it; prefill-only batches do not move.)
double decode_cost(int keys, int d, int esize) { return 64.0 + keys * (2.0 * d * esize) / 512.0; }
double prefill_cost(int keys, int rows, int d) { return 256.0 + keys * (rows * d * 4.0) / 65536.0; }

}  // namespace

pkv_status validate_problem(const pkv_problem* p) {
  if (!p) return fail(PKV_ERR_INVALID_ARG, "problem is NULL");
  if (p->batch < 0) return fail(PKV_ERR_INVALID_ARG, "batch < 0");
  if (p->num_heads_q <= 0 || p->num_heads_kv <= 0)
    return fail(PKV_ERR_INVALID_ARG, "head counts must be positive");
  if (p->num_heads_q % p->num_heads_kv != 0)
    return fail(PKV_ERR_INVALID_ARG, "num_heads_q (%d) %% num_heads_kv (%d) != 0", p->num_heads_q,
                p->num_heads_kv);
  // any group size: groups of more than 128 heads are cut into head sub-groups
  if (p->cache_dtype != PKV_BF16 && p->cache_dtype != PKV_FP8_E4M3)
    return fail(PKV_ERR_INVALID_ARG, "cache_dtype %d unknown", p->cache_dtype);
  if (p->head_dim != 64 && p->head_dim != 128 && p->head_dim != 256)
    return fail(PKV_ERR_UNSUPPORTED, "head_dim %d not in {64, 128, 256}", p->head_dim);
  if (p->page_size < 0 || p->page_size > 256 ||
      (p->page_size >= kBoxRows && p->page_size % kBoxRows != 0) ||
      (p->page_size > 0 && p->page_size < kBoxRows && (p->page_size & (p->page_size - 1)) != 0))
    return fail(PKV_ERR_UNSUPPORTED, "page_size %d: 0, 1, 2, 4 or a multiple of %d up to 256", p->page_size,
                kBoxRows);
  if (p->cache_capacity <= 0) return fail(PKV_ERR_INVALID_ARG, "cache_capacity must be positive");
  if (p->page_size > 0 && p->cache_capacity % p->page_size != 0)
    return fail(PKV_ERR_INVALID_ARG, "cache_capacity must be a multiple of page_size");
  if (p->num_pages <= 0) return fail(PKV_ERR_INVALID_ARG, "num_pages must be positive");
  if (p->page_size == 0 && p->num_pages < p->batch)
    return fail(PKV_ERR_INVALID_ARG, "contiguous cache: batch_size_cache (num_pages) < batch");
  if (!std::isfinite(p->softmax_scale) || !(p->softmax_scale > 0.0f))
    return fail(PKV_ERR_INVALID_ARG, "softmax_scale must be finite and positive");
  return PKV_OK;
}

}  // namespace pkv

using namespace pkv;

namespace {

pkv_status make_plan(const pkv_problem* problem, const int32_t* h_q_lens, const int32_t* h_cache_lens,
                     const int32_t* h_new_lens, int32_t num_sms, bool dynamic, pkv_plan_t* out_plan,
                     size_t* out_workspace_bytes) {
  if (!out_plan || !out_workspace_bytes) return fail(PKV_ERR_INVALID_ARG, "output pointers are NULL");
  *out_plan = nullptr;
  *out_workspace_bytes = 0;
  pkv_status st = validate_problem(problem);
  if (st != PKV_OK) return st;
  const pkv_problem& p = *problem;
  const int B = p.batch;
  if (B > 0 && (!h_q_lens || !h_cache_lens)) return fail(PKV_ERR_INVALID_ARG, "length arrays are NULL");
  if (num_sms <= 0) return fail(PKV_ERR_INVALID_ARG, "num_sms must be positive");

  const int G = p.num_heads_q / p.num_heads_kv;
  const int D = p.head_dim;
  const int esize = p.cache_dtype == PKV_BF16 ? 2 : 1;
  const int prefill_rows = kPrefillRowsTc;
  // tensor-core tiles: nh_tc heads of a group x tq query tokens (128 rows at
  // most); a group of more than 128 heads takes n_sub head sub-groups
  const int nh_tc = tc_group_heads(G);
  const int n_sub = (G + nh_tc - 1) / nh_tc;
  const int tq_prefill = prefill_rows / nh_tc;  // query tokens per tensor-core tile
  // A unit (sequence, kv head[, head sub-group]) is a decode unit (warp-MMA
  // tile) if its rows fit 16, else tensor-core tiles; units whose queries fit
  // one tile (decode steps of wide groups, short query runs) can be split
  // along the keys like decode units.
  const int dec_rows = decode_rows(D);  // rows of a warp-MMA decode tile (8 at D = 256)
  auto is_decode = [&](int lq) { return (int64_t)lq * G <= dec_rows; };
  auto splittable = [&](int lq) { return is_decode(lq) || lq <= tq_prefill; };
  // an item of a long query run holds up to two consecutive tiles (fp8 cache,
  // head dims up to 128; plans without decode tiles), which share its K/V tiles
  bool any_decode = false, any_prefill = false;
  for (int b = 0; b < B; ++b) {
    any_decode |= h_q_lens[b] > 0 && is_decode(h_q_lens[b]);
    any_prefill |= h_q_lens[b] > 0 && !is_decode(h_q_lens[b]);
  }
  const int tq_item = tq_prefill * (any_decode ? 1 : prefill_q_tiles(D, p.cache_dtype == PKV_FP8_E4M3));
  // decode-only plans over an fp8 cache at head dims up to 128, or a bf16 one
  // at head dim 64 (rows of 128 bytes), run two CTAs an SM
  const bool two_ctas = (p.cache_dtype == PKV_FP8_E4M3 ? D <= 128 : D == 64) && !any_prefill;
  const int cps = two_ctas ? 2 : 1;

  int64_t total_q = 0, total_new = 0, total_split_keys = 0;
  for (int b = 0; b < B; ++b) {
    int lq = h_q_lens[b], lc = h_cache_lens[b], ln = h_new_lens ? h_new_lens[b] : 0;
    if (lq < 0 || lc < 0 || ln < 0) return fail(PKV_ERR_INVALID_ARG, "negative length at sequence %d", b);
    if ((int64_t)lc + ln > p.cache_capacity)
      return fail(PKV_ERR_INVALID_ARG, "sequence %d: cache_len %d + new_len %d > capacity %d", b, lc, ln,
                  p.cache_capacity);
    total_q += lq;
    total_new += ln;
    if (dynamic && lq > 0 && !splittable(lq))
      return fail(PKV_ERR_UNSUPPORTED,
                  "dynamic plans take requests whose queries fit one tile (sequence %d: %d query tokens > %d)", b, lq,
                  std::max(tq_prefill, dec_rows / G));
    if (lq > 0 && splittable(lq))
      total_split_keys += (int64_t)(lc + ln) * p.num_heads_kv * (is_decode(lq) ? 1 : n_sub);
  }
  if (total_q > INT32_MAX / 2 || total_new > INT32_MAX / 2)
    return fail(PKV_ERR_UNSUPPORTED, "total tokens too large");

  // split-KV chunk: at least 2 splittable items per SM in decode-only plans, 4
  // when prefill tiles share the launch (their gaps want finer decode items),
  // chunks >= 512 keys.  Measured: the fp8 decode batch (two CTAs an SM) 59.1
  // against 60.9 us at 4, one of random lengths 61.7 against 64.9; the bf16
  // decode batch the same attention kernel and 100.4 against 101.8 us a call
  // (fewer partials to combine); the mixed batch 0.417 against 0.430 ms at 4.
  auto chunk_for = [&](int64_t items_per_sm) {
    const int64_t target = items_per_sm * num_sms;
    const int64_t c = (total_split_keys + target - 1) / target;
    return std::max<int64_t>(512, (c + kKvTile - 1) / kKvTile * kKvTile);
  };
  int64_t chunk = 1 << 30;
  if (total_split_keys > 0) chunk = chunk_for(any_prefill ? 4 : 2);
  // A decode-only plan whose units are placed as evenly whole (one item an SM
  // as the target) as in chunks of the half is not split at all: no partials
  // and no combine kernel (the bf16 decode batch: 98.1 against 100.3 us a
  // call, the same attention kernel).  Judged on the model costs of a
  // longest-first placement; batches with a few long sequences stay split.
  if (!any_prefill && total_split_keys > 0) {
    const int ctas = num_sms * cps;
    std::vector<double> c, load;
    c.reserve((size_t)B * 4);
    load.reserve((size_t)ctas);
    auto busiest = [&](int64_t ch) {  // the longest-first placement's largest CTA cost
      c.clear();
      for (int b = 0; b < B; ++b) {  // one cost per chunk; every kv head has the same
        if (h_q_lens[b] == 0) continue;
        const int lk = h_cache_lens[b] + (h_new_lens ? h_new_lens[b] : 0);
        const int n = lk <= ch ? 1 : (int)((lk + ch - 1) / ch);
        for (int k = 0; k < n; ++k)
          c.push_back(decode_cost((int)(std::min<int64_t>((int64_t)(k + 1) * ch, lk) - (int64_t)k * ch), D, esize));
      }
      std::sort(c.begin(), c.end(), std::greater<double>());
      load.assign((size_t)ctas, 0.0);  // a min-heap over the CTA loads
      for (double x : c)
        for (int hk = 0; hk < p.num_heads_kv; ++hk) {
          std::pop_heap(load.begin(), load.end(), std::greater<double>());
          load.back() += x;
          std::push_heap(load.begin(), load.end(), std::greater<double>());
        }
      return *std::max_element(load.begin(), load.end());
    };
    const int64_t whole = chunk_for(1);
    if (whole != chunk && busiest(whole) <= 1.02 * busiest(chunk)) chunk = whole;
  }
  auto nchunks_of = [&](int lk) { return lk <= chunk ? 1 : (int)((lk + chunk - 1) / chunk); };

  int64_t num_tiles_est = 0;
  for (int b = 0; b < B; ++b) {
    const int lq = h_q_lens[b], lk = h_cache_lens[b] + (h_new_lens ? h_new_lens[b] : 0);
    if (lq == 0) continue;
    num_tiles_est += (int64_t)p.num_heads_kv * (is_decode(lq) ? nchunks_of(lk)
                                                : (int64_t)n_sub * (splittable(lq) ? nchunks_of(lk)
                                                                                   : (lq + tq_item - 1) / tq_item));
  }
  std::vector<Tile> tiles;
  tiles.reserve((size_t)num_tiles_est);
  std::vector<CombineItem> combines;
  int64_t num_slots = 0;
  int32_t n_dec = 0, n_pre = 0;
  int64_t q_row = 0;
  for (int b = 0; b < B; ++b) {
    int lq = h_q_lens[b], lc = h_cache_lens[b], ln = h_new_lens ? h_new_lens[b] : 0;
    int lk = lc + ln;
    if (lq == 0) continue;
    for (int hk = 0; hk < p.num_heads_kv; ++hk) {
      const bool dec = is_decode(lq);
      for (int sg = 0; sg < (dec ? 1 : n_sub); ++sg) {
        const int h0 = dec ? 0 : sg * nh_tc;
        const int nh = dec ? G : std::min(nh_tc, G - h0);
        if (splittable(lq)) {
          // one query tile (all lq tokens), possibly cut into KV chunks
          const int nchunks = nchunks_of(lk);
          const int rows = lq * nh;
          const int stride = (rows + kDecodeRows - 1) / kDecodeRows;  // 16-row partial slots per chunk
          const int64_t slot0 = nchunks > 1 ? num_slots : -1;
          for (int c = 0; c < nchunks; ++c) {
            Tile t{};
            t.item.b = b;
            t.item.hk = hk;
            t.item.q_row0 = (int32_t)q_row;
            t.item.q_i0 = 0;
            t.item.n_q = lq;
            t.item.lq = lq;
            t.item.lk = lk;
            t.item.kv_begin = (int32_t)std::min<int64_t>((int64_t)c * chunk, lk);
            t.item.kv_end = (int32_t)std::min<int64_t>((int64_t)(c + 1) * chunk, lk);
            t.item.kind = dec ? kDecode : kPrefill;
            t.item.partial = nchunks > 1 ? (int32_t)(num_slots + (int64_t)c * stride) : -1;
            t.item.h0 = h0;
            t.item.nh = nh;
            const int keys = t.item.kv_end - t.item.kv_begin;
            t.cost = dec ? decode_cost(keys, D, esize)
                         : std::max(decode_cost(keys, D, esize), prefill_cost(keys, prefill_rows, D));
            tiles.push_back(t);
            if (dec) ++n_dec; else ++n_pre;
          }
          if (nchunks > 1) {
            CombineItem ci{};
            ci.b = b;
            ci.q_row0 = (int32_t)q_row;
            ci.n_q = lq;
            ci.hk = hk;
            ci.nsplit = nchunks;
            ci.slot0 = (int32_t)slot0;
            ci.slot_stride = stride;
            ci.h0 = h0;
            ci.nh = nh;
            combines.push_back(ci);
            num_slots += (int64_t)nchunks * stride;
          }
        } else {
          for (int i0 = 0; i0 < lq; i0 += tq_item) {
            int n = std::min(tq_item, lq - i0);
            int kv_end = lk;  // the keys of the item's last query token
            if (p.causal) kv_end = std::max(0, std::min(lk, i0 + n + lk - lq));
            Tile t{};
            t.item.b = b;
            t.item.hk = hk;
            t.item.q_row0 = (int32_t)(q_row + i0);
            t.item.q_i0 = i0;
            t.item.n_q = n;
            t.item.lq = lq;
            t.item.lk = lk;
            t.item.kv_begin = 0;
            t.item.kv_end = kv_end;
            t.item.kind = kPrefill;
            t.item.partial = -1;
            t.item.h0 = h0;
            t.item.nh = nh;
            // each query tile of the item attends the keys of its own last token
            t.cost = 0.0;
            for (int s = i0; s < i0 + n; s += tq_prefill) {
              const int ns = std::min(tq_prefill, i0 + n - s);
              const int ke = p.causal ? std::max(0, std::min(lk, s + ns + lk - lq)) : lk;
              t.cost += prefill_cost(ke, prefill_rows, D);
            }
            tiles.push_back(t);
            ++n_pre;
          }
        }
      }
    }
    q_row += lq;
  }
  if (num_slots > INT32_MAX / (kDecodeRows * 256))
    return fail(PKV_ERR_UNSUPPORTED, "too many split-KV partial slots");

  // longest processing time first onto the least-loaded CTA (ties: the lowest
  // CTA index), found with a tournament tree over the CTAs' (load, index)
  // pairs; each CTA keeps its items in the order they were assigned
  const int num_items = (int)tiles.size();
  const int num_ctas = std::max(1, std::min(num_sms * cps, num_items));
  std::vector<double> costs(num_items);
  for (int i = 0; i < num_items; ++i) costs[i] = tiles[i].cost;
  std::vector<int> order(num_items);
  for (int i = 0; i < num_items; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(), [&](int a, int c) { return costs[a] > costs[c]; });
  using Load = std::pair<double, int>;
  int leaves = 1;
  while (leaves < num_ctas) leaves *= 2;
  const Load none{HUGE_VAL, INT32_MAX};
  std::vector<Load> tree(2 * (size_t)leaves, none);  // node i: the lesser of nodes 2i and 2i+1
  for (int c = 0; c < num_ctas; ++c) tree[leaves + c] = {0.0, c};
  for (int i = leaves - 1; i >= 1; --i) tree[i] = std::min(tree[2 * i], tree[2 * i + 1]);
  std::vector<int> cta_of(num_items), cta_count(num_ctas, 0);
  for (int idx : order) {
    const int c = tree[1].second;
    cta_of[idx] = c;
    ++cta_count[c];
    int i = leaves + c;
    tree[i].first += costs[idx];
    for (i >>= 1; i >= 1; i >>= 1) tree[i] = std::min(tree[2 * i], tree[2 * i + 1]);
  }
  double max_cost = 0, sum_cost = 0;
  int max_items = 0;
  std::vector<Load> loads(tree.begin() + leaves, tree.begin() + leaves + num_ctas);
  std::sort(loads.begin(), loads.end());  // summed lightest first
  for (const Load& l : loads) {
    max_cost = std::max(max_cost, l.first);
    sum_cost += l.first;
  }
  for (int c = 0; c < num_ctas; ++c) max_items = std::max(max_items, cta_count[c]);

  // workspace layout
  WorkspaceLayout L{};
  size_t off = 0;
  L.status = off;
  off = align_up(off + 16, 256);
  L.items = off;
  off = align_up(off + sizeof(WorkItem) * (size_t)std::max(1, num_items), 256);
  L.cta_begin = off;
  off = align_up(off + sizeof(int32_t) * (size_t)(num_ctas + 1), 256);
  L.combine = off;
  off = align_up(off + sizeof(CombineItem) * (size_t)std::max<size_t>(1, combines.size()), 256);
  L.plan_lc = off;
  off = align_up(off + sizeof(int32_t) * (size_t)std::max(1, B), 256);
  size_t image_bytes = off;
  L.partial_o = off;
  off = align_up(off + sizeof(float) * (size_t)num_slots * kDecodeRows * D, 256);
  L.partial_lse = off;
  off = align_up(off + sizeof(float) * (size_t)num_slots * kDecodeRows, 256);
  L.total = off;

  pkv_plan_s* plan = new (std::nothrow) pkv_plan_s();
  if (!plan) return fail(PKV_ERR_INVALID_ARG, "out of host memory");
  plan->image = (unsigned char*)calloc(1, image_bytes);
  plan->item_cost = (double*)calloc((size_t)std::max(1, num_items), sizeof(double));
  if (!plan->image || !plan->item_cost) {
    free(plan->image);
    free(plan->item_cost);
    delete plan;
    return fail(PKV_ERR_INVALID_ARG, "out of host memory");
  }
  plan->problem = p;
  plan->num_ctas = num_items > 0 ? num_ctas : 0;
  plan->num_slots = (int32_t)num_slots;
  plan->total_q = (int32_t)total_q;
  plan->total_new = (int32_t)total_new;
  plan->max_items_per_cta = max_items;
  plan->num_decode_items = n_dec;
  plan->num_prefill_items = n_pre;
  plan->num_split_units = (int32_t)combines.size();
  plan->max_cta_cost = max_cost;
  plan->mean_cta_cost = num_ctas ? sum_cost / num_ctas : 0.0;
  plan->layout = L;
  plan->image_bytes = image_bytes;
  plan->num_items = num_items;
  plan->num_combine = (int32_t)combines.size();
  plan->dynamic = dynamic ? 1 : 0;

  WorkItem* items = (WorkItem*)(plan->image + L.items);
  int32_t* cta_begin = (int32_t*)(plan->image + L.cta_begin);
  cta_begin[0] = 0;
  for (int c = 0; c < num_ctas; ++c) cta_begin[c + 1] = cta_begin[c] + cta_count[c];
  std::vector<int32_t> fill(cta_begin, cta_begin + num_ctas);
  for (int idx : order) {
    const int k = fill[cta_of[idx]]++;
    items[k] = tiles[idx].item;
    plan->item_cost[k] = costs[idx];
  }
  if (!combines.empty()) memcpy(plan->image + L.combine, combines.data(), combines.size() * sizeof(CombineItem));
  int32_t* lc = (int32_t*)(plan->image + L.plan_lc);
  for (int b = 0; b < B; ++b) lc[b] = h_cache_lens[b];

  *out_plan = plan;
  *out_workspace_bytes = L.total;
  return PKV_OK;
}

}  // namespace

extern "C" pkv_status pkv_plan(const pkv_problem* problem, const int32_t* h_q_lens,
                               const int32_t* h_cache_lens, const int32_t* h_new_lens,
                               int32_t num_sms, pkv_plan_t* out_plan, size_t* out_workspace_bytes) {
  return make_plan(problem, h_q_lens, h_cache_lens, h_new_lens, num_sms, false, out_plan, out_workspace_bytes);
}

extern "C" pkv_status pkv_plan_decode_dynamic(const pkv_problem* problem, const int32_t* h_q_lens,
                                              const int32_t* h_max_cache_lens, const int32_t* h_new_lens,
                                              int32_t num_sms, pkv_plan_t* out_plan, size_t* out_workspace_bytes) {
  return make_plan(problem, h_q_lens, h_max_cache_lens, h_new_lens, num_sms, true, out_plan, out_workspace_bytes);
}

extern "C" pkv_status pkv_plan_get_stats(pkv_plan_t plan, pkv_plan_stats* s) {
  if (!plan || !s) return fail(PKV_ERR_INVALID_ARG, "NULL plan or stats");
  s->num_items = plan->num_items;
  s->num_decode_items = plan->num_decode_items;
  s->num_prefill_items = plan->num_prefill_items;
  s->num_split_units = plan->num_split_units;
  s->num_ctas = plan->num_ctas;
  s->total_q = plan->total_q;
  s->total_new = plan->total_new;
  s->max_items_per_cta = plan->max_items_per_cta;
  s->max_cta_cost = plan->max_cta_cost;
  s->mean_cta_cost = plan->mean_cta_cost;
  s->upload_bytes = (int64_t)plan->image_bytes;
  s->workspace_bytes = (int64_t)plan->layout.total;
  return PKV_OK;
}

extern "C" pkv_status pkv_plan_get_items(pkv_plan_t plan, pkv_work_item* h_items, int32_t capacity,
                                         int32_t* count) {
  if (!plan || !count) return fail(PKV_ERR_INVALID_ARG, "NULL plan or count");
  *count = plan->num_items;
  if (!h_items || capacity <= 0) return PKV_OK;
  const WorkItem* items = (const WorkItem*)(plan->image + plan->layout.items);
  const int32_t* cta_begin = (const int32_t*)(plan->image + plan->layout.cta_begin);
  int n = 0;
  for (int c = 0; c < plan->num_ctas && n < capacity; ++c) {
    for (int k = cta_begin[c]; k < cta_begin[c + 1] && n < capacity; ++k, ++n) {
      const WorkItem& w = items[k];
      pkv_work_item& o = h_items[n];
      o.seq = w.b;
      o.kv_head = w.hk;
      o.q_row0 = w.q_row0;
      o.q_index0 = w.q_i0;
      o.n_q = w.n_q;
      o.q_len = w.lq;
      o.kv_len = w.lk;
      o.kv_begin = w.kv_begin;
      o.kv_end = w.kv_end;
      o.kind = w.kind;
      o.partial_slot = w.partial;
      o.cta = c;
      o.head0 = w.h0;
      o.num_heads = w.nh;
      o.cost = plan->item_cost[k];
    }
  }
  return PKV_OK;
}

extern "C" void pkv_plan_destroy(pkv_plan_t plan) {
  if (!plan) return;
  free(plan->image);
  free(plan->item_cost);
  delete plan;
}
