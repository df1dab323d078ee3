"""fp64 NumPy reference of attention over a paged or contiguous KV cache.

TEST INFRASTRUCTURE ONLY (see the package docstring).  Plain, slow and direct:
no tiling, no online softmax, no fusion.  Each function names the passage of
the source pages it follows:

* flash-attention PR "Add flash_attn_varlen_func_with_kvcache" (FA2 page),
  section "Usage": packed q with cu_seqlens_q; optional new k/v appended into
  the cache in place; the cache alone is attended when no k/v are passed;
  cache shape (batch_size_cache, seqlen_cache, n_heads, head_dim).  Section
  "Minor Changes": per-sequence cache lengths (k_cache_seqlens) kept apart from
  the cumulative lengths of the new tokens (cu_seqlens_knew).
* TransformerEngine PR "Add KV cache for paged/non-paged attention" (TE page),
  backend table and notes: paged and non-paged caches in bshd format, one page
  table shared by K and V, the unfused backend converting paged to non-paged
  before attention.
* vLLM PR "[Kernel][Triton][FP8] Adding fp8 and variable length sequence
  support to Triton FAv2 kernel" (vLLM page), feature list: causal masking,
  grouped-query attention, 8-bit KV cache, variable sequence lengths.
* cutlass-sycl PR "Extend FlashAttention Prefill with KV cache": prefill over
  cached KV plus current KV, causal and non-causal; a per-sequence cached
  length (review comment on variable-length cached KV).

The pages do not write the attention formula out; they all assume the
textbook softmax(scale * Q K^T + mask) V, which is what ``attend`` computes.
Readings taken where the pages are silent (bottom-right causal alignment,
head mapping h // (Hq/Hkv), e4m3 "fn" format, rounding of the fp8 encode,
empty rows) are listed in the design notes and restated at each function.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional

import numpy as np


# ---------------------------------------------------------------------------
# number formats
# ---------------------------------------------------------------------------
def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """bf16 bit patterns -> float64 (exact: bf16 is the top half of fp32)."""
    u = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return u.view(np.float32).astype(np.float64)


def e4m3_decode(codes: np.ndarray) -> np.ndarray:
    """OCP FP8 E4M3 ("fn": bias 7, no infinities, S.1111.111 = NaN) -> float64.

    The pages only say "fp8" / "8-bit KV cache" (vLLM page, feature list; TE
    page, FP8 row of the backend table); e4m3 is the reading taken.  Closed
    form: normal (-1)^s 2^(e-7) (1 + m/8), subnormal (-1)^s 2^-6 (m/8).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = np.where(c >> 7 == 1, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = (c & 0x7).astype(np.float64)
    normal = s * np.ldexp(1.0 + m / 8.0, e - 7)
    sub = s * np.ldexp(m / 8.0, -6)
    out = np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, out)


def e4m3_encode(y: np.ndarray) -> np.ndarray:
    """float32 -> e4m3 code, round to nearest even, saturating at +-448.

    Reading taken for the encode (the pages give none): RNE onto the e4m3 grid,
    magnitudes >= 448 clamp to 448 (a "satfinite" conversion), NaN -> 0x7F.
    """
    with np.errstate(invalid="ignore", over="ignore", divide="ignore"):
        return _e4m3_encode(np.asarray(y, dtype=np.float32))


def _e4m3_encode(y: np.ndarray) -> np.ndarray:
    a = np.abs(y.astype(np.float64))
    a = np.where(np.isfinite(a), a, 448.0)
    sign = np.signbit(y).astype(np.uint8) << 7
    out = np.zeros(a.shape, dtype=np.uint8)
    sat = a >= 448.0
    sub = a < 2.0 ** -6
    # subnormal range: grid step 2^-9; q in 0..8 (q == 8 is the smallest normal, code 0x08)
    q_sub = np.rint(np.where(sub, a, 0.0) / 2.0 ** -9).astype(np.int64)
    # normal range: a = 2^e * (q/8), q in [8,16)
    with np.errstate(divide="ignore"):
        e = np.floor(np.log2(np.where(sub | sat, 1.0, a))).astype(np.int64)
    # guard floor(log2) against rounding at exact powers of two
    e = np.where(np.ldexp(1.0, e) > np.where(sub | sat, 1.0, a), e - 1, e)
    e = np.where(np.ldexp(1.0, e + 1) <= np.where(sub | sat, 1.0, a), e + 1, e)
    q = np.rint(np.where(sub | sat, 8.0, a) / np.ldexp(1.0, e - 3)).astype(np.int64)
    carry = q == 16
    e = np.where(carry, e + 1, e)
    q = np.where(carry, 8, q)
    code_norm = ((e + 7) << 3) | (q - 8)
    code = np.where(sub, q_sub, code_norm)
    code = np.where(sat, 0x7E, code)
    out = (code.astype(np.uint8) | sign).astype(np.uint8)
    out = np.where(np.isnan(y), np.uint8(0x7F), out)
    return out.astype(np.uint8)


def fp8_inverse_scale(scale: float) -> np.float32:
    """The single fp32 reciprocal 1/scale used by the encode (IEEE, RN)."""
    return np.float32(1.0) / np.float32(scale)


def fp8_quantize(x_bf16_bits: np.ndarray, scale: float) -> np.ndarray:
    """Cache encode of one value: e4m3(fp32(x) * fp32(1/scale)).

    One IEEE round-to-nearest fp32 multiply (no fused multiply-add), then the
    e4m3 encode above.  Per-tensor fp32 scales as in the 8-bit KV cache of the
    vLLM page's feature list; dequantisation is code * scale.
    """
    x = (np.asarray(x_bf16_bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)
    y = (x * fp8_inverse_scale(scale)).astype(np.float32)
    return e4m3_encode(y)


# ---------------------------------------------------------------------------
# cache addressing and the in-place append
# ---------------------------------------------------------------------------
def physical_slots(spec, block_table, b: int, pos: np.ndarray):
    """Index tuple of logical token positions ``pos`` of sequence ``b``.

    Paged: (block_table[b, pos // P], pos % P) into a (pages, P, Hkv, D) pool,
    one table for K and V (TE page, notes under the backend table).
    Contiguous: (b, pos) into (batch, seqlen_cache, Hkv, D) (FA2 page, Usage).
    """
    pos = np.asarray(pos, dtype=np.int64)
    if spec.page_size > 0:
        P = spec.page_size
        return (block_table[b, pos // P].astype(np.int64), pos % P)
    return (np.full(pos.shape, b, dtype=np.int64), pos)


def append_kv(spec, k_cache, v_cache, block_table, k_new, v_new, k_scale=1.0, v_scale=1.0):
    """Write the new tokens into copies of the caches (FA2 page, Usage: the
    cache is updated in place; Minor Changes: cache lengths vs cu_seqlens_knew).

    Token t of sequence b (t < new_lens[b]) lands at logical position
    cache_lens[b] + t.  bf16 caches store the bf16 bits unchanged; fp8 caches
    store ``fp8_quantize``.  Returns the new (k_cache, v_cache).
    """
    kc = np.array(k_cache, copy=True)
    vc = np.array(v_cache, copy=True)
    if k_new is None:
        return kc, vc
    cu = np.concatenate([[0], np.cumsum(spec.new_lens)]).astype(np.int64)
    for b in range(spec.batch):
        n = int(spec.new_lens[b])
        if n == 0:
            continue
        pos = int(spec.cache_lens[b]) + np.arange(n)
        idx = physical_slots(spec, block_table, b, pos)
        kb = k_new[cu[b]:cu[b] + n]
        vb = v_new[cu[b]:cu[b] + n]
        if spec.cache_dtype == "fp8":
            kb = fp8_quantize(kb, k_scale)
            vb = fp8_quantize(vb, v_scale)
        kc[idx] = kb
        vc[idx] = vb
    return kc, vc


def prepare_prefix(case):
    """fp8 cases carry their cached prefix as raw bf16: write it with the same
    append (into an empty cache), giving the cache state before this call."""
    spec = case.spec
    if case.prefix_k is None or spec.cache_dtype != "fp8":
        return case.k_cache, case.v_cache
    pspec = _with_lengths(spec, cache_lens=np.zeros(spec.batch, np.int32), new_lens=spec.cache_lens)
    return append_kv(pspec, case.k_cache, case.v_cache, case.block_table, case.prefix_k,
                     case.prefix_v, case.k_scale, case.v_scale)


def _with_lengths(spec, **kw):
    import copy
    s = copy.copy(spec)
    for k, v in kw.items():
        setattr(s, k, v)
    return s


def gather_sequence(spec, cache, block_table, b: int, n: int, scale: float = 1.0) -> np.ndarray:
    """Dense (n, Hkv, D) fp64 view of the first ``n`` cached tokens of ``b``.

    fp8 codes are dequantised as code * scale.  This is the paged -> non-paged
    conversion the TE page's unfused backend performs before attention.
    """
    idx = physical_slots(spec, block_table, b, np.arange(n))
    rows = cache[idx]
    if spec.cache_dtype == "fp8":
        return e4m3_decode(rows) * float(scale)
    return bf16_to_f64(rows)


# ---------------------------------------------------------------------------
# attention
# ---------------------------------------------------------------------------
def visible_mask(lq: int, lk: int, causal: bool) -> np.ndarray:
    """(lq, lk) boolean: may query i see key j?

    Non-causal: every key.  Causal (cutlass-sycl page: "both causal and
    non-causal"; vLLM page feature list): the queries are the last lq of lk
    positions, so query i sees keys j <= i + (lk - lq) (bottom-right alignment;
    the pages do not state the alignment, this is the reading taken).
    """
    i = np.arange(lq)[:, None]
    j = np.arange(lk)[None, :]
    if not causal:
        return np.ones((lq, lk), dtype=bool)
    return j <= i + (lk - lq)


def attend(q: np.ndarray, K: np.ndarray, V: np.ndarray, causal: bool, scale: float,
           return_weights: bool = False):
    """softmax(scale * q K^T + mask) V for one sequence, fp64.

    q: (lq, Hq, D); K, V: (lk, Hkv, D).  Query head h reads kv head h // G with
    G = Hq / Hkv (grouped-query attention, vLLM page feature list; the mapping
    is the reading taken).  Masked scores are -inf; a row with no visible key
    returns o = 0 and lse = -inf (reading taken; the pages are silent).
    Returns o (lq, Hq, D), lse (Hq, lq) natural-log, optionally the weights
    (Hq, lq, lk).
    """
    lq, hq, d = q.shape
    lk, hkv, _ = K.shape
    g = hq // hkv
    o = np.zeros((lq, hq, d), dtype=np.float64)
    lse = np.full((hq, lq), -np.inf, dtype=np.float64)
    w_all = np.zeros((hq, lq, lk), dtype=np.float64) if return_weights else None
    if lq == 0:
        return (o, lse, w_all) if return_weights else (o, lse)
    mask = visible_mask(lq, lk, causal)
    any_visible = mask.any(axis=1)
    for h in range(hq):
        hk = h // g
        s = (q[:, h, :] @ K[:, hk, :].T) * float(scale)          # (lq, lk)
        s = np.where(mask, s, -np.inf)
        m = np.max(s, axis=1, initial=-np.inf)
        m_safe = np.where(any_visible, m, 0.0)
        e = np.exp(s - m_safe[:, None])                              # masked -> 0 exactly
        den = e.sum(axis=1)
        w = np.divide(e, den[:, None], out=np.zeros_like(e), where=any_visible[:, None])
        o[:, h, :] = w @ V[:, hk, :]
        lse[h] = np.where(any_visible, m_safe + np.log(np.where(any_visible, den, 1.0)), -np.inf)
        if return_weights:
            w_all[h] = w
    return (o, lse, w_all) if return_weights else (o, lse)


def query_values(case, rows: np.ndarray) -> np.ndarray:
    """Query rows as attended: the bf16 values, or -- when the call quantises Q
    for the fp8 Q.K^T (``case.q_scale``; the fp8 "QKV" models of the vLLM page's
    feature list and lm-eval notes) -- their e4m3 codes with the same encode as
    the cache (one fp32 RN multiply by fp32(1/scale)), decoded times the scale."""
    if getattr(case, "q_scale", None) is None:
        return bf16_to_f64(rows)
    return e4m3_decode(fp8_quantize(rows, case.q_scale)) * float(np.float32(case.q_scale))


def forward(case, *, k_cache=None, v_cache=None):
    """The whole call: append the new K/V (if any), then attend every sequence.

    Returns dict(out (total_q, Hq, D) fp64, lse (Hq, total_q) fp64,
    k_cache, v_cache) where the caches are the post-append physical arrays.
    ``k_cache``/``v_cache`` override the starting cache (e.g. a prior step's).
    """
    spec = case.spec
    if k_cache is None:
        k_cache, v_cache = prepare_prefix(case)
    kc, vc = append_kv(spec, k_cache, v_cache, case.block_table, case.k_new, case.v_new,
                       case.k_scale, case.v_scale)
    out = np.zeros((spec.total_q, spec.hq, spec.d), dtype=np.float64)
    lse = np.full((spec.hq, spec.total_q), -np.inf, dtype=np.float64)
    cu_q = spec.cu_q
    kv_lens = spec.kv_lens
    for b in range(spec.batch):
        lq, lk = int(spec.q_lens[b]), int(kv_lens[b])
        if lq == 0:
            continue
        K = gather_sequence(spec, kc, case.block_table, b, lk, case.k_scale)
        V = gather_sequence(spec, vc, case.block_table, b, lk, case.v_scale)
        q = query_values(case, case.q[cu_q[b]:cu_q[b] + lq])
        o, l = attend(q, K, V, spec.causal, spec.softmax_scale)
        out[cu_q[b]:cu_q[b] + lq] = o
        lse[:, cu_q[b]:cu_q[b] + lq] = l
    return {"out": out, "lse": lse, "k_cache": kc, "v_cache": vc}


def forward_rows(case, k_cache_after, v_cache_after, rows: Iterable[tuple[int, int]]):
    """Oracle output for selected query rows (b, i) only, from post-append caches.

    Used at full problem sizes, where computing every row would take too long:
    each sampled row is computed exactly as ``attend`` would (same mask, same
    softmax), with its own dense gather.  Returns (o (n, Hq, D), lse (Hq, n)).
    """
    spec = case.spec
    rows = list(rows)
    cu_q = spec.cu_q
    kv_lens = spec.kv_lens
    o = np.zeros((len(rows), spec.hq, spec.d))
    lse = np.zeros((spec.hq, len(rows)))
    cache = {}
    for n, (b, i) in enumerate(rows):
        lq, lk = int(spec.q_lens[b]), int(kv_lens[b])
        if b not in cache:
            cache = {b: (gather_sequence(spec, k_cache_after, case.block_table, b, lk, case.k_scale),
                         gather_sequence(spec, v_cache_after, case.block_table, b, lk, case.v_scale))}
        K, V = cache[b]
        # query i is row i of a length-lq block; keep its causal horizon exact
        horizon = i + (lk - lq) + 1 if spec.causal else lk
        horizon = max(0, min(lk, horizon))
        q = query_values(case, case.q[cu_q[b] + i:cu_q[b] + i + 1])
        oi, li = attend(q, K[:horizon], V[:horizon], False, spec.softmax_scale)
        if horizon == 0:
            oi[:] = 0.0
            li[:] = -np.inf
        o[n] = oi[0]
        lse[:, n] = li[:, 0]
    return o, lse


def combine_partials(o_parts: np.ndarray, lse_parts: np.ndarray):
    """Merge attention over disjoint key chunks (split-KV).

    Each chunk i gives a normalised output o_i and its log-sum-exp lse_i; the
    result over the union of the chunks is
        lse = lse* + ln sum_i exp(lse_i - lse*),   lse* = max_i lse_i,
        o   = sum_i exp(lse_i - lse) o_i.
    FA2 page, Limitation / review (num_splits and split-KV for decoding) name
    the technique; this merge rule is the standard one it relies on.
    o_parts: (S, ..., D); lse_parts: (S, ...).  Chunks with lse = -inf (no
    visible key) get weight 0; if every chunk is empty the row is o = 0,
    lse = -inf.
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    m = np.max(lse_parts, axis=0)
    finite = np.isfinite(m)
    m_safe = np.where(finite, m, 0.0)
    w = np.exp(lse_parts - m_safe[None])
    w = np.where(np.isfinite(lse_parts), w, 0.0)
    tot = w.sum(axis=0)
    lse = np.where(finite, m_safe + np.log(np.where(finite, tot, 1.0)), -np.inf)
    wn = np.divide(w, tot[None], out=np.zeros_like(w), where=finite[None])
    o = np.sum(wn[..., None] * o_parts, axis=0)
    return o, lse


def split_forward(q, K, V, causal, scale, bounds):
    """Attention of one sequence computed chunk by chunk over keys [bounds[k],
    bounds[k+1]) and merged with ``combine_partials`` (used to pin the merge)."""
    lq, lk = q.shape[0], K.shape[0]
    mask = visible_mask(lq, lk, causal)
    o_parts, l_parts = [], []
    hq = q.shape[1]
    hkv = K.shape[1]
    g = hq // hkv
    for a, z in zip(bounds[:-1], bounds[1:]):
        o = np.zeros_like(q, dtype=np.float64)
        lse = np.full((hq, lq), -np.inf)
        for h in range(hq):
            hk = h // g
            s = (q[:, h, :] @ K[a:z, hk, :].T) * float(scale)
            s = np.where(mask[:, a:z], s, -np.inf)
            vis = mask[:, a:z].any(axis=1)
            m = np.where(vis, np.max(s, axis=1, initial=-np.inf), 0.0)
            e = np.exp(s - m[:, None])
            den = e.sum(axis=1)
            w = np.divide(e, den[:, None], out=np.zeros_like(e), where=vis[:, None])
            o[:, h] = w @ V[a:z, hk]
            lse[h] = np.where(vis, m + np.log(np.where(vis, den, 1.0)), -np.inf)
        o_parts.append(o)
        l_parts.append(lse)
    o, lse = combine_partials(np.stack(o_parts), np.stack([lp.T for lp in l_parts]))
    return o, lse.T


# ---------------------------------------------------------------------------
# algorithmic work (what a launch must at least move / compute)
# ---------------------------------------------------------------------------
def algorithmic_work(spec, with_new: bool = True) -> dict:
    """Bytes and flops a call must move / compute, counting valid tokens only.

    bytes: K and V of every attended token (cache element size), Q read and O
    write (bf16), new K/V read (bf16) and written (cache element size), block
    table entries used.  flops: 4 * D * Hq per visible (query, key) pair.
    """
    esz = 2 if spec.cache_dtype == "bf16" else 1
    lk = spec.kv_lens.astype(np.int64)
    lq = spec.q_lens.astype(np.int64)
    kv_read = int(lk.sum()) * spec.hkv * spec.d * 2 * esz
    q_o = int(lq.sum()) * spec.hq * spec.d * 2 * 2
    new_rw = 0
    if with_new:
        new_rw = int(spec.new_lens.sum()) * spec.hkv * spec.d * 2 * (2 + esz)
    bt = 0
    if spec.page_size:
        bt = int(sum((int(n) + spec.page_size - 1) // spec.page_size for n in lk)) * 4
    pairs = 0
    for a, k in zip(lq, lk):
        a, k = int(a), int(k)
        if spec.causal:
            i = np.arange(a)
            pairs += int(np.clip(i + 1 + k - a, 0, k).sum())
        else:
            pairs += a * k
    flops = 4 * spec.d * spec.hq * pairs
    return {"kv_bytes": kv_read, "bytes": kv_read + q_o + new_rw + bt, "flops": flops,
            "pairs": pairs}
