"""Seeded synthetic inputs for attention over a batched, variable-length KV cache.

This module only *draws* inputs: sequence lengths, request order, page
permutations / block tables, and bf16 (or raw fp32) tensor values.  It holds
none of the attention method's arithmetic (no append, no quantisation, no
scores, no softmax), so that both the CPU oracle and the CUDA path can consume
the same inputs without sharing any of the computation.

Conventions (shared by both sides, stated once here):

* bf16 tensors are numpy ``uint16`` arrays of bit patterns; ``fp8`` caches are
  numpy ``uint8`` arrays of OCP e4m3 ("fn") codes.
* Packed queries ``q``: ``(total_q, Hq, D)``; new K/V: ``(total_new, Hkv, D)``.
* Paged cache: ``(num_pages, page_size, Hkv, D)`` with a ``block_table`` of
  shape ``(batch, max_pages)``; contiguous cache: ``(batch, capacity, Hkv, D)``.
* ``cache_lens[b]`` is the cache length *before* the new tokens are appended.

Value recipe: N(0,1) fp32 draws rounded to nearest-even bf16.  Draw order:
lengths -> request order -> page permutation -> Q -> K/V cache prefix ->
K/V new (every config, generator ``numpy.random.Generator(PCG64(seed))``).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import numpy as np

BF16_NAN = np.uint16(0x7FC0)
FP8_NAN = np.uint8(0x7F)
FP8_MAX_CODE = np.uint8(0x7E)  # +448, the finite sentinel used in fp8 caches
SENTINEL_VALUE = 1.0e4          # finite sentinel written into unused bf16 slots


# ---------------------------------------------------------------------------
# bf16 bit helpers (input construction only)
# ---------------------------------------------------------------------------
def f32_to_bf16_bits(x: np.ndarray, check_nan: bool = True) -> np.ndarray:
    """Round float32 values to the nearest bf16 (ties to even); return bits."""
    # finite and infinite inputs cannot overflow 32 bits here; NaNs are patched below
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    t = u >> 16
    t &= 1
    t += np.uint32(0x7FFF)
    t += u
    t >>= 16
    out = t.astype(np.uint16)
    del t
    if not check_nan:
        return out
    nan = np.isnan(np.asarray(x, dtype=np.float32))
    if nan.any():
        out = out.copy()
        out[nan] = BF16_NAN
    return out


def bf16_bits_to_f32(u: np.ndarray) -> np.ndarray:
    """Widen bf16 bit patterns to float32 (exact)."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_bits_of(value: float) -> np.uint16:
    return f32_to_bf16_bits(np.array([value], dtype=np.float32))[0]


# ---------------------------------------------------------------------------
# problem description
# ---------------------------------------------------------------------------
@dataclass
class Spec:
    """Shape and options of one attention-over-KV-cache call."""

    batch: int
    hq: int
    hkv: int
    d: int
    page_size: int              # 0 = contiguous cache
    causal: bool
    softmax_scale: float        # stored as the fp32 value both sides use
    cache_dtype: str            # "bf16" | "fp8"
    q_lens: np.ndarray          # int32 [batch]
    cache_lens: np.ndarray      # int32 [batch], length before append
    new_lens: np.ndarray        # int32 [batch], tokens appended by this call
    capacity: int               # tokens one sequence's cache can hold
    name: str = "case"

    @property
    def g(self) -> int:
        return self.hq // self.hkv

    @property
    def paged(self) -> bool:
        return self.page_size > 0

    @property
    def total_q(self) -> int:
        return int(self.q_lens.sum())

    @property
    def total_new(self) -> int:
        return int(self.new_lens.sum())

    @property
    def kv_lens(self) -> np.ndarray:
        return (self.cache_lens + self.new_lens).astype(np.int32)

    @property
    def cu_q(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.q_lens)]).astype(np.int32)

    @property
    def cu_new(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.new_lens)]).astype(np.int32)


@dataclass
class Case:
    """A full set of inputs: spec, tensors, page map and (fp8) scales.

    ``k_cache``/``v_cache`` are the physical caches *before* this call's append.
    For bf16 caches the cached prefix is already in place; for fp8 caches the
    prefix is left as raw bf16 values in ``prefix_k``/``prefix_v`` and each side
    writes it with its own append (quantisation is part of the method).
    """

    spec: Spec
    q: np.ndarray                        # uint16 (total_q, Hq, D)
    k_new: Optional[np.ndarray]          # uint16 (total_new, Hkv, D) or None
    v_new: Optional[np.ndarray]
    k_cache: np.ndarray                  # uint16 / uint8 physical cache
    v_cache: np.ndarray
    block_table: Optional[np.ndarray]    # int32 (batch, max_pages) or None
    num_pages: int = 0
    poison_page: int = -1                # page every padding entry points at
    prefix_k: Optional[np.ndarray] = None  # uint16 (sum cache_lens, Hkv, D), fp8 only
    prefix_v: Optional[np.ndarray] = None
    k_scale: float = 1.0                 # fp32 per-tensor scales (fp8 only)
    v_scale: float = 1.0
    q_scale: Optional[float] = None      # fp8 only: Q quantised to e4m3 for Q K^T with this scale
    sentinel: str = "finite"             # "finite" | "nan" fill of unused slots
    extra: dict = field(default_factory=dict)

    @property
    def cu_prefix(self) -> np.ndarray:
        return np.concatenate([[0], np.cumsum(self.spec.cache_lens)]).astype(np.int32)


# ---------------------------------------------------------------------------
# drawing helpers
# ---------------------------------------------------------------------------
def _normal_bf16(rng: np.random.Generator, shape, mult: float = 1.0) -> np.ndarray:
    x = rng.standard_normal(size=shape, dtype=np.float32)
    if mult != 1.0:
        x *= np.float32(mult)
    return f32_to_bf16_bits(x, check_nan=False)   # N(0,1) draws are never NaN


def _amax_scale(*bits: np.ndarray) -> float:
    """Per-tensor fp8 scale = amax(|x|)/448 computed in fp32 (input choice)."""
    amax = np.float32(0.0)
    for b in bits:
        if b is not None and b.size:
            amax = max(amax, np.max(np.abs(bf16_bits_to_f32(b))))
    if amax == 0:
        amax = np.float32(1.0)
    return float(np.float32(amax) / np.float32(448.0))


def _fill_code(cache_dtype: str, sentinel: str):
    if cache_dtype == "bf16":
        return BF16_NAN if sentinel == "nan" else bf16_bits_of(SENTINEL_VALUE)
    return FP8_NAN if sentinel == "nan" else FP8_MAX_CODE


def make_case(spec: Spec, rng: np.random.Generator, *, block_table_width: Optional[int] = None,
              explicit_block_table: Optional[np.ndarray] = None, num_pages: Optional[int] = None,
              with_new: bool = True, sentinel: str = "finite", q_mult: float = 1.0,
              page_perm: bool = True, draw_values: bool = True) -> Case:
    """Draw a case for ``spec`` (lengths already fixed in the spec).

    Paged pool: exactly the pages each sequence needs for ``cache_lens +
    new_lens`` tokens, plus one poison page, seeded-permuted; block-table
    padding points at the poison page (never an out-of-range index).
    """
    B, Hq, Hkv, D = spec.batch, spec.hq, spec.hkv, spec.d
    esize_dtype = np.uint16 if spec.cache_dtype == "bf16" else np.uint8
    fill = _fill_code(spec.cache_dtype, sentinel)
    kv_lens = spec.kv_lens
    if np.any(kv_lens > spec.capacity):
        raise ValueError("cache capacity too small for cache_lens + new_lens")

    block_table = None
    poison = -1
    if spec.paged:
        P = spec.page_size
        pages_needed = [(int(n) + P - 1) // P for n in kv_lens]
        width = block_table_width or max(1, (spec.capacity + P - 1) // P)
        if explicit_block_table is not None:
            block_table = np.ascontiguousarray(explicit_block_table, dtype=np.int32)
            npages = int(num_pages)
        else:
            total = int(sum(pages_needed))
            npages = total + 1
            perm = rng.permutation(npages).astype(np.int32) if page_perm else np.arange(npages, dtype=np.int32)
            poison = int(perm[total])
            block_table = np.full((B, width), poison, dtype=np.int32)
            off = 0
            for b in range(B):
                n = pages_needed[b]
                block_table[b, :n] = perm[off:off + n]
                off += n
        cache_shape = (npages, P, Hkv, D)
    else:
        npages = 0
        cache_shape = (B, spec.capacity, Hkv, D)

    if not draw_values:   # lengths and page map only (host scheduling tests)
        return Case(spec=spec, q=None, k_new=None, v_new=None, k_cache=None, v_cache=None,
                    block_table=block_table, num_pages=npages, poison_page=poison, sentinel=sentinel)
    q = _normal_bf16(rng, (spec.total_q, Hq, D), q_mult)
    total_prefix = int(spec.cache_lens.sum())
    prefix_k = _normal_bf16(rng, (total_prefix, Hkv, D))
    prefix_v = _normal_bf16(rng, (total_prefix, Hkv, D))
    k_new = v_new = None
    if with_new:
        k_new = _normal_bf16(rng, (spec.total_new, Hkv, D))
        v_new = _normal_bf16(rng, (spec.total_new, Hkv, D))

    k_cache = np.full(cache_shape, fill, dtype=esize_dtype)
    v_cache = np.full(cache_shape, fill, dtype=esize_dtype)
    case = Case(spec=spec, q=q, k_new=k_new, v_new=v_new, k_cache=k_cache, v_cache=v_cache,
                block_table=block_table, num_pages=npages, poison_page=poison,
                sentinel=sentinel)
    if spec.cache_dtype == "bf16":
        place_prefix(case, prefix_k, prefix_v)
    else:
        case.prefix_k, case.prefix_v = prefix_k, prefix_v
        case.k_scale = _amax_scale(prefix_k, k_new)
        case.v_scale = _amax_scale(prefix_v, v_new)
    return case


def place_prefix(case: Case, prefix_k: np.ndarray, prefix_v: np.ndarray) -> None:
    """Copy logical bf16 prefix rows into the physical cache (pure indexing)."""
    spec = case.spec
    cu = case.cu_prefix
    for b in range(spec.batch):
        n = int(spec.cache_lens[b])
        if n == 0:
            continue
        pos = np.arange(n)
        if spec.paged:
            P = spec.page_size
            pages = case.block_table[b, pos // P]
            case.k_cache[pages, pos % P] = prefix_k[cu[b]:cu[b] + n]
            case.v_cache[pages, pos % P] = prefix_v[cu[b]:cu[b] + n]
        else:
            case.k_cache[b, :n] = prefix_k[cu[b]:cu[b] + n]
            case.v_cache[b, :n] = prefix_v[cu[b]:cu[b] + n]


def to_contiguous(case: Case) -> Case:
    """Same logical content as ``case`` with a contiguous cache (bf16 only).

    Used to pin paged == contiguous; a pure re-indexing of the physical cache.
    """
    spec = case.spec
    assert spec.paged and spec.cache_dtype == "bf16"
    cap = spec.capacity
    cspec = Spec(**{**spec.__dict__, "page_size": 0, "name": spec.name + "-contig"})
    fill = _fill_code("bf16", case.sentinel)
    kc = np.full((spec.batch, cap, spec.hkv, spec.d), fill, dtype=np.uint16)
    vc = np.full_like(kc, fill)
    P = spec.page_size
    for b in range(spec.batch):
        n = int(spec.cache_lens[b])
        pos = np.arange(n)
        pages = case.block_table[b, pos // P]
        kc[b, :n] = case.k_cache[pages, pos % P]
        vc[b, :n] = case.v_cache[pages, pos % P]
    return Case(spec=cspec, q=case.q, k_new=case.k_new, v_new=case.v_new, k_cache=kc, v_cache=vc,
                block_table=None, sentinel=case.sentinel)


def relabel_pages(case: Case, rng: np.random.Generator) -> Case:
    """Apply a random physical relabelling of the page pool (bf16 only)."""
    spec = case.spec
    assert spec.paged
    perm = rng.permutation(case.num_pages).astype(np.int32)  # old page p -> new perm[p]
    kc = np.empty_like(case.k_cache)
    vc = np.empty_like(case.v_cache)
    kc[perm] = case.k_cache
    vc[perm] = case.v_cache
    return Case(spec=spec, q=case.q, k_new=case.k_new, v_new=case.v_new, k_cache=kc, v_cache=vc,
                block_table=perm[case.block_table], num_pages=case.num_pages,
                poison_page=int(perm[case.poison_page]) if case.poison_page >= 0 else -1,
                prefix_k=case.prefix_k, prefix_v=case.prefix_v, k_scale=case.k_scale,
                v_scale=case.v_scale, sentinel=case.sentinel)


# ---------------------------------------------------------------------------
# the five workloads (sizes as stated for the method's benchmark configs)
# ---------------------------------------------------------------------------
def _scale(d: int) -> float:
    return float(np.float32(1.0 / math.sqrt(d)))


def config1(sentinel: str = "finite") -> Case:
    """Tiny paged GQA case: B=2, Hq=4, Hkv=2, D=64, P=16, cache lens {37,5},
    new tokens {3,1}, 8-page pool with block_table = permutation(8) as (2,4)."""
    rng = np.random.Generator(np.random.PCG64(1001))
    spec = Spec(batch=2, hq=4, hkv=2, d=64, page_size=16, causal=True, softmax_scale=_scale(64),
                cache_dtype="bf16", q_lens=np.array([3, 1], np.int32),
                cache_lens=np.array([37, 5], np.int32), new_lens=np.array([3, 1], np.int32),
                capacity=64, name="cfg1-tiny-paged")
    bt = rng.permutation(8).astype(np.int32).reshape(2, 4)
    return make_case(spec, rng, explicit_block_table=bt, num_pages=8, sentinel=sentinel)


def config2(sentinel: str = "finite", draw_values: bool = True) -> Case:
    """Decode: B=64, 1 query/new token each, Hq=32, Hkv=8, D=128, cache lens
    U[512,4096], paged P=16, block_table width 257."""
    rng = np.random.Generator(np.random.PCG64(1002))
    B = 64
    lc = rng.integers(512, 4096, size=B, endpoint=True).astype(np.int32)
    ones = np.ones(B, np.int32)
    spec = Spec(batch=B, hq=32, hkv=8, d=128, page_size=16, causal=True, softmax_scale=_scale(128),
                cache_dtype="bf16", q_lens=ones, cache_lens=lc, new_lens=ones.copy(),
                capacity=257 * 16, name="cfg2-decode-paged")
    return make_case(spec, rng, block_table_width=257, sentinel=sentinel, draw_values=draw_values)


def config3(causal: bool = True, sentinel: str = "finite", draw_values: bool = True) -> Case:
    """Prefill with a cached prefix, contiguous cache (8, 2048, 8, 128):
    B=8, 512 new q/k/v tokens on a 1536-token prefix, Hq=32, Hkv=8, D=128."""
    rng = np.random.Generator(np.random.PCG64(1003))
    B = 8
    n = np.full(B, 512, np.int32)
    spec = Spec(batch=B, hq=32, hkv=8, d=128, page_size=0, causal=causal, softmax_scale=_scale(128),
                cache_dtype="bf16", q_lens=n, cache_lens=np.full(B, 1536, np.int32), new_lens=n.copy(),
                capacity=2048, name="cfg3-prefill-contig-" + ("causal" if causal else "noncausal"))
    return make_case(spec, rng, sentinel=sentinel, draw_values=draw_values)


def config4(sentinel: str = "finite", draw_values: bool = True) -> Case:
    """Mixed in-flight batch, paged P=16: 64 requests in seeded order = 60 decode
    (1 token, cache len U[1024,8192]) + 4 prefill (2048 tokens on a U[0,2048]
    prefix); Hq=32, Hkv=8, D=128, causal; block_table width 513."""
    rng = np.random.Generator(np.random.PCG64(1004))
    dec_lc = rng.integers(1024, 8192, size=60, endpoint=True)
    pre_lc = rng.integers(0, 2048, size=4, endpoint=True)
    lc = np.concatenate([dec_lc, pre_lc]).astype(np.int32)
    lq = np.concatenate([np.ones(60), np.full(4, 2048)]).astype(np.int32)
    order = rng.permutation(64)
    lc, lq = lc[order], lq[order]
    spec = Spec(batch=64, hq=32, hkv=8, d=128, page_size=16, causal=True, softmax_scale=_scale(128),
                cache_dtype="bf16", q_lens=lq, cache_lens=lc, new_lens=lq.copy(),
                capacity=513 * 16, name="cfg4-mixed-paged")
    return make_case(spec, rng, block_table_width=513, sentinel=sentinel, draw_values=draw_values)


def config5(sentinel: str = "finite", batch: int = 64, seqlen: int = 2048) -> tuple[Case, Case]:
    """FP8-e4m3 paged cache (P=16, 129 pages per sequence): a causal prefill of
    ``seqlen`` tokens into an empty cache, then one decode token (kv len
    seqlen+1).  Per-tensor scales come from all seqlen+1 tokens' K (resp. V).

    Returns (prefill_case, decode_case).  The decode case's cache starts as the
    sentinel-filled pool: each side runs the prefill append first.
    """
    rng = np.random.Generator(np.random.PCG64(1005))
    B, L = batch, seqlen
    P = 16
    width = (L + 1 + P - 1) // P
    pre_spec = Spec(batch=B, hq=32, hkv=8, d=128, page_size=P, causal=True, softmax_scale=_scale(128),
                    cache_dtype="fp8", q_lens=np.full(B, L, np.int32), cache_lens=np.zeros(B, np.int32),
                    new_lens=np.full(B, L, np.int32), capacity=width * P, name="cfg5a-fp8-prefill")
    # pool sized for the decode step (L+1 tokens per sequence)
    pages_per_seq = width
    total = B * pages_per_seq
    perm = rng.permutation(total + 1).astype(np.int32)
    poison = int(perm[total])
    bt = perm[:total].reshape(B, pages_per_seq).copy()
    q_pre = _normal_bf16(rng, (B * L, 32, 128))
    k_all = _normal_bf16(rng, (B, L + 1, 8, 128))
    v_all = _normal_bf16(rng, (B, L + 1, 8, 128))
    q_dec = _normal_bf16(rng, (B, 32, 128))
    k_scale = _amax_scale(k_all)
    v_scale = _amax_scale(v_all)
    fill = _fill_code("fp8", sentinel)
    shape = (total + 1, P, 8, 128)
    pre = Case(spec=pre_spec, q=q_pre, k_new=np.ascontiguousarray(k_all[:, :L].reshape(B * L, 8, 128)),
               v_new=np.ascontiguousarray(v_all[:, :L].reshape(B * L, 8, 128)),
               k_cache=np.full(shape, fill, np.uint8), v_cache=np.full(shape, fill, np.uint8),
               block_table=bt, num_pages=total + 1, poison_page=poison,
               k_scale=k_scale, v_scale=v_scale, sentinel=sentinel)
    dec_spec = Spec(**{**pre_spec.__dict__, "q_lens": np.ones(B, np.int32),
                       "cache_lens": np.full(B, L, np.int32), "new_lens": np.ones(B, np.int32),
                       "name": "cfg5b-fp8-decode"})
    dec = Case(spec=dec_spec, q=q_dec, k_new=np.ascontiguousarray(k_all[:, L]),
               v_new=np.ascontiguousarray(v_all[:, L]), k_cache=pre.k_cache.copy(),
               v_cache=pre.v_cache.copy(), block_table=bt, num_pages=total + 1, poison_page=poison,
               prefix_k=pre.k_new, prefix_v=pre.v_new, k_scale=k_scale, v_scale=v_scale,
               sentinel=sentinel)
    return pre, dec


def random_case(seed: int, *, batch=None, hq=None, hkv=None, d=None, page_size=None, causal=None,
                cache_dtype="bf16", max_cache=40, max_new=8, with_new=True, sentinel="finite",
                q_equals_new=True, allow_zero=True) -> Case:
    """Small random case for property tests (all knobs seeded)."""
    rng = np.random.Generator(np.random.PCG64(seed))
    B = batch or int(rng.integers(1, 4))
    hkv_ = hkv or int(rng.choice([1, 2]))
    g = int(rng.choice([1, 2, 4]))
    hq_ = hq or hkv_ * g
    d_ = d or int(rng.choice([8, 16]))
    P = int(rng.choice([0, 1, 4, 16])) if page_size is None else page_size
    causal_ = bool(rng.integers(0, 2)) if causal is None else causal
    lo = 0 if allow_zero else 1
    lc = rng.integers(lo, max_cache + 1, size=B).astype(np.int32)
    ln = rng.integers(lo, max_new + 1, size=B).astype(np.int32) if with_new else np.zeros(B, np.int32)
    if q_equals_new and with_new:
        lq = ln.copy()
    else:
        lq = rng.integers(lo, max_new + 1, size=B).astype(np.int32)
    cap = int((lc + ln).max()) + int(rng.integers(0, 5))
    cap = max(cap, 1)
    if P:
        cap = ((cap + P - 1) // P) * P
    spec = Spec(batch=B, hq=hq_, hkv=hkv_, d=d_, page_size=P, causal=causal_,
                softmax_scale=float(np.float32(1.0 / math.sqrt(d_))), cache_dtype=cache_dtype,
                q_lens=lq, cache_lens=lc, new_lens=ln, capacity=cap, name=f"rand{seed}")
    return make_case(spec, rng, with_new=with_new, sentinel=sentinel)


def uniform_spec(name: str, batch: int, q_len: int, cache_len: int, *, hq=32, hkv=8, d=128,
                 page_size=16, causal=True, cache_dtype="bf16", capacity=None) -> Spec:
    """Equal-length batch (parity sweeps): every sequence has the same lengths."""
    cap = capacity or (cache_len + q_len)
    if page_size:
        cap = ((cap + page_size - 1) // page_size) * page_size
    return Spec(batch=batch, hq=hq, hkv=hkv, d=d, page_size=page_size, causal=causal,
                softmax_scale=float(np.float32(1.0 / math.sqrt(d))), cache_dtype=cache_dtype,
                q_lens=np.full(batch, q_len, np.int32), cache_lens=np.full(batch, cache_len, np.int32),
                new_lens=np.full(batch, q_len, np.int32), capacity=cap, name=name)


def subset_case(case: Case, seqs) -> Case:
    """The same inputs restricted to sequences ``seqs`` (pure indexing): used
    to check sampled sequences of a full-size workload against the oracle."""
    spec = case.spec
    seqs = [int(s) for s in seqs]
    cu_q, cu_n, cu_p = spec.cu_q, spec.cu_new, case.cu_prefix
    take = lambda arr, cu: (None if arr is None else
                            np.concatenate([arr[cu[b]:cu[b + 1]] for b in seqs], axis=0))
    sub = Spec(**{**spec.__dict__, "batch": len(seqs), "q_lens": spec.q_lens[seqs].copy(),
                  "cache_lens": spec.cache_lens[seqs].copy(), "new_lens": spec.new_lens[seqs].copy(),
                  "name": spec.name + "-subset"})
    num_pages, poison = case.num_pages, case.poison_page
    if spec.paged:
        # keep only the pages these sequences reference, renumbered in order
        rows = case.block_table[seqs]
        used = np.unique(rows)
        kc, vc = case.k_cache[used], case.v_cache[used]
        bt = np.searchsorted(used, rows).astype(np.int32)
        num_pages = int(used.size)
        poison = int(np.searchsorted(used, poison)) if poison in used else -1
    else:
        kc, vc, bt = case.k_cache[seqs].copy(), case.v_cache[seqs].copy(), None
    return Case(spec=sub, q=take(case.q, cu_q), k_new=take(case.k_new, cu_n), v_new=take(case.v_new, cu_n),
                k_cache=kc, v_cache=vc, block_table=bt, num_pages=num_pages, poison_page=poison,
                prefix_k=take(case.prefix_k, cu_p), prefix_v=take(case.prefix_v, cu_p), k_scale=case.k_scale,
                v_scale=case.v_scale, sentinel=case.sentinel)
