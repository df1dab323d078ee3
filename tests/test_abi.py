"""Host-side tests of the C ABI (no GPU): the library loads and exports every
symbol the header declares, host validation returns its status codes before
anything is launched, and the plan's work list covers every query row and key
exactly as the method requires."""
import ctypes
import os
import re

import numpy as np
import pytest

import synth

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def pkv():
    import paged_kv_variable_gb300 as m
    from paged_kv_variable_gb300 import build as b
    b.build()
    m.lib()
    return m


def _declared_symbols():
    text = open(os.path.join(ROOT, "include", "pkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(pkv_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(pkv):
    names = _declared_symbols()
    assert names, "no declarations found"
    assert sorted(names) == sorted(pkv.EXPORTED)
    for n in names:
        assert hasattr(pkv.lib(), n), n
    assert "sm_103a" in pkv.version()


def _problem(pkv, **kw):
    base = dict(batch=2, num_heads_q=4, num_heads_kv=2, head_dim=64, page_size=16, cache_capacity=64,
                num_pages=8, cache_dtype="bf16", causal=True, softmax_scale=0.125)
    base.update(kw)
    return pkv.make_problem(**base)


@pytest.mark.parametrize("kw,status", [
    (dict(num_heads_q=6, num_heads_kv=4), 1),
    (dict(head_dim=96), 2),
    (dict(head_dim=512), 2),
    (dict(page_size=3), 2),
    (dict(page_size=12), 2),
    (dict(page_size=512), 2),
    (dict(cache_capacity=0), 1),
    (dict(cache_capacity=40), 1),   # not a multiple of the page size
    (dict(softmax_scale=0.0), 1),
    (dict(softmax_scale=float("nan")), 1),
])
def test_plan_rejects_bad_problems(pkv, kw, status):
    with pytest.raises(pkv.PkvError) as e:
        pkv.plan(_problem(pkv, **kw), [1, 1], [3, 3], [1, 1], num_sms=4)
    assert e.value.status == status
    assert pkv.last_error()


def test_plan_rejects_overflowing_lengths(pkv):
    with pytest.raises(pkv.PkvError) as e:
        pkv.plan(_problem(pkv), [1, 1], [64, 3], [1, 1], num_sms=4)
    assert e.value.status == 1 and "capacity" in pkv.last_error()
    with pytest.raises(pkv.PkvError):
        pkv.plan(_problem(pkv), [1, -1], [3, 3], [1, 1], num_sms=4)


def _coverage(spec, items, num_sms):
    """Every (seq, query head, query token) is covered by exactly the tiles
    whose key ranges tile [0, limit) of that row without overlap."""
    G = spec.hq // spec.hkv
    cov = {}
    for it in items:
        b, hk = it["seq"], it["kv_head"]
        # (decode-only plans over an fp8 cache at head_dim <= 128: two CTAs an SM)
        two = spec.d <= 128 if spec.cache_dtype == "fp8" else spec.d == 64   # rows of 128 bytes or fewer
        cps = 2 if two and all(x["kind"] == 0 for x in items) else 1
        assert 0 <= it["cta"] < num_sms * cps
        assert it["kv_begin"] % 128 == 0 or it["kv_begin"] == it["kv_end"]
        assert 0 <= it["head0"] and it["head0"] + it["num_heads"] <= G
        for t in range(it["n_q"]):
            i = it["q_index0"] + t
            for h in range(it["head0"], it["head0"] + it["num_heads"]):
                cov.setdefault((b, hk * G + h, i), []).append((it["kv_begin"], it["kv_end"], it["partial_slot"]))
        rows = it["n_q"] * it["num_heads"]
        if it["kind"] == 0:
            assert rows <= 16 and it["num_heads"] == G
        else:
            # a tensor-core item holds two 128-row query tiles over an fp8 cache
            # at head_dim <= 128 in a plan without decode tiles (one when it is a
            # split-KV chunk), else one
            pairs = spec.d <= 128 and spec.cache_dtype == "fp8" and not any(x["kind"] == 0 for x in items)
            q_tiles = 2 if pairs and it["partial_slot"] < 0 else 1
            assert rows <= 128 * q_tiles and it["num_heads"] == min(128, G - it["head0"])
    for b in range(spec.batch):
        lq, lk = int(spec.q_lens[b]), int(spec.kv_lens[b])
        for hq in range(spec.hq):
            for i in range(lq):
                ranges = sorted(cov.pop((b, hq, i)))
                # ranges are disjoint, start at 0 and reach at least the row's horizon
                horizon = min(lk, i + lk - lq + 1) if spec.causal else lk
                pos = 0
                for a, z, _ in ranges:
                    assert a == pos
                    pos = z
                assert pos >= max(0, horizon) and pos <= lk
                if len(ranges) > 1:
                    assert all(s >= 0 for _, _, s in ranges)
                else:
                    assert ranges[0][2] == -1
    assert not cov


@pytest.mark.parametrize("which", ["cfg1", "cfg2", "cfg3", "cfg4", "rand", "mqa32", "g48", "g71", "g256", "g6"])
def test_plan_covers_every_row(pkv, which):
    wide = {"mqa32": (32, 1), "g48": (96, 2), "g71": (71, 1), "g256": (256, 1), "g6": (12, 2)}
    if which in wide:
        hq, hkv = wide[which]
        rng = np.random.default_rng(hq)
        case = synth.random_case(hq, batch=6, hq=hq, hkv=hkv, d=128, page_size=16, max_cache=3000, max_new=300,
                                 causal=True)
    elif which == "cfg1":
        case = synth.config1()
    elif which == "cfg2":
        case = synth.config2(draw_values=False)
    elif which == "cfg3":
        case = synth.config3(draw_values=False)
    elif which == "cfg4":
        case = synth.config4(draw_values=False)
    elif which == "rand":
        case = synth.random_case(7, batch=5, hq=8, hkv=2, d=128, page_size=16, max_cache=900, max_new=70)
    spec = case.spec
    prob = pkv.make_problem(batch=spec.batch, num_heads_q=spec.hq, num_heads_kv=spec.hkv, head_dim=spec.d,
                            page_size=spec.page_size, cache_capacity=spec.capacity,
                            num_pages=max(1, case.num_pages if spec.paged else spec.batch),
                            cache_dtype=spec.cache_dtype, causal=spec.causal, softmax_scale=spec.softmax_scale)
    for sms in (1, 13, 152):
        pl = pkv.plan(prob, spec.q_lens, spec.cache_lens, spec.new_lens, num_sms=sms)
        items = pl.items()
        st = pl.stats()
        assert st["num_items"] == len(items)
        assert st["total_q"] == spec.total_q and st["total_new"] == spec.total_new
        _coverage(spec, items, sms)
        if sms == 152 and which in ("cfg2", "cfg4"):
            assert st["num_ctas"] == 152
            assert st["max_cta_cost"] <= 1.15 * st["mean_cta_cost"]


def test_plan_accepts_zero_lengths(pkv):
    # zero kv length (a failure case reported for another scheduler) and zero query length
    prob = _problem(pkv, batch=3)
    pl = pkv.plan(prob, [2, 0, 1], [0, 5, 0], [0, 0, 1], num_sms=4)
    items = pl.items()
    assert sum(1 for it in items if it["seq"] == 1) == 0
    zero = [it for it in items if it["seq"] == 0]
    assert zero and all(it["kv_begin"] == it["kv_end"] == 0 for it in zero)


def test_dynamic_plan_decode_only(pkv):
    """A dynamic plan schedules decode units for the bounds and refuses
    requests whose queries need more than one tile."""
    spec = synth.config2(draw_values=False).spec
    prob = pkv.make_problem(batch=spec.batch, num_heads_q=spec.hq, num_heads_kv=spec.hkv, head_dim=spec.d,
                            page_size=spec.page_size, cache_capacity=spec.capacity, num_pages=100000,
                            cache_dtype=spec.cache_dtype, causal=spec.causal, softmax_scale=spec.softmax_scale)
    bounds = np.minimum(spec.cache_lens + 64, spec.capacity - 1).astype(np.int32)
    dyn = pkv.plan_decode_dynamic(prob, spec.q_lens, bounds, spec.new_lens, num_sms=152)
    fixed = pkv.plan(prob, spec.q_lens, bounds, spec.new_lens, num_sms=152)
    # the same work list as a plan for the bounds themselves
    assert dyn.items() == fixed.items() and dyn.workspace_bytes == fixed.workspace_bytes
    # queries of one request beyond one tensor-core tile (128 rows / G = 64 tokens at G = 2)
    with pytest.raises(pkv.PkvError) as e:
        pkv.plan_decode_dynamic(_problem(pkv, batch=2, cache_capacity=256), [1, 65], [3, 3], [1, 65], num_sms=4)
    assert e.value.status == 2 and "dynamic" in pkv.last_error()
    # a short query run that fits one tile is accepted
    pkv.plan_decode_dynamic(_problem(pkv, batch=2, cache_capacity=256), [1, 9], [3, 3], [1, 9], num_sms=4)


def test_empty_batch(pkv):
    pl = pkv.plan(_problem(pkv, batch=0), np.zeros(0, np.int32), np.zeros(0, np.int32), None, num_sms=4)
    assert pl.stats()["num_items"] == 0


class _FakeTensor:
    def __init__(self, ptr, shape, strides=None, esize=2):
        self._ptr, self.shape, self._esize = ptr, shape, esize
        if strides is None:
            strides, acc = [], 1
            for s in reversed(shape):
                strides.insert(0, acc)
                acc *= s
        self._strides = strides

    def data_ptr(self):
        return self._ptr

    def stride(self, i):
        return self._strides[i]

    def numel(self):
        return int(np.prod(self.shape))

    def dim(self):
        return len(self.shape)

    def element_size(self):
        return self._esize


def test_fwd_validation_before_any_launch(pkv):
    prob = _problem(pkv)
    pl = pkv.plan(prob, [3, 1], [37, 5], [3, 1], num_sms=4)
    ws = _FakeTensor(4096 * 256, (pl.workspace_bytes,), esize=1)
    q = _FakeTensor(1 << 20, (4, 4, 64))
    kc = _FakeTensor(1 << 24, (8, 16, 2, 64))
    i32 = _FakeTensor(1 << 16, (3,), esize=4)
    bt = _FakeTensor(1 << 17, (2, 4), esize=4)
    good = dict(q=q, out=q, cu_seqlens_q=i32, max_seqlen_q=3, k_cache=kc, v_cache=kc, cache_seqlens=i32,
                k_new=q, v_new=q, cu_seqlens_knew=i32, block_table=bt)

    def call(**over):
        kw = dict(good)
        kw.update(over)
        with pytest.raises(pkv.PkvError) as e:
            pkv.attn_varlen_kvcache_fwd(prob, pkv.make_args(**kw), pl, ws, stream=0)
        return e.value.status

    assert call(block_table=None) == 1
    assert call(k_cache=_FakeTensor((1 << 24) + 2, (8, 16, 2, 64))) == 1          # misaligned
    assert call(k_new=None, v_new=None, cu_seqlens_knew=None) == 1                  # plan expects new tokens
    assert call(q=_FakeTensor(1 << 20, (4, 4, 64), strides=[256, 66, 1])) == 1      # stride not 16 B multiple
    assert call(q_scale=i32) == 2      # quantised queries need an fp8 cache
    assert call(q_rows=3) == 1         # fewer q / out rows than the plan's 4 query rows
    assert call(q_rows=-1) == 1
    small = _FakeTensor(4096 * 256, (pl.workspace_bytes - 256,), esize=1)
    with pytest.raises(pkv.PkvError) as e:
        pkv.attn_varlen_kvcache_fwd(prob, pkv.make_args(**good), pl, small, stream=0)
    assert e.value.status == 3
    other = _problem(pkv, causal=False)
    with pytest.raises(pkv.PkvError) as e:
        pkv.attn_varlen_kvcache_fwd(other, pkv.make_args(**good), pl, ws, stream=0)
    assert e.value.status == 1
    fp8 = _problem(pkv, cache_dtype="fp8", head_dim=128)
    with pytest.raises(pkv.PkvError) as e:
        pkv.kv_append(fp8, pkv.make_args(**good), 4, None, stream=0)   # no scales
    assert e.value.status == 1


# ------------------------------------------------------------------ longest-processing-time assignment
def _lpt_heap(items, num_ctas):
    """Reference assignment with heapq: tiles in the plan's generation order
    (sequence, kv head, query tile, key chunk), stably sorted longest first,
    each given to the least-loaded CTA (ties: the lowest index); a CTA runs
    its tiles in the order it received them."""
    import heapq
    key = lambda it: (it["seq"], it["kv_head"], it["q_index0"], it["kv_begin"])
    gen = sorted(items, key=key)
    order = sorted(range(len(gen)), key=lambda k: -gen[k]["cost"])   # sorted() is stable
    heap = [(0.0, c) for c in range(num_ctas)]
    heapq.heapify(heap)
    lists = [[] for _ in range(num_ctas)]
    for k in order:
        load, c = heapq.heappop(heap)
        lists[c].append(key(gen[k]))
        heapq.heappush(heap, (load + gen[k]["cost"], c))
    return lists


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("sms", [1, 13, 152])
def test_plan_assignment_is_lpt(pkv, seed, sms):
    """The work list equals a heapq LPT over the plan's own tile costs, CTA by
    CTA and item by item (random mixed batches: decode units, split chunks,
    prefill tiles, zero lengths)."""
    rng = np.random.default_rng(seed)
    B = int(rng.integers(3, 40))
    lq = np.where(rng.random(B) < 0.7, 1, rng.integers(0, 700, B)).astype(np.int32)
    lc = rng.integers(0, 6000, B).astype(np.int32)
    cap = int((lc + lq).max() + 16) // 16 * 16 + 16
    prob = pkv.make_problem(batch=B, num_heads_q=8 * int(rng.choice([1, 2, 4])), num_heads_kv=8, head_dim=128,
                            page_size=16, cache_capacity=cap, num_pages=100000, cache_dtype="bf16", causal=True,
                            softmax_scale=0.088)
    pl = pkv.plan(prob, lq, lc, lq, num_sms=sms)
    items = pl.items()
    n_ctas = pl.stats()["num_ctas"]
    assert n_ctas == min(sms, len(items))
    got = [[] for _ in range(n_ctas)]
    for it in items:
        got[it["cta"]].append((it["seq"], it["kv_head"], it["q_index0"], it["kv_begin"]))
    assert got == _lpt_heap(items, n_ctas)


# ------------------------------------------------------------------ no-workspace entry point (host checks)
def test_noalloc_rejects_before_touching_its_scratch(pkv):
    """Host checks of the workspace-free call run before its fixed device
    array is resolved or written: a bad argument, or a plan needing more than
    the array's 32 MiB, is refused with no CUDA call at all (this test runs
    without a GPU)."""
    B, hkv, lk = 64, 8, 8191
    prob = pkv.make_problem(batch=B, num_heads_q=32, num_heads_kv=hkv, head_dim=128, page_size=16,
                            cache_capacity=8192, num_pages=B * 512, cache_dtype="bf16", causal=True,
                            softmax_scale=0.088)
    ones = np.ones(B, np.int32)
    big = pkv.plan(prob, ones, np.full(B, lk, np.int32), ones, num_sms=4096)   # 512-key chunks: many partials
    assert big.workspace_bytes > 32 << 20
    q = _FakeTensor(1 << 20, (B, 32, 128))
    kc = _FakeTensor(1 << 24, (B * 512, 16, hkv, 128))
    i32 = _FakeTensor(1 << 16, (B + 1,), esize=4)
    bt = _FakeTensor(1 << 17, (B, 512), esize=4)
    kn = _FakeTensor(1 << 18, (B, hkv, 128))
    good = dict(q=q, out=q, cu_seqlens_q=i32, max_seqlen_q=1, k_cache=kc, v_cache=kc, cache_seqlens=i32,
                k_new=kn, v_new=kn, cu_seqlens_knew=i32, block_table=bt)
    with pytest.raises(pkv.PkvError) as e:
        pkv.attn_varlen_kvcache_fwd_noalloc(prob, pkv.make_args(**good), big, stream=0)
    assert e.value.status == 3 and "fixed scratch" in pkv.last_error()
    small = pkv.plan(prob, ones, np.full(B, 100, np.int32), ones, num_sms=152)
    assert small.workspace_bytes <= 32 << 20
    bad = dict(good, block_table=None)
    with pytest.raises(pkv.PkvError) as e:
        pkv.attn_varlen_kvcache_fwd_noalloc(prob, pkv.make_args(**bad), small, stream=0)
    assert e.value.status == 1 and "block_table" in pkv.last_error()
    with pytest.raises(pkv.PkvError) as e:       # new tokens missing: caught before any copy
        pkv.attn_varlen_kvcache_fwd_noalloc(prob, pkv.make_args(**dict(good, k_new=None, v_new=None)), small,
                                            stream=0)
    assert e.value.status == 1


@pytest.mark.parametrize("hq,hkv", [(32, 1), (64, 2), (200, 1), (256, 2)])
def test_wide_groups_plan(pkv, hq, hkv):
    """Groups of more than 16 heads: decode steps become tensor-core tiles of
    the whole group (split along the keys when long); groups of more than 128
    heads are cut into sub-groups of 128; a dynamic plan accepts them."""
    G = hq // hkv
    B = 5
    prob = pkv.make_problem(batch=B, num_heads_q=hq, num_heads_kv=hkv, head_dim=128, page_size=16,
                            cache_capacity=16384, num_pages=100000, cache_dtype="bf16", causal=True,
                            softmax_scale=0.088)
    ones = np.ones(B, np.int32)
    lc = np.array([9000, 100, 0, 16000, 3000], np.int32)
    pl = pkv.plan(prob, ones, lc, ones, num_sms=152)
    items = pl.items()
    assert all(it["kind"] == 1 for it in items)
    subs = {(it["head0"], it["num_heads"]) for it in items}
    want = {(h0, min(128, G - h0)) for h0 in range(0, G, 128)}
    assert subs == want
    assert pl.stats()["num_split_units"] > 0
    dyn = pkv.plan_decode_dynamic(prob, ones, lc, ones, num_sms=152)
    assert dyn.items() == items
    with pytest.raises(pkv.PkvError):   # more query tokens than one tile holds: not a dynamic-plan request
        pkv.plan_decode_dynamic(prob, np.full(B, 200, np.int32), lc, np.full(B, 200, np.int32), num_sms=152)


def test_two_query_tile_items_only_for_fp8_prefill_plans(pkv):
    """Items of two 128-row query tiles (sharing each K/V tile) appear for an
    fp8 cache at head_dim <= 128 in plans without decode tiles, and nowhere
    else: not for a bf16 cache, not at head_dim 256, not beside a decode unit."""
    def items(dtype, d, q_lens):
        prob = pkv.make_problem(batch=len(q_lens), num_heads_q=8, num_heads_kv=2, head_dim=d, page_size=16,
                                cache_capacity=4096, num_pages=1024, cache_dtype=dtype, causal=True,
                                softmax_scale=0.125)
        lc = [100] * len(q_lens)
        return pkv.plan(prob, q_lens, lc, q_lens, num_sms=13).items()
    tq = 128 // 4
    pairs = [it for it in items("fp8", 128, [300, 70]) if it["n_q"] > tq]
    assert pairs and all(it["n_q"] <= 2 * tq for it in pairs)
    assert any(it["n_q"] > tq for it in items("fp8", 64, [300, 70]))
    assert not any(it["n_q"] > tq for it in items("bf16", 128, [300, 70]))
    assert not any(it["n_q"] > tq for it in items("fp8", 256, [300, 70]))
    mixed = items("fp8", 128, [300, 1])
    assert any(it["kind"] == 0 for it in mixed) and not any(it["n_q"] > tq for it in mixed)


def test_decode_only_split_policy(pkv):
    """Decode-only plans: units that balance as well placed whole (within 2%
    of the split placement, on the planner's costs) are not split, so no
    combine runs; a batch with a few long sequences is still split; a plan
    with prefill tiles splits its decode units finer (four items an SM); an
    fp8 cache at head_dim <= 128, or a bf16 one at head_dim 64, runs two
    CTAs an SM."""
    def plan(dtype, q_lens, lc):
        B = len(lc)
        prob = pkv.make_problem(batch=B, num_heads_q=32, num_heads_kv=8, head_dim=128, page_size=16,
                                cache_capacity=65552, num_pages=200000, cache_dtype=dtype, causal=True,
                                softmax_scale=0.088)
        q = np.asarray(q_lens, np.int32)
        return pkv.plan(prob, q, np.asarray(lc, np.int32), q, num_sms=152).stats()
    rng = np.random.default_rng(5)
    lc = rng.integers(512, 4097, 64)
    even = plan("bf16", [1] * 64, lc)
    assert even["num_split_units"] == 0 and even["num_items"] == 64 * 8 and even["num_ctas"] == 152
    skewed = plan("bf16", [1] * 64, [65536] * 8 + [1024] * 56)
    assert skewed["num_split_units"] > 0
    assert skewed["max_cta_cost"] <= 1.1 * skewed["mean_cta_cost"]
    fp8 = plan("fp8", [1] * 64, [2048] * 64)
    assert fp8["num_ctas"] == 2 * 152 and fp8["num_split_units"] == 0
    # rows of 128 bytes over a bf16 cache (head_dim 64) run two CTAs an SM too
    prob64 = pkv.make_problem(batch=64, num_heads_q=32, num_heads_kv=8, head_dim=64, page_size=16,
                              cache_capacity=65552, num_pages=200000, cache_dtype="bf16", causal=True,
                              softmax_scale=0.125)
    ones = np.ones(64, np.int32)
    assert pkv.plan(prob64, ones, np.full(64, 2048, np.int32), ones, num_sms=152).stats()["num_ctas"] == 2 * 152
    # one prefill request in the batch: the decode units are cut for four items an SM
    mixed = plan("bf16", [1] * 63 + [512], list(lc[:63]) + [1000])
    assert mixed["num_prefill_items"] > 0 and mixed["num_split_units"] > 0 and mixed["num_ctas"] == 152
