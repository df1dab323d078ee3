"""GPU parity: the CUDA path (through the C ABI) against the CPU oracle.

Bar: cache appends bit-exact; outputs within max-abs 2e-2 / mean-abs 2e-3
(bf16 cache) or max-abs 6e-2 (fp8 cache); LSE within 2e-3.  Small cases are
compared element by element; the full-size workloads on sampled query rows
(every head of the row) and on the whole post-append cache.
"""
import numpy as np
import pytest

import oracle
import synth
from tests import harness as H

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    torch = pytest.importorskip("torch")
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from paged_kv_variable_gb300 import build
    build.build()


def tol_for(case):
    return H.FP8_TOL if case.spec.cache_dtype == "fp8" else H.BF16_TOL


def run_full(case, num_sms=None, check_cache=True):
    g = H.GpuCase(case, num_sms=num_sms)
    g.write_prefix()
    g.run()
    assert g.status() == 0, g.pkv.last_error()
    ref = oracle.forward(case)
    H.compare_out(g.out, ref["out"], tol_for(case))
    H.compare_lse(g.lse, ref["lse"])
    if check_cache:
        assert np.array_equal(H.to_numpy_bits(g.k_cache), ref["k_cache"]), "k cache differs"
        assert np.array_equal(H.to_numpy_bits(g.v_cache), ref["v_cache"]), "v cache differs"
    return g, ref


@pytest.mark.parametrize("sentinel", ["finite", "nan"])
def test_config1_tiny_paged(sentinel):
    run_full(synth.config1(sentinel=sentinel))


@pytest.mark.parametrize("seed", range(40))
def test_random_bf16(seed):
    run_full(H.gpu_random_case(seed, sentinel="nan" if seed % 3 == 0 else "finite"))


@pytest.mark.parametrize("seed", range(16))
def test_random_fp8(seed):
    run_full(H.gpu_random_case(100 + seed, cache_dtype="fp8", sentinel="nan" if seed % 2 else "finite"))


@pytest.mark.parametrize("P,q8", [(16, False), (0, False), (1, False), (4, False), (8, False), (64, False),
                                  (16, True), (0, True)])
def test_fp8_head_dim_64(P, q8):
    """fp8 cache at D = 64 (64-byte e4m3 rows, 64-byte TMA swizzle): a mixed
    batch of decode steps (one split along the keys), short query runs and
    prefills on cached prefixes; with q_scale, Q.K^T on e4m3 MMAs (warp MMAs
    on decode tiles, tcgen05 kind::f8f6f4 on 64-byte-swizzled tiles)."""
    import dataclasses
    spec = synth.Spec(batch=5, hq=16, hkv=4, d=64, page_size=P, causal=True,
                      softmax_scale=float(np.float32(1.0 / np.sqrt(64))), cache_dtype="fp8",
                      q_lens=np.array([1, 300, 1, 6, 140], np.int32), cache_lens=np.array([3000, 100, 0, 900, 37], np.int32),
                      new_lens=np.array([1, 300, 1, 6, 140], np.int32), capacity=3008, name="fp8-d64")
    case = synth.make_case(spec, np.random.default_rng(900 + P))
    if q8:
        amax = float(np.abs(synth.bf16_bits_to_f32(case.q)).max())
        case = dataclasses.replace(case, q_scale=float(np.float32(amax / 448.0)))
    g, _ = run_full(case, num_sms=16)
    assert g.plan.stats()["num_split_units"] > 0


@pytest.mark.parametrize("dtype,P,hq,hkv,q8", [("bf16", 16, 16, 4, False), ("bf16", 0, 16, 4, False),
                                               ("bf16", 256, 32, 4, False), ("bf16", 1, 8, 1, False),
                                               ("fp8", 16, 16, 4, False), ("fp8", 0, 32, 2, False),
                                               ("fp8", 8, 16, 4, True), ("bf16", 16, 64, 2, False)])
def test_head_dim_256(dtype, P, hq, hkv, q8):
    """head_dim 256 (64-key tiles: three 64-column S buffers beside a
    256-column O in tensor memory, 32 KB stages): a mixed batch of decode steps
    (split along the keys), a short query run and prefills on cached prefixes,
    GQA groups of 4 and 8 (decode tiles of at most 8 rows) and wider groups
    (tensor-core tiles), bf16 and fp8 caches, with and without q_scale."""
    import dataclasses
    spec = synth.Spec(batch=5, hq=hq, hkv=hkv, d=256, page_size=P, causal=True,
                      softmax_scale=float(np.float32(1.0 / np.sqrt(256))), cache_dtype=dtype,
                      q_lens=np.array([1, 200, 1, 3, 90], np.int32), cache_lens=np.array([2500, 100, 600, 0, 41], np.int32),
                      new_lens=np.array([1, 200, 1, 3, 90], np.int32), capacity=2560, name="d256")
    case = synth.make_case(spec, np.random.default_rng(2560 + P + hq))
    if q8:
        amax = float(np.abs(synth.bf16_bits_to_f32(case.q)).max())
        case = dataclasses.replace(case, q_scale=float(np.float32(amax / 448.0)))
    g, _ = run_full(case, num_sms=24)
    assert g.plan.stats()["num_split_units"] > 0


@pytest.mark.parametrize("seed", range(6))
def test_random_head_dim_256(seed):
    """Random batches at head_dim 256 (both cache dtypes, causal or not, the
    page sizes of the random cases)."""
    case = H.gpu_random_case(2600 + seed, d=256, cache_dtype="fp8" if seed % 2 else "bf16",
                             sentinel="nan" if seed % 3 == 0 else "finite")
    run_full(case)


@pytest.mark.parametrize("layout", ["head_pad", "base_offset"])
@pytest.mark.parametrize("cache_dtype", ["bf16", "fp8"])
def test_output_rows_not_32_byte_aligned(layout, cache_dtype):
    """Output rows on 16 but not 32 bytes (a padded head stride, or a base 16
    bytes past a 32-byte boundary): the 16-byte store path, same results."""
    import torch
    case = synth.random_case(7, batch=3, hq=8, hkv=2, d=128, page_size=16, causal=True, cache_dtype=cache_dtype,
                             max_cache=300, max_new=200, allow_zero=False)
    spec = case.spec
    g = H.GpuCase(case)
    g.write_prefix()
    shape = (spec.total_q, spec.hq, spec.d)
    if layout == "head_pad":
        big = torch.full((spec.total_q, spec.hq, spec.d + 8), float("nan"), dtype=torch.bfloat16, device="cuda")
        g.out = big[:, :, :spec.d]
        assert (g.out.stride(1) * 2) % 32 == 16
    else:
        big = torch.full((spec.total_q * spec.hq * spec.d + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
        g.out = big[8:].view(shape)
        assert g.out.data_ptr() % 32 == 16
    g.run()
    assert g.status() == 0, g.pkv.last_error()
    ref = oracle.forward(case)
    H.compare_out(g.out.contiguous(), ref["out"], tol_for(case))
    H.compare_lse(g.lse, ref["lse"])


@pytest.mark.parametrize("seed", range(8))
def test_cache_only_and_ragged_queries(seed):
    # no new K/V (cache-only attention) and query lengths unrelated to new lengths
    run_full(H.gpu_random_case(200 + seed, with_new=(seed % 2 == 0), q_equals_new=False))


def test_zero_lengths_and_empty_rows():
    spec = synth.Spec(batch=4, hq=8, hkv=2, d=128, page_size=16, causal=True, softmax_scale=0.0883883461356163,
                      cache_dtype="bf16", q_lens=np.array([3, 0, 5, 2], np.int32),
                      cache_lens=np.array([0, 7, 0, 1], np.int32), new_lens=np.array([0, 2, 5, 0], np.int32),
                      capacity=32, name="zeros")
    case = synth.make_case(spec, np.random.default_rng(5))
    g, ref = run_full(case)
    # sequence 0 sees no key at all: zeros and -inf
    assert np.all(ref["out"][:3] == 0)


@pytest.mark.parametrize("g_", [1, 2, 4, 8, 16])
def test_group_sizes_decode_and_prefill(g_):
    for seed, lq in ((300 + g_, 1), (310 + g_, 40)):
        rng = np.random.default_rng(seed)
        spec = synth.uniform_spec(f"g{g_}", 3, lq, int(rng.integers(100, 400)), hq=2 * g_, hkv=2, d=128)
        run_full(synth.make_case(spec, rng))


@pytest.mark.parametrize("hq,hkv,lq,lc,P,dtype,sms", [
    (32, 1, 1, 3000, 16, "bf16", 16),     # MQA decode, split along the keys
    (32, 1, 200, 500, 16, "bf16", 152),   # MQA prefill: 4 tokens per tile
    (64, 2, 1, 1500, 0, "bf16", 8),       # G = 32 decode, contiguous cache, split
    (96, 2, 3, 700, 16, "bf16", 152),     # G = 48: a short query run in one tile
    (71, 1, 5, 900, 32, "bf16", 4),       # G = 71 (prime): one token per tile, split
    (256, 1, 2, 600, 16, "bf16", 152),    # G = 256: two head sub-groups of 128
    (200, 1, 1, 2500, 16, "bf16", 8),     # G = 200: sub-groups of 128 and 72, split
    (12, 2, 9, 300, 16, "bf16", 152),     # G = 6: 54 rows in one tile
    (24, 8, 1, 800, 16, "bf16", 152),     # G = 3: a decode tile of 3 rows
    (32, 1, 1, 2000, 16, "fp8", 16),      # MQA decode on an fp8 cache, split
    (64, 2, 130, 200, 16, "fp8", 152),    # G = 32 prefill on an fp8 cache
    (64, 1, 1, 1000, 64, "bf16", 152),    # G = 64 decode, D = 64 below
])
def test_wide_and_odd_groups(hq, hkv, lq, lc, P, dtype, sms):
    """Any group size (MQA and GQA beyond 16 heads per kv head): rows of more
    than 16 go to tensor-core tiles that hold the whole group (up to 128 heads,
    larger groups cut into sub-groups), split along the keys when a unit's
    queries fit one tile; small odd groups stay on decode tiles."""
    d = 64 if (hq, hkv, lc, P) == (64, 1, 1000, 64) else 128
    rng = np.random.default_rng(hq * 1000 + lq + lc)
    spec = synth.uniform_spec(f"g{hq // hkv}", 3, lq, lc, hq=hq, hkv=hkv, d=d, page_size=P, cache_dtype=dtype)
    case = synth.make_case(spec, rng)
    g, _ = run_full(case, num_sms=sms)
    if sms <= 16 and lq == 1:
        assert g.plan.stats()["num_split_units"] > 0


def test_wide_group_mixed_batch_and_quantised_queries():
    """An MQA batch mixing decode steps, short query runs and long prefills in
    one launch; then the same on an fp8 cache with quantised queries."""
    import dataclasses
    spec = synth.Spec(batch=5, hq=32, hkv=1, d=128, page_size=16, causal=True,
                      softmax_scale=float(np.float32(1.0 / np.sqrt(128))), cache_dtype="bf16",
                      q_lens=np.array([1, 300, 1, 4, 37], np.int32), cache_lens=np.array([2500, 100, 0, 900, 0], np.int32),
                      new_lens=np.array([1, 300, 1, 4, 37], np.int32), capacity=2512, name="mqa-mixed")
    run_full(synth.make_case(spec, np.random.default_rng(55)), num_sms=24)
    fspec = dataclasses.replace(spec, cache_dtype="fp8")
    case = synth.make_case(fspec, np.random.default_rng(56))
    amax = float(np.abs(synth.bf16_bits_to_f32(case.q)).max())
    run_full(dataclasses.replace(case, q_scale=float(np.float32(amax / 448.0))), num_sms=24)


def test_long_decode_is_split_and_matches():
    rng = np.random.default_rng(11)
    spec = synth.uniform_spec("long", 2, 1, 9000, hq=8, hkv=2, d=128, page_size=64)
    case = synth.make_case(spec, rng)
    g, _ = run_full(case, num_sms=8)
    assert g.plan.stats()["num_split_units"] > 0


def test_split_counts_agree():
    case = synth.random_case(21, batch=4, hq=8, hkv=2, d=128, page_size=32, causal=True, max_cache=3000,
                             max_new=1, allow_zero=False)
    outs = []
    for sms in (1, 5, 37, 152):
        g, _ = run_full(case, num_sms=sms)
        outs.append(H.bf16_to_f64(g.out))
    for o in outs[1:]:
        assert np.max(np.abs(o - outs[0])) <= 1e-2


def test_deterministic_and_poison_independent():
    a = H.gpu_random_case(31, page_size=16, sentinel="finite")
    b = H.gpu_random_case(31, page_size=16, sentinel="nan")
    ga = H.GpuCase(a)
    ga.run()
    ga2 = H.GpuCase(a)
    ga2.run()
    gb = H.GpuCase(b)
    gb.run()
    first = H.to_numpy_bits(ga.out)
    assert np.array_equal(first, H.to_numpy_bits(ga2.out))
    assert np.array_equal(first, H.to_numpy_bits(gb.out))


def test_paged_equals_contiguous_and_relabel():
    case = synth.random_case(41, batch=3, hq=8, hkv=2, d=128, page_size=16, causal=True, max_cache=500,
                             max_new=40, allow_zero=False)
    ga = H.GpuCase(case)
    ga.run()
    gc = H.GpuCase(synth.to_contiguous(case))
    gc.run()
    gr = H.GpuCase(synth.relabel_pages(case, np.random.default_rng(3)))
    gr.run()
    base = H.to_numpy_bits(ga.out)
    assert np.array_equal(base, H.to_numpy_bits(gc.out))
    assert np.array_equal(base, H.to_numpy_bits(gr.out))


def test_fused_append_equals_append_then_attend():
    import torch
    case = H.gpu_random_case(51, page_size=32)
    fused = H.GpuCase(case)
    fused.run()
    sep = H.GpuCase(case)
    spec = case.spec
    sep.pkv.kv_append(sep.problem, sep.args(), spec.total_new, sep.workspace)
    # the attention alone over the advanced cache lengths
    adv = synth.Spec(**{**spec.__dict__, "cache_lens": spec.kv_lens, "new_lens": np.zeros_like(spec.new_lens)})
    import paged_kv_variable_gb300 as pkv
    pl = pkv.plan(sep.problem, adv.q_lens, adv.cache_lens, None)
    ws = pkv.workspace_tensor(pl.workspace_bytes)
    pl.upload(ws)
    a = pkv.make_args(q=sep.q, out=sep.out, lse=sep.lse, cu_seqlens_q=sep.cu_q, max_seqlen_q=int(spec.q_lens.max()),
                      k_cache=sep.k_cache, v_cache=sep.v_cache, cache_seqlens=H.i32(adv.cache_lens),
                      block_table=sep.block_table)
    pkv.attn_varlen_kvcache_fwd(sep.problem, a, pl, ws)
    assert pkv.get_status(ws) == 0
    assert np.array_equal(H.to_numpy_bits(fused.out), H.to_numpy_bits(sep.out))
    assert torch.equal(fused.k_cache, sep.k_cache)


def test_device_status_on_bad_block_table_entry():
    # an out-of-range page number is never dereferenced: the append skips the
    # row, the gather reads zeros, and the status word reports it
    case = synth.config1()
    g = H.GpuCase(case)
    bt = g.block_table.clone()
    bt[0, 1] = 10_000
    g.block_table = bt
    g.run()
    assert g.status() == 6


def test_device_status_on_plan_mismatch():
    case = synth.config1()
    g = H.GpuCase(case)
    g.cache_lens[1] += 1
    g.run()
    assert g.status() == 7


# ------------------------------------------------------------------ full-size workloads
def _sample_rows(spec, n, seed):
    rng = np.random.default_rng(seed)
    rows = []
    seqs = [b for b in range(spec.batch) if spec.q_lens[b] > 0]
    for _ in range(n):
        b = int(rng.choice(seqs))
        i = int(rng.integers(0, int(spec.q_lens[b])))
        rows.append((b, i))
    # always include the first and last query of the longest sequence
    bl = int(np.argmax(spec.q_lens))
    rows += [(bl, 0), (bl, int(spec.q_lens[bl]) - 1)]
    return rows


def check_sampled(case, g, n_rows=48, seed=0, full_cache=True):
    """bf16 caches: the whole post-append cache bit-exact, then sampled rows
    from the oracle's own post-append cache.  fp8 (full_cache=False): the
    oracle writes and attends only the sampled sequences."""
    spec = case.spec
    rows = _sample_rows(spec, n_rows, seed)
    tol = tol_for(case)
    out = g.out.float().cpu().double().numpy()
    lse = g.lse.cpu().double().numpy()
    cu = spec.cu_q
    if full_cache:
        kc0, vc0 = oracle.prepare_prefix(case)
        kc, vc = oracle.append_kv(spec, kc0, vc0, case.block_table, case.k_new, case.v_new, case.k_scale,
                                  case.v_scale)
        assert np.array_equal(H.to_numpy_bits(g.k_cache), kc), "k cache differs"
        assert np.array_equal(H.to_numpy_bits(g.v_cache), vc), "v cache differs"
        o, l = oracle.forward_rows(case, kc, vc, rows)
        idx = [cu[b] + i for b, i in rows]
        err = np.abs(out[idx] - o)
        assert err.max() <= tol["max_abs"], float(err.max())
        assert err.mean() <= tol["mean_abs"], float(err.mean())
        assert np.max(np.abs(lse[:, idx] - l)) <= H.LSE_TOL
        return
    by_seq = {}
    for b, i in rows:
        by_seq.setdefault(b, []).append(i)
    for b, idx in by_seq.items():
        sub = synth.subset_case(case, [b])
        kc0, vc0 = oracle.prepare_prefix(sub)
        kc, vc = oracle.append_kv(sub.spec, kc0, vc0, sub.block_table, sub.k_new, sub.v_new, sub.k_scale,
                                  sub.v_scale)
        o, l = oracle.forward_rows(sub, kc, vc, [(0, i) for i in idx])
        got = out[[cu[b] + i for i in idx]]
        err = np.abs(got - o)
        assert err.max() <= tol["max_abs"], (b, float(err.max()))
        assert err.mean() <= tol["mean_abs"], (b, float(err.mean()))
        gl = lse[:, [cu[b] + i for i in idx]]
        assert np.max(np.abs(gl - l)) <= H.LSE_TOL


def check_every_row(case, g):
    """The whole post-append cache bit-exact and EVERY output row (all heads)
    against ``oracle.forward`` of the full workload."""
    ref = oracle.forward(case)
    assert np.array_equal(H.to_numpy_bits(g.k_cache), ref["k_cache"]), "k cache differs"
    assert np.array_equal(H.to_numpy_bits(g.v_cache), ref["v_cache"]), "v cache differs"
    H.compare_out(g.out, ref["out"], tol_for(case))
    H.compare_lse(g.lse, ref["lse"])
    return ref


@pytest.mark.slow
def test_config2_decode_full():
    case = synth.config2()
    g = H.GpuCase(case)
    g.run()
    assert g.status() == 0
    check_every_row(case, g)


@pytest.mark.slow
@pytest.mark.parametrize("causal", [True, False])
def test_config3_prefill_full(causal):
    """Every one of the 4096 query rows (x 32 heads) of the cached-prefix
    prefill: 16 query tiles per kv head, the epilogue deferred across items."""
    case = synth.config3(causal=causal)
    g = H.GpuCase(case)
    g.run()
    assert g.status() == 0
    check_every_row(case, g)


@pytest.mark.slow
def test_config4_mixed_full():
    """Every row of the mixed batch: 60 decode rows and the 4 x 2048 rows of
    the prefill requests, one launch."""
    case = synth.config4()
    g = H.GpuCase(case)
    g.run()
    assert g.status() == 0
    check_every_row(case, g)


@pytest.mark.slow
def test_config5_fp8_prefill_then_decode():
    pre, dec = synth.config5()
    g = H.GpuCase(pre)
    g.run()
    assert g.status() == 0
    check_sampled(pre, g, n_rows=24, full_cache=False)
    # fp8 append bit-exact on sampled sequences
    spec = pre.spec
    for b in (0, 17, 63):
        sub = synth.subset_case(pre, [b])
        kc, vc = oracle.append_kv(sub.spec, sub.k_cache, sub.v_cache, sub.block_table, sub.k_new, sub.v_new,
                                  sub.k_scale, sub.v_scale)
        pages = pre.block_table[b]
        local = sub.block_table[0]          # the subset renumbers its pages
        assert np.array_equal(H.to_numpy_bits(g.k_cache[pages.tolist()]), kc[local])
        assert np.array_equal(H.to_numpy_bits(g.v_cache[pages.tolist()]), vc[local])
    # every row of two whole sequences (first and last of the batch)
    out = g.out.float().cpu().double().numpy()
    lse = g.lse.cpu().double().numpy()
    cu = spec.cu_q
    for b in (0, spec.batch - 1):
        ref = oracle.forward(synth.subset_case(pre, [b]))
        rows = slice(int(cu[b]), int(cu[b + 1]))
        err = np.abs(out[rows] - ref["out"])
        assert err.max() <= H.FP8_TOL["max_abs"] and err.mean() <= H.FP8_TOL["mean_abs"], (b, float(err.max()))
        assert np.max(np.abs(lse[:, rows] - ref["lse"])) <= H.LSE_TOL
    # decode step on the cache the prefill left (token 2049): every row
    gd = H.GpuCase(dec)
    gd.k_cache.copy_(g.k_cache)
    gd.v_cache.copy_(g.v_cache)
    gd.run()
    assert gd.status() == 0
    ref = oracle.forward(dec)
    H.compare_out(gd.out, ref["out"], H.FP8_TOL)
    H.compare_lse(gd.lse, ref["lse"])
    assert np.array_equal(H.to_numpy_bits(gd.k_cache), ref["k_cache"]), "k cache differs"


# ------------------------------------------------------------------ widening: ragged page list, CUDA graphs
def test_ragged_page_list_equals_block_table():
    import torch
    case = synth.random_case(71, batch=5, hq=8, hkv=2, d=128, page_size=16, causal=True, max_cache=700,
                             max_new=60, allow_zero=True)
    spec = case.spec
    g = H.GpuCase(case)
    g.run()
    assert g.status() == 0
    base = H.to_numpy_bits(g.out)
    # kv_indices / kv_indptr: only the pages each sequence uses, concatenated
    P = spec.page_size
    counts = [(int(n) + P - 1) // P for n in spec.kv_lens]
    flat = np.concatenate([case.block_table[b, :counts[b]] for b in range(spec.batch)] + [np.zeros(0, np.int32)])
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    r = H.GpuCase(case)
    a = r.pkv.make_args(q=r.q, out=r.out, lse=r.lse, cu_seqlens_q=r.cu_q, max_seqlen_q=int(spec.q_lens.max()),
                        k_cache=r.k_cache, v_cache=r.v_cache, cache_seqlens=r.cache_lens, k_new=r.k_new,
                        v_new=r.v_new, cu_seqlens_knew=r.cu_new, block_table=H.i32(flat),
                        page_indptr=H.i32(indptr))
    r.pkv.attn_varlen_kvcache_fwd(r.problem, a, r.plan, r.workspace)
    assert r.status() == 0
    assert np.array_equal(base, H.to_numpy_bits(r.out))
    assert torch.equal(g.k_cache, r.k_cache) and torch.equal(g.v_cache, r.v_cache)
    ref = oracle.forward(case)
    H.compare_out(r.out, ref["out"], H.BF16_TOL)
    H.compare_lse(r.lse, ref["lse"])


@pytest.mark.parametrize("hq,hkv,cache_dtype", [(16, 4, "bf16"), (32, 1, "bf16"), (16, 4, "fp8")])
def test_non_contiguous_query_rows(hq, hkv, cache_dtype):
    """Query / output rows placed anywhere (the non-contiguous Q/O layout:
    row offsets per sequence in cu_seqlens_q, lengths from the plan, gaps and
    any order) with a ragged page list holding spare pages (KV lengths from
    cache_seqlens alone): decode units (split along the keys), a short query
    run and prefill tiles match the oracle, and the rows in the gaps are never
    written."""
    import torch
    spec = synth.Spec(batch=5, hq=hq, hkv=hkv, d=128, page_size=16, causal=True,
                      softmax_scale=float(np.float32(1.0 / np.sqrt(128))), cache_dtype=cache_dtype,
                      q_lens=np.array([1, 300, 1, 5, 140], np.int32), cache_lens=np.array([3000, 100, 700, 0, 33], np.int32),
                      new_lens=np.array([1, 300, 1, 5, 140], np.int32), capacity=3008, name="gapped-q")
    case = synth.make_case(spec, np.random.default_rng(800 + hq))
    rng = np.random.default_rng(801)
    order = rng.permutation(spec.batch)                 # sequences laid out in this order
    gaps = rng.integers(1, 40, spec.batch)              # rows left free before each one
    starts = np.zeros(spec.batch, np.int64)
    row = 0
    for b in order:
        row += int(gaps[b])
        starts[b] = row
        row += int(spec.q_lens[b])
    q_rows = row + 7
    g = H.GpuCase(case, num_sms=24)
    assert g.plan.stats()["num_split_units"] > 0
    g.write_prefix()
    cu = spec.cu_q
    qbig = torch.full((q_rows, hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    for b in range(spec.batch):
        qbig[starts[b]:starts[b] + spec.q_lens[b]] = g.q[cu[b]:cu[b + 1]]
    obig = torch.full((q_rows, hq, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    lbig = torch.full((hq, q_rows), float("nan"), dtype=torch.float32, device="cuda")
    P = spec.page_size
    width = case.block_table.shape[1]
    counts = [min((int(n) + P - 1) // P + 1, width) for n in spec.kv_lens]   # a spare page where the row has one
    flat = np.concatenate([case.block_table[b, :counts[b]] for b in range(spec.batch)])
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    assert flat.size == indptr[-1]
    a = g.pkv.make_args(q=qbig, out=obig, lse=lbig, cu_seqlens_q=H.i32(np.append(starts, q_rows)),
                        max_seqlen_q=int(spec.q_lens.max()), k_cache=g.k_cache, v_cache=g.v_cache,
                        cache_seqlens=g.cache_lens, k_new=g.k_new, v_new=g.v_new, cu_seqlens_knew=g.cu_new,
                        block_table=H.i32(flat), page_indptr=H.i32(indptr),
                        k_scale=g.k_scale if cache_dtype == "fp8" else None,
                        v_scale=g.v_scale if cache_dtype == "fp8" else None, q_rows=q_rows)
    g.pkv.attn_varlen_kvcache_fwd(g.problem, a, g.plan, g.workspace)
    assert g.status() == 0, g.pkv.last_error()
    ref = oracle.forward(case)
    used = np.zeros(q_rows, bool)
    got = torch.empty_like(g.out)
    got_lse = torch.empty((hq, spec.total_q), dtype=torch.float32, device="cuda")
    for b in range(spec.batch):
        used[starts[b]:starts[b] + spec.q_lens[b]] = True
        got[cu[b]:cu[b + 1]] = obig[starts[b]:starts[b] + spec.q_lens[b]]
        got_lse[:, cu[b]:cu[b + 1]] = lbig[:, starts[b]:starts[b] + spec.q_lens[b]]
    H.compare_out(got, ref["out"], tol_for(case))
    H.compare_lse(got_lse, ref["lse"])
    free = torch.from_numpy(~used).cuda()
    assert torch.isnan(obig[free].float()).all() and torch.isnan(lbig[:, free]).all(), "a gap row was written"


@pytest.mark.parametrize("cache_dtype,P", [("bf16", 16), ("bf16", 1), ("fp8", 16), ("bf16", 64)])
def test_ragged_page_list_prefill_against_oracle(cache_dtype, P):
    """Prefill-heavy batches (several 128-row query tiles per kv head, cached
    prefixes, a decode request among them) addressed through a ragged page
    list that holds more pages than each sequence uses (the kv_indptr /
    kv_indices form), against the oracle."""
    spec = synth.Spec(batch=4, hq=16, hkv=4, d=128, page_size=P, causal=True,
                      softmax_scale=float(np.float32(1.0 / np.sqrt(128))), cache_dtype=cache_dtype,
                      q_lens=np.array([300, 1, 129, 520], np.int32), cache_lens=np.array([700, 900, 0, 33], np.int32),
                      new_lens=np.array([300, 1, 129, 520], np.int32), capacity=1024, name="ragged-prefill")
    case = synth.make_case(spec, np.random.default_rng(700 + P))
    counts = [(int(n) + P - 1) // P + 1 for n in spec.kv_lens]     # one spare page per sequence
    counts = [min(c, case.block_table.shape[1]) for c in counts]
    flat = np.concatenate([case.block_table[b, :counts[b]] for b in range(spec.batch)])
    indptr = np.concatenate([[0], np.cumsum(counts)]).astype(np.int32)
    r = H.GpuCase(case)
    r.write_prefix()
    a = r.pkv.make_args(q=r.q, out=r.out, lse=r.lse, cu_seqlens_q=r.cu_q, max_seqlen_q=int(spec.q_lens.max()),
                        k_cache=r.k_cache, v_cache=r.v_cache, cache_seqlens=r.cache_lens, k_new=r.k_new,
                        v_new=r.v_new, cu_seqlens_knew=r.cu_new, block_table=H.i32(flat),
                        page_indptr=H.i32(indptr), k_scale=r.k_scale if cache_dtype == "fp8" else None,
                        v_scale=r.v_scale if cache_dtype == "fp8" else None)
    r.pkv.attn_varlen_kvcache_fwd(r.problem, a, r.plan, r.workspace)
    assert r.status() == 0, r.pkv.last_error()
    ref = oracle.forward(case)
    H.compare_out(r.out, ref["out"], tol_for(case))
    H.compare_lse(r.lse, ref["lse"])
    assert np.array_equal(H.to_numpy_bits(r.k_cache), ref["k_cache"]), "k cache differs"


@pytest.mark.parametrize("kind", ["decode", "mixed"])
def test_cuda_graph_capture_and_replay(kind):
    import torch
    if kind == "decode":
        rng = np.random.default_rng(81)
        case = synth.make_case(synth.uniform_spec("graph-decode", 6, 1, 1500, hq=8, hkv=2, d=128, page_size=16), rng)
    else:
        case = H.gpu_random_case(82, page_size=16, max_cache=600, max_new=70)
    g = H.GpuCase(case)
    g.run()                                   # first call outside capture (one-time set-up)
    torch.cuda.synchronize()
    assert g.status() == 0
    first = H.to_numpy_bits(g.out)
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    graph = torch.cuda.CUDAGraph()
    args = g.args()
    with torch.cuda.graph(graph, stream=stream):
        g.pkv.attn_varlen_kvcache_fwd(g.problem, args, g.plan, g.workspace, stream=stream)
    g.out.fill_(float("nan"))
    torch.cuda.synchronize()
    graph.replay()
    torch.cuda.synchronize()
    assert np.array_equal(first, H.to_numpy_bits(g.out))   # the append rewrites the same values
    # new queries in the captured buffers: the replay attends them
    rng = np.random.default_rng(83)
    case.q = synth.f32_to_bf16_bits(rng.standard_normal(case.q.shape, dtype=np.float32))
    g.q.copy_(H.bf16_tensor(case.q))
    graph.replay()
    torch.cuda.synchronize()
    assert g.status() == 0
    ref = oracle.forward(case)
    H.compare_out(g.out, ref["out"], H.BF16_TOL)


@pytest.mark.parametrize("cache_dtype,ragged,hq,hkv", [("bf16", False, 8, 2), ("bf16", True, 8, 2),
                                                        ("fp8", False, 8, 2), ("bf16", False, 32, 1)])
def test_dynamic_plan_graph_decode_steps(cache_dtype, ragged, hq, hkv):
    """One dynamic plan and one captured graph serve several decode steps while
    cache_seqlens grows on the device; every step matches the oracle (bf16 and
    fp8 caches, padded block table or ragged page list, GQA and MQA with 32
    heads per kv head on tensor-core tiles)."""
    import dataclasses
    import math
    import torch
    steps = 5
    rng = np.random.default_rng(91)
    B, d, P = 6, 128, 16
    base = rng.integers(100, 1500, B).astype(np.int32)
    base[0] = 0                         # a sequence that starts empty
    total = base + steps                # the tokens the steps will append are drawn up front
    cap = int((total.max() + 1 + P - 1) // P * P)
    spec = synth.Spec(batch=B, hq=hq, hkv=hkv, d=d, page_size=P, causal=True,
                      softmax_scale=float(np.float32(1.0 / math.sqrt(d))), cache_dtype=cache_dtype,
                      q_lens=np.ones(B, np.int32), cache_lens=total.astype(np.int32),
                      new_lens=np.ones(B, np.int32), capacity=cap, name="dynamic-decode")
    case = synth.make_case(spec, rng)
    g = H.GpuCase(case)
    g.write_prefix()                    # fp8: the whole drawn prefix, quantised by the library's append
    bounds = (base + steps - 1).astype(np.int32)
    plan = g.pkv.plan_decode_dynamic(g.problem, spec.q_lens, bounds, spec.new_lens)
    assert plan.stats()["num_split_units"] > 0          # split chunks that early steps leave empty
    ws = g.pkv.workspace_tensor(plan.workspace_bytes)
    plan.upload(ws)
    cu_total = np.concatenate([[0], np.cumsum(total)]).astype(np.int64)

    def token(pos_of_b):                 # the drawn K/V of one position per sequence (bf16 bits)
        if cache_dtype == "fp8":
            rows = [cu_total[b] + p for b, p in enumerate(pos_of_b)]
            return case.prefix_k[rows], case.prefix_v[rows]
        k = np.stack([case.k_cache[case.block_table[b, p // P], p % P] for b, p in enumerate(pos_of_b)])
        v = np.stack([case.v_cache[case.block_table[b, p // P], p % P] for b, p in enumerate(pos_of_b)])
        return k, v

    extra = {}
    if ragged:
        counts = [(int(t) + 1 + P - 1) // P for t in total]
        flat = np.concatenate([case.block_table[b, :counts[b]] for b in range(B)])
        extra = dict(block_table=H.i32(flat), page_indptr=H.i32(np.concatenate([[0], np.cumsum(counts)])))
    args = g.pkv.make_args(q=g.q, out=g.out, lse=g.lse, cu_seqlens_q=g.cu_q, max_seqlen_q=1, k_cache=g.k_cache,
                           v_cache=g.v_cache, cache_seqlens=g.cache_lens, k_new=g.k_new, v_new=g.v_new,
                           cu_seqlens_knew=g.cu_new, k_scale=g.k_scale if cache_dtype == "fp8" else None,
                           v_scale=g.v_scale if cache_dtype == "fp8" else None,
                           **(extra or dict(block_table=g.block_table)))
    kt, vt = token(base)
    g.k_new.copy_(H.bf16_tensor(kt))
    g.v_new.copy_(H.bf16_tensor(vt))
    g.cache_lens.copy_(H.i32(base))
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    stream.wait_stream(torch.cuda.current_stream())
    g.pkv.attn_varlen_kvcache_fwd(g.problem, args, plan, ws, stream=stream)   # first call outside capture
    stream.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        g.pkv.attn_varlen_kvcache_fwd(g.problem, args, plan, ws, stream=stream)
    tol = H.FP8_TOL if cache_dtype == "fp8" else H.BF16_TOL
    for s in range(steps):
        lc = (base + s).astype(np.int32)
        kt, vt = token(lc)
        q = synth.f32_to_bf16_bits(rng.standard_normal((B, hq, d), dtype=np.float32))
        g.cache_lens.copy_(H.i32(lc))
        g.k_new.copy_(H.bf16_tensor(kt))
        g.v_new.copy_(H.bf16_tensor(vt))
        g.q.copy_(H.bf16_tensor(q))
        g.out.fill_(float("nan"))
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        assert g.pkv.get_status(ws) == 0
        step = dict(q=q, k_new=kt, v_new=vt)
        if cache_dtype == "fp8":          # the oracle writes its own prefix: the first lc tokens
            rows = np.concatenate([np.arange(cu_total[b], cu_total[b] + lc[b]) for b in range(B)]).astype(np.int64)
            step.update(prefix_k=case.prefix_k[rows], prefix_v=case.prefix_v[rows])
        step_case = dataclasses.replace(case, spec=dataclasses.replace(spec, cache_lens=lc), **step)
        ref = oracle.forward(step_case)
        H.compare_out(g.out, ref["out"], tol)
        H.compare_lse(g.lse, ref["lse"])
    # a length past the plan's bound is reported
    g.cache_lens.copy_(H.i32(bounds + 1))
    graph.replay()
    torch.cuda.synchronize()
    assert g.pkv.get_status(ws) == 7


@pytest.mark.parametrize("P,cache_dtype,d", [(8, "bf16", 128), (8, "bf16", 64), (24, "bf16", 128), (8, "fp8", 128),
                                             (1, "bf16", 128), (2, "bf16", 64), (4, "bf16", 128), (4, "fp8", 128),
                                             (1, "fp8", 128)])
def test_small_and_odd_pages(P, cache_dtype, d):
    """Pages of 8 tokens (one 8-row TMA box each), of 24 (three boxes) and of
    1, 2 or 4 tokens (rows gathered one by one): random decode + prefill
    batches against the oracle, and paged == contiguous."""
    case = synth.random_case(100 + P + d, batch=4, hq=8, hkv=2, d=d, page_size=P, causal=True, max_cache=700,
                             max_new=70, cache_dtype=cache_dtype)
    g = H.GpuCase(case)
    g.write_prefix()
    g.run()
    assert g.status() == 0
    ref = oracle.forward(case)
    tol = H.FP8_TOL if cache_dtype == "fp8" else H.BF16_TOL
    H.compare_out(g.out, ref["out"], tol)
    H.compare_lse(g.lse, ref["lse"])
    if cache_dtype == "bf16":
        c = H.GpuCase(synth.to_contiguous(case))
        c.run()
        assert c.status() == 0
        assert np.array_equal(H.to_numpy_bits(g.out), H.to_numpy_bits(c.out))


@pytest.mark.parametrize("P,cache_dtype", [(1, "bf16"), (4, "bf16"), (2, "fp8")])
def test_small_pages_decode(P, cache_dtype):
    """Decode batches (split-KV chunks included) over pages of 1, 2 and 4 tokens."""
    rng = np.random.default_rng(140 + P)
    spec = synth.uniform_spec("small-page-decode", 6, 1, 2500, hq=16, hkv=4, d=128, page_size=P,
                              cache_dtype=cache_dtype)
    case = synth.make_case(spec, rng)
    # (decode-only plans aim at two items an SM: 16 SMs to have them split)
    g = H.GpuCase(case, num_sms=16)
    assert g.plan.stats()["num_split_units"] > 0
    g.write_prefix()
    g.run()
    assert g.status() == 0
    ref = oracle.forward(case)
    H.compare_out(g.out, ref["out"], H.FP8_TOL if cache_dtype == "fp8" else H.BF16_TOL)
    H.compare_lse(g.lse, ref["lse"])


@pytest.mark.parametrize("P,G,split", [(16, 4, False), (16, 4, True), (0, 8, False), (8, 1, True)])
def test_fp8_quantised_queries_decode(P, G, split):
    """fp8 cache with q_scale: Q quantised to e4m3 and Q.K^T on fp8 tensor cores
    (decode tiles), against the oracle's quantised-query reading."""
    import dataclasses
    rng = np.random.default_rng(160 + P + G)
    spec = synth.uniform_spec("fp8-q8-decode", 5, 1, 1800 if split else 400, hq=2 * G, hkv=2, d=128, page_size=P,
                              cache_dtype="fp8")
    case = synth.make_case(spec, rng)
    amax = float(np.abs(synth.bf16_bits_to_f32(case.q)).max())
    case = dataclasses.replace(case, q_scale=float(np.float32(amax / 448.0)))
    g = H.GpuCase(case, num_sms=8 if split else 152)
    assert (g.plan.stats()["num_split_units"] > 0) == split
    g.write_prefix()
    g.run()                                          # q_scale goes in with the other arguments
    assert g.status() == 0
    ref = oracle.forward(case)
    H.compare_out(g.out, ref["out"], H.FP8_TOL)
    H.compare_lse(g.lse, ref["lse"])


@pytest.mark.parametrize("d,G,causal,P,q8", [(128, 4, True, 16, False), (64, 8, False, 0, False),
                                              (128, 1, True, 32, True), (128, 16, True, 16, False),
                                              (64, 2, True, 16, True), (128, 4, False, 1, False)])
def test_fp8_two_query_tile_items(d, G, causal, P, q8):
    """Prefill-only batches over an fp8 cache, whose items hold two query tiles
    sharing each K/V tile: ragged query runs leave single-tile items and tiles
    with fewer rows, the first tile of a causal item attending fewer key tiles
    than the second; every row against the oracle."""
    import dataclasses
    rng = np.random.default_rng(700 + d + G + P + int(causal) + int(q8))
    tq = 128 // G
    lq = np.array([2 * tq + 5, 3 * tq + tq // 2, tq + 1, 4 * tq], np.int32)
    lc = np.array([0, 130, 7, 300], np.int32)
    spec = synth.Spec(batch=4, hq=2 * G, hkv=2, d=d, page_size=P, causal=causal,
                      softmax_scale=float(np.float32(1.0 / np.sqrt(d))), cache_dtype="fp8",
                      q_lens=lq, cache_lens=lc, new_lens=lq.copy(),
                      capacity=int(((lc + lq).max() + 15) // 16 * 16 + 16), name="fp8-two-query-tiles")
    case = synth.make_case(spec, rng)
    if q8:
        amax = float(np.abs(synth.bf16_bits_to_f32(case.q)).max())
        case = dataclasses.replace(case, q_scale=float(np.float32(amax / 448.0)))
    g = H.GpuCase(case)
    items = g.plan.items()
    assert all(it["kind"] == 1 for it in items)
    assert any(it["n_q"] > tq for it in items), "no item holds two query tiles"
    g.write_prefix()
    g.run()
    assert g.status() == 0, g.pkv.last_error()
    ref = oracle.forward(case)
    H.compare_out(g.out, ref["out"], H.FP8_TOL)
    H.compare_lse(g.lse, ref["lse"])
    assert np.array_equal(H.to_numpy_bits(g.k_cache), ref["k_cache"]), "k cache differs"


@pytest.mark.parametrize("P,G,causal,mixed", [(16, 4, True, False), (0, 4, False, False), (16, 8, True, True),
                                              (32, 2, True, False)])
def test_fp8_quantised_queries_prefill(P, G, causal, mixed):
    """fp8 cache with q_scale on prefill tiles: Q quantised to e4m3 and Q.K^T as
    tcgen05 kind::f8f6f4 MMAs on the raw cache tiles (P.V in f16), against the
    oracle's quantised-query reading; ragged lengths leave partial tiles."""
    import dataclasses
    rng = np.random.default_rng(300 + P + G + int(mixed))
    if mixed:
        spec = synth.Spec(batch=4, hq=2 * G, hkv=2, d=128, page_size=P, causal=causal,
                          softmax_scale=float(np.float32(1.0 / np.sqrt(128))), cache_dtype="fp8",
                          q_lens=np.array([1, 300, 1, 77], np.int32), cache_lens=np.array([900, 150, 40, 0], np.int32),
                          new_lens=np.array([1, 300, 1, 77], np.int32), capacity=1216, name="fp8-q8-mixed")
    else:
        spec = synth.uniform_spec("fp8-q8-prefill", 3, 200, 333, hq=2 * G, hkv=2, d=128, page_size=P,
                                  causal=causal, cache_dtype="fp8")
    case = synth.make_case(spec, rng)
    amax = float(np.abs(synth.bf16_bits_to_f32(case.q)).max())
    case = dataclasses.replace(case, q_scale=float(np.float32(amax / 448.0)))
    g = H.GpuCase(case)
    assert g.plan.stats()["num_prefill_items"] > 0
    g.write_prefix()
    g.run()
    assert g.status() == 0, g.pkv.last_error()
    ref = oracle.forward(case)
    H.compare_out(g.out, ref["out"], H.FP8_TOL)
    H.compare_lse(g.lse, ref["lse"])
    assert np.array_equal(H.to_numpy_bits(g.k_cache), ref["k_cache"]), "k cache differs"



@pytest.mark.parametrize("dtype,sms,q8,d", [("fp8", 152, False, 128), ("fp8", 12, False, 128), ("fp8", 152, True, 128),
                                            ("bf16", 152, False, 128), ("bf16", 8, False, 128),
                                            ("bf16", 152, False, 64), ("fp8", 152, False, 64)])
def test_decode_random_lengths_whole_and_split(dtype, sms, q8, d):
    """Decode batches of random lengths U[512, 4096] with the full GQA shape
    (Hq=32, Hkv=8, D=128 or 64, pages of 16, poisoned unused slots): at a few
    SMs the planner places the 192 units whole (no partials, no combine), at
    152 SMs (two CTAs an SM where rows are 128 bytes or fewer) it splits them
    to fill the CTAs; every row against the oracle, the cache byte for byte."""
    import dataclasses
    rng = np.random.default_rng(7100 + sms + (1 if q8 else 0))
    B = 24
    lc = rng.integers(512, 4097, B).astype(np.int32)
    ones = np.ones(B, np.int32)
    spec = synth.Spec(batch=B, hq=32, hkv=8, d=d, page_size=16, causal=True,
                      softmax_scale=float(np.float32(1.0 / np.sqrt(d))), cache_dtype=dtype, q_lens=ones,
                      cache_lens=lc, new_lens=ones.copy(), capacity=4112, name="decode-rand")
    case = synth.make_case(spec, rng, sentinel="nan")
    if q8:
        amax = float(np.abs(synth.bf16_bits_to_f32(case.q)).max())
        case = dataclasses.replace(case, q_scale=float(np.float32(amax / 448.0)))
    g, _ = run_full(case, num_sms=sms)
    st = g.plan.stats()
    assert (st["num_split_units"] > 0) == (sms == 152)
    two = d <= 128 if dtype == "fp8" else d == 64   # rows of 128 bytes or fewer: two CTAs an SM
    assert st["num_ctas"] == sms * (2 if two else 1)
