"""Pins of the CPU oracle against things other than itself (no GPU).

* a pure-Python brute force (tests/bruteforce.py) on the tiny paged case and
  on 200 random tiny cases (bf16 and fp8 caches, paged and contiguous);
* hand-derived golden values (tests/golden/*.json);
* PyTorch's fp64 scaled_dot_product_attention with an explicit mask;
* invariants: softmax rows sum to 1, masked weights are exactly 0, page
  relabelling / layout changes / key permutations leave the output unchanged,
  split-KV merge equals the unsplit result, the append touches only its slots;
* special cases with closed forms (one key, constant keys, decode causal ==
  non-causal, empty rows).
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle
import synth
from tests import bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _expr(s):
    s = str(s)
    if s == "-inf":
        return -math.inf
    if "ln(" in s:
        return float(eval(s.replace("ln(", "math.log("), {"math": math}))
    return float(Fraction(s))


# ---------------------------------------------------------------------------
# golden hand cases
# ---------------------------------------------------------------------------
def _hand_cases():
    with open(os.path.join(GOLDEN, "attention_hand_cases.json")) as f:
        return json.load(f)


@pytest.mark.parametrize("case", _hand_cases()["cases"], ids=lambda c: c["name"])
def test_golden_hand_attention(case):
    q = np.array([[[_expr(x) for x in hd] for hd in tok] for tok in case["q"]])
    K = np.array(case["k"], dtype=np.float64)
    V = np.array(case["v"], dtype=np.float64)
    o, lse = oracle.attend(q, K, V, case["causal"], case["scale"])
    exp_o = np.array([[[_expr(x) for x in hd] for hd in tok] for tok in case["o"]])
    exp_l = np.array([[_expr(x) for x in row] for row in case["lse"]])
    np.testing.assert_allclose(o, exp_o, rtol=0, atol=1e-13)
    fin = np.isfinite(exp_l)
    assert np.array_equal(np.isfinite(lse), fin)
    np.testing.assert_allclose(lse[fin], exp_l[fin], rtol=0, atol=1e-13)


@pytest.mark.parametrize("vc", _hand_cases()["visible_counts"], ids=lambda v: str(v["q_lens"]))
def test_golden_visible_counts(vc):
    counts = []
    for lq, lc, ln in zip(vc["q_lens"], vc["cache_lens"], vc["new_lens"]):
        counts += list(oracle.visible_mask(lq, lc + ln, True).sum(axis=1))
    assert counts == vc["counts"]


# ---------------------------------------------------------------------------
# brute force
# ---------------------------------------------------------------------------
def _check_against_bruteforce(case, tol=1e-12):
    ref = oracle.forward(case)
    out, lse, kc, vc = bruteforce.run(case)
    out = np.array(out, dtype=np.float64).reshape(ref["out"].shape)
    lse = np.array(lse, dtype=np.float64).reshape(ref["lse"].shape)
    np.testing.assert_allclose(ref["out"], out, rtol=0, atol=tol)
    fin = np.isfinite(lse)
    assert np.array_equal(np.isfinite(ref["lse"]), fin)
    np.testing.assert_allclose(ref["lse"][fin], lse[fin], rtol=0, atol=tol)
    # appended / cached contents, position by position
    spec = case.spec
    for (b, pos, hk), codes in kc.items():
        idx = oracle.physical_slots(spec, case.block_table, b, np.array([pos]))
        got = ref["k_cache"][idx][0, hk]
        assert list(int(x) for x in got) == codes
        got = ref["v_cache"][idx][0, hk]
        assert list(int(x) for x in got) == vc[b, pos, hk]


@pytest.mark.parametrize("sentinel", ["finite", "nan"])
def test_bruteforce_config1(sentinel):
    _check_against_bruteforce(synth.config1(sentinel=sentinel))


@pytest.mark.parametrize("seed", range(200))
def test_bruteforce_random(seed):
    dtype = "fp8" if seed % 4 == 3 else "bf16"
    case = synth.random_case(seed, cache_dtype=dtype, with_new=(seed % 5 != 0),
                             q_equals_new=(seed % 7 != 0), sentinel="nan" if seed % 3 == 0 else "finite")
    _check_against_bruteforce(case)


# ---------------------------------------------------------------------------
# library cross-check
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(20))
def test_sdpa_crosscheck(seed):
    torch = pytest.importorskip("torch")
    case = synth.random_case(1000 + seed, max_cache=64, max_new=12, allow_zero=False)
    spec = case.spec
    ref = oracle.forward(case)
    cu = spec.cu_q
    for b in range(spec.batch):
        lq, lk = int(spec.q_lens[b]), int(spec.kv_lens[b])
        K = oracle.gather_sequence(spec, ref["k_cache"], case.block_table, b, lk)
        V = oracle.gather_sequence(spec, ref["v_cache"], case.block_table, b, lk)
        q = oracle.bf16_to_f64(case.q[cu[b]:cu[b] + lq])
        tq = torch.from_numpy(q).permute(1, 0, 2)                  # (Hq, lq, D)
        tk = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(spec.g, 0)
        tv = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(spec.g, 0)
        i = torch.arange(lq)[:, None]
        j = torch.arange(lk)[None, :]
        mask = (j <= i + (lk - lq)) if spec.causal else torch.ones(lq, lk, dtype=torch.bool)
        o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=mask,
                                                             scale=spec.softmax_scale)
        got = ref["out"][cu[b]:cu[b] + lq]
        np.testing.assert_allclose(got, o.permute(1, 0, 2).numpy(), rtol=0, atol=1e-12)


# ---------------------------------------------------------------------------
# invariants and closed forms
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(10))
def test_softmax_rows(seed):
    rng = np.random.default_rng(seed)
    lq, lk, hq, hkv, d = 5, 17, 4, 2, 8
    q = rng.standard_normal((lq, hq, d)) * 3
    K = rng.standard_normal((lk, hkv, d))
    V = rng.standard_normal((lk, hkv, d))
    for causal in (True, False):
        o, lse, w = oracle.attend(q, K, V, causal, 0.3, return_weights=True)
        mask = oracle.visible_mask(lq, lk, causal)
        np.testing.assert_allclose(w.sum(axis=2), 1.0, rtol=0, atol=1e-12)
        assert np.all(w >= 0) and np.all(w <= 1)
        assert np.all(w[:, ~mask] == 0.0)
        # o is exactly the weights applied to V
        for h in range(hq):
            np.testing.assert_allclose(o[:, h], w[h] @ V[:, h // 2], atol=1e-12)


def test_single_key_returns_value_row():
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 4, 8))
    K = rng.standard_normal((1, 2, 8))
    V = rng.standard_normal((1, 2, 8))
    o, lse = oracle.attend(q, K, V, True, 0.5)
    for h in range(4):
        assert np.array_equal(o[0, h], V[0, h // 2])
        assert lse[h, 0] == pytest.approx(0.5 * q[0, h] @ K[0, h // 2], abs=1e-14)


def test_constant_keys_give_mean_of_visible_values():
    rng = np.random.default_rng(4)
    lq, lk = 3, 9
    q = rng.standard_normal((lq, 2, 4))
    K = np.tile(rng.standard_normal((1, 1, 4)), (lk, 1, 1))
    V = rng.standard_normal((lk, 1, 4))
    o, lse = oracle.attend(q, K, V, True, 1.0)
    for i in range(lq):
        n = i + (lk - lq) + 1
        np.testing.assert_allclose(o[i, 0], V[:n, 0].mean(axis=0), atol=1e-13)
        np.testing.assert_allclose(lse[0, i], q[i, 0] @ K[0, 0] + math.log(n), atol=1e-12)


def test_decode_causal_equals_noncausal():
    rng = np.random.default_rng(5)
    q = rng.standard_normal((1, 4, 8))
    K = rng.standard_normal((30, 2, 8))
    V = rng.standard_normal((30, 2, 8))
    a = oracle.attend(q, K, V, True, 0.2)
    b = oracle.attend(q, K, V, False, 0.2)
    assert np.array_equal(a[0], b[0]) and np.array_equal(a[1], b[1])


def test_prefill_from_empty_cache_is_lower_triangular():
    m = oracle.visible_mask(7, 7, True)
    assert np.array_equal(m, np.tril(np.ones((7, 7), dtype=bool)))
    m = oracle.visible_mask(3, 8, True)   # bottom-right: last row sees everything
    assert m[-1].all() and m[0].sum() == 6


def test_empty_rows_are_zero_with_minus_inf_lse():
    q = np.ones((3, 1, 2))
    K = np.ones((1, 1, 2))
    V = np.full((1, 1, 2), 5.0)
    o, lse = oracle.attend(q, K, V, True, 1.0)
    assert np.all(o[:2] == 0) and np.all(np.isneginf(lse[0, :2]))
    assert np.all(o[2] == 5.0)
    o, lse = oracle.attend(np.ones((2, 1, 2)), np.zeros((0, 1, 2)), np.zeros((0, 1, 2)), False, 1.0)
    assert np.all(o == 0) and np.all(np.isneginf(lse))


@pytest.mark.parametrize("seed", range(8))
def test_noncausal_key_permutation_invariance(seed):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((4, 4, 8))
    K = rng.standard_normal((23, 2, 8))
    V = rng.standard_normal((23, 2, 8))
    p = rng.permutation(23)
    a = oracle.attend(q, K, V, False, 0.4)
    b = oracle.attend(q, K[p], V[p], False, 0.4)
    np.testing.assert_allclose(a[0], b[0], atol=1e-13)
    np.testing.assert_allclose(a[1], b[1], atol=1e-13)


@pytest.mark.parametrize("seed", range(6))
def test_page_relabel_and_contiguous_equivalence(seed):
    case = synth.random_case(300 + seed, page_size=4, max_cache=30, max_new=6, allow_zero=False)
    ref = oracle.forward(case)
    rel = synth.relabel_pages(case, np.random.default_rng(seed))
    r2 = oracle.forward(rel)
    assert np.array_equal(ref["out"], r2["out"]) and np.array_equal(ref["lse"], r2["lse"])
    con = synth.to_contiguous(case)
    r3 = oracle.forward(con)
    np.testing.assert_allclose(ref["out"], r3["out"], rtol=0, atol=1e-13)
    np.testing.assert_allclose(ref["lse"], r3["lse"], rtol=0, atol=1e-13)


def test_config1_paged_equals_contiguous():
    case = synth.config1()
    ref = oracle.forward(case)
    r3 = oracle.forward(synth.to_contiguous(case))
    np.testing.assert_allclose(ref["out"], r3["out"], rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", range(10))
def test_split_merge_equals_unsplit(seed):
    rng = np.random.default_rng(seed)
    lq, lk = int(rng.integers(1, 6)), int(rng.integers(6, 60))
    q = rng.standard_normal((lq, 4, 8)) * 2
    K = rng.standard_normal((lk, 2, 8))
    V = rng.standard_normal((lk, 2, 8))
    cuts = sorted(set(rng.integers(1, lk, size=int(rng.integers(1, 5))).tolist()))
    bounds = [0] + cuts + [lk]
    for causal in (True, False):
        o, lse = oracle.attend(q, K, V, causal, 0.35)
        o2, lse2 = oracle.split_forward(q, K, V, causal, 0.35, bounds)
        np.testing.assert_allclose(o2, o, rtol=0, atol=1e-13)
        np.testing.assert_allclose(lse2, lse, rtol=0, atol=1e-13)


def test_split_merge_handles_empty_chunk():
    # causal decode-like row where a later chunk is fully masked
    q = np.ones((1, 1, 2))
    K = np.arange(12, dtype=float).reshape(6, 1, 2) / 10
    V = np.arange(12, dtype=float).reshape(6, 1, 2)
    o, lse = oracle.attend(q[:, :, :], K, V, True, 1.0)
    lq = 1
    o2, l2 = oracle.split_forward(q, K, V, True, 1.0, [0, 3, 6])
    np.testing.assert_allclose(o2, o, atol=1e-13)
    o_parts = np.stack([o, np.zeros_like(o)])
    l_parts = np.stack([lse.T, np.full_like(lse.T, -np.inf)])
    o3, l3 = oracle.combine_partials(o_parts, l_parts)
    np.testing.assert_allclose(o3, o, atol=1e-15)


@pytest.mark.parametrize("seed", range(6))
def test_append_touches_only_its_slots(seed):
    for dtype in ("bf16", "fp8"):
        case = synth.random_case(500 + seed, cache_dtype=dtype, max_cache=30, max_new=9)
        spec = case.spec
        kc0, vc0 = oracle.prepare_prefix(case)
        kc, vc = oracle.append_kv(spec, kc0, vc0, case.block_table, case.k_new, case.v_new,
                                  case.k_scale, case.v_scale)
        touched = np.zeros(kc.shape[:2], dtype=bool)
        cu = spec.cu_new
        for b in range(spec.batch):
            for t in range(int(spec.new_lens[b])):
                pos = int(spec.cache_lens[b]) + t
                idx = oracle.physical_slots(spec, case.block_table, b, np.array([pos]))
                touched[idx] = True
                row_k = kc[idx][0]
                want = case.k_new[cu[b] + t]
                if dtype == "fp8":
                    want = oracle.fp8_quantize(want, case.k_scale)
                assert np.array_equal(row_k, want)
        assert np.array_equal(kc[~touched], kc0[~touched])
        assert np.array_equal(vc[~touched], vc0[~touched])


def test_algorithmic_work_closed_forms():
    case = synth.config3(causal=True, draw_values=False)
    w = oracle.algorithmic_work(case.spec)
    assert w["pairs"] == 8 * (512 * 1536 + 512 * 513 // 2)
    case = synth.config3(causal=False, draw_values=False)
    assert oracle.algorithmic_work(case.spec)["pairs"] == 8 * 512 * 2048
    spec = synth.config2(draw_values=False).spec
    w = oracle.algorithmic_work(spec)
    assert w["kv_bytes"] == int(spec.kv_lens.sum()) * 8 * 128 * 2 * 2


# ---------------------------------------------------------------------------
# forward_rows: the per-row oracle the full-size parity tests sample from
# ---------------------------------------------------------------------------
def _rows_equal_forward(case):
    """forward_rows over EVERY query row equals forward() row by row: its own
    causal horizon, per-sequence gather and empty-row handling against the
    whole-sequence masked softmax."""
    spec = case.spec
    ref = oracle.forward(case)
    rows = [(b, i) for b in range(spec.batch) for i in range(int(spec.q_lens[b]))]
    if not rows:
        return
    # visit the rows in a shuffled order: the gather cache of forward_rows
    # must not depend on the rows of one sequence arriving together
    order = np.random.default_rng(len(rows)).permutation(len(rows))
    rows = [rows[k] for k in order]
    o, lse = oracle.forward_rows(case, ref["k_cache"], ref["v_cache"], rows)
    idx = [int(spec.cu_q[b]) + i for b, i in rows]
    np.testing.assert_allclose(o, ref["out"][idx], rtol=0, atol=1e-13)
    want = ref["lse"][:, idx]
    fin = np.isfinite(want)
    assert np.array_equal(np.isfinite(lse), fin)
    assert np.all(np.isneginf(lse[~fin]))
    np.testing.assert_allclose(lse[fin], want[fin], rtol=0, atol=1e-13)


@pytest.mark.parametrize("seed", range(60))
def test_forward_rows_equals_forward_random(seed):
    # causal and non-causal, Lq != Ln (and Lq > Lk: rows with an empty causal
    # horizon), zero lengths, paged / contiguous, bf16 / fp8, GQA group sizes
    case = synth.random_case(4000 + seed, causal=(seed % 2 == 0), cache_dtype="fp8" if seed % 5 == 4 else "bf16",
                             with_new=(seed % 7 != 6), q_equals_new=(seed % 3 != 0), max_cache=50, max_new=12)
    _rows_equal_forward(case)


def test_forward_rows_equals_forward_config1():
    _rows_equal_forward(synth.config1())
    _rows_equal_forward(synth.config1(sentinel="nan"))


def test_forward_rows_empty_horizons():
    """Rows that see no key: Lk = 0, and causal Lq > Lk (the first Lq - Lk rows)."""
    spec = synth.Spec(batch=3, hq=4, hkv=2, d=16, page_size=4, causal=True, softmax_scale=0.25,
                      cache_dtype="bf16", q_lens=np.array([3, 5, 2], np.int32),
                      cache_lens=np.array([0, 1, 6], np.int32), new_lens=np.array([0, 1, 2], np.int32),
                      capacity=8, name="empty-horizons")
    case = synth.make_case(spec, np.random.default_rng(9))
    ref = oracle.forward(case)
    assert np.all(ref["out"][:3] == 0) and np.all(np.isneginf(ref["lse"][:, :3]))   # Lk = 0
    assert np.all(ref["out"][3:6] == 0) and np.all(np.isfinite(ref["lse"][:, 6:8]))  # Lq 5 on Lk 2
    _rows_equal_forward(case)


def test_forward_rows_equals_forward_mixed_subset():
    """Sequences of the mixed in-flight batch: a 2048-token prefill request on
    its cached prefix and three long decode requests."""
    full = synth.config4()
    pre = [b for b in range(full.spec.batch) if full.spec.q_lens[b] > 1][0]
    dec = [b for b in range(full.spec.batch) if full.spec.q_lens[b] == 1][:3]
    _rows_equal_forward(synth.subset_case(full, [dec[0], pre, dec[1], dec[2]]))


# ---------------------------------------------------------------------------
# byte and flop counts behind the roofline numbers, counted by hand
# ---------------------------------------------------------------------------
def test_algorithmic_work_hand_count_config1():
    """The tiny paged workload counted by hand: B=2, Hq=4, Hkv=2, D=64, page
    16, cache lengths {37, 5}, new tokens = queries {3, 1}, so Lk = {40, 6}."""
    import bench
    spec = synth.config1().spec
    kv_read = (40 + 6) * 2 * 64 * 2 * 2       # keys x kv heads x D x (K, V) x 2 bytes
    q_read_o_write = (3 + 1) * 4 * 64 * 2 * 2  # query rows x q heads x D x 2 bytes x (read q, write out)
    new_kv = (3 + 1) * 2 * 64 * 2 * (2 + 2)   # new tokens x kv heads x D x (K, V) x (read bf16 + write bf16)
    table = (3 + 1) * 4                        # pages used: ceil(40/16) + ceil(6/16), 4 bytes each
    assert (kv_read, q_read_o_write, new_kv, table) == (23552, 4096, 4096, 16)
    # causal pairs: sequence 0 rows see 38, 39, 40 keys; sequence 1's row sees 6
    pairs = 38 + 39 + 40 + 6
    w = oracle.algorithmic_work(spec)
    assert w["kv_bytes"] == kv_read
    assert w["bytes"] == kv_read + q_read_o_write + new_kv + table == 31760
    assert w["pairs"] == pairs == 123
    assert w["flops"] == 4 * 64 * 4 * pairs
    sw = bench.step_work(spec)
    assert sw["attn_bytes"] == kv_read + q_read_o_write + table == 27664
    assert sw["append_bytes"] == new_kv
    assert sw["bytes"] == w["bytes"] and sw["flops"] == w["flops"]
    # fp8 cache: K/V are read and written one byte each, new K/V still read as bf16
    fspec = synth.Spec(**{**spec.__dict__, "cache_dtype": "fp8"})
    fw = oracle.algorithmic_work(fspec)
    assert fw["bytes"] == (40 + 6) * 2 * 64 * 2 * 1 + q_read_o_write + (3 + 1) * 2 * 64 * 2 * (2 + 1) + table
    assert bench.step_work(fspec)["bytes"] == fw["bytes"]
    # non-causal: every query row sees every key of its sequence
    nspec = synth.Spec(**{**spec.__dict__, "causal": False})
    assert oracle.algorithmic_work(nspec)["pairs"] == 3 * 40 + 1 * 6 == bench.step_work(nspec)["flops"] // (4 * 64 * 4)
