"""Pins of the oracle's fp8 e4m3 codec (no GPU): golden format facts, an
independent nearest-code search, PyTorch's float8_e4m3fn conversions, and
round trips over every code and every bf16 bit pattern."""
import json
import math
import os

import numpy as np
import pytest

import oracle
import synth
from tests import bruteforce

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden():
    with open(os.path.join(GOLDEN, "e4m3_codes.json")) as f:
        return json.load(f)


def _num(s):
    try:
        return float(s)          # keeps the sign of "-0"
    except ValueError:
        return float(eval(s, {"__builtins__": {}}, {"nan": float("nan")}))


def test_golden_decode():
    for code, val in _golden()["decode"]:
        got = oracle.e4m3_decode(np.array([int(code, 16)], np.uint8))[0]
        want = _num(val)
        if math.isnan(want):
            assert math.isnan(got)
        else:
            assert got == want and math.copysign(1, got) == math.copysign(1, want)


def test_golden_encode():
    for x, code, why in _golden()["encode_rne_satfinite"]:
        got = oracle.e4m3_encode(np.array([_num(x)], np.float32))[0]
        assert got == int(code, 16), why


def test_decode_all_codes_matches_torch():
    torch = pytest.importorskip("torch")
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.e4m3_decode(codes)
    theirs = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    nan = np.isnan(theirs)
    assert np.array_equal(np.isnan(ours), nan)
    assert np.array_equal(ours[~nan], theirs[~nan])
    assert nan.sum() == 2


def test_decode_matches_bitfield_formula():
    for c in range(256):
        a = oracle.e4m3_decode(np.array([c], np.uint8))[0]
        b = bruteforce.fp8_value(c)
        assert (math.isnan(a) and math.isnan(b)) or a == b


def test_roundtrip_every_finite_code():
    codes = np.array([c for c in range(256) if (c & 0x7F) != 0x7F], np.uint8)
    back = oracle.e4m3_encode(oracle.e4m3_decode(codes).astype(np.float32))
    assert np.array_equal(back, codes)


def test_every_bf16_pattern_against_torch_cast():
    torch = pytest.importorskip("torch")
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    x = (bits.astype(np.uint32) << 16).view(np.float32)
    ours = oracle.e4m3_encode(x)
    finite = np.isfinite(x)
    inrange = finite & (np.abs(x) < 464.0)       # below the 448/480 midpoint torch rounds too
    theirs = torch.from_numpy(x.copy()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(ours[inrange], theirs[inrange])
    big = finite & (np.abs(x) >= 448.0)
    assert np.all((ours[big] & 0x7F) == 0x7E)
    assert np.array_equal(ours[big] >> 7, np.signbit(x[big]).astype(np.uint8))
    assert np.all(ours[np.isnan(x)] == 0x7F)


def test_encode_against_nearest_code_search():
    rng = np.random.default_rng(0)
    vals = np.concatenate([rng.standard_normal(400) * 50,
                           rng.standard_normal(200) * 0.01,
                           rng.uniform(-600, 600, 100)]).astype(np.float32)
    # exact midpoints between neighbouring codes
    grid = np.sort(np.unique(oracle.e4m3_decode(np.arange(0, 0x7F, dtype=np.uint8))))
    mids = ((grid[:-1] + grid[1:]) / 2).astype(np.float32)
    vals = np.concatenate([vals, mids, -mids])
    ours = oracle.e4m3_encode(vals)
    for v, c in zip(vals, ours):
        assert c == bruteforce.fp8_nearest(float(v)), v


def test_quantize_uses_single_fp32_multiply():
    # a value whose product with 1/scale lands exactly on a tie only when the
    # multiply is rounded to fp32 first (fma-free): check against explicit fp32 math
    rng = np.random.default_rng(1)
    scale = float(np.float32(3.7) / np.float32(448.0))
    inv = np.float32(1.0) / np.float32(scale)
    x_bits = (rng.standard_normal(5000).astype(np.float32).view(np.uint32) >> 16).astype(np.uint16)
    x = (x_bits.astype(np.uint32) << 16).view(np.float32)
    want = oracle.e4m3_encode((x * inv).astype(np.float32))
    assert np.array_equal(oracle.fp8_quantize(x_bits, scale), want)


# ---------------------------------------------------------------------------
# quantised queries (Q . K^T on fp8): the same encode as the cache
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("seed", range(12))
def test_quantised_queries_against_bruteforce(seed):
    """Oracle with q_scale vs the brute force's own nearest-code encode of Q."""
    import dataclasses
    from tests import bruteforce
    case = synth.random_case(500 + seed, cache_dtype="fp8")
    amax = float(np.abs(synth.bf16_bits_to_f32(case.q)).max())
    case = dataclasses.replace(case, q_scale=float(np.float32(max(amax, 1e-3) / 448.0)))
    ref = oracle.forward(case)
    out, lse, _, _ = bruteforce.run(case)
    np.testing.assert_allclose(ref["out"], np.array(out, dtype=np.float64).reshape(ref["out"].shape), rtol=0,
                               atol=1e-12)
    lse_b = np.array(lse, dtype=np.float64).reshape(ref["lse"].shape)
    assert np.array_equal(np.isfinite(ref["lse"]), np.isfinite(lse_b))
    fin = np.isfinite(lse_b)
    np.testing.assert_allclose(ref["lse"][fin], lse_b[fin], rtol=0, atol=1e-12)


def test_quantised_queries_identity_on_representable_values():
    """Queries that are e4m3 codes times the scale quantise to themselves: the
    call with q_scale then equals the plain call."""
    import dataclasses
    case = synth.random_case(77, cache_dtype="fp8", batch=3)
    q_scale = float(np.float32(0.03125))           # a power of two: code * scale is exact in bf16
    rng = np.random.default_rng(3)
    codes = rng.integers(0, 0x7E, size=case.q.shape, dtype=np.int64).astype(np.uint8)
    codes[rng.random(case.q.shape) < 0.5] |= 0x80
    vals = (oracle.e4m3_decode(codes) * q_scale).astype(np.float32)
    q_bits = synth.f32_to_bf16_bits(vals)
    assert np.array_equal(synth.bf16_bits_to_f32(q_bits), vals)   # exactly representable
    plain = dataclasses.replace(case, q=q_bits)
    quant = dataclasses.replace(plain, q_scale=q_scale)
    a, b = oracle.forward(plain), oracle.forward(quant)
    assert np.array_equal(a["out"], b["out"]) and np.array_equal(a["lse"], b["lse"])
