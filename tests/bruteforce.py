"""Pure-Python brute force of the whole call, written independently of the
oracle: its own cache walk, its own fp8 encode (nearest-code search over all
254 finite codes) and decode (bit fields), triple loops with ``math.exp``.
Only for tiny inputs."""
import math


def bf16(bits):
    import struct
    return struct.unpack("<f", struct.pack("<I", int(bits) << 16))[0]


def fp8_value(code):
    code = int(code)
    s = -1.0 if code & 0x80 else 1.0
    e = (code >> 3) & 0xF
    m = code & 7
    if e == 15 and m == 7:
        return float("nan")
    if e == 0:
        return s * (m / 8.0) * 2.0 ** -6
    return s * (1.0 + m / 8.0) * 2.0 ** (e - 7)


_FINITE = [c for c in range(256) if not ((c >> 3) & 0xF == 15 and c & 7 == 7)]


def fp8_nearest(y):
    """Nearest finite e4m3 code to y (ties -> even mantissa), clamped to +-448."""
    if y != y:
        return 0x7F
    best = None
    for c in _FINITE:
        v = fp8_value(c)
        if (v == 0.0) and (c & 0x80) != (0x80 if math.copysign(1.0, y) < 0 else 0):
            continue  # keep the sign of zero
        err = abs(v - y)
        key = (err, c & 1)
        if best is None or key < best[0]:
            best = (key, c)
    return best[1]


def f32mul(a, b):
    import numpy as np
    return float(np.float32(a) * np.float32(b))


def run(case):
    """Returns (out[t][h][d], lse[h][t]) as nested lists of floats."""
    spec = case.spec
    B, Hq, Hkv, D, P = spec.batch, spec.hq, spec.hkv, spec.d, spec.page_size
    G = Hq // Hkv
    fp8 = spec.cache_dtype == "fp8"

    def loc(b, pos):
        if P:
            return (int(case.block_table[b][pos // P]), pos % P)
        return (b, pos)

    # logical cache: dict (b, pos, hk) -> list of D cache codes/bits
    kc = {}
    vc = {}

    def read_phys(arr, b, pos, hk):
        a, s = loc(b, pos)
        return [int(x) for x in arr[a][s][hk]]

    lc = [int(x) for x in spec.cache_lens]
    ln = [int(x) for x in spec.new_lens]
    inv_k = float(__import__("numpy").float32(1.0) / __import__("numpy").float32(case.k_scale))
    inv_v = float(__import__("numpy").float32(1.0) / __import__("numpy").float32(case.v_scale))

    def enc(bits, inv):
        return fp8_nearest(f32mul(bf16(bits), inv))

    # cached prefix
    pre = 0
    for b in range(B):
        for pos in range(lc[b]):
            for hk in range(Hkv):
                if fp8 and case.prefix_k is not None:
                    kc[b, pos, hk] = [enc(x, inv_k) for x in case.prefix_k[pre + pos][hk]]
                    vc[b, pos, hk] = [enc(x, inv_v) for x in case.prefix_v[pre + pos][hk]]
                else:
                    kc[b, pos, hk] = read_phys(case.k_cache, b, pos, hk)
                    vc[b, pos, hk] = read_phys(case.v_cache, b, pos, hk)
        pre += lc[b]
    # new tokens
    off = 0
    for b in range(B):
        for t in range(ln[b]):
            for hk in range(Hkv):
                kr = [int(x) for x in case.k_new[off + t][hk]]
                vr = [int(x) for x in case.v_new[off + t][hk]]
                if fp8:
                    kr = [enc(x, inv_k) for x in kr]
                    vr = [enc(x, inv_v) for x in vr]
                kc[b, lc[b] + t, hk] = kr
                vc[b, lc[b] + t, hk] = vr
        off += ln[b]

    def val(code, scale):
        return fp8_value(code) * scale if fp8 else bf16(code)

    total_q = sum(int(x) for x in spec.q_lens)
    out = [[[0.0] * D for _ in range(Hq)] for _ in range(total_q)]
    lse = [[-math.inf] * total_q for _ in range(Hq)]
    t0 = 0
    for b in range(B):
        lq = int(spec.q_lens[b])
        lk = lc[b] + ln[b]
        for i in range(lq):
            for h in range(Hq):
                hk = h // G
                qv = [bf16(x) for x in case.q[t0 + i][h]]
                if getattr(case, "q_scale", None) is not None:  # Q quantised for Q K^T
                    np_ = __import__("numpy")
                    inv_q = float(np_.float32(1.0) / np_.float32(case.q_scale))
                    qs = float(np_.float32(case.q_scale))
                    qv = [fp8_value(fp8_nearest(f32mul(x, inv_q))) * qs for x in qv]
                scores = []
                for j in range(lk):
                    if spec.causal and j > i + lk - lq:
                        continue
                    kv = [val(x, case.k_scale) for x in kc[b, j, hk]]
                    s = sum(qv[d] * kv[d] for d in range(D)) * spec.softmax_scale
                    scores.append((j, s))
                if not scores:
                    continue
                m = max(s for _, s in scores)
                den = sum(math.exp(s - m) for _, s in scores)
                o = [0.0] * D
                for j, s in scores:
                    w = math.exp(s - m) / den
                    vv = [val(x, case.v_scale) for x in vc[b, j, hk]]
                    for d in range(D):
                        o[d] += w * vv[d]
                out[t0 + i][h] = o
                lse[h][t0 + i] = m + math.log(den)
        t0 += lq
    return out, lse, kc, vc
