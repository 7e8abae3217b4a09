"""Pins of the CPU oracle against facts that do not come from the oracle itself.

Each test names what fixes the expected value: a hand-worked fixture under tests/golden/
(with its citation), a closed form, a brute-force integer sum, a full stable sort, an fp64
evaluation within a derived rounding bound, or an identity the layer must satisfy
(forced all-experts = dense loop, identical experts, batch invariance, the pages' IDOT
accuracy).  CPU only.
"""
import json
import math
import os
from fractions import Fraction

import numpy as np
import pytest

from gen import gen
from gen import workloads as W
from oracle import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
EPS32 = 2.0 ** -24  # unit roundoff of fp32


def golden(name):
    with open(os.path.join(GOLDEN, name)) as fh:
        return json.load(fh)


def decode_nibbles(packed):
    """independent int4 decode: two's complement, low nibble = even element"""
    p = packed.astype(np.int16)
    lo = p & 15
    hi = p >> 4
    lo = np.where(lo >= 8, lo - 16, lo)
    hi = np.where(hi >= 8, hi - 16, hi)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 2,), dtype=np.int16)
    out[..., 0::2] = lo
    out[..., 1::2] = hi
    return out


def round_half_away(fr):
    """exact rational rounding, half away from zero"""
    s = 1 if fr >= 0 else -1
    a = abs(fr)
    n = math.floor(a)
    if a - n >= Fraction(1, 2):
        n += 1
    return s * n


# ------------------------------------------------------------------ generator ----------

def test_generator_splitmix64_published_vector():
    g = golden("splitmix64.json")
    got = [gen.draw_raw_host(g["seed"], n) for n in range(5)]
    assert got == [int(v) for v in g["outputs"]]


def test_generator_normal_moments():
    z = gen.normal_host((1 << 18,), 0, 0, gen.T_X, 0)
    assert abs(float(z.mean())) < 0.01
    assert abs(float(z.std()) - 1.0) < 0.01
    # Irwin-Hall(12) is bounded by 6 sigma and the 16-bit grid is exact in fp32
    assert np.abs(z).max() <= 6.0
    assert np.all(z * 65536.0 == np.round(z * 65536.0))


# ------------------------------------------------------------------ formats ------------

def test_int4_nibble_exhaustive():
    """all 256 (lo, hi) code pairs pack into distinct bytes and decode back"""
    codes = np.array([(a, b) for a in range(-8, 8) for b in range(-8, 8)], dtype=np.int8).ravel()
    packed = np.empty(codes.size // 2, dtype=np.uint8)
    O.lib().orc_pack_i4_row(codes.ctypes.data, codes.size, packed.ctypes.data)
    assert sorted(packed.tolist()) == list(range(256))
    assert np.array_equal(decode_nibbles(packed), codes)
    for j in range(0, codes.size, 37):
        assert O.lib().orc_i4_get(packed.ctypes.data, j) == codes[j]


def test_int4_pack_golden():
    g = golden("int4_pack.json")
    codes = np.array(g["codes"], dtype=np.int8)
    packed = np.empty(codes.size // 2, dtype=np.uint8)
    O.lib().orc_pack_i4_row(codes.ctypes.data, codes.size, packed.ctypes.data)
    assert [f"{b:02x}" for b in packed] == g["bytes_hex"]


def test_int4_row_quant_golden():
    g = golden("int4_row_quant.json")
    w = np.array([g["w"]], dtype=np.float32)
    packed, s = O.quantize_i4_rows(w)
    assert s[0] == np.float32(np.float32(0.7) / np.float32(7))
    assert decode_nibbles(packed)[0].tolist() == g["codes"]


def test_int4_row_quant_bounds():
    rng = np.random.default_rng(1)
    w = (rng.standard_normal((64, 256)) * rng.uniform(0.001, 3, (64, 1))).astype(np.float32)
    w[3] = 0.0
    packed, s = O.quantize_i4_rows(w)
    q = decode_nibbles(packed).astype(np.float64)
    amax = np.abs(w).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(7)).astype(np.float32))
    assert s[3] == 0 and np.all(q[3] == 0)
    assert q.min() >= -7 and q.max() <= 7
    live = s > 0
    err = np.abs(w[live].astype(np.float64) - s[live, None].astype(np.float64) * q[live])
    assert np.all(err <= s[live, None] * (0.5 + 1e-5))
    arg = np.abs(w).argmax(axis=1)
    ext = q[np.arange(64), arg]
    assert np.all(np.abs(ext[live]) == 7)
    assert np.all(np.sign(ext[live]) == np.sign(w[np.arange(64), arg][live]))


def test_q8_golden():
    g = golden("q8_block.json")
    x = np.array([-15.875] + [np.float32(0.3) * np.float32(j - 16) for j in range(1, 32)],
                 dtype=np.float32)
    q, d = O.quantize_q8(x)
    assert d[0] == np.float32(g["scale"])
    assert q.tolist() == g["codes"]


def test_q8_exact_rational_rounding():
    """codes equal exact-rational round(x / d) wherever x/d is not within 1e-4 of a tie"""
    rng = np.random.default_rng(2)
    x = (rng.standard_normal(32 * 200) * rng.uniform(0.01, 10, 32 * 200)).astype(np.float32)
    x[64:96] = 0.0
    q, d = O.quantize_q8(x)
    xb = x.reshape(-1, 32)
    amax = np.abs(xb).max(axis=1)
    assert np.array_equal(d, (amax / np.float32(127)).astype(np.float32))
    assert d[2] == 0 and np.all(q[64:96] == 0)
    qb = q.reshape(-1, 32)
    checked = 0
    for b in range(xb.shape[0]):
        if d[b] == 0:
            continue
        for j in range(32):
            r = Fraction(float(xb[b, j])) / Fraction(float(d[b]))
            frac = abs(r - math.floor(r))
            if abs(frac - Fraction(1, 2)) < Fraction(1, 10000):
                continue
            assert qb[b, j] == max(-127, min(127, round_half_away(r)))
            checked += 1
        assert abs(int(qb[b, np.abs(xb[b]).argmax()])) == 127
    assert checked > 6000


# ------------------------------------------------------------------ integer dots -------

def test_block_dot_brute_force():
    rng = np.random.default_rng(3)
    cols = 256
    packed = rng.integers(0, 256, (16, cols // 2), dtype=np.uint8)
    packed[0] = 0x88  # every code -8
    qx = rng.integers(-127, 128, cols, dtype=np.int8)
    qx[:32] = -127
    W4 = decode_nibbles(packed).astype(np.int64)
    for r in range(16):
        for b in range(cols // 32):
            ref = int(np.sum(W4[r, 32 * b:32 * b + 32] * qx[32 * b:32 * b + 32].astype(np.int64)))
            got = O.lib().orc_block_dot(packed[r].ctypes.data, qx.ctypes.data, b)
            assert got == ref
    assert O.lib().orc_block_dot(packed[0].ctypes.data, qx.ctypes.data, 0) == 32 * 8 * 127


def test_matvec_accumulators_brute_force():
    rng = np.random.default_rng(4)
    rows, cols = 40, 512
    packed = rng.integers(0, 256, (rows, cols // 2), dtype=np.uint8)
    s = rng.uniform(0.001, 0.01, rows).astype(np.float32)
    x = rng.standard_normal(cols).astype(np.float32)
    qx, dx = O.quantize_q8(x)
    out, A = O.i4_matvec(packed, s, cols, qx, dx, want_A=True)
    W4 = decode_nibbles(packed).astype(np.int64)
    ref = (W4.reshape(rows, -1, 32) * qx.astype(np.int64).reshape(1, -1, 32)).sum(axis=2)
    assert np.array_equal(A, ref)
    # fp64 value from the same integers, within the canonical sum's rounding bound
    exact = s.astype(np.float64) * (ref * dx.astype(np.float64)).sum(axis=1)
    mag = np.abs(s.astype(np.float64)) * (np.abs(ref) * dx.astype(np.float64)).sum(axis=1)
    nb = cols // 32
    bound = (math.ceil(nb / 32) + 5 + 2) * EPS32 * mag
    assert np.all(np.abs(out.astype(np.float64) - exact) <= bound)


# ------------------------------------------------------------------ int8 rows ----------

def test_int8_row_quant_golden():
    g = golden("int8_row_quant.json")
    w = np.array([g["w"]], dtype=np.float32)
    q, s = O.quantize_i8_rows(w)
    assert s[0] == np.float32(np.float32(1.27) / np.float32(127))
    assert q[0].tolist() == g["codes"]


def test_int8_row_quant_bounds():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((64, 256)) * rng.uniform(0.001, 3, (64, 1))).astype(np.float32)
    w[5] = 0.0
    q8, s = O.quantize_i8_rows(w)
    q = q8.astype(np.float64)
    amax = np.abs(w).max(axis=1)
    assert np.array_equal(s, (amax / np.float32(127)).astype(np.float32))
    assert s[5] == 0 and np.all(q[5] == 0)
    assert q.min() >= -127 and q.max() <= 127
    live = s > 0
    err = np.abs(w[live].astype(np.float64) - s[live, None].astype(np.float64) * q[live])
    assert np.all(err <= s[live, None] * (0.5 + 1e-5))
    # the largest magnitude of every live row lands on +-127 with its sign
    arg = np.abs(w).argmax(axis=1)
    ext = q[np.arange(64), arg]
    assert np.all(np.abs(ext[live]) == 127)
    assert np.all(np.sign(ext[live]) == np.sign(w[np.arange(64), arg][live]))


def test_int8_codes_round_trip_exhaustively():
    # a row holding every code -127..127 times a power-of-two step is reproduced exactly
    codes = np.arange(-127, 128, dtype=np.float32)
    w = (codes * np.float32(2.0 ** -7)).reshape(1, -1)
    w = np.concatenate([w, np.zeros((1, 1), np.float32)], axis=1)  # 256 columns
    q, s = O.quantize_i8_rows(w)
    assert s[0] == np.float32(2.0 ** -7)
    assert np.array_equal(q[0, :255].astype(np.int64), codes.astype(np.int64))


def test_i8_block_dot_brute_force():
    rng = np.random.default_rng(12)
    cols = 256
    W = rng.integers(-127, 128, (16, cols), dtype=np.int8)
    W[0] = -127
    qx = rng.integers(-127, 128, cols, dtype=np.int8)
    qx[:32] = -127
    for r in range(16):
        for b in range(cols // 32):
            ref = int(np.sum(W[r, 32 * b:32 * b + 32].astype(np.int64) * qx[32 * b:32 * b + 32].astype(np.int64)))
            assert O.lib().orc_i8_block_dot(W[r].ctypes.data, qx.ctypes.data, b) == ref
    assert O.lib().orc_i8_block_dot(W[0].ctypes.data, qx.ctypes.data, 0) == 32 * 127 * 127


def test_i8_matvec_accumulators_brute_force():
    rng = np.random.default_rng(13)
    rows, cols = 40, 512
    W = rng.integers(-127, 128, (rows, cols), dtype=np.int8)
    s = rng.uniform(0.0001, 0.001, rows).astype(np.float32)
    x = rng.standard_normal(cols).astype(np.float32)
    qx, dx = O.quantize_q8(x)
    out, A = O.i8_matvec(W, s, cols, qx, dx, want_A=True)
    ref = (W.astype(np.int64).reshape(rows, -1, 32) * qx.astype(np.int64).reshape(1, -1, 32)).sum(axis=2)
    assert np.array_equal(A, ref)
    # fp64 value from the same integers, within the canonical sum's rounding bound
    exact = s.astype(np.float64) * (ref * dx.astype(np.float64)).sum(axis=1)
    mag = np.abs(s.astype(np.float64)) * (np.abs(ref) * dx.astype(np.float64)).sum(axis=1)
    nb = cols // 32
    bound = (math.ceil(nb / 32) + 5 + 2) * EPS32 * mag
    assert np.all(np.abs(out.astype(np.float64) - exact) <= bound)


# ------------------------------------------------------------------ int2 rows ---------

def decode_i2(packed):
    """independent int2 decode: two's-complement 2-bit fields, lowest bits = element 4i"""
    p = packed.astype(np.int16)
    out = np.empty(packed.shape[:-1] + (packed.shape[-1] * 4,), dtype=np.int16)
    for k in range(4):
        c = (p >> (2 * k)) & 3
        out[..., k::4] = np.where(c >= 2, c - 4, c)
    return out


def test_int2_decode_golden():
    for case in golden("int2_rows.json")["decode"]:
        row = np.array([case["byte"]], dtype=np.uint8)
        got = [O.lib().orc_i2_get(row.ctypes.data, k) for k in range(4)]
        assert got == case["codes"], case["why"]


def test_int2_row_quant_golden():
    rows = golden("int2_rows.json")["rows"]
    w = np.array([r["w"] for r in rows], dtype=np.float32)
    packed, s = O.quantize_i2_rows(w)
    assert s.tolist() == [float(np.float32(0.3)), 1.0, 0.0]
    for i, r in enumerate(rows):
        assert packed[i].tolist() == r["bytes"], r["why"]
        got = [O.lib().orc_i2_get(packed[i].ctypes.data, j) for j in range(8)]
        assert got == r["codes"], r["why"]


def test_int2_pack_exhaustive():
    """all 256 four-code tuples over [-2, 1] pack into distinct bytes and decode back"""
    codes = np.array([(a, b, c, e) for a in range(-2, 2) for b in range(-2, 2)
                      for c in range(-2, 2) for e in range(-2, 2)], dtype=np.int8).ravel()
    packed = np.empty(codes.size // 4, dtype=np.uint8)
    O.lib().orc_pack_i2_row(codes.ctypes.data, codes.size, packed.ctypes.data)
    assert sorted(packed.tolist()) == list(range(256))
    assert np.array_equal(decode_i2(packed), codes)
    got = np.array([O.lib().orc_i2_get(packed.ctypes.data, j) for j in range(codes.size)])
    assert np.array_equal(got, codes)


def test_int2_row_quant_bounds():
    rng = np.random.default_rng(14)
    w = (rng.standard_normal((64, 256)) * rng.uniform(0.001, 3, (64, 1))).astype(np.float32)
    w[9] = 0.0
    packed, s = O.quantize_i2_rows(w)
    q = decode_i2(packed).astype(np.float64)
    amax = np.abs(w).max(axis=1)
    assert np.array_equal(s, amax)
    assert s[9] == 0 and np.all(q[9] == 0)
    assert q.min() >= -1 and q.max() <= 1
    live = s > 0
    err = np.abs(w[live].astype(np.float64) - s[live, None].astype(np.float64) * q[live])
    assert np.all(err <= s[live, None] * (0.5 + 1e-6))
    arg = np.abs(w).argmax(axis=1)
    ext = q[np.arange(64), arg]
    assert np.all(ext[live] == np.sign(w[np.arange(64), arg][live]))


def test_i2_block_dot_brute_force():
    rng = np.random.default_rng(15)
    cols = 256
    W = rng.integers(0, 256, (16, cols // 4), dtype=np.uint8)  # every field pattern, -2 included
    W[0] = 0xAA
    qx = rng.integers(-127, 128, cols, dtype=np.int8)
    qx[:32] = -127
    Wd = decode_i2(W).astype(np.int64)
    for r in range(16):
        for b in range(cols // 32):
            ref = int(np.sum(Wd[r, 32 * b:32 * b + 32] * qx[32 * b:32 * b + 32].astype(np.int64)))
            assert O.lib().orc_i2_block_dot(W[r].ctypes.data, qx.ctypes.data, b) == ref
    assert O.lib().orc_i2_block_dot(W[0].ctypes.data, qx.ctypes.data, 0) == 32 * 2 * 127


def test_i2_matvec_accumulators_brute_force():
    rng = np.random.default_rng(16)
    rows, cols = 40, 512
    W = rng.integers(0, 256, (rows, cols // 4), dtype=np.uint8)
    s = rng.uniform(0.0001, 0.001, rows).astype(np.float32)
    x = rng.standard_normal(cols).astype(np.float32)
    qx, dx = O.quantize_q8(x)
    out, A = O.i2_matvec(W, s, cols, qx, dx, want_A=True)
    ref = (decode_i2(W).astype(np.int64).reshape(rows, -1, 32)
           * qx.astype(np.int64).reshape(1, -1, 32)).sum(axis=2)
    assert np.array_equal(A, ref)
    exact = s.astype(np.float64) * (ref * dx.astype(np.float64)).sum(axis=1)
    mag = np.abs(s.astype(np.float64)) * (np.abs(ref) * dx.astype(np.float64)).sum(axis=1)
    nb = cols // 32
    bound = (math.ceil(nb / 32) + 5 + 2) * EPS32 * mag
    assert np.all(np.abs(out.astype(np.float64) - exact) <= bound)


def test_i2_i4_i8_rows_of_equal_codes_agree():
    """codes in [-1, 1] stored as int2, int4 and int8 rows give the same accumulators and the
    same fp32 outputs: the three formats differ only in how a code is stored"""
    rng = np.random.default_rng(17)
    rows, cols = 24, 1024
    codes = rng.integers(-1, 2, (rows, cols), dtype=np.int8)
    s = rng.uniform(0.001, 0.01, rows).astype(np.float32)
    x = rng.standard_normal(cols).astype(np.float32)
    qx, dx = O.quantize_q8(x)
    p2 = np.empty((rows, cols // 4), dtype=np.uint8)
    p4 = np.empty((rows, cols // 2), dtype=np.uint8)
    for r in range(rows):
        O.lib().orc_pack_i2_row(codes[r].ctypes.data, cols, p2[r].ctypes.data)
        O.lib().orc_pack_i4_row(codes[r].ctypes.data, cols, p4[r].ctypes.data)
    o2, A2 = O.i2_matvec(p2, s, cols, qx, dx, want_A=True)
    o4, A4 = O.i4_matvec(p4, s, cols, qx, dx, want_A=True)
    o8, A8 = O.i8_matvec(codes, s, cols, qx, dx, want_A=True)
    assert np.array_equal(A2, A8) and np.array_equal(A4, A8)
    assert np.array_equal(o2.view(np.uint32), o8.view(np.uint32))
    assert np.array_equal(o4.view(np.uint32), o8.view(np.uint32))


# ------------------------------------------------------------------ canonical fp32 -----

def ulp32(v):
    v = abs(v)
    if v < 2.0 ** -126:
        return 2.0 ** -149
    return 2.0 ** (math.floor(math.log2(v)) - 23)


def test_exp_within_two_ulp():
    xs = np.concatenate([np.linspace(-87.0, 88.7, 20001), np.linspace(-1, 1, 4001),
                         np.array([0.0, -0.0, 1e-30, -1e-30, 88.72, -87.33])]).astype(np.float32)
    ys = O.exp(xs)
    worst = 0.0
    for x, y in zip(xs.tolist(), ys.tolist()):
        ref = math.exp(x)
        worst = max(worst, abs(y - ref) / ulp32(ref))
    assert worst <= 2.0, worst
    assert O.lib().orc_exp(0.0) == 1.0
    assert O.lib().orc_exp(1.0) == np.float32(math.e)
    assert math.isinf(O.lib().orc_exp(89.5)) and math.isinf(O.lib().orc_exp(1e30))
    assert O.lib().orc_exp(-110.0) == 0.0 and O.lib().orc_exp(float("-inf")) == 0.0
    assert math.isnan(O.lib().orc_exp(float("nan")))
    # subnormal range stays within 1 subnormal ulp
    for x in (-90.0, -95.5, -100.0, -103.0):
        assert abs(O.lib().orc_exp(x) - math.exp(x)) <= 2.0 ** -149


def test_sigmoid_and_silu_special_values():
    assert O.lib().orc_sigmoid(0.0) == 0.5
    assert O.lib().orc_sigmoid(200.0) == 1.0
    assert O.lib().orc_sigmoid(-200.0) == 0.0
    assert O.lib().orc_silu_mul(0.0, 3.0) == 0.0
    assert O.lib().orc_silu_mul(-200.0, 1.0) == 0.0  # -200/inf = -0
    assert O.lib().orc_silu_mul(200.0, 0.5) == 100.0
    rng = np.random.default_rng(5)
    for g, u in rng.standard_normal((500, 2)).astype(np.float32) * 4:
        ref = float(g) / (1 + math.exp(-float(g))) * float(u)
        got = O.lib().orc_silu_mul(float(g), float(u))
        assert abs(got - ref) <= 6 * EPS32 * abs(ref) + 1e-38


def test_pairwise32_is_a_tree():
    """[2^24, 1, 1, 1, 0...]: the pairwise tree gives (2^24+1 -> 2^24) + (1+1) = 2^24 + 2 exactly,
    while a left-to-right sum would lose both ones and give 2^24."""
    p = np.zeros(32, dtype=np.float32)
    p[:4] = [2.0 ** 24, 1, 1, 1]
    assert O.pairwise32(p) == 2.0 ** 24 + 2
    # level structure: a pair sum at positions (30, 31) is added last
    p = np.zeros(32, dtype=np.float32)
    p[0], p[30], p[31] = 2.0 ** 24, 1, 1
    assert O.pairwise32(p) == 2.0 ** 24 + 2


def test_canon_dot_groups_are_contiguous():
    """n = 64 -> 32 groups of 2 adjacent elements.  a0 = 2^24, a1 = -2^24 cancel inside group 0
    and a32 = a33 = 1 share group 16: result 2 (= the exact sum).  Groups made of strided elements
    ({0,32}, {1,33}, ...) would give 2^24 (+1 lost) - 2^24 + 1 = 1 instead."""
    a = np.zeros(64, dtype=np.float32)
    a[0], a[1], a[32], a[33] = 2.0 ** 24, -2.0 ** 24, 1, 1
    assert O.canon_dot(a, np.ones(64, dtype=np.float32)) == 2.0


def test_canon_dot_error_bound():
    rng = np.random.default_rng(6)
    for n in (32, 100, 512, 6144):
        a = rng.standard_normal(n).astype(np.float32)
        b = rng.standard_normal(n).astype(np.float32)
        exact = float(np.dot(a.astype(np.float64), b.astype(np.float64)))
        mag = float(np.abs(a.astype(np.float64) * b.astype(np.float64)).sum())
        bound = (math.ceil(n / 32) + 5) * EPS32 * mag
        assert abs(O.canon_dot(a, b) - exact) <= bound


def test_canon_blocksum_exact_on_small_integers():
    """power-of-two scales and small integer accumulators: every partial is exact, so the
    canonical sum equals the integer closed form"""
    rng = np.random.default_rng(7)
    for nb in (8, 16, 64, 192):
        A = rng.integers(-28448, 28449, nb).astype(np.int32)
        d = (2.0 ** rng.integers(-6, 0, nb)).astype(np.float32)
        exact = sum(Fraction(int(a)) * Fraction(float(x)) for a, x in zip(A, d))
        assert Fraction(O.canon_blocksum(d, A)) == exact


# ------------------------------------------------------------------ router -------------

def test_topk_equals_full_stable_sort():
    rng = np.random.default_rng(8)
    for E, K in ((32, 4), (256, 8), (16, 16)):
        for _ in range(20):
            sel = (rng.integers(0, 12, E) / 8.0).astype(np.float32)  # many ties
            ids = O.topk(sel, K)
            ref = np.argsort(-sel.astype(np.float64), kind="stable")[:K]
            assert ids.tolist() == ref.tolist()
    assert sorted(O.topk(np.zeros(16, np.float32), 16).tolist()) == list(range(16))


def test_router_logits_scores_weights():
    wl = W.WORKLOADS["glm_decode_t1"]
    Wr = W.router_host(wl, 0)
    x = W.x_host(wl, 1)[0]
    logits, scores, ids, w = O.route_token(Wr, None, x, wl.K)
    exact = Wr.astype(np.float64) @ x.astype(np.float64)
    mag = np.abs(Wr.astype(np.float64)) @ np.abs(x.astype(np.float64))
    assert np.all(np.abs(logits - exact) <= (192 + 5) * EPS32 * mag)
    sig = 1.0 / (1.0 + np.exp(-logits.astype(np.float64)))
    assert np.all(np.abs(scores - sig) <= 8 * EPS32 * sig)
    assert ids.tolist() == np.argsort(-scores.astype(np.float64), kind="stable")[:wl.K].tolist()
    assert abs(float(w.astype(np.float64).sum()) - 1.0) <= 2 * wl.K * EPS32
    ref_w = scores[ids].astype(np.float64) / scores[ids].astype(np.float64).sum()
    assert np.all(np.abs(w - ref_w) <= 4 * wl.K * EPS32 * ref_w)


def test_router_bias_changes_selection_not_weights():
    wl = W.WORKLOADS["glm_verify_t4"]
    Wr = W.router_host(wl, 0)
    bias = W.bias_host(wl, 0)
    S = set(np.nonzero(bias)[0].tolist())
    x = W.x_host(wl, 4)
    for t in range(4):
        _, scores, ids, w = O.route_token(Wr, bias, x[t], wl.K)
        assert S <= set(ids.tolist())
        sel = scores.astype(np.float64) + bias
        assert ids.tolist() == np.argsort(-sel, kind="stable")[:wl.K].tolist()
        ref_w = scores[ids].astype(np.float64) / scores[ids].astype(np.float64).sum()
        assert np.all(np.abs(w - ref_w) <= 4 * wl.K * EPS32)


def test_rmsnorm_closed_form():
    gamma = W.gamma_host(W.WORKLOADS["glm_stack16_t1"], 0)
    assert gamma.min() >= 0.9 and gamma.max() < 1.1
    c = np.float32(0.75)
    out = O.rmsnorm(np.full(6144, c, np.float32), gamma, 1e-6)
    ref = gamma.astype(np.float64) * 0.75 / math.sqrt(0.5625 + 1e-6)
    assert np.all(np.abs(out - ref) <= 8 * EPS32 * np.abs(ref))
    x = W.x_host(W.WORKLOADS["glm_stack16_t1"], 1)[0]
    out = O.rmsnorm(x, gamma, 1e-6)
    xd = x.astype(np.float64)
    ref = xd / math.sqrt((xd * xd).mean() + 1e-6) * gamma
    assert np.all(np.abs(out - ref) <= 16 * EPS32 * np.abs(ref) + 1e-12)


# ------------------------------------------------------------------ batch union --------

def test_union_bucket_brute_force():
    rng = np.random.default_rng(9)
    for T, K, E in ((1, 8, 256), (4, 8, 256), (7, 4, 32), (16, 8, 64)):
        ids = np.stack([rng.choice(E, K, replace=False) for _ in range(T)]).astype(np.int32)
        ub = O.union_bucket(ids, E, 1)
        distinct = sorted(set(ids.ravel().tolist()))
        assert ub["union_ids"].tolist() == distinct + [E]
        p = 0
        for s, e in enumerate(distinct):
            pairs = [(t, k) for t in range(T) for k in range(K) if ids[t, k] == e]
            assert ub["offsets"][s] == p
            for (t, k) in pairs:
                assert ub["pair_token"][p] == t and ub["pair_rank"][p] == k and ub["inv"][t, k] == p
                p += 1
        assert ub["offsets"][len(distinct)] == T * K
        assert ub["pair_token"][T * K:].tolist() == list(range(T))
        assert np.all(ub["pair_rank"][T * K:] == -1)
        assert ub["offsets"][-1] == T * K + T


# ------------------------------------------------------------------ one expert ---------

def test_expert_ffn_against_fp64():
    wl = W.WORKLOADS["tiny_t1"]
    rec, sc = O.expert_record(wl, 0, 5)
    x = W.x_host(wl, 1)[0]
    qx, dx = O.quantize_q8(x)
    r = O.expert_ffn(rec, sc, wl.d, wl.f, qx, dx, want_A=True)
    d, f = wl.d, wl.f
    Wg = decode_nibbles(rec[:f * d // 2].reshape(f, d // 2)).astype(np.int64)
    Wu = decode_nibbles(rec[f * d // 2:f * d].reshape(f, d // 2)).astype(np.int64)
    Wd = decode_nibbles(rec[f * d:].reshape(d, f // 2)).astype(np.int64)
    Ag = (Wg.reshape(f, -1, 32) * qx.astype(np.int64).reshape(1, -1, 32)).sum(axis=2)
    assert np.array_equal(r["Ag"], Ag)
    g64 = sc[:f].astype(np.float64) * (Ag * dx.astype(np.float64)).sum(axis=1)
    mag = sc[:f].astype(np.float64) * (np.abs(Ag) * dx.astype(np.float64)).sum(axis=1)
    assert np.all(np.abs(r["g"] - g64) <= 10 * EPS32 * mag)
    Au = (Wu.reshape(f, -1, 32) * qx.astype(np.int64).reshape(1, -1, 32)).sum(axis=2)
    assert np.array_equal(r["Au"], Au)
    h64 = r["g"].astype(np.float64) / (1 + np.exp(-r["g"].astype(np.float64))) * r["u"]
    assert np.all(np.abs(r["h"] - h64) <= 8 * EPS32 * np.abs(h64) + 1e-30)
    # h codes are the q8 quantisation of h (independent closed-form check of each block)
    hb = r["h"].reshape(-1, 32)
    assert np.array_equal(r["dh"], (np.abs(hb).max(axis=1) / np.float32(127)).astype(np.float32))
    err = np.abs(hb - r["dh"][:, None] * r["qh"].reshape(-1, 32).astype(np.float32))
    assert np.all(err <= r["dh"][:, None] * 0.5001)
    Ad = (Wd.reshape(d, -1, 32) * r["qh"].astype(np.int64).reshape(1, -1, 32)).sum(axis=2)
    assert np.array_equal(r["Ad"], Ad)
    e64 = sc[2 * f:].astype(np.float64) * (Ad * r["dh"].astype(np.float64)).sum(axis=1)
    mag = sc[2 * f:].astype(np.float64) * (np.abs(Ad) * r["dh"].astype(np.float64)).sum(axis=1)
    assert np.all(np.abs(r["e"] - e64) <= 10 * EPS32 * mag)


# ------------------------------------------------------------------ experts of other widths

def _packed(codes, bits):
    """rows of codes in the int8 (one per byte), int4 or int2 row format"""
    codes = np.ascontiguousarray(codes, dtype=np.int8)
    if bits == 8:
        return codes.view(np.uint8).ravel().copy()
    rows, cols = codes.shape
    out = np.empty((rows, cols * bits // 8), dtype=np.uint8)
    pack = O.lib().orc_pack_i4_row if bits == 4 else O.lib().orc_pack_i2_row
    for r in range(rows):
        pack(codes[r].ctypes.data, cols, out[r].ctypes.data)
    return out.ravel()


def _expert_record(cg, cu, cd, bits):
    return np.concatenate([_packed(m, bits) for m in (cg, cu, cd)])


def test_expert_of_equal_codes_is_the_same_in_every_width():
    """an expert whose codes fit every width gives the same bits stored as int2, int4 or int8
    rows (the record layout differs only in the bytes per code), and 4-bit rows give
    orc_expert_ffn's result"""
    rng = np.random.default_rng(18)
    d, f = 512, 256
    sc = rng.uniform(0.002, 0.02, 2 * f + d).astype(np.float32)
    qx, dx = O.quantize_q8(rng.standard_normal(d).astype(np.float32))
    keys = ("qh", "dh", "e", "g", "u", "h")
    cg, cu, cd = (rng.integers(-1, 2, shp, dtype=np.int8) for shp in ((f, d), (f, d), (d, f)))
    outs = [O.expert_ffn_bits(b, _expert_record(cg, cu, cd, b), sc, d, f, qx, dx) for b in (2, 4, 8)]
    for o in outs[1:]:
        for k in keys:
            assert np.array_equal(o[k].view(np.uint8), outs[0][k].view(np.uint8)), k
    cg, cu, cd = (rng.integers(-7, 8, shp, dtype=np.int8) for shp in ((f, d), (f, d), (d, f)))
    r4 = _expert_record(cg, cu, cd, 4)
    o4 = O.expert_ffn_bits(4, r4, sc, d, f, qx, dx)
    o8 = O.expert_ffn_bits(8, _expert_record(cg, cu, cd, 8), sc, d, f, qx, dx)
    ref = O.expert_ffn(r4, sc, d, f, qx, dx)
    for k in keys:
        assert np.array_equal(o8[k].view(np.uint8), o4[k].view(np.uint8)), k
        assert np.array_equal(o4[k].view(np.uint8), ref[k].view(np.uint8)), k
    with pytest.raises(ValueError):
        O.expert_ffn_bits(3, r4, sc, d, f, qx, dx)


def test_int8_expert_against_fp64():
    """full-range int8 rows: every step against fp64 evaluated from brute-force integer sums"""
    rng = np.random.default_rng(19)
    d, f = 512, 256
    cg, cu, cd = (rng.integers(-127, 128, shp, dtype=np.int8) for shp in ((f, d), (f, d), (d, f)))
    sc = (rng.uniform(0.5, 2.0, 2 * f + d) / 127 * 0.02).astype(np.float32)
    qx, dx = O.quantize_q8(rng.standard_normal(d).astype(np.float32))
    r = O.expert_ffn_bits(8, _expert_record(cg, cu, cd, 8), sc, d, f, qx, dx)
    q64 = qx.astype(np.int64).reshape(1, -1, 32)
    for name, codes, s, out in (("g", cg, sc[:f], r["g"]), ("u", cu, sc[f:2 * f], r["u"])):
        A = (codes.astype(np.int64).reshape(f, -1, 32) * q64).sum(axis=2)
        v64 = s.astype(np.float64) * (A * dx.astype(np.float64)).sum(axis=1)
        mag = s.astype(np.float64) * (np.abs(A) * dx.astype(np.float64)).sum(axis=1)
        assert np.all(np.abs(out - v64) <= 10 * EPS32 * mag), name
    h64 = r["g"].astype(np.float64) / (1 + np.exp(-r["g"].astype(np.float64))) * r["u"]
    assert np.all(np.abs(r["h"] - h64) <= 8 * EPS32 * np.abs(h64) + 1e-30)
    hb = r["h"].reshape(-1, 32)
    assert np.array_equal(r["dh"], (np.abs(hb).max(axis=1) / np.float32(127)).astype(np.float32))
    err = np.abs(hb - r["dh"][:, None] * r["qh"].reshape(-1, 32).astype(np.float32))
    assert np.all(err <= r["dh"][:, None] * 0.5001)
    Ad = (cd.astype(np.int64).reshape(d, -1, 32) * r["qh"].astype(np.int64).reshape(1, -1, 32)).sum(axis=2)
    e64 = sc[2 * f:].astype(np.float64) * (Ad * r["dh"].astype(np.float64)).sum(axis=1)
    mag = sc[2 * f:].astype(np.float64) * (np.abs(Ad) * r["dh"].astype(np.float64)).sum(axis=1)
    assert np.all(np.abs(r["e"] - e64) <= 10 * EPS32 * mag)


def test_layer_of_equal_codes_is_the_same_in_every_width():
    """a whole layer (routing, union, experts, fixed-order combine) whose expert codes fit
    every width gives the same bits with int2, int4 or int8 expert records; the fp64 output
    agrees too"""
    wl = W.WORKLOADS["tiny_t1"]
    d, f = wl.d, wl.f
    rng = np.random.default_rng(20)
    L = O.Layer(wl)
    codes = {e: [rng.integers(-1, 2, shp, dtype=np.int8) for shp in ((f, d), (f, d), (d, f))]
             for e in range(wl.E + wl.n_shared)}
    scs = {e: rng.uniform(0.005, 0.05, 2 * f + d).astype(np.float32) for e in codes}
    x = W.x_host(wl, 3, 7)
    outs = {}
    for bits in (2, 4, 8):
        recs = {e: (_expert_record(*codes[e], bits), scs[e]) for e in codes}
        outs[bits] = O.forward(wl, x, L.Wr, L.bias, L.gamma, recs, wbits=bits)
    assert int(outs[4]["n_union"][0]) > wl.K  # several experts, shared one included
    for bits in (2, 8):
        for k in ("y", "y64", "qh", "dh", "e", "ids", "w", "offsets"):
            assert np.array_equal(np.ascontiguousarray(outs[bits][k]).view(np.uint8),
                                  np.ascontiguousarray(outs[4][k]).view(np.uint8)), (bits, k)
    assert normwise_rel64(outs[8]["y"], outs[8]["y64"]) < 1e-5


def normwise_rel64(a, ref):
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(np.asarray(a, dtype=np.float64) - ref).max() / np.abs(ref).max())


# ------------------------------------------------------------------ layer identities ---

def _layer_inputs(wl, layer=0):
    L = O.Layer(wl, layer)
    L.ensure(range(wl.E + wl.n_shared))
    return L


def test_forced_all_experts_equals_dense_loop():
    """K = E: every expert is selected; the layer must equal a dense loop over experts that
    calls the single-expert FFN directly (no union or bucketing), combined in rank order."""
    base = W.WORKLOADS["tiny_t1"]
    wl = W.Workload("tiny_dense", d=base.d, f=base.f, E=base.E, K=base.E, n_shared=1, T=2)
    L = _layer_inputs(wl)
    x = W.x_host(wl, 2)
    out = L.forward(x, want_y64=True)
    for t in range(2):
        qx, dx = O.quantize_q8(x[t])
        es = O.expert_ffn(*L.recs[wl.E], wl.d, wl.f, qx, dx)["e"].astype(np.float64)
        acc = es.copy()
        for k in range(wl.K):
            ex = int(out["ids"][t, k])
            ek = O.expert_ffn(*L.recs[ex], wl.d, wl.f, qx, dx)["e"]
            assert np.array_equal(out["e"][out["inv"][t, k]], ek)  # bit-exact per expert
            acc += float(out["w"][t, k]) * ek.astype(np.float64)
        assert sorted(out["ids"][t].tolist()) == list(range(wl.E))
        scale = np.abs(acc).max()
        assert np.abs(out["y"][t] - acc).max() <= 1e-5 * scale


def test_identical_experts_closed_form():
    """all experts identical: y = shared(x) + FFN(x) * sum(w) = shared + FFN(x), whatever the routing"""
    wl = W.WORKLOADS["tiny_t1"]
    rec, sc = O.expert_record(wl, 0, 3)
    srec, ssc = O.expert_record(wl, 0, wl.E)
    recs = {e: (rec, sc) for e in range(wl.E)}
    recs[wl.E] = (srec, ssc)
    Wr = W.router_host(wl, 0)
    x = W.x_host(wl, 3)
    out = O.forward(wl, x, Wr, None, None, recs)
    for t in range(3):
        qx, dx = O.quantize_q8(x[t])
        e = O.expert_ffn(rec, sc, wl.d, wl.f, qx, dx)["e"].astype(np.float64)
        es = O.expert_ffn(srec, ssc, wl.d, wl.f, qx, dx)["e"].astype(np.float64)
        ref = es + e
        assert np.abs(out["y"][t] - ref).max() <= 1e-5 * np.abs(ref).max()


def test_batch_invariance():
    """a token's output does not depend on the batch it is verified in (draft and verify
    compute the same function): forward(T=4)[t] == forward(T=1, x_t) bit for bit"""
    for name in ("tiny_t1",):
        wl = W.WORKLOADS[name]
        L = _layer_inputs(wl)
        x = W.x_host(wl, 4, token0=10)
        yb = L.forward(x, want_dump=False, want_y64=False)["y"]
        for t in range(4):
            y1 = L.forward(x[t:t + 1], want_dump=False, want_y64=False)["y"]
            assert np.array_equal(yb[t], y1[0])


def test_norm_layer_is_residual_of_plain_layer():
    """with RMSNorm: y = x + MoE(RMSNorm(x)); the plain layer run on RMSNorm(x) gives MoE(.), and
    the residual is one fp32 add, so the two agree bit for bit"""
    base = W.WORKLOADS["tiny_t1"]
    wl_n = W.Workload("tiny_norm", d=base.d, f=base.f, E=base.E, K=base.K, n_shared=1, T=2,
                      has_norm=True)
    L = _layer_inputs(wl_n)
    x = W.x_host(wl_n, 2)
    out = L.forward(x)
    gamma = W.gamma_host(wl_n, 0)
    xn = np.stack([O.rmsnorm(x[t], gamma, wl_n.rms_eps) for t in range(2)])
    assert np.array_equal(out["xn"], xn)
    plain = O.forward(base, xn, L.Wr, None, None, L.recs, want_dump=False, want_y64=False)["y"]
    assert np.array_equal(out["y"], (x + plain).astype(np.float32))


def test_fp32_canonical_output_within_fp64():
    wl = W.WORKLOADS["tiny_t1"]
    L = _layer_inputs(wl)
    x = W.x_host(wl, 4)
    out = L.forward(x)
    err = np.abs(out["y"] - out["y64"]).max() / np.abs(out["y64"]).max()
    assert err <= 1e-5


def test_idot_accuracy_band():
    """The pages report about 0.3% RMS error for the int8-activation integer-dot path against
    float dequant-on-use (on real activations).  Closed form for these synthetic inputs: rounding
    a block of 32 to int8 adds error of RMS amax/(127*sqrt(12)); relative to the operand's RMS
    that is p_x for x (enters g and u independently) and p_h for h = SiLU(g)*u, so the layer's
    relative RMS error is about sqrt(2 p_x^2 + p_h^2), ~1% for Gaussian x (h is heavier-tailed
    than real activations).  The measured error must sit within 0.8x..1.2x of that: a path with
    twice the error, or one that skips the re-quantisation of h (about 0.7x), fails.  The
    measured 1.10% lies above the <= 1% band first proposed for this check, and above the
    pages' ~0.3%: the prediction, not the band, is what Gaussian synthetic inputs give."""
    wl = W.WORKLOADS["tiny_t1"]
    L = _layer_inputs(wl)
    x = W.x_host(wl, 16)
    out = L.forward(x)
    y64 = O.dequant64(wl, out["xn"], out["ids"], out["w"], L.recs)
    rel = np.sqrt(((out["y"] - y64) ** 2).mean()) / np.sqrt((y64 ** 2).mean())

    def block_noise(v):
        b = v.reshape(-1, 32).astype(np.float64)
        return np.abs(b).max(axis=1).mean() / (127 * math.sqrt(12)) / math.sqrt((b ** 2).mean())

    pred = math.sqrt(2 * block_noise(out["xn"]) ** 2 + block_noise(out["h"]) ** 2)
    assert 0.8 * pred <= rel <= 1.2 * pred, (rel, pred)
    assert 5e-3 <= rel <= 1.5e-2


def test_expert_size_matches_pages():
    """≈19 MB int4 per expert (colibrì 架构概述 §2; README 核心概念)"""
    wl = W.WORKLOADS["glm_decode_t1"]
    assert wl.expert_bytes == 18_915_328
    assert round(wl.expert_bytes / 1e6) == 19
