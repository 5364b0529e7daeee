"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these re-types the oracle's own formula: each compares it with a
different formulation (exact rational arithmetic, closed forms, hand-derived
tables from the pages, brute-force rank counting, invariants).
"""
import math
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(1234)


def _bits_of(vals):
    """bf16 bits of values that are exactly representable in bf16 (via exact f32)."""
    f = np.asarray(vals, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not representable in bf16"
    return (b >> 16).astype(np.uint16)


def _rand_bf16(shape, scale=1.0):
    x = (RNG.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)   # truncation: any bf16 pattern will do


def _frac_of_bits(bits):
    return Fraction(float(O.bf16_to_f64(np.array([bits]))[0]))


def _round_frac_bf16(v: Fraction) -> Fraction:
    """Correct RNE rounding of an exact rational to bf16 (8 significant bits), by
    exact comparison; the independent check of f64_to_bf16."""
    if v == 0:
        return Fraction(0)
    s = -1 if v < 0 else 1
    a = abs(v)
    e = math.floor(math.log2(a))
    while Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    q = Fraction(2) ** (max(e, -126) - 7)          # quantum: 8 significant bits
    n = a / q
    lo = math.floor(n)
    rem = n - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    return s * lo * q


# ----------------------------------------------------------------------- bf16 rounding
def test_bf16_roundtrip_all_patterns():
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    exp = (bits >> 7) & 0xFF
    finite = bits[exp != 0xFF]
    assert np.array_equal(O.f64_to_bf16(O.bf16_to_f64(finite)), finite)


def test_bf16_rounding_from_f32_matches_integer_rne():
    # the classic integer form of RNE on f32 bit patterns is an independent formulation
    x = (RNG.standard_normal(200000) * 10.0 ** RNG.integers(-30, 30, 200000)).astype(np.float32)
    b = x.view(np.uint32).astype(np.uint64)
    ref = ((b + 0x7FFF + ((b >> 16) & 1)) >> 16).astype(np.uint16)
    assert np.array_equal(O.f64_to_bf16(x.astype(np.float64)), ref)


def test_bf16_rounding_is_single_step_from_f64():
    # 1 + 2**-8 + 2**-30 lies above the midpoint of 1 and 1 + 2**-7: it must round up,
    # although going through f32 first would land exactly on the midpoint and tie to 1.
    got = O.bf16_to_f64(O.f64_to_bf16(np.array([1 + 2.0 ** -8 + 2.0 ** -30, 1 + 2.0 ** -8])))
    assert got[0] == 1 + 2.0 ** -7 and got[1] == 1.0


def test_bf16_rounding_exact_rationals():
    vals = RNG.standard_normal(300) * 10.0 ** RNG.integers(-5, 5, 300)
    got = O.bf16_to_f64(O.f64_to_bf16(vals))
    for v, g in zip(vals, got):
        assert Fraction(float(g)) == _round_frac_bf16(Fraction(float(v)))


# ----------------------------------------------------------------------- e2m1 / e8m0
def _quant_at_unit_scale(values):
    """Quantise each value in a block whose amax is 6 (scale 2**0)."""
    out = []
    for v in values:
        blk = np.zeros(32)
        blk[0] = v
        blk[1] = 6.0
        codes, scales, _ = O.fp4_quant_e8m0(_bits_of(blk)[None, :])
        assert scales[0, 0] == 127
        out.append(int(codes[0, 0]))
    return out


def test_e2m1_golden_ties():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "e2m1_rne.txt")) if l.strip() and l[0] != "#"]
    vals = [float(r[0]) for r in rows]
    want = [int(r[1]) for r in rows]
    assert _quant_at_unit_scale(vals) == want


def test_e2m1_exhaustive_thresholds():
    # every non-negative bf16 value up to 6, in increasing order: the code must be
    # non-decreasing and switch exactly at the grid midpoints, with the midpoint
    # itself going to the even code (0.25->0, 0.75->2, 1.25->2, 1.75->4, 2.5->4, 3.5->6, 5->6)
    bits = np.arange(0, 0x7F80, dtype=np.uint32).astype(np.uint16)
    vals = O.bf16_to_f64(bits)
    vals = vals[vals <= 6.0]
    blocks = np.zeros((vals.size, 32))
    blocks[:, 0] = vals
    blocks[:, 1] = 6.0
    codes, scales, deq = O.fp4_quant_e8m0(_bits_of(blocks))
    assert np.all(scales[:, 0] == 127)
    c = codes[:, 0].astype(int)
    mids = [(0.25, 0), (0.75, 2), (1.25, 2), (1.75, 4), (2.5, 4), (3.5, 6), (5.0, 6)]
    expect = np.zeros(vals.size, dtype=int)
    for k, (m, at) in enumerate(mids):
        expect = np.where(vals > m, k + 1, expect)
        expect = np.where(vals == m, at, expect)
    assert np.array_equal(c, expect)
    assert np.all(np.diff(c) >= 0)
    # the negated inputs give the same magnitude with the sign bit set
    codes_n, _, _ = O.fp4_quant_e8m0(_bits_of(-blocks))
    assert np.array_equal(codes_n[:, 0].astype(int), expect | 8)


def test_e8m0_closed_forms():
    def scale_byte(amax):
        blk = np.zeros(32)
        blk[5] = amax
        return int(O.fp4_quant_e8m0(_bits_of(blk)[None, :])[1][0, 0])
    assert scale_byte(6.0) == 127                  # 6 / 6 = 1 = 2**0
    assert scale_byte(6.03125) == 128              # next bf16 above 6 needs 2**1
    assert scale_byte(3.0) == 126                  # 3 / 6 = 0.5 = 2**-1
    assert scale_byte(3.015625) == 127             # next bf16 above 3
    assert scale_byte(1.0) == 125                  # 1/6 -> 2**-2 (0.25 >= 1/6 > 0.125)
    assert scale_byte(2.0 ** 100) == 127 + 98      # 6 * 2**98 = 1.5 * 2**100
    assert scale_byte(0.0) == 1                    # floor 6 * 2**-126 -> 2**-126
    assert scale_byte(2.0 ** -130) == 1            # subnormal amax still floored
    assert scale_byte(6.0 * 2.0 ** -126) == 1


def test_e8m0_minimal_power_of_two():
    x = _rand_bf16((4000, 32), scale=1.0)
    x[::7] = _rand_bf16((x[::7].shape), scale=1e-20)
    x[1::7] = _rand_bf16((x[1::7].shape), scale=1e20)
    codes, scales, deq = O.fp4_quant_e8m0(x)
    amax = np.maximum(np.abs(O.bf16_to_f64(x)).max(axis=1), 6 * 2.0 ** -126)
    e = scales[:, 0].astype(int) - 127
    assert np.all(np.ldexp(6.0, e) >= amax)
    assert np.all(np.ldexp(6.0, e - 1) < amax)
    # every dequantised value is the scale times a grid value of the right sign
    xv = O.bf16_to_f64(x)
    assert np.all(np.abs(deq) <= 6.0 * np.ldexp(1.0, e)[:, None])
    assert np.all((deq == 0) | (np.sign(deq) == np.sign(xv)))


def test_quant_error_bound_and_idempotence():
    x = _rand_bf16((2000, 128))
    codes, scales, deq = O.fp4_quant_e8m0(x)
    e = np.repeat(scales.astype(int) - 127, 32, axis=1)
    xv = O.bf16_to_f64(x)
    # largest grid gap is 2 (between 4 and 6): error at most half of it, times the scale
    assert np.all(np.abs(xv - deq) <= np.ldexp(1.0, e))
    # re-quantising the dequantised values reproduces the same values (the scale may
    # shrink when amax rounded down, e.g. 3.2 -> 3, but every value stays on the grid)
    deq_bits = O.f64_to_bf16(deq)
    _, _, d2 = O.fp4_quant_e8m0(deq_bits)
    assert np.array_equal(d2, deq)


# ----------------------------------------------------------------------- 68-byte row
def test_key_row_layout_golden():
    rows = [l.split() for l in open(os.path.join(GOLDEN, "key_row_layout.txt")) if l.strip() and l[0] != "#"]
    hd, mx, _ = map(int, rows[0])
    assert O.key_row_bytes(hd) == mx == O.KEY_ROW_BYTES


def test_row_pack_roundtrip():
    x = _rand_bf16((50, 128))
    codes, scales, deq = O.fp4_quant_e8m0(x)
    rows = O.pack_row68(codes, scales)
    assert rows.shape == (50, 68) and rows.dtype == np.uint8
    c2, s2 = O.unpack_row68(rows)
    assert np.array_equal(c2, codes) and np.array_equal(s2, scales)
    assert np.array_equal(O.dequant_row68(rows), deq)
    # element 0 in the low nibble of byte 0, element 1 in the high nibble
    assert rows[3, 0] == (codes[3, 0] | (codes[3, 1] << 4))
    assert np.array_equal(rows[:, 64:], scales)


# ----------------------------------------------------------------------- YaRN / RoPE
def test_yarn_reduces_to_plain_rope():
    cos, sin = O.yarn_freqs_cis(64, 3, 10000.0, 1.0, 4096, 32, 1)
    f = (10000.0 ** (-np.arange(32) * 2 / 64)).astype(np.float32)
    assert np.array_equal(cos[0], np.ones(32, np.float32)) and np.array_equal(sin[0], np.zeros(32, np.float32))
    assert np.array_equal(cos[1], np.cos(f.astype(np.float64)).astype(np.float32))
    cos0, sin0 = O.yarn_freqs_cis(64, 3, 10000.0, 16.0, 0, 32, 1)   # original_seq_len 0: no YaRN
    assert np.array_equal(cos0[1], cos[1]) and np.array_equal(sin0[2], sin[2])


def test_yarn_correction_range_closed_form():
    # theta 160000, L 4096, dim 64: c(32) = 64 ln(4096/(64 pi)) / (2 ln 160000) = 8.05...,
    # c(1) = 64 ln(4096/(2 pi)) / (2 ln 160000) = 17.30...  ->  low = 8, high = 18.
    c32 = 64 * math.log(4096 / (64 * math.pi)) / (2 * math.log(160000))
    c1 = 64 * math.log(4096 / (2 * math.pi)) / (2 * math.log(160000))
    assert 8 < c32 < 8.1 and 17.2 < c1 < 17.4
    _, sin = O.yarn_freqs_cis(64, 2, 160000.0, 16.0, 4096, 32, 1)
    f = 160000.0 ** (-np.arange(32) * 2 / 64)
    angle1 = np.arcsin(sin[1].astype(np.float64))
    # dims 0..8 keep the base frequency, dims 18.. are divided by the factor, between is a ramp
    assert np.allclose(angle1[:9], f[:9], rtol=1e-6)
    assert np.allclose(angle1[18:], f[18:] / 16.0, rtol=1e-6)
    mid = angle1[9:18] / f[9:18]
    ramp = (np.arange(9, 18) - 8) / 10.0
    assert np.allclose(mid, 1 - ramp + ramp / 16.0, rtol=1e-6)


def test_yarn_unit_circle():
    cos, sin = O.yarn_freqs_cis(64, 5000, 160000.0, 16.0, 4096, 32, 1)
    r = cos.astype(np.float64) ** 2 + sin.astype(np.float64) ** 2
    assert np.all(np.abs(r - 1) < 4e-7)


def test_rope_identity_and_quarter_turn():
    x = _rand_bf16((7, 128))
    x[x == 0x8000] = 0x3F80
    ones = np.ones((1, 32), np.float32)
    zeros = np.zeros((1, 32), np.float32)
    assert np.array_equal(O.rope_interleaved(x, ones, zeros, np.zeros(7, int), 64), x)
    # cos 0, sin 1: (x0, x1) -> (-x1, x0) exactly, only in the last 64 dims
    y = O.rope_interleaved(x, zeros, ones, np.zeros(7, int), 64)
    assert np.array_equal(y[:, :64], x[:, :64])
    assert np.array_equal(y[:, 64::2], x[:, 65::2] ^ 0x8000)
    assert np.array_equal(y[:, 65::2], x[:, 64::2])


def test_rope_pairs_use_their_own_column():
    x = _rand_bf16((1, 128))
    cos = np.ones((1, 32), np.float32)
    sin = np.zeros((1, 32), np.float32)
    cos[0, 5], sin[0, 5] = 0.0, 1.0      # only pair 5 (dims 64+10, 64+11) turns
    y = O.rope_interleaved(x, cos, sin, np.zeros(1, int), 64)
    changed = np.nonzero(y[0] != x[0])[0]
    assert set(changed) <= {74, 75}
    assert y[0, 74] == x[0, 75] ^ 0x8000 and y[0, 75] == x[0, 74]


def test_rope_preserves_pair_norm():
    x = _rand_bf16((200, 128))
    cos, sin = O.yarn_freqs_cis(64, 1000, 160000.0, 16.0, 4096, 32, 1)
    pos = RNG.integers(0, 1000, 200)
    y = O.rope_interleaved(x, cos, sin, pos, 64)
    a = O.bf16_to_f64(x[:, 64:]).reshape(200, 32, 2)
    b = O.bf16_to_f64(y[:, 64:]).reshape(200, 32, 2)
    na, nb = np.hypot(a[..., 0], a[..., 1]), np.hypot(b[..., 0], b[..., 1])
    assert np.all(np.abs(na - nb) <= 2 ** -7 * na + 1e-30)


# A rotation whose result depends on the f32 operation order. x0 = x1 = 1 + 2^-7 (bf16
# 0x3F81), c = 1 - 2^-24 (f32 0x3F7FFFFF), s = 1 - 2^-23 (f32 0x3F7FFFFE). By hand:
#   x0*c = 1 + 2^-7 - 2^-24 - 2^-31 lies 2^-24 - 2^-31 above L = 1 + 2^-7 - 2^-23 and
#          2^-24 + 2^-31 below 1 + 2^-7, so it rounds to L in f32;
#   x1*s = 1 + 2^-7 - 2^-23 - 2^-30 lies 2^-30 below L, so it also rounds to L;
#   y0 = f32(L - L) = +0  (bf16 0x0000).
# With a fused multiply-add (f32(x0*c - f32(x1*s))) y0 would be 2^-24 - 2^-31, and exact
# arithmetic would give 2^-24 + 2^-31: both nonzero. y1 = f32(L + L) = 2 + 2^-6 - 2^-22,
# which rounds to bf16 2 + 2^-6 (0x4001).
_ROPE_ORDER_X = 0x3F81
_ROPE_ORDER_C = np.array([0x3F7FFFFF], np.uint32).view(np.float32)[0]
_ROPE_ORDER_S = np.array([0x3F7FFFFE], np.uint32).view(np.float32)[0]


def test_rope_f32_rounds_each_product_then_the_sum():
    """The RoPE reading (products rounded to f32, then their difference / sum rounded to
    f32, no fused multiply-add) on a hand-derived case where the order decides the result."""
    x = np.zeros((1, 128), np.uint16)
    x[0, 64] = x[0, 65] = _ROPE_ORDER_X
    cos = np.ones((1, 32), np.float32)
    sin = np.zeros((1, 32), np.float32)
    cos[0, 0], sin[0, 0] = _ROPE_ORDER_C, _ROPE_ORDER_S
    y = O.rope_interleaved(x, cos, sin, np.zeros(1, int), 64)
    assert y[0, 64] == 0x0000
    assert y[0, 65] == 0x4001


# A case where the rotation order still shows after the fp4 quantiser. x0 = -0.75 (bf16
# 0xBF40), x1 = 1 + 2^-7 (0x3F81), c = f32 0x3F2EE23C, s = 0.5; a second pair holds 1.5
# (unrotated), which fixes block 2's scale at 2^-2 (amax 1.5 -> e = -2, byte 125). By hand:
#   x0*s = -0.375 exactly; x1*c = 0.6884765625 + 2.79e-8 rounds in f32 to 0.6884765625;
#   y1 = f32(-0.375 + 0.6884765625) = 0.3134765625 = 0.3125 + 2^-10, the midpoint between
#   bf16 0.3125 and 0.314453125, so it rounds to even: 0.3125. At scale 2^-2 that is 1.25,
#   the e2m1 tie between 1.0 (code 2) and 1.5 (code 3): code 2.
# A fused multiply-add would keep the 2.79e-8, round y1 up to bf16 0.314453125 and give
# code 3. This is the case the GPU parity test drives through the query prep.
ROPE_TIE_Q = (0xBF40, 0x3F81)
ROPE_TIE_CS = (np.array([0x3F2EE23C], np.uint32).view(np.float32)[0], np.float32(0.5))


def test_rope_order_shows_after_quantisation():
    x = np.zeros((1, 1, 1, 128), np.uint16)
    x[..., 64], x[..., 65] = ROPE_TIE_Q
    x[..., 66] = 0x3FC0                                   # 1.5, rotated by the identity pair
    cos = np.ones((1, 32), np.float32)
    sin = np.zeros((1, 32), np.float32)
    cos[0, 0], sin[0, 0] = ROPE_TIE_CS
    rows, _, qrot = O.prep_queries(x, np.full((1, 1, 1), 0x3F80, np.uint16), cos, sin, 0, 64, 1)
    assert qrot[0, 0, 0, 65] == 0x3EA0                    # bf16 0.3125
    codes, scales = O.unpack_row68(rows[0, 0, 0])
    assert scales[2] == 125
    assert codes[65] == 2


# --------------------------------------------------------------------- query prep
def test_query_head_weight_factor_matches_the_pages_constants():
    """w' = weights * softmax_scale * n_heads^-0.5 with softmax_scale = index_head_dim^-0.5
    (index-keys page, Indexer.__init__ softmax_scale, Indexer.forward weights line). For
    index_head_dim 128: H 8 -> 1/32, H 32 -> 1/64, H 128 -> 1/128 exactly; H 64 ->
    0.011048543456..., H 16 -> 0.022097086912... (decimal constants, not recomputed)."""
    table_c = np.ones((4, 32), np.float32)
    table_s = np.zeros((4, 32), np.float32)
    exact = {8: 0.03125, 32: 0.015625, 128: 0.0078125}
    approx = {64: 0.011048543456039806, 16: 0.022097086912079612}
    for H in (8, 16, 32, 64, 128):
        q = _rand_bf16((1, 2, H, 128))
        w = _rand_bf16((1, 2, H), scale=3.0)
        _, wprime, _ = O.prep_queries(q, w, table_c, table_s, 0, 64, H)
        ratio = wprime / O.bf16_to_f64(w)
        ok = np.isfinite(ratio)
        if H in exact:
            assert np.array_equal(wprime, O.bf16_to_f64(w) * exact[H])
        else:
            assert np.all(np.abs(ratio[ok] - approx[H]) <= 1e-15)
    # a unit weight gives the factor itself
    one = np.full((1, 1, 64), 0x3F80, np.uint16)
    _, wp, _ = O.prep_queries(_rand_bf16((1, 1, 64, 128)), one, table_c, table_s, 0, 64, 64)
    assert np.all(np.abs(wp - 0.011048543456039806) < 1e-16)


def test_query_rope_position_is_start_pos_plus_row():
    """Row s of a chunk starting at start_pos is rotated at position start_pos + s (index-keys
    page, Indexer.forward: freqs_cis[start_pos:end_pos] applied to q). A table whose pair-0
    cosine encodes the position ((p + 1) / 4096, exact in bf16 for p < 255) and whose sines
    are zero turns the query value 1.0 at the pair's first element into that position."""
    max_pos = 200
    cos = np.ones((max_pos, 32), np.float32)
    sin = np.zeros((max_pos, 32), np.float32)
    cos[:, 0] = (np.arange(max_pos) + 1) / 4096.0
    for start, S in ((0, 3), (100, 5), (190, 10)):
        q = np.zeros((2, S, 4, 128), np.uint16)
        q[..., 64] = 0x3F80                                   # 1.0 at the first rotated dim
        w = np.full((2, S, 4), 0x3F80, np.uint16)
        _, _, qrot = O.prep_queries(q, w, cos, sin, start, 64, 4)
        got = O.bf16_to_f64(qrot[..., 64]) * 4096.0 - 1.0
        want = np.broadcast_to((start + np.arange(S))[None, :, None], got.shape)
        assert np.array_equal(got, want)


# ----------------------------------------------------------------------- wk / RMSNorm
def test_linear_is_correctly_rounded_exact_sum():
    x = _rand_bf16((6, 128))
    w = _rand_bf16((9, 128), scale=128 ** -0.5)
    y = O.linear_bf16(x, w)
    for i in range(6):
        for o in range(9):
            exact = sum(_frac_of_bits(x[i, j]) * _frac_of_bits(w[o, j]) for j in range(128))
            assert _frac_of_bits(y[i, o]) == _round_frac_bf16(exact)


def test_query_projection_unflattens_feature_h_times_128_plus_d():
    """q = wq_b(qr) unflattened to [H][128]: feature o = h * 128 + d, each the correctly
    rounded exact sum (checked by brute force with fractions on a tiny case)."""
    qr = _rand_bf16((2, 3, 64))
    wq = _rand_bf16((2 * 128, 64), scale=64 ** -0.5)
    q = O.project_queries(qr, wq, 2)
    assert q.shape == (2, 3, 2, 128)
    for b, s, h, dd in [(0, 0, 0, 0), (0, 2, 1, 5), (1, 1, 0, 127), (1, 2, 1, 64), (0, 1, 1, 100)]:
        o = h * 128 + dd
        exact = sum(_frac_of_bits(qr[b, s, j]) * _frac_of_bits(wq[o, j]) for j in range(64))
        assert _frac_of_bits(q[b, s, h, dd]) == _round_frac_bf16(exact)


def test_rmsnorm_against_high_precision():
    from decimal import Decimal, getcontext
    getcontext().prec = 60
    x = _rand_bf16((5, 128))
    w = _rand_bf16((128,), scale=0.3)
    w = O.f64_to_bf16(O.bf16_to_f64(w) + 1.0)
    eps = 1e-6
    y = O.rmsnorm_bf16(x, w, eps)
    eps_d = Decimal(float(np.float32(eps)))
    for i in range(5):
        xs = [Decimal(float(v)) for v in O.bf16_to_f64(x[i])]
        ms = sum(v * v for v in xs) / 128
        r = 1 / (ms + eps_d).sqrt()
        for j in range(128):
            exact = Decimal(float(O.bf16_to_f64(w[j:j + 1])[0])) * xs[j] * r
            ref = _round_frac_bf16(Fraction(exact))
            assert _frac_of_bits(y[i, j]) == ref


def test_rmsnorm_unit_rms_and_scale_invariance():
    x = _rand_bf16((20, 128))
    ones = O.f64_to_bf16(np.ones(128))
    y = O.bf16_to_f64(O.rmsnorm_bf16(x, ones, 0.0))
    rms = np.sqrt(np.mean(y * y, axis=1))
    assert np.all(np.abs(rms - 1) < 2 ** -8)
    x4 = O.f64_to_bf16(O.bf16_to_f64(x) * 4.0)     # exact power-of-two scaling
    assert np.array_equal(O.rmsnorm_bf16(x4, ones, 0.0), O.rmsnorm_bf16(x, ones, 0.0))


# ----------------------------------------------------------------------- publish positions
def test_key_slots_prefill_and_decode():
    s, p = O.key_slots(0, 5, 4)
    assert list(s) == [0, 1, 2, 3, 4] and list(p) == [0, 4, 8, 12, 16]
    s, p = O.key_slots(32767, 1, 4)                 # token 32767 completes group 8191
    assert list(s) == [8191] and list(p) == [32764]
    with pytest.raises(ValueError):
        O.key_slots(32766, 1, 4)                    # group still filling: nothing to publish


# ----------------------------------------------------------------------- scores
def test_scores_exact_rational_tiny():
    H, T = 2, 5                                     # H=2: w' = w / sqrt(128*2) = w / 16, exact
    q = _rand_bf16((1, 3, H, 128))
    k = _rand_bf16((1, T, 128))
    w = _rand_bf16((1, 3, H))
    qc, qs, qd = O.fp4_quant_e8m0(q)
    kc, ks, kd = O.fp4_quant_e8m0(k)
    qrows = O.pack_row68(qc, qs)
    krows = O.pack_row68(kc, ks)
    wprime = O.bf16_to_f64(w) / 16.0
    vis = np.array([T, T, 3])
    sc = O.index_scores(qrows, wprime, krows, T, vis)
    for s in range(3):
        for t in range(T):
            if t >= vis[s]:
                assert sc[0, s, t] == -np.inf
                continue
            tot = Fraction(0)
            for h in range(H):
                dot = sum(Fraction(float(qd[0, s, h, d])) * Fraction(float(kd[0, t, d])) for d in range(128))
                tot += Fraction(float(wprime[0, s, h])) * max(dot, Fraction(0))
            assert abs(Fraction(float(sc[0, s, t])) - tot) <= abs(tot) * Fraction(1, 2 ** 50)


def test_scores_head_permutation_and_linearity():
    q = _rand_bf16((1, 4, 8, 128))
    k = _rand_bf16((1, 10, 128))
    qc, qs, _ = O.fp4_quant_e8m0(q)
    kc, ks, _ = O.fp4_quant_e8m0(k)
    qr, kr = O.pack_row68(qc, qs), O.pack_row68(kc, ks)
    w = RNG.standard_normal((1, 4, 8))
    vis = np.full(4, 10)
    base = O.index_scores(qr, w, kr, 10, vis)
    perm = RNG.permutation(8)
    assert np.allclose(O.index_scores(qr[:, :, perm], w[:, :, perm], kr, 10, vis), base, rtol=1e-13)
    assert np.array_equal(O.index_scores(qr, 2 * w, kr, 10, vis), 2 * base)
    w0 = w.copy()
    w0[..., 3] = 0
    # zero weight drops a head; the head's relu keeps negative dots out
    one_head = O.index_scores(qr[:, :, 3:4], np.ones((1, 4, 1)), kr, 10, vis)
    assert np.all(one_head >= 0)
    assert np.allclose(O.index_scores(qr, w0, kr, 10, vis) + w[..., 3:4] * one_head, base, rtol=1e-12, atol=1e-12)


def test_visible_lens_causal_rule():
    v = O.visible_lens(0, 12, 4)
    assert list(v) == [0, 0, 0, 1, 1, 1, 1, 2, 2, 2, 2, 3]     # arange(1..S) // ratio
    assert list(O.visible_lens(32767, 1, 4)) == [8192]           # decode: end_pos // ratio


# ----------------------------------------------------------------------- top-k
def _brute_topk(row, vis, k, offset, width):
    """Rank counting: position t is kept iff fewer than k finite visible entries beat it."""
    keep = []
    for t in range(min(vis, len(row))):
        if not np.isfinite(row[t]):
            continue
        beats = sum(1 for u in range(min(vis, len(row)))
                    if np.isfinite(row[u]) and (row[u] > row[t] or (row[u] == row[t] and u < t)))
        if beats < k:
            keep.append(t + offset)
    return keep + [-1] * (width - len(keep))


def test_topk_brute_force_with_ties():
    for trial in range(300):
        T = int(RNG.integers(1, 14))
        k = int(RNG.integers(1, 8))
        row = RNG.integers(-3, 4, T).astype(np.float64)     # many exact ties
        if trial % 3 == 0:
            row[RNG.random(T) < 0.3] = -np.inf
        vis = int(RNG.integers(0, T + 1))
        off = int(RNG.integers(0, 5))
        got = O.topk_positions(row[None, :], np.array([vis]), k, off, T)[0]
        assert list(got) == _brute_topk(row, vis, min(k, T), off, k)


def test_topk_invariants_random():
    R, T, k = 50, 300, 40
    sc = RNG.standard_normal((R, T))
    vis = RNG.integers(0, T + 1, R)
    for r in range(R):
        sc[r, vis[r]:] = -np.inf
    out = O.topk_positions(sc, vis, k, 0, T)
    for r in range(R):
        valid = out[r][out[r] >= 0]
        assert np.all(np.diff(valid) > 0)                               # ascending
        assert np.all(out[r][len(valid):] == -1)                        # -1 trailing
        assert len(valid) == min(k, vis[r])
        if len(valid):
            unsel = np.setdiff1d(np.arange(vis[r]), valid)
            if len(unsel):
                assert sc[r, valid].min() >= sc[r, unsel].max()


def test_short_context_rows_golden():
    for line in open(os.path.join(GOLDEN, "short_context_fill.txt")):
        if not line.strip() or line[0] == "#":
            continue
        pos, row = line.split(":")
        pos = int(pos)
        want = [int(v) for v in row.split()]
        T = 6 * 4                                     # any width >= the visible count
        vis = O.visible_lens(0, pos + 1, 4)[-1:]
        sc = RNG.standard_normal((1, T))
        sc[0, vis[0]:] = -np.inf
        assert list(O.topk_positions(sc, vis, 6, 0, T)[0]) == want


# ----------------------------------------------------------------------- candidate blocks
def test_select_candidate_blocks_brute_force():
    for trial in range(200):
        cbs = int(RNG.integers(1, 5))
        T = int(RNG.integers(1, 25))
        cbk = int(RNG.integers(1, 6))
        vis = int(RNG.integers(0, T + 1))
        row = RNG.integers(-4, 5, T).astype(np.float64)
        row[vis:] = -np.inf
        got = O.select_candidate_blocks(row[None, :], np.array([vis]), cbk, cbs)[0]
        nblk = -(-T // cbs)
        best = {}
        for j in range(nblk):
            if j * cbs < vis:
                best[j] = max(row[j * cbs:min((j + 1) * cbs, T)])
        kept = sorted(j for j in best
                      if sum(1 for i in best if best[i] > best[j] or (best[i] == best[j] and i < j)) < cbk)
        assert list(got) == kept + [-1] * (cbk - len(kept))


def test_candidate_blocks_contain_argmax_and_all_when_few():
    sc = RNG.standard_normal((30, 200))
    vis = RNG.integers(1, 201, 30)
    for r in range(30):
        sc[r, vis[r]:] = -np.inf
    blocks = O.select_candidate_blocks(sc, vis, 4, 16)
    for r in range(30):
        assert int(np.argmax(sc[r])) // 16 in blocks[r]
    many = O.select_candidate_blocks(sc, vis, 20, 16)
    for r in range(30):
        kept = many[r][many[r] >= 0]
        assert list(kept) == list(range(-(-vis[r] // 16)))


def test_level_two_mask_emits_only_kept_positions():
    T = 256
    sc = RNG.standard_normal((10, T))
    vis = np.full(10, T)
    blocks = O.select_candidate_blocks(sc, vis, 3, 32)
    keep = O.candidate_mask(blocks, T, 32)
    assert np.all(keep.sum(axis=1) == 96)
    masked = np.where(keep, RNG.standard_normal((10, T)), -np.inf)
    out = O.topk_positions(masked, vis, 200, 0, T)
    for r in range(10):
        v = out[r][out[r] >= 0]
        assert len(v) == 96 and np.all(keep[r, v])


# ----------------------------------------------------------------------- composition
def test_forward_tiny_composition():
    from workloads import WORKLOADS, ROPE
    import torch
    wl = WORKLOADS["tiny_prefill"]
    as_bits = lambda t: t.view(torch.int16).numpy().view(np.uint16)
    q, w, lat = as_bits(wl.q()), as_bits(wl.w()), as_bits(wl.latent())
    wk, knw = as_bits(wl.wk()), as_bits(wl.k_norm_w())
    cos, sin = O.yarn_freqs_cis(wl.rope_dim, wl.max_pos, ROPE.theta, ROPE.factor, ROPE.original_seq_len,
                                ROPE.beta_fast, ROPE.beta_slow)
    slots, rows, _ = O.publish_keys(lat, wk, knw, cos, sin, 0, wl.ratio, wl.rope_dim, wl.norm_eps)
    cache = np.zeros((wl.B, wl.T_cap, 68), np.uint8)
    cache[:, slots] = rows
    top, _, sc = O.forward(q, w, cache, cos, sin, 0, wl.ratio, wl.rope_dim, wl.topk, wl.offset)
    assert top.shape == (1, 256, 16)
    assert np.all(top[0, :3] == -1)                                   # rows 0..2 see nothing
    vis = O.visible_lens(0, 256, 4)
    for s in range(256):
        n = min(vis[s], 16)
        assert np.all(top[0, s, :n] >= 0) and np.all(top[0, s, n:] == -1)
        if vis[s] <= 16:
            assert list(top[0, s, :n]) == list(range(n))


# ----------------------------------------------------------------------------- FP8 rows
def _torch_e4m3_codes(x_f32: np.ndarray) -> np.ndarray:
    """PyTorch's float32 -> float8_e4m3fn conversion (round to nearest even) as bytes."""
    torch = pytest.importorskip("torch")
    return torch.from_numpy(np.ascontiguousarray(x_f32, dtype=np.float32)).to(torch.float8_e4m3fn) \
        .view(torch.uint8).numpy()


def test_e4m3_rounding_exhaustive_against_torch():
    """Every finite bf16 value in [-448, 448] (which includes every e4m3 midpoint, so every
    tie) rounds like PyTorch's float8_e4m3fn conversion, sign kept for values that round
    to zero. Each row carries 448 so that its scale is 2**0."""
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    v = O.bf16_to_f64(bits)
    ok = np.isfinite(v) & (np.abs(v) <= 448.0)
    vals = bits[ok]
    n = (len(vals) + 126) // 127 * 127
    padded = np.concatenate([vals, np.zeros(n - len(vals), np.uint16)]).reshape(-1, 127)
    rows = np.concatenate([np.full((padded.shape[0], 1), O.f32_to_bf16(np.float32(448.0)), np.uint16), padded],
                          axis=1)
    codes, e, _ = O.fp8_quant_ue8m0(rows)
    assert np.all(e == 0)
    ref = _torch_e4m3_codes(O.bf16_to_f64(rows).astype(np.float32))
    assert np.array_equal(codes, ref)


def test_e4m3_golden_ties():
    """Hand-worked ties between neighbouring e4m3 values go to the even code."""
    cases = {1.0625: 1.0, 1.1875: 1.25, 17.0: 16.0, 19.0: 20.0, 0.0029296875: 0.00390625, 0.0009765625: 0.0,
             -0.0009765625: -0.0, 440.0: 448.0, 424.0: 416.0}
    for x, want in cases.items():
        row = np.zeros(128, np.uint16)
        row[0] = O.f32_to_bf16(np.float32(448.0))
        row[1] = O.f32_to_bf16(np.float32(x))
        _, e, deq = O.fp8_quant_ue8m0(row[None])
        assert e[0] == 0 and deq[0, 1] == want and math.copysign(1.0, deq[0, 1]) == math.copysign(1.0, want), x


def test_ue8m0_fp8_closed_forms():
    """The scale is the smallest power of two 2**e with 448 * 2**e >= amax; all-zero rows
    take the floor 2**-126."""
    for amax, want in [(448.0, 0), (450.0, 1), (224.0, -1), (225.0, 0), (0.875, -9), (0.0, -126), (2.0 ** -127, -126),
                       (3.5 * 2.0 ** 100, 93)]:
        row = np.zeros(128, np.uint16)
        row[5] = O.f32_to_bf16(np.float32(amax))
        assert O.bf16_to_f64(row[5]) == amax, amax
        _, e, _ = O.fp8_quant_ue8m0(row[None])
        assert e[0] == want, (amax, e[0], want)


def test_fp8_error_bound_and_row_bytes():
    """|x - deq| is within half an e4m3 step: 2**-4 |x| for normal values, 2**(e-10) at the
    subnormal end; the row is the 128 codes then the f32 scale little-endian."""
    rng = np.random.default_rng(3)
    x = (rng.standard_normal((64, 128)) * np.exp(rng.uniform(-20, 20, (64, 1)))).astype(np.float32)
    bits = O.f32_to_bf16(x)
    codes, e, deq = O.fp8_quant_ue8m0(bits)
    xv = O.bf16_to_f64(bits)
    assert np.all(np.abs(xv - deq) <= np.maximum(np.abs(xv) * 2.0 ** -4, np.ldexp(1.0, e[:, None] - 10)))
    rows = O.pack_row132(codes, e)
    assert rows.shape == (64, 132) and np.array_equal(rows[:, :128], codes)
    sc = rows[:, 128:].copy().view("<f4")[:, 0]
    assert np.array_equal(sc.astype(np.float64), np.ldexp(1.0, e))
    one = O.pack_row132(np.zeros((1, 128), np.uint8), np.array([0]))
    assert list(one[0, 128:]) == [0x00, 0x00, 0x80, 0x3F]
    assert np.array_equal(O.dequant_row132(rows), deq)


def test_fp8_scores_against_torch_dequantisation():
    """index_scores on FP8 rows equals sum_h w' relu(q . k) with q and k dequantised by
    PyTorch's e4m3 conversion times the rows' scales (one head with w' = 1 reduces to
    relu(q . k))."""
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(5)
    q = O.f32_to_bf16(rng.standard_normal((1, 3, 4, 128)).astype(np.float32))
    k = O.f32_to_bf16((rng.standard_normal((1, 9, 128)) * 3).astype(np.float32))
    qr, kr = O.quantise_rows(q, "fp8"), O.quantise_rows(k, "fp8")
    w = rng.standard_normal((1, 3, 4))

    def deq(rows):
        vals = torch.from_numpy(np.ascontiguousarray(rows[..., :128])).view(torch.float8_e4m3fn).float().numpy()
        sc = np.ascontiguousarray(rows[..., 128:]).view("<f4")[..., 0]
        return vals.astype(np.float64) * sc[..., None]
    dq, dk = deq(qr), deq(kr)
    ref = np.einsum("sht,sh->st", np.maximum(np.einsum("shd,td->sht", dq[0], dk[0]), 0.0), w[0])
    got = O.index_scores(qr, w, kr, 9, np.full(3, 9))[0]
    assert np.allclose(got, ref, rtol=0, atol=1e-12 * np.abs(ref).max())
    one = O.index_scores(qr[:, :, :1], np.ones((1, 3, 1)), kr, 9, np.full(3, 9))[0]
    assert np.allclose(one, np.maximum(dq[0, :, 0] @ dk[0].T, 0.0), rtol=0, atol=1e-12)
