"""Pins of the upstream-producer oracle functions (compress module page: Compressor.forward,
fp4_quant_e4m3_inplace, LATENT_BLOCK; index-keys page: weights_proj) against what the pages
and the mathematics fix, never against the oracle's own formulas: torch's e4m3 conversion,
hand-derived scale ties, closed forms of the softmax pooling (uniform gates give the mean,
a dominant gate picks its token, shifts and token order do not matter) and a 60-digit
decimal evaluation of the RMSNorm."""
import math
import os
from decimal import Decimal, getcontext
from fractions import Fraction

import numpy as np
import torch

import oracle as O

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
RNG = np.random.default_rng(77)


def _bits(vals):
    f = np.asarray(vals, dtype=np.float32)
    b = f.view(np.uint32)
    assert np.all((b & 0xFFFF) == 0), "value not representable in bf16"
    return (b >> 16).astype(np.uint16)


def _rand_bf16(shape, scale=1.0):
    x = (RNG.standard_normal(shape) * scale).astype(np.float32)
    return (x.view(np.uint32) >> 16).astype(np.uint16)


# ----------------------------------------------------------------------------- e4m3 scale rounding
def test_e4m3_round_matches_torch_on_every_grid_point_and_midpoint():
    g = O.E4M3_GRID
    mids = (g[:-1] + g[1:]) / 2
    quarter = np.concatenate([g[:-1] + (g[1:] - g[:-1]) * f for f in (0.25, 0.49, 0.51, 0.75)])
    y = np.concatenate([g, mids, quarter]).astype(np.float32)           # all exact in f32
    want = torch.from_numpy(y).to(torch.float8_e4m3fn).view(torch.uint8).numpy() & 0x7F
    got = O.e4m3_round(y.astype(np.float64))
    assert np.array_equal(got, want)


def test_e4m3_round_saturates_at_448():
    assert O.E4M3_GRID[O.e4m3_round(np.array([448.0, 464.0, 1e6]))].tolist() == [448.0, 448.0, 448.0]


# ----------------------------------------------------------------------------- fp4 with e4m3 scales
def test_latent_quant_closed_forms():
    # all zero: amax floored at 6 * 2^-9, scale 2^-9 (the smallest e4m3 value), codes 0
    codes, sc, deq = O.fp4_quant_e4m3(np.zeros((1, 16), np.uint16))
    assert O.E4M3_GRID[sc[0, 0]] == 2.0 ** -9 and not codes.any() and not deq.any()
    # amax 6: scale 1, the codes are the e2m1 golden table's
    vals, want = [], []
    for line in open(os.path.join(GOLDEN, "e2m1_rne.txt")):
        line = line.split("#")[0].strip()
        if line:
            v, c = line.split()
            vals.append(float(v))
            want.append(int(c))
    for i in range(0, len(vals), 15):
        blk = [6.0] + vals[i:i + 15]
        blk += [0.0] * (16 - len(blk))
        codes, sc, _ = O.fp4_quant_e4m3(_bits(blk)[None])
        assert O.E4M3_GRID[sc[0, 0]] == 1.0
        assert codes[0, 1:1 + len(vals[i:i + 15])].tolist() == want[i:i + 15]
    # amax 6.375: amax / 6 = 1.0625 ties between e4m3 1.0 (even code) and 1.125 -> scale 1.0,
    # and 6.375 / 1 saturates onto 6 (code 7)
    codes, sc, deq = O.fp4_quant_e4m3(_bits([6.375] + [0.0] * 15)[None])
    assert O.E4M3_GRID[sc[0, 0]] == 1.0 and codes[0, 0] == 7 and O.bf16_to_f64(deq[0, 0]) == 6.0
    # amax 7.125: 1.1875 ties between 1.125 (odd code) and 1.25 (even) -> scale 1.25; 7.125 / 1.25
    # = 5.7 -> 6 (code 7) -> 7.5; -0.3125 / 1.25 = -0.25 ties to 0 keeping the sign (code 8)
    codes, sc, deq = O.fp4_quant_e4m3(_bits([7.125, -0.3125] + [0.0] * 14)[None])
    assert O.E4M3_GRID[sc[0, 0]] == 1.25 and codes[0, 0] == 7 and codes[0, 1] == 8
    assert O.bf16_to_f64(deq[0, 0]) == 7.5 and deq[0, 1] == 0x8000


def test_latent_quant_error_bound():
    x = _rand_bf16((64, 128), scale=3.0)
    codes, sc, deq = O.fp4_quant_e4m3(x)
    xv = O.bf16_to_f64(x).reshape(64, 8, 16)
    dv = O.bf16_to_f64(deq).reshape(64, 8, 16)
    s = O.E4M3_GRID[sc][..., None]
    amax = np.max(np.abs(xv), axis=-1, keepdims=True)
    assert np.all(s >= amax / 6.0 * (1 - 2.0 ** -4))     # e4m3 keeps 4 significant bits
    assert np.all(np.abs(dv - xv) <= s + 1e-300)           # at most half of the widest e2m1 gap (2)
    inside = np.abs(xv) <= 6 * s
    assert np.all(np.abs(dv - xv)[inside] <= s.repeat(16, -1)[inside])
    # dequantised values are sign * grid * scale exactly
    mags = O.E2M1_GRID[codes.reshape(64, 8, 16) & 7] * s
    assert np.array_equal(np.abs(dv), mags)


# ----------------------------------------------------------------------------- weights_proj
def test_weights_proj_is_the_correctly_rounded_linear():
    x = _rand_bf16((2, 3, 96))
    wp = _rand_bf16((8, 96), scale=96 ** -0.5)
    w = O.weights_proj(x, wp)
    assert w.shape == (2, 3, 8)
    fr = lambda b: Fraction(float(O.bf16_to_f64(np.array([b]))[0]))
    for (i, j, h) in [(0, 0, 0), (1, 2, 7), (0, 1, 3)]:
        exact = sum(fr(x[i, j, k]) * fr(wp[h, k]) for k in range(96))
        got = fr(w[i, j, h])
        # the nearest bf16 to the exact sum (ties even): no other bf16 is closer
        ulp = Fraction(2) ** (math.floor(math.log2(abs(float(exact)))) - 7)
        assert abs(got - exact) <= ulp / 2


# ----------------------------------------------------------------------------- compressor
def _rms_decimal(p, w, eps):
    getcontext().prec = 60
    pd = [Decimal(float(v)) for v in p]
    ms = sum(v * v for v in pd) / len(pd)
    r = 1 / (ms + Decimal(float(np.float32(eps)))).sqrt()
    return [Decimal(float(wi)) * v * r for wi, v in zip(w, pd)]


def _nearest_bf16_ok(got_bits, exact_dec):
    """got is the bf16 nearest to the exact value (within half an ulp)."""
    for b, e in zip(got_bits, exact_dec):
        g = Decimal(float(O.bf16_to_f64(np.array([b]))[0]))
        if e == 0:
            assert g == 0
            continue
        ulp = Decimal(2) ** (math.floor(math.log2(abs(float(e)))) - 7)
        assert abs(g - e) <= ulp / 2 * (1 + Decimal(10) ** -30)


def test_compressor_ratio_one_is_the_normed_projection():
    x = _rand_bf16((1, 3, 64))
    wkv = _rand_bf16((16, 64), scale=0.125)
    wg = _rand_bf16((16, 64), scale=0.125)
    nw = O.f64_to_bf16(O.bf16_to_f64(_rand_bf16((16,), 0.3)) + 1.0)
    lat = O.compress_latent(x, wkv, wg, nw, 1, 1e-6)
    for t in range(3):
        kv = [sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(O.bf16_to_f64(x[0, t]), O.bf16_to_f64(wkv[d])))
              for d in range(16)]
        _nearest_bf16_ok(lat[0, t], _rms_decimal([float(v) for v in kv], O.bf16_to_f64(nw), 1e-6))


def test_compressor_uniform_gates_give_the_mean():
    x = _rand_bf16((2, 8, 32))
    wkv = _rand_bf16((16, 32), scale=0.2)
    wg = np.zeros((16, 32), np.uint16)                      # every score 0: uniform softmax
    nw = np.full(16, 0x3F80, np.uint16)
    lat = O.compress_latent(x, wkv, wg, nw, 4, 1e-6)
    assert lat.shape == (2, 2, 16)
    kv = O.bf16_to_f64(x) @ O.bf16_to_f64(wkv).T
    for b in range(2):
        for g in range(2):
            mean = kv[b, 4 * g:4 * g + 4].mean(axis=0)
            _nearest_bf16_ok(lat[b, g], _rms_decimal(mean, np.ones(16), 1e-6))


def test_compressor_dominant_gate_picks_its_token():
    """A gate feature that is 1 on one token of each group and 0 elsewhere, weighted 400 in
    every gate row, gives that token a softmax weight 1 - O(e^-390): the latent is the
    ratio-1 latent of that token."""
    ratio, G, dim, hd = 4, 3, 40, 16
    x = _rand_bf16((1, G * ratio, dim), scale=0.5)
    x[..., 0] = 0
    pick = [1, 3, 0]
    for g, k in enumerate(pick):
        x[0, g * ratio + k, 0] = 0x3F80
    wkv = _rand_bf16((hd, dim), scale=0.2)
    wkv[:, 0] = 0
    wg = _rand_bf16((hd, dim), scale=0.01)
    wg[:, 0] = _bits([400.0])[0]
    nw = O.f64_to_bf16(O.bf16_to_f64(_rand_bf16((hd,), 0.3)) + 1.0)
    lat = O.compress_latent(x, wkv, wg, nw, ratio, 1e-6)
    one = O.compress_latent(x, wkv, wg, nw, 1, 1e-6)
    for g, k in enumerate(pick):
        assert np.array_equal(lat[0, g], one[0, g * ratio + k])


def test_compressor_shift_and_token_order_invariance():
    ratio, dim, hd = 4, 32, 16
    x = _rand_bf16((1, 8, dim))
    wkv = _rand_bf16((hd, dim), scale=0.2)
    wg = _rand_bf16((hd, dim), scale=0.2)
    nw = np.full(hd, 0x3F80, np.uint16)
    base = O.compress_latent(x, wkv, wg, nw, ratio, 1e-6)
    # token order inside a group
    perm = np.array([2, 0, 3, 1, 5, 7, 4, 6])
    assert np.all(np.abs(O.bf16_to_f64(O.compress_latent(x[:, perm], wkv, wg, nw, ratio, 1e-6)) -
                         O.bf16_to_f64(base)) <= 2.0 ** -7 * np.abs(O.bf16_to_f64(base)))
    # a feature equal on every token adds the same amount to all gate scores of a group
    x2 = x.copy()
    x2[..., 0] = 0x4000                                       # 2.0 on every token
    wkv2 = wkv.copy()
    wkv2[:, 0] = 0
    wg2 = wg.copy()
    wg2[:, 0] = _bits([3.0])[0]
    x0 = x.copy()
    x0[..., 0] = 0
    a = O.compress_latent(x2, wkv2, wg2, nw, ratio, 1e-6)
    b = O.compress_latent(x0, wkv2, wg2, nw, ratio, 1e-6)
    assert np.all(np.abs(O.bf16_to_f64(a) - O.bf16_to_f64(b)) <= 2.0 ** -7 * np.abs(O.bf16_to_f64(b)))
