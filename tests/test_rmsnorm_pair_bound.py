"""The error bound behind the key publish's f32-pair RMSNorm route.

The GPU evaluates y = (w x) / sqrt(mean(x^2) + eps) in unevaluated f32 pairs (TwoSum sums of
the exact squares, an rsqrtf estimate with one second-order correction, an exact product of
the high part) and keeps that value only where it lies more than 2^-38 |P| from the bf16
rounding midpoint next to it; elsewhere it runs the f64 evaluation. That is sound when the
pair is within 2^-41 of the exact value. This test replays the same sequence of f32
operations in numpy (every step rounded to f32 as the device does, an rsqrtf-like estimate
off by up to 2.5 ulp) on seeded keys of several scales and checks the bound against the
exact value, so a change to the sequence that loosens it fails here, on the CPU.
"""
import numpy as np

F32, F64 = np.float32, np.float64


def _rn(x):
    return x.astype(F32)


def _add(a, b):
    return _rn(a.astype(F64) + b.astype(F64))


def _sub(a, b):
    return _rn(a.astype(F64) - b.astype(F64))


def _mul(a, b):
    return _rn(a.astype(F64) * b.astype(F64))


def _fma(a, b, c):
    # an f32 FMA: the product of two f32 values is exact in f64, and the f64 sum is within
    # 2^-53 of exact before the one f32 rounding
    return _rn(a.astype(F64) * b.astype(F64) + c.astype(F64))


def _two_sum(a, b):
    s = _add(a, b)
    z = _sub(s, a)
    return s, _add(_sub(a, _sub(s, z)), _sub(b, z))


def _bf16(x):
    b = x.astype(F32).view(np.uint32).astype(np.uint64)
    return (((b + 0x7FFF + ((b >> 16) & 1)) >> 16) << 16).astype(np.uint32).view(F32)


def test_pair_route_is_within_2_to_the_minus_41():
    rng = np.random.default_rng(20261203)
    n = 6000
    scale = (2.0 ** rng.uniform(-20, 20, size=(n, 1))).astype(F32)
    x = _bf16(rng.standard_normal((n, 128)).astype(F32) * scale)
    w = _bf16(rng.uniform(-1.5, 1.5, size=(n, 128)).astype(F32))
    eps = F32(1e-6)
    # sum of squares: exact squares, a TwoSum tree like the warp butterflies and warp pairs
    sh, sl = _mul(x, x), np.zeros((n, 128), F32)
    while sh.shape[1] > 1:
        t, e = _two_sum(sh[:, 0::2], sh[:, 1::2])
        sl = _add(_add(sl[:, 0::2], sl[:, 1::2]), e)
        sh = t
    mh, ml = _mul(sh[:, 0], np.full(n, 1 / 128, F32)), _mul(sl[:, 0], np.full(n, 1 / 128, F32))
    vh, vl = _two_sum(mh, np.full(n, eps, F32))
    vl = _add(vl, ml)
    vh, vl = _two_sum(vh, vl)
    # an rsqrtf-like estimate: within 2.5 ulp of 1/sqrt(vh)
    r0 = _rn(1.0 / np.sqrt(vh.astype(F64)) * (1 + rng.uniform(-2.5, 2.5, size=n) * 2.0 ** -23))
    p = _mul(r0, r0)
    pe = _fma(r0, r0, -p)
    q = _mul(vh, p)
    qe = _fma(vh, p, -q)
    d = _sub(_sub(np.ones(n, F32), q), _add(qe, _fma(vh, pe, _mul(vl, p))))
    rl = _mul(r0, _fma(np.full(n, 0.375, F32), _mul(d, d), _mul(np.full(n, 0.5, F32), d)))
    wx = _mul(w, x)
    r0b, rlb = np.broadcast_to(r0[:, None], wx.shape), np.broadcast_to(rl[:, None], wx.shape)
    ph = _mul(wx, r0b)
    pl = _fma(wx, rlb, _fma(wx, r0b, -ph))
    Ph, Pl = _two_sum(ph, pl)
    got = Ph.astype(F64) + Pl.astype(F64)
    # the exact value (f64 of exact bf16 products and sums is within 2^-50 of it here)
    ms = (x.astype(F64) ** 2).sum(axis=1) / 128
    exact = wx.astype(F64) / np.sqrt(ms + F64(eps))[:, None]
    nz = exact != 0
    rel = np.abs(got[nz] - exact[nz]) / np.abs(exact[nz])
    assert rel.max() < 2.0 ** -41, f"worst 2^{np.log2(rel.max()):.1f}"
