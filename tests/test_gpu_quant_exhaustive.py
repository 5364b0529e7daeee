"""The GPU quantiser on every finite bf16 pattern and on the golden ties, through the
query prep (indexer_prep_q), bit-exact against the oracle.

A RoPE table of (cos, sin) = (1, 0) everywhere turns the rotation into the identity (the
one exception, -0 - (-0) = +0 in a rotated pair, is the same IEEE operation on both
sides), so the bf16 patterns reach the e2m1 / e8m0 quantiser as given:
  * every finite pattern in ascending bit order, 128 per head vector (blocks of 32 close
    patterns: every code and scale byte), and again rolled by 64 dims so each pattern is
    also seen in the other half of a vector;
  * the e2m1 ties and thresholds of tests/golden/e2m1_rne.txt at scales 2^-126 .. 2^120,
    each block anchored by 6 * 2^e so that its scale is 2^e;
  * the rotation-order case of the oracle pins, where rounding each f32 product before
    the sum leaves a bf16 midpoint on an e2m1 tie (code 2; a fused multiply-add gives 3).
"""
import os

import numpy as np
import pytest
import torch

import oracle as O
from tests import cases as C
from tests.test_oracle_pins import ROPE_TIE_CS, ROPE_TIE_Q

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "e2m1_rne.txt")


@pytest.fixture(scope="module")
def X():
    import sparse_attention_top_indexer_gb300 as X
    X.load_library()
    return X


def _identity_table(max_pos: int):
    cos = np.ones((max_pos, 32), np.float32)
    sin = np.zeros((max_pos, 32), np.float32)
    return cos, sin


def _gpu_table(cos, sin):
    return torch.from_numpy(np.ascontiguousarray(np.stack([cos, sin], axis=-1))).cuda()


def _prep_both(X, q_bits: np.ndarray, cos, sin, H: int):
    """q_bits uint16 [1, S, H, 128] through indexer_prep_q and the oracle; returns both rows."""
    S = q_bits.shape[1]
    d = X.make_dims(n_heads=H, ratio=4, index_topk=16)
    q = torch.from_numpy(q_bits.view(np.int16)).view(torch.bfloat16).cuda()
    w_bits = np.full((1, S, H), 0x3F80, np.uint16)
    w = torch.from_numpy(w_bits.view(np.int16)).view(torch.bfloat16).cuda()
    rows = torch.empty((1, S, H, 68), dtype=torch.uint8, device="cuda")
    wp = torch.empty((1, S, H), dtype=torch.float32, device="cuda")
    X.indexer_prep_q(d, q, w, 0, _gpu_table(cos, sin), rows, wp)
    ref, _, _ = O.prep_queries(q_bits, w_bits, cos, sin, 0, 64, H)
    return rows.cpu().numpy(), ref


def _finite_patterns() -> np.ndarray:
    p = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    return p[((p >> 7) & 0xFF) != 0xFF]                   # 65024 finite patterns


@pytest.mark.parametrize("roll", [0, 64])
def test_every_finite_bf16_pattern(X, roll):
    pats = _finite_patterns()
    H = 8
    per_row = H * 128
    S = -(-pats.size // per_row)
    buf = np.zeros(S * per_row, np.uint16)
    buf[:pats.size] = pats
    q = np.roll(buf.reshape(S, H, 128), roll, axis=-1).reshape(1, S, H, 128)
    cos, sin = _identity_table(S)
    got, ref = _prep_both(X, q, cos, sin, H)
    bad = np.any(got != ref, axis=-1)
    assert not bad.any(), f"{bad.sum()} of {bad.size} head vectors differ"
    # the identity table left the values as given, so the quantiser saw every pattern: the
    # rows equal a direct quantisation except where a -0 in a rotated pair became +0
    direct_codes, direct_scales = O.unpack_row68(O.quantise_rows(q))
    codes, scales = O.unpack_row68(got)
    assert np.array_equal(scales, direct_scales)
    moved = codes != direct_codes
    assert np.all(q[moved] == 0x8000) and np.all(codes[moved] == 0)


def test_golden_ties_at_many_scales(X):
    vals = []
    for line in open(GOLDEN):
        line = line.split("#")[0].strip()
        if line:
            vals.append(float(line.split()[0]))
    vals = np.array(vals)                                   # at scale 1
    exps = list(range(-126, 121, 7))
    H = 8
    blocks = []
    for e in exps:
        for i in range(0, len(vals), 31):
            chunk = vals[i:i + 31] * 2.0 ** e
            blk = np.zeros(32)
            blk[0] = 6.0 * 2.0 ** e                          # anchor: the block's scale is 2^e
            blk[1:1 + len(chunk)] = chunk
            blocks.append(blk)
    while len(blocks) % (4 * H):
        blocks.append(np.zeros(32))
    arr = np.array(blocks).astype(np.float32)
    assert np.all(np.isfinite(arr))
    bits = (arr.view(np.uint32) >> 16).astype(np.uint16)
    assert np.array_equal(O.bf16_to_f64(bits), arr.astype(np.float64)), "tie values must be exact in bf16"
    S = len(blocks) // (4 * H)
    q = bits.reshape(1, S, H, 128)
    cos, sin = _identity_table(S)
    got, ref = _prep_both(X, q, cos, sin, H)
    assert np.array_equal(got, ref)


def test_rotation_order_case_on_the_gpu(X):
    H = 8
    q = np.zeros((1, 1, H, 128), np.uint16)
    q[0, 0, 3, 64], q[0, 0, 3, 65] = ROPE_TIE_Q
    q[0, 0, 3, 66] = 0x3FC0
    cos, sin = _identity_table(1)
    cos[0, 0], sin[0, 0] = ROPE_TIE_CS
    got, ref = _prep_both(X, q, cos, sin, H)
    assert np.array_equal(got, ref)
    codes, scales = O.unpack_row68(got[0, 0, 3])
    assert scales[2] == 125 and codes[65] == 2
