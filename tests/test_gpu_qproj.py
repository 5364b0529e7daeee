"""GPU parity of the fused query projection (indexer_prep_q_proj: q = wq_b(qr), RoPE and the
fp4 quantiser in one kernel) against the oracle, through the C ABI."""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from tests import cases as C
from workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    import sparse_attention_top_indexer_gb300 as X
    X.load_library()
    return X


def _ws(X):
    ws = torch.empty(X.STATUS_BYTES, dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    return ws


# qp_a: one ragged 128-row tile, K of two stages; qp_b: H = 8 (four 256-feature tiles), three
# row tiles, positions from 7; qp_c: 256 tiles (more than one per CTA: both accumulators and
# the stage ring across tiles), the prefill q_lora_rank; qp_d: three sequences at start_pos 4093
@pytest.mark.parametrize("name,B,S,H,Kq,start", [("qp_a", 2, 37, 64, 128, 0), ("qp_b", 1, 300, 8, 1280, 7),
                                                 ("qp_c", 1, 1024, 64, 1280, 0), ("qp_d", 3, 50, 16, 640, 4093)])
def test_qproj_parity(X, name, B, S, H, Kq, start):
    wl = dataclasses.replace(WORKLOADS["prefill"], name=name, B=B, S=S, H=H, start_pos=start, q_lora_rank=Kq)
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    qr, wq, w = wl.qr("cuda"), wl.wq_b("cuda"), wl.w("cuda")
    rows = torch.empty((B, S, H, 68), dtype=torch.uint8, device="cuda")
    wp = torch.empty((B, S, H), dtype=torch.float32, device="cuda")
    qo = torch.empty((B, S, H, 128), dtype=torch.bfloat16, device="cuda")
    ws = _ws(X)
    X.indexer_prep_q_proj(d, qr, wq, w, start, table, rows, wp, ws, q_out=qo)
    X.indexer_status(ws)
    # q: the exactly rounded projection, except where the f32 accumulation moves the sum across
    # a bf16 rounding midpoint; every value within the f32 accumulation bound of the exact sum:
    # |q - exact| <= 2^-8 |exact| (the bf16 rounding) + Kq 2^-24 sum_j |qr_j wq_j|
    ref_q = O.project_queries(C.bits(qr), C.bits(wq), H)
    got_q = C.bits(qo)
    diff = got_q != ref_q
    assert diff.mean() < 1e-3, f"{diff.mean():.2e} of q differ"
    a64, b64 = O.bf16_to_f64(C.bits(qr)).reshape(-1, Kq), O.bf16_to_f64(C.bits(wq))
    exact = (a64 @ b64.T).reshape(got_q.shape)
    mag = (np.abs(a64) @ np.abs(b64).T).reshape(got_q.shape)
    acc_bound = Kq * 2.0 ** -24 * mag
    g64, r64 = O.bf16_to_f64(got_q), O.bf16_to_f64(ref_q)
    err = np.abs(g64 - exact)
    assert np.all(err <= 2.0 ** -8 * np.abs(exact) + acc_bound + 2.0 ** -133)
    # a value differs only where the exact sum lies within the accumulation bound of the bf16
    # rounding midpoint between the two results (or, where the sum cancels, of either result)
    mid = 0.5 * (g64 + r64)
    near_mid = np.abs(exact - mid) <= acc_bound + 2.0 ** -133
    assert np.all(near_mid[diff] | (err[diff] <= acc_bound[diff] + 2.0 ** -133))
    # rows and w': the oracle's query prep of the GPU's own q (the quantiser decides in the
    # kernel's precision), bit-exact
    ref_rows, ref_w, _ = O.prep_queries(got_q, C.bits(w), cos, sin, start, wl.rope_dim, H)
    got = rows.cpu().numpy()
    assert np.array_equal(got, ref_rows), f"{np.sum(np.any(got != ref_rows, axis=-1))} query rows differ"
    assert np.allclose(wp.cpu().numpy(), ref_w, rtol=2e-7, atol=0)
    # end to end from qr: the oracle's rows of its own (exactly rounded) q differ from the
    # kernel's only in head vectors that hold one of the q values counted above
    ref_rows_e2e, _, _ = O.prep_queries(ref_q, C.bits(w), cos, sin, start, wl.rope_dim, H)
    row_diff = np.any(got != ref_rows_e2e, axis=-1)
    assert np.all(np.any(diff, axis=-1)[row_diff]), "a query row differs without a differing q value"
    assert row_diff.mean() <= np.any(diff, axis=-1).mean()
    # without q_out: the same rows
    rows2 = torch.zeros_like(rows)
    X.indexer_prep_q_proj(d, qr, wq, w, start, table, rows2, wp, ws)
    X.indexer_status(ws)
    assert torch.equal(rows, rows2)


def test_qproj_rejects_what_it_does_not_take(X):
    wl = dataclasses.replace(WORKLOADS["prefill"], name="qp_err", B=1, S=8, H=8, q_lora_rank=128)
    table = C.gpu_table(wl.max_pos)
    qr, wq, w = wl.qr("cuda"), wl.wq_b("cuda"), wl.w("cuda")
    rows = torch.empty((1, 8, 8, 68), dtype=torch.uint8, device="cuda")
    wp = torch.empty((1, 8, 8), dtype=torch.float32, device="cuda")
    ws = _ws(X)
    with pytest.raises(X.IndexerError) as e:   # FP8 query rows are not written by this kernel
        X.indexer_prep_q_proj(C.dims_of(wl, key_format=1), qr, wq, w, 0, table, rows, wp, ws)
    assert e.value.code == -3
    with pytest.raises(X.IndexerError) as e:   # q_lora_rank not a multiple of 64
        X.indexer_prep_q_proj(C.dims_of(wl), qr[..., :96].contiguous(), wq[:, :96].contiguous(), w, 0, table, rows,
                              wp, ws)
    assert e.value.code == -3
