"""The FP8 key format (132-byte rows: 128 e4m3 codes + an f32 power-of-two scale)
through the C ABI, against the oracle: key publish and query prep bit for bit, scores
within tolerance and indices exact up to boundary swaps, for decode (single-row kernel,
split and fused), prefill (several-row kernel), the two-level decode and a mixed batch
through a page pool.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from tests import cases as C
from workloads import MIXED, WORKLOADS

pytestmark = pytest.mark.gpu

FP8 = 1


@pytest.fixture(scope="module")
def X():
    import sparse_attention_top_indexer_gb300 as X
    X.load_library()
    return X


def _decode(B=6, start=8191, H=64, topk=512, **kw):
    return dataclasses.replace(WORKLOADS["decode"], name=f"fp8_dec_{B}_{H}", B=B, start_pos=start, H=H, topk=topk,
                               key_format=FP8, **kw)


def _forward(X, wl, q, w, table, cache, cand_in=None, want_cand=False, want_scores=True):
    d = C.dims_of(wl)
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda") if want_scores else None
    cand = torch.empty((wl.B, wl.S, wl.cand_topk_blocks), dtype=torch.int32, device="cuda") if want_cand else None
    X.indexer_forward(d, q, w, wl.start_pos, table, cache, top, ws, cand_in=cand_in, cand_out=cand, scores_out=sc)
    X.indexer_status(ws)
    return top, cand, sc


def test_fp8_publish_bit_exact(X):
    wl = _decode(B=3, start=4095)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    assert cache.shape[-1] == X.PAGE_BYTES_FP8
    assert np.array_equal(C.fp8_pages_to_rows(cache), C.oracle_cache(wl, cos, sin))


def test_fp8_query_prep_bit_exact(X):
    for wl in (_decode(B=5, start=4095, H=32), dataclasses.replace(WORKLOADS["prefill"], name="fp8_prep", S=1536,
                                                                       key_format=FP8)):
        d = C.dims_of(wl)
        table = C.gpu_table(wl.max_pos)
        cos, sin = C.oracle_table(wl.max_pos)
        q, w = wl.q("cuda"), wl.w("cuda")
        rows = torch.empty((wl.B, wl.S, wl.H, X.ROW_BYTES_FP8), dtype=torch.uint8, device="cuda")
        wp = torch.empty((wl.B, wl.S, wl.H), dtype=torch.float32, device="cuda")
        X.indexer_prep_q(d, q, w, wl.start_pos, table, rows, wp)
        ref_rows, ref_w, _ = O.prep_queries(C.bits(q), C.bits(w), cos, sin, wl.start_pos, wl.rope_dim, wl.H,
                                            fmt="fp8")
        assert np.array_equal(rows.cpu().numpy(), ref_rows), wl.name
        assert np.allclose(wp.cpu().numpy(), ref_w, rtol=2e-7, atol=0)


@pytest.mark.parametrize("B,H,start,topk", [(6, 64, 8191, 512), (3, 128, 4095, 256), (4, 16, 2047, 100)])
def test_fp8_decode_forward_and_split(X, B, H, start, topk):
    wl = _decode(B=B, start=start, H=H, topk=topk)
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    ref_cache = C.oracle_cache(wl, cos, sin)
    q, w = wl.q("cuda"), wl.w("cuda")
    top, _, sc = _forward(X, wl, q, w, table, cache)
    ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, wl.start_pos, wl.ratio, wl.rope_dim,
                                   wl.topk, wl.offset)
    C.assert_scores_close(sc.cpu().numpy(), ref_sc)
    swaps = C.compare_topk(top.cpu().numpy().reshape(-1, wl.topk), ref_top.reshape(-1, wl.topk),
                           ref_sc.reshape(-1, wl.T), wl.offset)
    # the split entry points give the fused forward's results bit for bit
    rows = torch.empty((wl.B, 1, wl.H, X.ROW_BYTES_FP8), dtype=torch.uint8, device="cuda")
    wp = torch.empty((wl.B, 1, wl.H), dtype=torch.float32, device="cuda")
    X.indexer_prep_q(d, q, w, wl.start_pos, table, rows, wp)
    ws = torch.empty(X.STATUS_BYTES, dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    sc2 = torch.empty_like(sc)
    X.indexer_scores(d, rows, wp, wl.start_pos, cache, sc2, ws)
    top2 = torch.empty_like(top)
    X.indexer_topk(d, sc2, wl.start_pos, top2)
    X.indexer_status(ws)
    assert torch.equal(sc2, sc) and torch.equal(top2, top)
    C.record_swaps(f"fp8/decode B{B} H{H}", swaps, wl.B, int((top >= 0).sum()))


@pytest.mark.parametrize("S,H,topk", [(256, 8, 16), (2048, 64, 128), (1024, 128, 64)])
def test_fp8_prefill_forward(X, S, H, topk):
    wl = dataclasses.replace(WORKLOADS["prefill"], name=f"fp8_pf_{S}_{H}", S=S, H=H, topk=topk, key_format=FP8)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    ref_cache = C.oracle_cache(wl, cos, sin)
    assert np.array_equal(C.fp8_pages_to_rows(cache), ref_cache)
    q, w = wl.q("cuda"), wl.w("cuda")
    top, _, sc = _forward(X, wl, q, w, table, cache)
    ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, wl.start_pos, wl.ratio, wl.rope_dim,
                                   wl.topk, wl.offset)
    C.assert_scores_close(sc.cpu().numpy(), ref_sc)
    swaps = C.compare_topk(top.cpu().numpy().reshape(-1, wl.topk), ref_top.reshape(-1, wl.topk),
                           ref_sc.reshape(-1, wl.T), wl.offset)
    C.record_swaps(f"fp8/prefill S{S} H{H}", swaps, wl.B * wl.S, int((top >= 0).sum()))


def test_fp8_two_level_decode(X):
    wl = _decode(B=4, start=32767, topk=1024, cand_topk_blocks=32, cand_block_size=64)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    ref_cache = C.oracle_cache(wl, cos, sin)
    q1, w1 = wl.q("cuda", tag="q1"), wl.w("cuda", tag="w1")
    _, cand, sc1 = _forward(X, wl, q1, w1, table, cache, want_cand=True)
    _, ref_cand, ref_sc1 = O.forward(C.bits(q1), C.bits(w1), ref_cache, cos, sin, wl.start_pos, wl.ratio,
                                     wl.rope_dim, wl.topk, wl.offset, cand_topk_blocks=wl.cand_topk_blocks,
                                     cand_block_size=wl.cand_block_size, want_candidates=True)
    C.assert_scores_close(sc1.cpu().numpy(), ref_sc1)
    got = cand.cpu().numpy()
    for r in range(wl.B):   # a block may swap only where its max ties the last kept block's
        g, o = set(got[r, 0]), set(ref_cand[r, 0])
        if g != o:
            bm = np.array([ref_sc1[r, 0, j * 64:(j + 1) * 64].max() for j in range(wl.T // 64)])
            kth = np.sort(bm)[::-1][wl.cand_topk_blocks - 1]
            for j in g ^ o:
                assert abs(bm[j] - kth) <= C.SCORE_ATOL + C.SCORE_RTOL * abs(kth)
    q2, w2 = wl.q("cuda", tag="q2"), wl.w("cuda", tag="w2")
    top2, _, _ = _forward(X, wl, q2, w2, table, cache, cand_in=torch.from_numpy(ref_cand).cuda(),
                          want_scores=False)   # the kept-pages-only path
    ref_top2, _, ref_sc2 = O.forward(C.bits(q2), C.bits(w2), ref_cache, cos, sin, wl.start_pos, wl.ratio,
                                     wl.rope_dim, wl.topk, wl.offset, cand_in=ref_cand,
                                     cand_block_size=wl.cand_block_size)
    swaps = C.compare_topk(top2.cpu().numpy().reshape(-1, wl.topk), ref_top2.reshape(-1, wl.topk),
                           ref_sc2.reshape(-1, wl.T), wl.offset)
    C.record_swaps("fp8/two-level level two", swaps, wl.B, int((top2 >= 0).sum()))


def test_fp8_mixed_batch_page_pool(X):
    m = dataclasses.replace(MIXED["mixed_small"], key_format=FP8)
    d = X.make_dims(n_heads=m.H, ratio=m.ratio, index_topk=m.topk, offset=m.offset, rope_dim=m.rope_dim,
                    head_dim=m.D, norm_eps=m.norm_eps, key_format=FP8)
    table = C.gpu_table(m.max_pos)
    cos, sin = C.oracle_table(m.max_pos)
    pool = X.new_key_pool(m.num_pages, key_format=FP8)
    bt = m.block_table()
    lat, pos, slots = [], [], []
    for b in range(m.n_seq):
        T = m.T_list[b]
        if T:
            j = torch.arange(T)
            lat.append(m.latent(b))
            pos.append(j * m.ratio)
            slots.append(bt[b, j // 64].long() * 64 + j % 64)
    ws = torch.empty(X.STATUS_BYTES, dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    X.indexer_publish_k_paged(d, torch.cat(lat).cuda(), m.wk("cuda"), m.k_norm_w("cuda"), table,
                              torch.cat(pos).to(torch.int32).cuda(), torch.cat(slots).to(torch.int32).cuda(), pool, ws)
    X.indexer_status(ws)
    wsf = torch.empty(X.indexer_workspace_size_paged(d, m.Q, m.n_seq, m.T_max), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(wsf)
    top = torch.empty((m.Q, m.topk), dtype=torch.int32, device="cuda")
    sc = torch.empty((m.Q, m.T_max), dtype=torch.float32, device="cuda")
    q, w = m.q("cuda"), m.w("cuda")
    X.indexer_forward_paged(d, q, w, torch.tensor([sp for sp, _ in m.seqs], dtype=torch.int32, device="cuda"),
                            torch.tensor(m.q_start, dtype=torch.int32, device="cuda"), m.T_max, table, pool, bt.cuda(),
                            top, wsf, scores_out=sc)
    X.indexer_status(wsf)
    top, sc = top.cpu().numpy(), sc.cpu().numpy()
    qb, wb = C.bits(q), C.bits(w)
    pool_np = pool.cpu().numpy()
    for b, (sp, S) in enumerate(m.seqs):
        T = m.T_list[b]
        _, rows, _ = O.publish_keys(C.bits(m.latent(b))[None], C.bits(m.wk()), C.bits(m.k_norm_w()), cos, sin, 0,
                                    m.ratio, m.rope_dim, m.norm_eps, fmt="fp8")
        if T:
            assert np.array_equal(C.pool_to_rows(pool_np, bt[b], T), rows[0]), f"sequence {b}: pool rows"
        if S == 0:
            continue
        r0 = m.q_start[b]
        keys = np.zeros((1, max(T, 1), 132), np.uint8)
        if T:
            keys[0, :T] = rows[0]
        ref_top, _, ref_sc = O.forward(qb[None, r0:r0 + S], wb[None, r0:r0 + S], keys, cos, sin, sp, m.ratio,
                                       m.rope_dim, m.topk, m.offset)
        C.assert_scores_close(sc[r0:r0 + S, :T], ref_sc[0, :, :T])
        C.compare_topk(top[r0:r0 + S], ref_top[0], ref_sc[0, :, :T].reshape(S, T), m.offset)
