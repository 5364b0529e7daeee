"""The page pool and mixed batches through the C ABI, against the oracle.

Keys are published through a slot mapping into a pool of 64-key pages dealt to the
sequences in a seeded random order; indexer_forward_paged then runs batches that mix
decode rows, a prefill chunk at start_pos > 0, a prefill from 0, an empty sequence and a
one-key sequence. Each sequence is checked against the oracle run on that sequence alone
(its own start_pos, rows and keys); a uniform batch put through the pool must equal
indexer_forward bit for bit.
"""
import dataclasses
import types

import numpy as np
import pytest
import torch

import oracle as O
from tests import cases as C
from workloads import MIXED, WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    import sparse_attention_top_indexer_gb300 as X
    X.load_library()
    return X


def _dims(X, m, **over):
    kw = dict(n_heads=m.H, ratio=m.ratio, index_topk=m.topk, offset=m.offset, rope_dim=m.rope_dim, head_dim=m.D,
              cand_topk_blocks=m.cand_topk_blocks, cand_block_size=m.cand_block_size, norm_eps=m.norm_eps)
    kw.update(over)
    return X.make_dims(**kw)


def _status_ws(X):
    ws = torch.empty(X.STATUS_BYTES, dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    return ws


def _publish_pool(X, m, d, table):
    """Every sequence's keys 0 .. T_b - 1 through one paged publish; returns (pool, block table)."""
    pool = X.new_key_pool(m.num_pages)
    bt = m.block_table()
    lat, pos, slots = [], [], []
    for b in range(m.n_seq):
        T = m.T_list[b]
        if T == 0:
            continue
        j = torch.arange(T)
        lat.append(m.latent(b))
        pos.append(j * m.ratio)
        slots.append(bt[b, j // 64].long() * 64 + j % 64)
    ws = _status_ws(X)
    X.indexer_publish_k_paged(d, torch.cat(lat).cuda(), m.wk("cuda"), m.k_norm_w("cuda"), table,
                              torch.cat(pos).to(torch.int32).cuda(), torch.cat(slots).to(torch.int32).cuda(), pool, ws)
    X.indexer_status(ws)
    return pool, bt


def _oracle_keys(m, b, cos, sin):
    """The oracle's rows of sequence b's keys, [T_b, 68]."""
    _, rows, _ = O.publish_keys(C.bits(m.latent(b))[None], C.bits(m.wk()), C.bits(m.k_norm_w()), cos, sin, 0,
                                m.ratio, m.rope_dim, m.norm_eps)
    return rows[0]


def _forward_paged(X, m, d, q, w, table, pool, bt, cand_in=None, want_cand=False, want_scores=True):
    ws = torch.empty(X.indexer_workspace_size_paged(d, m.Q, m.n_seq, m.T_max), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    top = torch.full((m.Q, m.topk), -7, dtype=torch.int32, device="cuda")
    sc = torch.full((m.Q, m.T_max), 7.0, dtype=torch.float32, device="cuda") if want_scores else None
    cand = torch.empty((m.Q, d.cand_topk_blocks), dtype=torch.int32, device="cuda") if want_cand else None
    seq_pos = torch.tensor([sp for sp, _ in m.seqs], dtype=torch.int32, device="cuda")
    q_start = torch.tensor(m.q_start, dtype=torch.int32, device="cuda")
    X.indexer_forward_paged(d, q, w, seq_pos, q_start, m.T_max, table, pool, bt.cuda(), top, ws, cand_in=cand_in,
                            cand_out=cand, scores_out=sc)
    X.indexer_status(ws)
    return top, cand, sc


@pytest.mark.parametrize("name", ["mixed_small", "mixed_decode"])
def test_publish_paged_matches_oracle(X, name):
    m = MIXED[name]
    d = _dims(X, m)
    table = C.gpu_table(m.max_pos)
    cos, sin = C.oracle_table(m.max_pos)
    pool, bt = _publish_pool(X, m, d, table)
    pool_np = pool.cpu().numpy()
    for b in range(m.n_seq):
        if m.T_list[b]:
            got = C.pool_to_rows(pool_np, bt[b], m.T_list[b])
            assert np.array_equal(got, _oracle_keys(m, b, cos, sin)), f"sequence {b}: pool rows differ"
    owned = set(bt[bt >= 0].tolist())
    spare = [p for p in range(m.num_pages) if p not in owned]
    assert len(spare) == m.spare_pages and not pool_np[spare].any(), "a page no sequence owns was written"


@pytest.mark.parametrize("name", ["mixed_small", "mixed_decode"])
def test_forward_paged_mixed_against_oracle(X, name):
    m = MIXED[name]
    d = _dims(X, m)
    table = C.gpu_table(m.max_pos)
    cos, sin = C.oracle_table(m.max_pos)
    pool, bt = _publish_pool(X, m, d, table)
    q, w = m.q("cuda"), m.w("cuda")
    top, _, sc = _forward_paged(X, m, d, q, w, table, pool, bt)
    top, sc = top.cpu().numpy(), sc.cpu().numpy()
    qb, wb = C.bits(q), C.bits(w)
    swaps = 0
    for b, (sp, S) in enumerate(m.seqs):
        if S == 0:
            continue
        r0, T = m.q_start[b], m.T_list[b]
        keys = np.zeros((1, max(T, 1), 68), np.uint8)
        if T:
            keys[0, :T] = _oracle_keys(m, b, cos, sin)
        ref_top, _, ref_sc = O.forward(qb[None, r0:r0 + S], wb[None, r0:r0 + S], keys, cos, sin, sp, m.ratio,
                                       m.rope_dim, m.topk, m.offset)
        C.assert_scores_close(sc[r0:r0 + S, :T], ref_sc[0, :, :T])
        swaps += C.compare_topk(top[r0:r0 + S], ref_top[0], ref_sc[0, :, :T].reshape(S, T), m.offset)
    C.record_swaps(f"paged/{name}", swaps, int(top.shape[0]), int((top >= 0).sum()))


@pytest.mark.parametrize("name", ["decode", "tiny_prefill"])
def test_forward_paged_uniform_equals_forward(X, name):
    """A uniform batch (B sequences of S rows at one start_pos) put through a shuffled pool
    gives the sequence-major forward's scores and indices bit for bit."""
    wl = WORKLOADS[name]
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    q, w = wl.q("cuda"), wl.w("cuda")
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    top_u = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    sc_u = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda")
    X.indexer_forward(d, q, w, wl.start_pos, table, cache, top_u, ws, scores_out=sc_u)
    X.indexer_status(ws)
    # the same pages, shuffled into a pool
    pps = cache.shape[1]
    flat = cache.reshape(-1, X.PAGE_BYTES)
    perm = torch.randperm(flat.shape[0], generator=torch.Generator().manual_seed(1))
    pool = flat[perm.cuda()].contiguous()
    inv = torch.empty_like(perm)
    inv[perm] = torch.arange(perm.numel())
    bt = inv.view(wl.B, pps).to(torch.int32)
    m = types.SimpleNamespace(Q=wl.B * wl.S, n_seq=wl.B, T_max=wl.T, topk=wl.topk, seqs=[(wl.start_pos, wl.S)] * wl.B,
                              q_start=[b * wl.S for b in range(wl.B + 1)])
    top_p, _, sc_p = _forward_paged(X, m, d, q.view(-1, wl.H, wl.D), w.view(-1, wl.H), table, pool, bt)
    assert torch.equal(sc_p.view(wl.B, wl.S, wl.T), sc_u), "scores differ"
    assert torch.equal(top_p.view(wl.B, wl.S, wl.topk), top_u), "indices differ"


def test_forward_paged_two_level(X):
    """Level one publishes candidate blocks (cand_out) from a decode-only batch; level two
    (independent q, w) scores only the pages of the kept blocks and ranks their keys."""
    m = dataclasses.replace(MIXED["mixed_decode"], cand_topk_blocks=16, cand_block_size=64)
    d = _dims(X, m)
    table = C.gpu_table(m.max_pos)
    cos, sin = C.oracle_table(m.max_pos)
    pool, bt = _publish_pool(X, m, d, table)
    q1, w1 = m.q("cuda", tag="q1"), m.w("cuda", tag="w1")
    top1, cand, sc1 = _forward_paged(X, m, d, q1, w1, table, pool, bt, want_cand=True)
    q2, w2 = m.q("cuda", tag="q2"), m.w("cuda", tag="w2")
    ref_cands = []
    for b, (sp, S) in enumerate(m.seqs):
        keys = _oracle_keys(m, b, cos, sin)[None]
        _, rc, rsc = O.forward(C.bits(q1)[None, b:b + 1], C.bits(w1)[None, b:b + 1], keys, cos, sin, sp, m.ratio,
                               m.rope_dim, m.topk, m.offset, cand_topk_blocks=16, cand_block_size=64,
                               want_candidates=True)
        C.assert_scores_close(sc1.cpu().numpy()[b:b + 1, :m.T_list[b]], rsc[0])
        got = cand.cpu().numpy()[b]
        if not np.array_equal(got, rc[0, 0]):   # a swap only where a block max ties the 16th within tolerance
            T = m.T_list[b]
            bm = np.array([rsc[0, 0, j * 64:min((j + 1) * 64, T)].max() for j in range((T + 63) // 64)])
            kth = np.sort(bm)[::-1][15]
            for j in set(got) ^ set(rc[0, 0]):
                assert abs(bm[j] - kth) <= C.SCORE_ATOL + C.SCORE_RTOL * abs(kth)
        ref_cands.append(rc[0])
    ref_cand = np.concatenate(ref_cands)                      # [Q, 16]
    top2, _, _ = _forward_paged(X, m, d, q2, w2, table, pool, bt, cand_in=torch.from_numpy(ref_cand).cuda(),
                                want_scores=False)
    top2 = top2.cpu().numpy()
    swaps = 0
    for b, (sp, S) in enumerate(m.seqs):
        keys = _oracle_keys(m, b, cos, sin)[None]
        rt, _, rsc = O.forward(C.bits(q2)[None, b:b + 1], C.bits(w2)[None, b:b + 1], keys, cos, sin, sp, m.ratio,
                               m.rope_dim, m.topk, m.offset, cand_in=ref_cand[None, b:b + 1],
                               cand_block_size=64)
        swaps += C.compare_topk(top2[b:b + 1], rt[0], rsc[0].reshape(1, -1), m.offset)
    C.record_swaps("paged/two-level level two", swaps, int(top2.shape[0]), int((top2 >= 0).sum()))


def test_paged_bad_metadata_is_reported(X):
    """A block-table entry outside the pool and a row table out of order are reported by
    indexer_status as INDEXER_ERR_RANGE; nothing outside the buffers is touched."""
    m = MIXED["mixed_small"]
    d = _dims(X, m)
    table = C.gpu_table(m.max_pos)
    pool, bt = _publish_pool(X, m, d, table)
    q, w = m.q("cuda"), m.w("cuda")
    bad_bt = bt.clone()
    bad_bt[1, 3] = 1 << 20
    with pytest.raises(X.IndexerError) as e:
        _forward_paged(X, m, d, q, w, table, pool, bad_bt)
    assert e.value.code == -4
    # rows out of order: no sequence is scored, every row is all -1
    seq_pos = torch.tensor([sp for sp, _ in m.seqs], dtype=torch.int32, device="cuda")
    q_start = torch.tensor(m.q_start, dtype=torch.int32, device="cuda")
    q_start[2] = 200
    ws = torch.empty(X.indexer_workspace_size_paged(d, m.Q, m.n_seq, m.T_max), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    top = torch.full((m.Q, m.topk), -7, dtype=torch.int32, device="cuda")
    X.indexer_forward_paged(d, q, w, seq_pos, q_start, m.T_max, table, pool, bt.cuda(), top, ws)
    with pytest.raises(X.IndexerError) as e:
        X.indexer_status(ws)
    assert e.value.code == -4
    assert bool((top == -1).all())
    # a slot mapping entry outside the pool is skipped and reported
    ws2 = _status_ws(X)
    lat = m.latent(1)[:2].cuda()
    X.indexer_publish_k_paged(d, lat, m.wk("cuda"), m.k_norm_w("cuda"), table,
                              torch.tensor([0, 4], dtype=torch.int32, device="cuda"),
                              torch.tensor([m.num_pages * 64, -1], dtype=torch.int32, device="cuda"), pool, ws2)
    with pytest.raises(X.IndexerError) as e:
        X.indexer_status(ws2)
    assert e.value.code == -4


def test_paged_publish_few_keys_with_padding(X):
    """A decode-sized slot mapping (40 entries, the cluster-per-key publish) with padding
    entries (-1) interleaved: every real key lands at its slot bit-exact, and no other row of
    the pool is written."""
    m = MIXED["mixed_small"]
    d = _dims(X, m)
    table = C.gpu_table(m.max_pos)
    cos, sin = C.oracle_table(m.max_pos)
    n = 40
    slots = torch.arange(n, dtype=torch.int32) * 3 + 130   # spread over pages 2 .. 3
    slots[::5] = -1
    pos = torch.arange(n, dtype=torch.int32) * m.ratio
    pool = X.new_key_pool(m.num_pages)
    ws = _status_ws(X)
    X.indexer_publish_k_paged(d, m.latent(0)[:n].cuda(), m.wk("cuda"), m.k_norm_w("cuda"), table, pos.cuda(),
                              slots.cuda(), pool, ws)
    X.indexer_status(ws)
    got = C.pages_to_rows(pool)
    ref = _oracle_keys(m, 0, cos, sin)[:n]
    real = slots >= 0
    assert np.array_equal(got[slots[real].numpy()], ref[real.numpy()])
    untouched = np.ones(got.shape[0], dtype=bool)
    untouched[slots[real].numpy()] = False
    assert not got[untouched].any()


def test_paged_unowned_rows_are_empty(X):
    """Rows past q_start[n_seq] belong to no sequence: all -1, and the owned rows are
    unaffected."""
    m = MIXED["mixed_small"]
    d = _dims(X, m)
    table = C.gpu_table(m.max_pos)
    pool, bt = _publish_pool(X, m, d, table)
    q, w = m.q("cuda"), m.w("cuda")
    top_all, _, _ = _forward_paged(X, m, d, q, w, table, pool, bt, want_scores=False)
    sub = dataclasses.replace(m, seqs=m.seqs[:3])   # the first three sequences' rows only
    ws = torch.empty(X.indexer_workspace_size_paged(d, m.Q, 3, m.T_max), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    top = torch.full((m.Q, m.topk), -7, dtype=torch.int32, device="cuda")
    seq_pos = torch.tensor([sp for sp, _ in sub.seqs], dtype=torch.int32, device="cuda")
    q_start = torch.tensor(sub.q_start, dtype=torch.int32, device="cuda")
    X.indexer_forward_paged(d, q, w, seq_pos, q_start, m.T_max, table, pool, bt[:3].contiguous().cuda(), top, ws)
    X.indexer_status(ws)
    n = sub.q_start[-1]
    assert torch.equal(top[:n], top_all[:n])
    assert bool((top[n:] == -1).all())
