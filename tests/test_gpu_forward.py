"""indexer_forward on the five workloads, through the C ABI, against the oracle.

Decode workloads are compared on every row; the two large prefills on sampled
rows (the oracle recomputes just those rows from the same seeded inputs), and on
properties that hold at any size for every row.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from tests import cases as C
from workloads import WORKLOADS, Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    import sparse_attention_top_indexer_gb300 as X
    X.load_library()
    return X


def _run_forward(X, wl: Workload, q, w, table, cache, cand_in=None, want_cand=False, want_scores=True,
                 dims=None):
    d = dims or C.dims_of(wl)
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda") if want_scores else None
    cand = torch.empty((wl.B, wl.S, wl.cand_topk_blocks), dtype=torch.int32, device="cuda") if want_cand else None
    X.indexer_forward(d, q, w, wl.start_pos, table, cache, top, ws, cand_in=cand_in, cand_out=cand, scores_out=sc)
    X.indexer_status(ws)
    return top, cand, sc


def _check_properties(top: np.ndarray, wl: Workload):
    vis = O.visible_lens(wl.start_pos, wl.S, wl.ratio)
    k_eff = min(wl.topk, wl.T)
    t = top.reshape(wl.B, wl.S, wl.topk)
    nvalid = (t >= 0).sum(-1)
    assert np.array_equal(nvalid, np.broadcast_to(np.minimum(vis, k_eff), (wl.B, wl.S)))
    nxt, cur = t[..., 1:], t[..., :-1]
    assert np.all((nxt < 0) | (nxt > cur)), "valid indices not strictly ascending"
    assert np.all((nxt < 0) | (cur >= 0)), "-1 padding not trailing"
    assert np.all((t < 0) | ((t >= wl.offset) & (t < wl.offset + vis[None, :, None])))


@pytest.mark.parametrize("name", ["tiny_prefill", "decode"])
def test_forward_full_compare(X, name):
    wl = WORKLOADS[name]
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    ref_cache = C.oracle_cache(wl, cos, sin)
    assert np.array_equal(C.pages_to_rows(cache), ref_cache)
    q, w = wl.q("cuda"), wl.w("cuda")
    top, _, sc = _run_forward(X, wl, q, w, table, cache)
    ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, wl.start_pos, wl.ratio, wl.rope_dim,
                                   wl.topk, wl.offset)
    C.assert_scores_close(sc.cpu().numpy(), ref_sc)
    swaps = C.compare_topk(top.cpu().numpy().reshape(-1, wl.topk), ref_top.reshape(-1, wl.topk),
                           ref_sc.reshape(-1, wl.T), wl.offset)
    _check_properties(top.cpu().numpy(), wl)
    C.record_swaps(f"forward/{name}", swaps, wl.B * wl.S, int((top >= 0).sum()))


def test_forward_two_level_decode(X):
    wl = WORKLOADS["two_level_decode"]
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    ref_cache = C.oracle_cache(wl, cos, sin)
    assert np.array_equal(C.pages_to_rows(cache), ref_cache)
    # level one: the candidate source layer (its own q, w) publishes its blocks and its top-k
    q1, w1 = wl.q("cuda", tag="q1"), wl.w("cuda", tag="w1")
    top1, cand, sc1 = _run_forward(X, wl, q1, w1, table, cache, want_cand=True)
    ref_top1, ref_cand, ref_sc1 = O.forward(C.bits(q1), C.bits(w1), ref_cache, cos, sin, wl.start_pos, wl.ratio,
                                            wl.rope_dim, wl.topk, wl.offset, cand_topk_blocks=wl.cand_topk_blocks,
                                            cand_block_size=wl.cand_block_size, want_candidates=True)
    C.assert_scores_close(sc1.cpu().numpy(), ref_sc1)
    C.compare_topk(top1.cpu().numpy().reshape(-1, wl.topk), ref_top1.reshape(-1, wl.topk),
                   ref_sc1.reshape(-1, wl.T), wl.offset)
    got_cand = cand.cpu().numpy()
    if not np.array_equal(got_cand, ref_cand):
        # a block may swap only where its max score ties the 64th block's within tolerance
        for r in range(wl.B):
            g, o = set(got_cand[r, 0]), set(ref_cand[r, 0])
            blk_max = np.array([ref_sc1[r, 0, j * 64:(j + 1) * 64].max() for j in range(wl.T // 64)])
            kth = np.sort(blk_max)[::-1][wl.cand_topk_blocks - 1]
            for j in g ^ o:
                assert abs(blk_max[j] - kth) <= C.SCORE_ATOL + C.SCORE_RTOL * abs(kth)
    # level two: a consumer with independent q, w, restricted to the oracle's kept blocks
    q2, w2 = wl.q("cuda", tag="q2"), wl.w("cuda", tag="w2")
    cand_t = torch.from_numpy(ref_cand).cuda()
    top2, _, sc2 = _run_forward(X, wl, q2, w2, table, cache, cand_in=cand_t)
    ref_top2, _, ref_sc2 = O.forward(C.bits(q2), C.bits(w2), ref_cache, cos, sin, wl.start_pos, wl.ratio,
                                     wl.rope_dim, wl.topk, wl.offset, cand_in=ref_cand,
                                     cand_block_size=wl.cand_block_size)
    swaps = C.compare_topk(top2.cpu().numpy().reshape(-1, wl.topk), ref_top2.reshape(-1, wl.topk),
                           ref_sc2.reshape(-1, wl.T), wl.offset)
    # every emitted position lies in a kept block
    keep = O.candidate_mask(ref_cand.reshape(wl.B, -1), wl.T, wl.cand_block_size)
    t2 = top2.cpu().numpy().reshape(wl.B, -1)
    for r in range(wl.B):
        v = t2[r][t2[r] >= 0]
        assert len(v) == wl.topk and np.all(keep[r, v])
    C.record_swaps("forward/two_level_decode level two", swaps, wl.B * wl.S, int((top2 >= 0).sum()))


def _sample_rows(wl: Workload, n_rand: int, seed: int):
    rng = np.random.default_rng(seed)
    fixed = [0, 1, 2, 3, 4, 63, 64, wl.topk * wl.ratio - 2, wl.topk * wl.ratio - 1, wl.topk * wl.ratio,
             wl.S // 2, wl.S - 2, wl.S - 1]
    rows = sorted(set([r for r in fixed if 0 <= r < wl.S] + list(rng.integers(0, wl.S, n_rand))))
    return rows


# prefill_t4096: 16384 rows over 4096 keys, the many-rows top-k with 16 keys per thread.
# h8_t8192 / h32_t6144: 16 and 4 query rows per score tile over long rows (groups of up to
# 64 tiles): slow epilogues that let an MMA warp run rounds ahead of an accumulator's
# releases (each accumulator's release barrier is per MMA warp, so no parity wait is ambiguous)
_SAMPLED = {"prefill": WORKLOADS["prefill"], "large_prefill": WORKLOADS["large_prefill"],
            "prefill_t4096": dataclasses.replace(WORKLOADS["prefill"], name="prefill_t4096", S=16384, topk=1024),
            "h8_t8192": dataclasses.replace(WORKLOADS["large_prefill"], name="h8_t8192", B=1, H=8),
            "h32_t6144": dataclasses.replace(WORKLOADS["large_prefill"], name="h32_t6144", B=1, S=24576, H=32)}


@pytest.mark.parametrize("name,n_rand", [("prefill", 40), ("large_prefill", 24), ("prefill_t4096", 24),
                                         ("h8_t8192", 16), ("h32_t6144", 16)])
def test_forward_prefill_sampled(X, name, n_rand):
    wl = _SAMPLED[name]
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    ref_cache = C.oracle_cache(wl, cos, sin)
    assert np.array_equal(C.pages_to_rows(cache), ref_cache)
    q, w = wl.q("cuda"), wl.w("cuda")
    top, _, sc = _run_forward(X, wl, q, w, table, cache)
    top_np = top.cpu().numpy()
    _check_properties(top_np, wl)
    w_cpu = w.cpu()
    rows = _sample_rows(wl, n_rand, 11)
    total_swaps = 0
    for b in range(wl.B):
        flat = [b * wl.S + s for s in rows]
        q_sub = wl.q_rows(flat).unsqueeze(0)                      # [1, R, H, D]
        w_sub = w_cpu[b, rows].unsqueeze(0)
        pos = np.array(rows) + wl.start_pos
        q_rows_o, w_o, _ = O.prep_queries(C.bits(q_sub), C.bits(w_sub), cos, sin, wl.start_pos, wl.rope_dim, wl.H,
                                          row_positions=pos)
        vis = O.visible_lens(wl.start_pos, len(rows), wl.ratio, row_positions=pos)
        ref_sc = O.index_scores(q_rows_o, w_o, ref_cache[b:b + 1], wl.T, vis)[0]
        ref_top = O.topk_positions(ref_sc, vis, wl.topk, wl.offset, wl.T)
        if sc is not None:
            C.assert_scores_close(sc[b, rows].cpu().numpy(), ref_sc)
        total_swaps += C.compare_topk(top_np[b, rows], ref_top, ref_sc, wl.offset)
    C.record_swaps(f"forward/{name} sampled rows", total_swaps, wl.B * len(rows),
                   int((top_np[:, rows] >= 0).sum()))


# ----------------------------------------------------------------------------- edge cases
@pytest.mark.parametrize("S,start,topk", [(3, 0, 8), (1, 2, 8), (9, 0, 64), (130, 0, 4)])
def test_forward_edges(X, S, start, topk):
    """S < ratio (no visible key), decode before the first group, topk > T, ragged T."""
    wl = dataclasses.replace(WORKLOADS["prefill"], name=f"edge{S}_{start}", B=2, S=S, start_pos=start, topk=topk,
                             H=32)
    table = C.gpu_table(max(wl.max_pos, 8))
    cos, sin = C.oracle_table(max(wl.max_pos, 8))
    T_cap = max(128, wl.T_cap)
    cache = X.new_key_cache(wl.B, T_cap)
    ref_cache = np.zeros((wl.B, T_cap, 68), np.uint8)
    if wl.T > 0:
        cache = C.gpu_cache(wl, table)
        ref_cache = C.oracle_cache(wl, cos, sin)
    q, w = wl.q("cuda"), wl.w("cuda")
    top, _, sc = _run_forward(X, wl, q, w, table, cache, want_scores=wl.T > 0)
    ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, wl.start_pos, wl.ratio, wl.rope_dim,
                                   wl.topk, wl.offset)
    if wl.T > 0:
        C.assert_scores_close(sc.cpu().numpy(), ref_sc)
        C.compare_topk(top.cpu().numpy().reshape(-1, topk), ref_top.reshape(-1, topk), ref_sc.reshape(-1, wl.T), 0)
    else:
        assert np.all(top.cpu().numpy() == -1)
    _check_properties(top.cpu().numpy(), wl)


def test_short_context_rows_exact(X):
    """Rows with vis <= k_eff are [0 .. vis) + offset then -1, whatever the scores."""
    wl = dataclasses.replace(WORKLOADS["large_prefill"], name="short", B=1, S=600, topk=128)
    table = C.gpu_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    top, _, _ = _run_forward(X, wl, wl.q("cuda"), wl.w("cuda"), table, cache, want_scores=False)
    top = top.cpu().numpy()[0]
    vis = O.visible_lens(0, wl.S, wl.ratio)
    for s in range(wl.S):
        if vis[s] <= 128:
            want = [i + wl.offset for i in range(vis[s])] + [-1] * (128 - vis[s])
            assert list(top[s]) == want


@pytest.mark.parametrize("ratio,S,start,H,fmt,topk", [
    (1, 96, 0, 64, 0, 32),        # no compression
    (2, 200, 0, 16, 0, 40),       # ratio 2 prefill
    (4, 300, 1000, 64, 0, 128),   # chunked prefill: 300 rows at start_pos 1000
    (1, 1, 511, 32, 0, 64),       # ratio 1 decode (every token completes a group)
    (2, 64, 640, 128, 1, 100),    # FP8, ratio 2, 128 heads, a chunk at start_pos 640
])
def test_forward_ratios_and_chunks(X, ratio, S, start, H, fmt, topk):
    """Compression ratios 1 and 2 and chunked prefill (start_pos > 0, S > 1) against the
    oracle on every row."""
    wl = dataclasses.replace(WORKLOADS["prefill"], name=f"r{ratio}_{S}_{start}_{fmt}", B=2, S=S, start_pos=start,
                             ratio=ratio, H=H, topk=topk, key_format=fmt)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    ref_cache = C.oracle_cache(wl, cos, sin)
    assert np.array_equal(C.any_pages_to_rows(cache), ref_cache)
    q, w = wl.q("cuda"), wl.w("cuda")
    top, _, sc = _run_forward(X, wl, q, w, table, cache)
    ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, wl.start_pos, wl.ratio, wl.rope_dim,
                                   wl.topk, wl.offset)
    C.assert_scores_close(sc.cpu().numpy(), ref_sc)
    swaps = C.compare_topk(top.cpu().numpy().reshape(-1, topk), ref_top.reshape(-1, topk), ref_sc.reshape(-1, wl.T),
                           wl.offset)
    _check_properties(top.cpu().numpy(), wl)
    C.record_swaps(f"forward/ratio {ratio} S{S} start {start} fmt {fmt}", swaps, wl.B * wl.S, int((top >= 0).sum()))
