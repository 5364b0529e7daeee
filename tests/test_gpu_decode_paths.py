"""indexer_forward on decode shapes (one query row per sequence) against the separate
entry points and the oracle.

Its scores and indices must equal, bit for bit, what indexer_prep_q + indexer_scores +
indexer_topk produce on the same inputs, also when the call is repeated on one workspace
and when a prefill call shares the workspace.
"""
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


def _split_path(X, wl, d, q, w, table, cache):
    rows = torch.empty((wl.B, 1, wl.H, 68), dtype=torch.uint8, device="cuda")
    wp = torch.empty((wl.B, 1, wl.H), dtype=torch.float32, device="cuda")
    X.indexer_prep_q(d, q, w, wl.start_pos, table, rows, wp)
    sc = torch.empty((wl.B, 1, wl.T), dtype=torch.float32, device="cuda")
    ws = torch.empty(X.STATUS_BYTES, dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    X.indexer_scores(d, rows, wp, wl.start_pos, cache, sc, ws)
    top = torch.empty((wl.B, 1, wl.topk), dtype=torch.int32, device="cuda")
    X.indexer_topk(d, sc, wl.start_pos, top)
    X.indexer_status(ws)
    return sc, top


def _fused(X, wl, d, q, w, table, cache, ws):
    sc = torch.empty((wl.B, 1, wl.T), dtype=torch.float32, device="cuda")
    top = torch.empty((wl.B, 1, wl.topk), dtype=torch.int32, device="cuda")
    X.indexer_forward(d, q, w, wl.start_pos, table, cache, top, ws, scores_out=sc)
    return sc, top


@pytest.mark.parametrize("name,B,H,start,topk", [
    ("f_dec", 3, 64, 4095, 256),        # 1024 keys, 8 pages per row over several CTAs
    ("f_rag", 5, 8, 1999, 100),          # 500 keys: ragged last page, N padded to 16
    ("f_h16", 2, 16, 511, 64),           # one page
    ("f_h32", 4, 32, 8191, 1023),        # 2048 keys
    ("f_h128", 2, 128, 16383, 2047),     # 4096 keys, one CTA per SM
    ("f_full", 32, 64, 32767, 2048),     # the decode workload's shape
])
def test_fused_equals_split_and_oracle(X, name, B, H, start, topk):
    wl = dataclasses.replace(WORKLOADS["decode"], name=name, B=B, H=H, start_pos=start, topk=topk)
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    q, w = wl.q("cuda"), wl.w("cuda")
    sc_ref, top_ref = _split_path(X, wl, d, q, w, table, cache)
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, 1, wl.start_pos), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    for rep in range(3):
        sc, top = _fused(X, wl, d, q, w, table, cache, ws)
        X.indexer_status(ws)
        assert torch.equal(sc.view(torch.int32), sc_ref.view(torch.int32)), f"rep {rep}: scores differ"
        assert torch.equal(top, top_ref), f"rep {rep}: indices differ"
    if B * wl.T <= 8 * 4096:   # oracle check on the smaller shapes
        cos, sin = C.oracle_table(wl.max_pos)
        ref_cache = C.oracle_cache(wl, cos, sin)
        ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, wl.start_pos, wl.ratio,
                                       wl.rope_dim, wl.topk, wl.offset)
        C.assert_scores_close(sc.cpu().numpy(), ref_sc)
        C.compare_topk(top.cpu().numpy().reshape(-1, wl.topk), ref_top.reshape(-1, wl.topk),
                       ref_sc.reshape(-1, wl.T), wl.offset)


def test_fused_workspace_shared_with_prefill(X):
    """Decode and prefill calls interleaved on one workspace."""
    dec = dataclasses.replace(WORKLOADS["decode"], name="f_share", B=4, start_pos=4095, topk=300)
    pre = dataclasses.replace(WORKLOADS["prefill"], name="f_share_p", B=2, S=600, topk=64)
    dd, dp = C.dims_of(dec), C.dims_of(pre)
    n = max(X.indexer_workspace_size(dd, dec.B, 1, dec.start_pos), X.indexer_workspace_size(dp, pre.B, pre.S, 0))
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    t_dec, t_pre = C.gpu_table(dec.max_pos), C.gpu_table(pre.max_pos)
    c_dec, c_pre = C.gpu_cache(dec, t_dec), C.gpu_cache(pre, t_pre)
    qd, wd = dec.q("cuda"), dec.w("cuda")
    _, top_ref = _split_path(X, dec, dd, qd, wd, t_dec, c_dec)
    for _ in range(2):
        top_p = torch.empty((pre.B, pre.S, pre.topk), dtype=torch.int32, device="cuda")
        X.indexer_forward(dp, pre.q("cuda"), pre.w("cuda"), 0, t_pre, c_pre, top_p, ws)
        _, top = _fused(X, dec, dd, qd, wd, t_dec, c_dec, ws)
        X.indexer_status(ws)
        assert torch.equal(top, top_ref)


@pytest.mark.parametrize("B,start,cbk,cbs,topk", [
    (8, 131071, 64, 64, 2048),   # the two-level workload's shape: 64 blocks of 64 of 32768 keys
    (3, 8191, 20, 48, 300),      # blocks straddling page boundaries
    (2, 4095, 7, 100, 64),       # few kept keys (700) for top-64
    (4, 32767, 16, 128, 2047),   # kept keys (2048) just above k
])
def test_level_two_kept_blocks_only(X, B, start, cbk, cbs, topk):
    """Level two with one query row and no score output scores and ranks only the kept
    blocks' keys; its indices must equal the full-width path's (scores_out given)."""
    wl = dataclasses.replace(WORKLOADS["two_level_decode"], name=f"sp{B}_{cbs}", B=B, start_pos=start, topk=topk,
                             cand_topk_blocks=cbk, cand_block_size=cbs)
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    q, w = wl.q("cuda", tag="q2"), wl.w("cuda", tag="w2")
    nblk = -(-wl.T // cbs)
    rng = np.random.default_rng(B * 1000 + cbs)
    cand = np.full((B, 1, cbk), -1, np.int32)
    for b in range(B):
        n = cbk if b % 2 == 0 else cbk // 2          # some rows padded with -1
        cand[b, 0, :n] = np.sort(rng.choice(nblk, n, replace=False))
    if B > 2:                                         # one row unsorted, with a repeated block
        cand[1, 0, :3] = cand[1, 0, [2, 0, 0]]
    cand_t = torch.from_numpy(cand).cuda()
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, 1, wl.start_pos), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    sc = torch.empty((wl.B, 1, wl.T), dtype=torch.float32, device="cuda")
    top_full = torch.empty((wl.B, 1, wl.topk), dtype=torch.int32, device="cuda")
    X.indexer_forward(d, q, w, wl.start_pos, table, cache, top_full, ws, cand_in=cand_t, scores_out=sc)
    top_kept = torch.empty_like(top_full)
    X.indexer_forward(d, q, w, wl.start_pos, table, cache, top_kept, ws, cand_in=cand_t)
    X.indexer_status(ws)
    assert torch.equal(top_kept, top_full)
    if B * wl.T <= 16384:
        cos, sin = C.oracle_table(wl.max_pos)
        ref_cache = C.oracle_cache(wl, cos, sin)
        ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, wl.start_pos, wl.ratio, wl.rope_dim,
                                       wl.topk, wl.offset, cand_in=cand, cand_block_size=cbs)
        C.compare_topk(top_kept.cpu().numpy().reshape(-1, wl.topk), ref_top.reshape(-1, wl.topk),
                       ref_sc.reshape(-1, wl.T), wl.offset)


@pytest.mark.parametrize("name,B,H,start,fmt", [
    ("fp_dec", 32, 64, 32767, 0),     # decode: publish and query prep in one launch
    ("fp_h16", 5, 16, 4095, 0),
    ("fp_fp8", 8, 64, 8191, 1),
    ("fp_pf", 1, 64, 0, 0),           # prefill: the separate launches
])
def test_forward_publish_equals_separate_calls(X, name, B, H, start, fmt):
    """indexer_forward_publish leaves the same cache, scores and indices as
    indexer_publish_k followed by indexer_forward."""
    base = WORKLOADS["decode"] if start > 0 else WORKLOADS["tiny_prefill"]
    wl = dataclasses.replace(base, name=name, B=B, H=H, start_pos=start, key_format=fmt,
                             topk=min(base.topk, 512))
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    if start > 0:
        cache_a = X.new_key_cache(wl.B, wl.T_cap, key_format=fmt)
        X.indexer_publish_k(d, wl.latent("cuda"), wl.wk("cuda"), wl.k_norm_w("cuda"), table, 0, cache_a)
        lat = wl.decode_latent("cuda")
    else:
        cache_a = X.new_key_cache(wl.B, wl.T_cap, key_format=fmt)
        lat = wl.latent("cuda")
    cache_b = cache_a.clone()
    q, w = wl.q("cuda"), wl.w("cuda")
    outs = []
    for cache, fused in ((cache_a, False), (cache_b, True)):
        ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos), dtype=torch.uint8, device="cuda")
        X.indexer_workspace_init(ws)
        top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
        sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda")
        if fused:
            X.indexer_forward_publish(d, lat, wl.wk("cuda"), wl.k_norm_w("cuda"), q, w, wl.start_pos, table, cache,
                                      top, ws, scores_out=sc)
        else:
            X.indexer_publish_k(d, lat, wl.wk("cuda"), wl.k_norm_w("cuda"), table, wl.start_pos, cache)
            X.indexer_forward(d, q, w, wl.start_pos, table, cache, top, ws, scores_out=sc)
        X.indexer_status(ws)
        outs.append((top, sc))
    assert torch.equal(cache_a, cache_b), "caches differ"
    assert torch.equal(outs[0][1], outs[1][1]), "scores differ"
    assert torch.equal(outs[0][0], outs[1][0]), "indices differ"


@pytest.mark.parametrize("start", [32767, 0])
def test_forward_publish_host_equals_device(X, start):
    """indexer_forward_publish_host (inputs and indices in pinned host memory, copied by the
    call on its stream) leaves the same cache and indices as indexer_forward_publish."""
    base = WORKLOADS["decode"] if start > 0 else WORKLOADS["tiny_prefill"]
    wl = dataclasses.replace(base, name=f"fph{start}", B=6 if start > 0 else 2, topk=min(base.topk, 512))
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cache_a = X.new_key_cache(wl.B, wl.T_cap)
    if start > 0:
        X.indexer_publish_k(d, wl.latent("cuda"), wl.wk("cuda"), wl.k_norm_w("cuda"), table, 0, cache_a)
        lat = wl.decode_latent("cuda")
    else:
        lat = wl.latent("cuda")
    cache_b = cache_a.clone()
    q, w = wl.q("cuda"), wl.w("cuda")
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    X.indexer_forward_publish(d, lat, wl.wk("cuda"), wl.k_norm_w("cuda"), q, w, wl.start_pos, table, cache_a, top, ws)
    X.indexer_status(ws)
    n = X.indexer_workspace_size_host(d, wl.B, wl.S, wl.start_pos, lat.shape[1], lat.shape[2])
    assert n > ws.numel()
    ws_h = torch.empty(n, dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws_h)
    top_h = torch.full((wl.B, wl.S, wl.topk), -7, dtype=torch.int32).pin_memory()
    X.indexer_forward_publish_host(d, lat.cpu().pin_memory(), wl.wk("cuda"), wl.k_norm_w("cuda"), q.cpu().pin_memory(),
                                   w.cpu().pin_memory(), wl.start_pos, table, cache_b, top_h, ws_h)
    torch.cuda.synchronize()
    X.indexer_status(ws_h)
    assert torch.equal(cache_a, cache_b), "caches differ"
    assert torch.equal(top.cpu(), top_h), "indices differ"
    # a token that completes no group (G == 0): the forward alone, on the published cache
    wl0 = dataclasses.replace(wl, start_pos=wl.start_pos + 1) if start > 0 else None
    if wl0 is not None:
        d0 = C.dims_of(wl0)
        table0 = C.gpu_table(wl0.max_pos)   # one more position than the publishing step's
        ws0 = torch.empty(X.indexer_workspace_size(d0, wl0.B, wl0.S, wl0.start_pos), dtype=torch.uint8,
                          device="cuda")
        X.indexer_workspace_init(ws0)
        top0 = torch.empty_like(top)
        X.indexer_forward(d0, q, w, wl0.start_pos, table0, cache_a, top0, ws0)
        X.indexer_status(ws0)
        n0 = X.indexer_workspace_size_host(d0, wl0.B, wl0.S, wl0.start_pos, 0, lat.shape[2])
        ws0h = torch.empty(n0, dtype=torch.uint8, device="cuda")
        X.indexer_workspace_init(ws0h)
        top0h = torch.full_like(top_h, -7).pin_memory()
        X.indexer_forward_publish_host(d0, torch.empty((wl.B, 0, lat.shape[2]), dtype=torch.bfloat16),
                                       wl.wk("cuda"), wl.k_norm_w("cuda"), q.cpu().pin_memory(), w.cpu().pin_memory(),
                                       wl0.start_pos, table0, cache_b, top0h, ws0h)
        torch.cuda.synchronize()
        X.indexer_status(ws0h)
        assert torch.equal(top0.cpu(), top0h), "indices differ without a key to publish"
    with pytest.raises(X.IndexerError) as e:   # the workspace must hold the staging too
        X.indexer_forward_publish_host(d, lat.cpu().pin_memory(), wl.wk("cuda"), wl.k_norm_w("cuda"),
                                       q.cpu().pin_memory(), w.cpu().pin_memory(), wl.start_pos, table, cache_b, top_h,
                                       ws)
    assert e.value.code == -5
