"""The bounded device waits, exercised without a fault: the several-row score kernel is
launched with its producer role held back (indexer_scores_hold_test), so no query row, key
tile or MMA is ever requested and every other role's mbarrier wait runs out after a short
limit. The kernel must report the timeout through the workspace status word, write no
score, leave nothing in flight, and the same stream must then run an ordinary forward
that matches the oracle.
"""
import dataclasses
import time

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


@pytest.mark.parametrize("fmt", [0, 1])
def test_held_producer_times_out_and_the_stream_recovers(X, fmt):
    wl = dataclasses.replace(WORKLOADS["prefill"], name=f"hold{fmt}", B=1, S=600, topk=64, key_format=fmt)
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    q, w = wl.q("cuda"), wl.w("cuda")
    rows = torch.empty((wl.B, wl.S, wl.H, X.row_bytes(fmt)), dtype=torch.uint8, device="cuda")
    wp = torch.empty((wl.B, wl.S, wl.H), dtype=torch.float32, device="cuda")
    X.indexer_prep_q(d, q, w, wl.start_pos, table, rows, wp)
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    X.indexer_status(ws)                                      # clean before the test
    scores = torch.full((wl.B, wl.S, wl.T), float("nan"), dtype=torch.float32, device="cuda")
    t0 = time.perf_counter()
    X.indexer_scores_hold_test(d, rows, wp, wl.start_pos, cache, scores, ws, wait_ns=2_000_000)
    with pytest.raises(X.IndexerError) as err:
        X.indexer_status(ws)                                  # synchronises; reads and clears the word
    elapsed = time.perf_counter() - t0
    assert err.value.code == -8, err.value
    assert elapsed < 10.0
    assert torch.isnan(scores).all(), "a held kernel wrote scores"
    X.indexer_status(ws)                                      # the word was cleared
    # the same stream and workspace run an ordinary forward that matches the oracle
    top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda")
    X.indexer_forward(d, q, w, wl.start_pos, table, cache, top, ws, scores_out=sc)
    X.indexer_status(ws)
    ref_cache = C.oracle_cache(wl, cos, sin)
    ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, wl.start_pos, wl.ratio, wl.rope_dim,
                                   wl.topk, wl.offset)
    C.assert_scores_close(sc.cpu().numpy(), ref_sc)
    swaps = C.compare_topk(top.cpu().numpy().reshape(-1, wl.topk), ref_top.reshape(-1, wl.topk),
                           ref_sc.reshape(-1, wl.T), wl.offset)
    C.record_swaps(f"after a held kernel fmt {fmt}", swaps, wl.S, int((top >= 0).sum()))
