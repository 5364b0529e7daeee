"""indexer_forward_noalloc: the forward for callers that cannot allocate device memory
when they call the indexer (for instance a plugin whose host runtime owns the whole
device memory pool, or a server whose memory budget is fixed at start-up). It uses the
library's fixed static scratch instead of a caller workspace, and its results must
equal indexer_forward's on consecutive calls, whatever the previous call left in the
scratch.

Collected last on purpose, so that a run stopping at the first failure has already run
every other test.
"""
import dataclasses

import numpy as np
import pytest
import torch

from tests import cases as C
from workloads import WORKLOADS

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    import sparse_attention_top_indexer_gb300 as X
    X.load_library()
    return X


def _reference(X, wl, q, w, table, cache):
    d = C.dims_of(wl)
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda")
    X.indexer_forward(d, q, w, wl.start_pos, table, cache, top, ws, scores_out=sc)
    X.indexer_status(ws)
    return top.cpu().numpy(), sc.cpu().numpy()


@pytest.mark.parametrize("name,over,with_scores", [
    ("decode", dict(B=8), True),          # 8 sequences x 8192 keys, top-2048
    ("decode", dict(B=8), False),         # the scores live in the static scratch only
    ("tiny_prefill", dict(), True),       # 256 rows, 8 heads, including short-context rows
    ("tiny_prefill", dict(), False),
])
def test_noalloc_matches_forward_on_two_calls(X, name, over, with_scores):
    wl = dataclasses.replace(WORKLOADS[name], **over)
    table = C.gpu_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    q, w = wl.q("cuda"), wl.w("cuda")
    ref_top, ref_sc = _reference(X, wl, q, w, table, cache)
    d = C.dims_of(wl)
    for _ in range(2):
        top = torch.full((wl.B, wl.S, wl.topk), 7, dtype=torch.int32, device="cuda")
        sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda") if with_scores else None
        X.indexer_forward_noalloc(d, q, w, wl.start_pos, table, cache, top, scores_out=sc)
        X.indexer_noalloc_status()
        assert np.array_equal(top.cpu().numpy(), ref_top)
        if with_scores:
            got = sc.cpu().numpy()
            assert np.array_equal(np.isneginf(got), np.isneginf(ref_sc))
            fin = np.isfinite(ref_sc)
            assert np.all(np.abs(got[fin] - ref_sc[fin]) <= C.SCORE_ATOL + C.SCORE_RTOL * np.abs(ref_sc[fin]))


def test_noalloc_two_level_decode(X):
    """Level one (candidate blocks out) and level two (the kept blocks' pages only) through the
    static scratch: indices and blocks equal indexer_forward's with a workspace."""
    wl = dataclasses.replace(WORKLOADS["two_level_decode"], B=4)
    d = C.dims_of(wl)
    assert X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos) <= X.NOALLOC_SCRATCH_BYTES
    table = C.gpu_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    q1, w1 = wl.q("cuda", tag="q1"), wl.w("cuda", tag="w1")
    q2, w2 = wl.q("cuda", tag="q2"), wl.w("cuda", tag="w2")
    ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos), dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    shape = (wl.B, wl.S, wl.topk)
    cshape = (wl.B, wl.S, wl.cand_topk_blocks)
    ref1, refc = torch.empty(shape, dtype=torch.int32, device="cuda"), torch.empty(cshape, dtype=torch.int32,
                                                                                 device="cuda")
    ref2 = torch.empty(shape, dtype=torch.int32, device="cuda")
    X.indexer_forward(d, q1, w1, wl.start_pos, table, cache, ref1, ws, cand_out=refc)
    X.indexer_forward(d, q2, w2, wl.start_pos, table, cache, ref2, ws, cand_in=refc)
    X.indexer_status(ws)
    for _ in range(2):
        t1, c1 = torch.full(shape, 7, dtype=torch.int32, device="cuda"), torch.full(cshape, 7, dtype=torch.int32,
                                                                                   device="cuda")
        t2 = torch.full(shape, 7, dtype=torch.int32, device="cuda")
        X.indexer_forward_noalloc(d, q1, w1, wl.start_pos, table, cache, t1, cand_out=c1)
        X.indexer_forward_noalloc(d, q2, w2, wl.start_pos, table, cache, t2, cand_in=c1)
        X.indexer_noalloc_status()
        assert torch.equal(t1, ref1) and torch.equal(c1, refc) and torch.equal(t2, ref2)


def test_noalloc_rejected_call_leaves_the_scratch_alone(X):
    """A call that fails its argument checks enqueues nothing; the status reader still
    reports a clean state afterwards."""
    wl = dataclasses.replace(WORKLOADS["decode"], B=2)
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    q, w = wl.q("cuda"), wl.w("cuda")
    top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    X.indexer_forward_noalloc(d, q, w, wl.start_pos, table, cache, top)
    X.indexer_noalloc_status()
    with pytest.raises(X.IndexerError) as err:       # the table is too short for the query positions
        X.indexer_forward_noalloc(d, q, w, wl.start_pos, table[:100], cache, top)
    assert err.value.code == -4
    X.indexer_noalloc_status()


def test_noalloc_rejects_sizes_beyond_its_scratch(X):
    wl = WORKLOADS["prefill"]       # 8192 x 2048 f32 scores alone need 64 MiB
    d = C.dims_of(wl)
    need = X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos)
    assert need > X.NOALLOC_SCRATCH_BYTES
    q = torch.zeros((wl.B, wl.S, wl.H, wl.D), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((wl.B, wl.S, wl.H), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((wl.max_pos, 32, 2), dtype=torch.float32, device="cuda")
    cache = X.new_key_cache(wl.B, wl.T_cap)
    top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    with pytest.raises(X.IndexerError) as err:
        X.indexer_forward_noalloc(d, q, w, 0, table, cache, top)
    assert err.value.code == -5 and str(need) in str(err.value)
