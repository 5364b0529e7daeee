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


@pytest.mark.parametrize("name,over", [
    ("decode", dict(B=8)),          # 8 sequences x 8192 keys, top-2048
    ("tiny_prefill", dict()),       # 256 rows, 8 heads, including short-context rows
])
def test_noalloc_matches_forward_on_two_calls(X, name, over):
    wl = dataclasses.replace(WORKLOADS[name], **over)
    table = C.gpu_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    q, w = wl.q("cuda"), wl.w("cuda")
    ref_top, ref_sc = _reference(X, wl, q, w, table, cache)
    d = C.dims_of(wl)
    for _ in range(2):
        top = torch.full((wl.B, wl.S, wl.topk), 7, dtype=torch.int32, device="cuda")
        sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda")
        X.indexer_forward_noalloc(d, q, w, wl.start_pos, table, cache, top, scores_out=sc)
        torch.cuda.synchronize()
        assert np.array_equal(top.cpu().numpy(), ref_top)
        got = sc.cpu().numpy()
        assert np.array_equal(np.isneginf(got), np.isneginf(ref_sc))
        fin = np.isfinite(ref_sc)
        assert np.all(np.abs(got[fin] - ref_sc[fin]) <= C.SCORE_ATOL + C.SCORE_RTOL * np.abs(ref_sc[fin]))


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
