"""Row-major key rows (the pages' indexer-cache layout: one 68- or 132-byte row per
compressed position) <-> the library's 64-key pages, through the C ABI.

The oracle's rows (pack_row68 / pack_row132 of the oracle's key publish) are the
reference: imported rows must give the pages the GPU publishes itself, exported pages
must give the oracle's rows, both bit for bit, and a forward over an imported cache
must select what a forward over the GPU-published cache selects.
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


@pytest.mark.parametrize("fmt", [0, 1])
def test_rows_pages_round_trip_against_oracle(X, fmt):
    wl = dataclasses.replace(WORKLOADS["prefill"], name=f"layout{fmt}", B=2, S=1000, key_format=fmt)  # T = 250
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    pages = C.gpu_cache(wl, table)                         # GPU publish, [B, T_cap/64, page bytes]
    ref = C.oracle_cache(wl, cos, sin)                     # oracle rows [B, T_cap, row bytes]
    d = C.dims_of(wl)
    rb = X.row_bytes(fmt)
    # pages -> rows: the oracle's rows for the published keys, the rest untouched
    rows = torch.full((wl.B, wl.T_cap, rb), 0xA5, dtype=torch.uint8, device="cuda")
    X.indexer_cache_to_rows(d, pages, rows, n_keys=wl.T)
    got = rows.cpu().numpy()
    assert np.array_equal(got[:, :wl.T], ref[:, :wl.T])
    assert np.all(got[:, wl.T:] == 0xA5)
    # rows -> pages: the oracle's rows give the GPU's published pages
    ref_rows = torch.from_numpy(np.ascontiguousarray(ref)).cuda()
    imported = X.new_key_cache(wl.B, wl.T_cap, key_format=fmt)
    X.indexer_cache_from_rows(d, ref_rows, imported, n_keys=wl.T)
    torch.cuda.synchronize()
    assert torch.equal(imported, pages)


def test_page_pool_round_trip_and_ragged_keys(X):
    """A page pool is n_seq = num_pages sequences of 64 keys; any bytes survive both ways,
    and keys past n_keys of the destination are left as they were."""
    d = X.make_dims(n_heads=64, ratio=4, index_topk=16)
    g = torch.Generator(device="cuda").manual_seed(5)
    pool = torch.randint(0, 256, (37, X.PAGE_BYTES), dtype=torch.uint8, device="cuda", generator=g)
    rows = torch.empty((37, 64, 68), dtype=torch.uint8, device="cuda")
    X.indexer_cache_to_rows(d, pool.view(37, 1, X.PAGE_BYTES), rows)
    back = torch.zeros_like(pool)
    X.indexer_cache_from_rows(d, rows, back.view(37, 1, X.PAGE_BYTES))
    torch.cuda.synchronize()
    assert torch.equal(back, pool)
    # the permutation itself, against the byte formula of the page layout
    ref_rows = C.pages_to_rows(pool.view(37, 1, X.PAGE_BYTES).cpu().numpy())
    assert np.array_equal(rows.cpu().numpy(), ref_rows)
    # ragged: 100 of 128 keys per sequence
    cache = torch.full((3, 2, X.PAGE_BYTES), 0x5A, dtype=torch.uint8, device="cuda")
    src = torch.randint(0, 256, (3, 128, 68), dtype=torch.uint8, device="cuda", generator=g)
    X.indexer_cache_from_rows(d, src, cache, n_keys=100)
    as_rows = C.pages_to_rows(cache.cpu().numpy())
    assert np.array_equal(as_rows[:, :100], src.cpu().numpy()[:, :100])
    assert np.all(as_rows[:, 100:] == 0x5A)


def test_forward_over_imported_rows_selects_the_same(X):
    wl = WORKLOADS["decode"]
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    pages = C.gpu_cache(wl, table)
    ref = C.oracle_cache(wl, cos, sin)
    d = C.dims_of(wl)
    imported = X.new_key_cache(wl.B, wl.T_cap)
    X.indexer_cache_from_rows(d, torch.from_numpy(np.ascontiguousarray(ref)).cuda(), imported, n_keys=wl.T)
    q, w = wl.q("cuda"), wl.w("cuda")
    outs = []
    for cache in (pages, imported):
        ws = torch.empty(X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos), dtype=torch.uint8, device="cuda")
        X.indexer_workspace_init(ws)
        top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
        X.indexer_forward(d, q, w, wl.start_pos, table, cache, top, ws)
        X.indexer_status(ws)
        outs.append(top.cpu())
    assert torch.equal(outs[0], outs[1])
