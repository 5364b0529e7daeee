"""Head-parallel scoring on one GPU: the index heads split into `world` shards, each
shard's partial scores from the library (indexer_prep_q with n_heads_total, then
indexer_scores), summed the way the ranks' all-reduce would sum them, then indexer_topk.
The sum must match the full-head scores of the same kernels within f32 rounding, the
oracle within the score tolerance, and the selection the oracle's up to boundary swaps.
Only the exchange itself (an NCCL all-reduce between GPUs) is not run here: one GPU."""
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


@pytest.mark.parametrize("name,over,world", [
    ("prefill", dict(S=700, topk=128), 2),             # several-row kernel, 32 heads per shard
    ("prefill", dict(S=300, topk=64), 8),              # 8 heads per shard
    ("decode", dict(B=6), 4),                          # single-row kernel, 16 heads per shard
    ("two_level_decode", dict(B=2), 2),                # level two: the kept blocks' mask in each shard
])
def test_shards_sum_to_the_full_scores(X, name, over, world):
    from sparse_attention_top_indexer_gb300.head_parallel import forward_head_parallel, head_range, shard_dims
    wl = dataclasses.replace(WORKLOADS[name], **over)
    d = C.dims_of(wl)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    q, w = wl.q("cuda"), wl.w("cuda")
    ws = torch.empty(max(X.STATUS_BYTES, X.indexer_workspace_size(d, wl.B, wl.S, wl.start_pos)), dtype=torch.uint8,
                     device="cuda")
    X.indexer_workspace_init(ws)
    ref_cache = C.oracle_cache(wl, cos, sin)
    cand = None
    if wl.two_level:   # the level-one blocks from the oracle's own level-one scores
        _, ref_cand, _ = O.forward(C.bits(wl.q(tag="q1")), C.bits(wl.w(tag="w1")), ref_cache, cos, sin,
                                   wl.start_pos, wl.ratio, wl.rope_dim, wl.topk, wl.offset,
                                   cand_topk_blocks=wl.cand_topk_blocks, cand_block_size=wl.cand_block_size,
                                   want_candidates=True)
        cand = torch.from_numpy(ref_cand).cuda()
    # every shard's partial scores, summed as the all-reduce would
    parts = []
    for r in range(world):
        h0, h1 = head_range(wl.H, world, r)
        sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda")
        top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
        parts.append(sc)
        forward_head_parallel(d, q[:, :, h0:h1].contiguous(), w[:, :, h0:h1].contiguous(), wl.start_pos, table,
                              cache, top, ws, sc, world, cand_in=cand, all_reduce=lambda t: None)
    total = torch.stack(parts).sum(0)
    top = torch.empty((wl.B, wl.S, wl.topk), dtype=torch.int32, device="cuda")
    X.indexer_topk(d, total, wl.start_pos, top)
    X.indexer_status(ws)
    # the full-head kernels on the same inputs
    rows = torch.empty((wl.B, wl.S, wl.H, 68), dtype=torch.uint8, device="cuda")
    wp = torch.empty((wl.B, wl.S, wl.H), dtype=torch.float32, device="cuda")
    X.indexer_prep_q(d, q, w, wl.start_pos, table, rows, wp)
    full = torch.empty_like(total)
    X.indexer_scores(d, rows, wp, wl.start_pos, cache, full, ws, cand_blocks=cand)
    X.indexer_status(ws)
    a, b = total.cpu().numpy(), full.cpu().numpy()
    assert np.array_equal(np.isneginf(a), np.isneginf(b))
    fin = np.isfinite(b)
    # f32 sums in another order: the shards' partials are O(1) and may cancel, so the bound is
    # on the size of the terms, not of the total
    assert np.all(np.abs(a[fin] - b[fin]) <= 4e-6 + 1e-5 * np.abs(b[fin]))
    # the oracle
    ref_top, _, ref_sc = O.forward(C.bits(q), C.bits(w), ref_cache, cos, sin, wl.start_pos, wl.ratio, wl.rope_dim,
                                   wl.topk, wl.offset, cand_in=None if cand is None else ref_cand,
                                   cand_block_size=wl.cand_block_size)
    C.assert_scores_close(a, ref_sc)
    swaps = C.compare_topk(top.cpu().numpy().reshape(-1, wl.topk), ref_top.reshape(-1, wl.topk),
                           ref_sc.reshape(-1, wl.T), wl.offset)
    C.record_swaps(f"head-parallel/{name} world {world}", swaps, wl.B * wl.S, int((top >= 0).sum()))
    sd = shard_dims(d, world)
    assert (sd.n_heads, sd.n_heads_total) == (wl.H // world, wl.H)


def test_shard_weight_factor_is_the_models(X):
    """A shard's w' uses the model's head count: w * (128 * n_heads_total)^-0.5."""
    wl = dataclasses.replace(WORKLOADS["prefill"], name="hp_w", S=3, H=64)
    table = C.gpu_table(wl.max_pos)
    w = wl.w("cuda")[:, :, :16].contiguous()
    q = wl.q("cuda")[:, :, :16].contiguous()
    d = X.make_dims(n_heads=16, ratio=4, index_topk=8, n_heads_total=64)
    rows = torch.empty((1, 3, 16, 68), dtype=torch.uint8, device="cuda")
    wp = torch.empty((1, 3, 16), dtype=torch.float32, device="cuda")
    X.indexer_prep_q(d, q, w, 0, table, rows, wp)
    want = w.float() * 0.011048543456039806
    assert torch.allclose(wp, want, rtol=2e-7, atol=0)
