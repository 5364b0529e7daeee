"""GPU parity: every step of the CUDA path against the CPU oracle, through the C ABI.

Sizes span several 128-key tiles and ragged tails; the full workloads are covered
element by element where the oracle is fast enough and on sampled rows otherwise.
"""
import dataclasses

import numpy as np
import pytest
import torch

import oracle as O
from tests import cases as C
from workloads import WORKLOADS, Workload, normal_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def X():
    import sparse_attention_top_indexer_gb300 as X
    X.load_library()
    return X


def _ws(X, dims, B, S, start_pos):
    n = max(X.indexer_workspace_size(dims, B, S, start_pos), X.STATUS_BYTES)
    ws = torch.empty(n, dtype=torch.uint8, device="cuda")
    X.indexer_workspace_init(ws)
    return ws


# ----------------------------------------------------------------------------- RoPE table
@pytest.mark.parametrize("max_pos", [1, 300, 131072])
def test_rope_table_bit_exact(X, max_pos):
    cos, sin = C.oracle_table(max_pos)
    t = C.gpu_table(max_pos).cpu().numpy()
    assert np.array_equal(t[..., 0].view(np.uint32), cos.view(np.uint32))
    assert np.array_equal(t[..., 1].view(np.uint32), sin.view(np.uint32))


# ----------------------------------------------------------------------------- key publish
@pytest.mark.parametrize("B,G", [(1, 64), (3, 517)])
def test_publish_prefill_bit_exact(X, B, G):
    wl = dataclasses.replace(WORKLOADS["tiny_prefill"], name=f"pub{B}x{G}", B=B, S=G * 4)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    got = C.pages_to_rows(C.gpu_cache(wl, table))
    ref = C.oracle_cache(wl, cos, sin)
    assert np.array_equal(got, ref), f"{np.sum(np.any(got != ref, axis=-1))} rows differ"


def test_publish_decode_slot(X):
    wl = dataclasses.replace(WORKLOADS["decode"], B=2, name="pubdec")
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = X.new_key_cache(wl.B, wl.T_cap)
    lat = wl.decode_latent("cuda")
    X.indexer_publish_k(C.dims_of(wl), lat, wl.wk("cuda"), wl.k_norm_w("cuda"), table, wl.start_pos, cache)
    got = C.pages_to_rows(cache)
    slots, rows, _ = O.publish_keys(C.bits(lat), C.bits(wl.wk()), C.bits(wl.k_norm_w()), cos, sin, wl.start_pos,
                                    wl.ratio, wl.rope_dim, wl.norm_eps)
    assert list(slots) == [8191]
    assert np.array_equal(got[:, 8191], rows[:, 0])
    assert not got[:, :8191].any()


# RMSNorm over the ranges of k_pre: keys far outside the f32 route's range (2^70 and 2^-60
# latents take the f64 evaluation), all-zero keys, magnitudes 2^32 apart inside one key
# (wk rows scaled 2^(o/4 - 16)), zero and negative norm weights; the cluster path (40
# decode keys), four threads per output (200 keys) and one (600 keys).
@pytest.mark.parametrize("B,G,start", [(40, 1, 32767), (1, 200, 0), (1, 600, 0)])
@pytest.mark.parametrize("fmt", ["mxfp4", "fp8"])
def test_publish_norm_ranges(X, B, G, start, fmt):
    wl = dataclasses.replace(WORKLOADS["decode"], name="pubnorm", key_format=1 if fmt == "fp8" else 0)
    D, n = wl.D, B * G
    g = torch.Generator().manual_seed(4242 + G)
    key_scale = torch.tensor([1.0, 2.0 ** 70, 2.0 ** -60, 0.0, 2.0 ** 20, 2.0 ** -30, 1e-3])[torch.arange(n) % 7]
    lat = (torch.randn(n, D, generator=g) * key_scale[:, None]).to(torch.bfloat16).reshape(B, G, D)
    row_scale = 2.0 ** (torch.arange(128, dtype=torch.float32) / 4.0 - 16.0)
    wk = (torch.randn(128, D, generator=g) * row_scale[:, None]).to(torch.bfloat16)
    knorm = torch.randn(128, generator=g).to(torch.bfloat16)
    knorm[::7] = 0
    T_cap = wl.T_cap if start else (G + 63) // 64 * 64
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = X.new_key_cache(B, T_cap, key_format=wl.key_format)
    X.indexer_publish_k(C.dims_of(wl), lat.cuda(), wk.cuda(), knorm.cuda(), table, start, cache)
    slots, rows, _ = O.publish_keys(C.bits(lat), C.bits(wk), C.bits(knorm), cos, sin, start, wl.ratio, wl.rope_dim,
                                    wl.norm_eps, fmt=fmt)
    got = C.any_pages_to_rows(cache)[:, slots]
    assert np.array_equal(got, rows), f"{np.sum(np.any(got != rows, axis=-1))} of {n} keys differ"


# ----------------------------------------------------------------------------- query prep
# qf: 80040 vectors, the bulk-copy kernel (above 16384 vectors; 64 vectors per CTA) with a
# ragged last batch of 40
@pytest.mark.parametrize("name,B,S,H,start", [("qa", 2, 37, 64, 0), ("qb", 1, 256, 8, 0), ("qc", 32, 1, 64, 32767),
                                              ("qd", 3, 5, 16, 1000), ("qe", 2, 9, 128, 7), ("qf", 5, 2001, 8, 3)])
def test_prep_q_bit_exact(X, name, B, S, H, start):
    wl = dataclasses.replace(WORKLOADS["prefill"], name=name, B=B, S=S, H=H, start_pos=start)
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    q, w = wl.q("cuda"), wl.w("cuda")
    rows = torch.empty((B, S, H, 68), dtype=torch.uint8, device="cuda")
    wp = torch.empty((B, S, H), dtype=torch.float32, device="cuda")
    X.indexer_prep_q(C.dims_of(wl), q, w, start, table, rows, wp)
    ref_rows, ref_w, _ = O.prep_queries(C.bits(q), C.bits(w), cos, sin, start, 64, H)
    got = rows.cpu().numpy()
    assert np.array_equal(got, ref_rows), f"{np.sum(np.any(got != ref_rows, axis=-1))} query rows differ"
    assert np.allclose(wp.cpu().numpy(), ref_w, rtol=2e-7, atol=0)


def test_prep_q_rope_dim_32(X):
    wl = dataclasses.replace(WORKLOADS["prefill"], name="rd32", B=1, S=11, H=32, rope_dim=32)
    table = C.gpu_table(wl.max_pos, 32)
    cos, sin = C.oracle_table(wl.max_pos, 32)
    q, w = wl.q("cuda"), wl.w("cuda")
    rows = torch.empty((1, 11, 32, 68), dtype=torch.uint8, device="cuda")
    wp = torch.empty((1, 11, 32), dtype=torch.float32, device="cuda")
    X.indexer_prep_q(C.dims_of(wl), q, w, 0, table, rows, wp)
    ref_rows, _, _ = O.prep_queries(C.bits(q), C.bits(w), cos, sin, 0, 32, 32)
    assert np.array_equal(rows.cpu().numpy(), ref_rows)


# ----------------------------------------------------------------------------- scores
def _scores_case(X, wl: Workload, cand=None):
    table = C.gpu_table(wl.max_pos)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.gpu_cache(wl, table)
    ref_cache = C.oracle_cache(wl, cos, sin)
    assert np.array_equal(C.pages_to_rows(cache), ref_cache)
    q, w = wl.q("cuda"), wl.w("cuda")
    d = C.dims_of(wl)
    rows = torch.empty((wl.B, wl.S, wl.H, 68), dtype=torch.uint8, device="cuda")
    wp = torch.empty((wl.B, wl.S, wl.H), dtype=torch.float32, device="cuda")
    X.indexer_prep_q(d, q, w, wl.start_pos, table, rows, wp)
    sc = torch.empty((wl.B, wl.S, wl.T), dtype=torch.float32, device="cuda")
    ws = _ws(X, d, wl.B, wl.S, wl.start_pos)
    X.indexer_scores(d, rows, wp, wl.start_pos, cache, sc, ws, cand_blocks=cand)
    X.indexer_status(ws)
    ref_rows, ref_w, _ = O.prep_queries(C.bits(q), C.bits(w), cos, sin, wl.start_pos, wl.rope_dim, wl.H)
    vis = O.visible_lens(wl.start_pos, wl.S, wl.ratio)
    ref = O.index_scores(ref_rows, ref_w, ref_cache, wl.T, vis)
    if cand is not None:
        keep = O.candidate_mask(cand.cpu().numpy().reshape(wl.B * wl.S, -1), wl.T, wl.cand_block_size)
        ref = np.where(keep.reshape(ref.shape), ref, -np.inf)
    return sc.cpu().numpy(), ref


@pytest.mark.parametrize("name,B,S,H,start,T_extra", [
    ("s_tiny", 1, 256, 8, 0, 0),          # the tiny prefill: QG = 32 rows x 8 heads per tile
    ("s_rag", 2, 300, 64, 0, 0),          # 75 keys: one ragged tile, 4-row groups, ragged group
    ("s_h16", 1, 1030, 16, 0, 0),         # 257 keys: three tiles, last with a single key
    ("s_h32", 1, 64, 32, 0, 0),
    ("s_h128", 1, 520, 128, 0, 0),
    ("s_dec", 3, 1, 64, 4095, 0),         # decode, 1024 keys split over CTAs
    ("s_dec8", 2, 1, 8, 2047, 0),         # decode with N padded to 16
    ("s_chunk", 2, 7, 64, 1021, 0),       # chunked prefill: start_pos > 0, S > 1
])
def test_scores_parity(X, name, B, S, H, start, T_extra):
    wl = dataclasses.replace(WORKLOADS["prefill"], name=name, B=B, S=S, H=H, start_pos=start)
    got, ref = _scores_case(X, wl)
    C.assert_scores_close(got, ref)


def test_scores_candidate_mask(X):
    wl = dataclasses.replace(WORKLOADS["two_level_decode"], name="s_cand", B=2, start_pos=8191,
                             cand_topk_blocks=5, cand_block_size=64)
    rng = np.random.default_rng(7)
    nblk = -(-wl.T // 64)
    cand = np.full((2, 1, 5), -1, np.int32)
    for b in range(2):
        cand[b, 0, :4] = np.sort(rng.choice(nblk, 4, replace=False))
    got, ref = _scores_case(X, wl, cand=torch.from_numpy(cand).cuda())
    C.assert_scores_close(got, ref)


# ----------------------------------------------------------------------------- selection kernels
def _synthetic_scores(seed, R, T, ties=False):
    g = normal_bf16(seed, "syn_scores", (R, T)).float()
    if ties:
        g = torch.round(g * 2) / 2        # many exact ties
    return g


@pytest.mark.parametrize("S,start,T_over,topk,offset,ties", [
    (1, 8191, None, 2048, 0, False), (1, 8191, None, 2048, 0, True), (300, 0, None, 16, 5, True),
    (5, 131067, None, 2048, 0, False), (64, 0, None, 100, 8192, False), (3, 10, None, 1, 0, True),
])
def test_topk_kernel_bit_exact(X, S, start, T_over, topk, offset, ties):
    B, ratio = 2, 4
    T = (start + S) // ratio
    sc = _synthetic_scores(S * 7 + start, B * S, T, ties).view(B, S, T)
    vis = O.visible_lens(start, S, ratio)
    for s in range(S):
        sc[:, s, vis[s]:] = float("-inf")
    d = X.make_dims(n_heads=64, ratio=ratio, index_topk=topk, offset=offset)
    out = torch.empty((B, S, topk), dtype=torch.int32, device="cuda")
    X.indexer_topk(d, sc.cuda(), start, out)
    ref = O.topk_positions(sc.double().numpy().reshape(B * S, T), np.tile(vis, B), topk, offset, T)
    assert np.array_equal(out.cpu().numpy().reshape(B * S, topk), ref)


# Many rows (prefill): the register-capped 256-thread builds with 8, 16 and 32 keys a thread
# (rows of 2048, 2524 / 3025 and 8192 keys; 3025 is not a multiple of four floats, so its rows
# take the scalar loads), short-context and selected rows mixed, ties.
@pytest.mark.parametrize("B,S,start,topk,offset,ties", [
    (2, 2560, 30208, 2048, 8192, False),   # T 8192, every row selected
    (2, 4096, 6000, 2048, 0, True),        # T 2524: about half the rows take the short fill
    (1, 8192, 0, 512, 0, False),           # T 2048, the 2048-key prefill's shape
    (1, 4100, 8000, 1000, 3, True),        # T 3025: rows not 16-byte aligned
])
def test_topk_many_rows_bit_exact(X, B, S, start, topk, offset, ties):
    ratio = 4
    T = (start + S) // ratio
    sc = _synthetic_scores(S + start + B, B * S, T, ties).view(B, S, T)
    vis = O.visible_lens(start, S, ratio)
    for s in range(S):
        sc[:, s, vis[s]:] = float("-inf")
    d = X.make_dims(n_heads=64, ratio=ratio, index_topk=topk, offset=offset)
    out = torch.empty((B, S, topk), dtype=torch.int32, device="cuda")
    X.indexer_topk(d, sc.cuda(), start, out)
    ref = O.topk_positions(sc.double().numpy().reshape(B * S, T), np.tile(vis, B), topk, offset, T)
    got = out.cpu().numpy().reshape(B * S, topk)
    assert np.array_equal(got, ref), f"{np.sum(np.any(got != ref, axis=-1))} of {B * S} rows differ"


@pytest.mark.parametrize("T,cbs,cbk,ties", [(32768, 64, 64, False), (1000, 64, 8, True), (100, 7, 40, True)])
def test_candidate_kernel_bit_exact(X, T, cbs, cbk, ties):
    B, S, ratio = 3, 1, 4
    start = T * ratio - 1
    sc = _synthetic_scores(T + cbs, B * S, T, ties).view(B, S, T)
    d = X.make_dims(n_heads=64, ratio=ratio, index_topk=16, cand_topk_blocks=cbk, cand_block_size=cbs)
    out = torch.empty((B, S, cbk), dtype=torch.int32, device="cuda")
    X.indexer_select_candidate_blocks(d, sc.cuda(), start, out)
    vis = O.visible_lens(start, S, ratio)
    ref = O.select_candidate_blocks(sc.double().numpy().reshape(B * S, T), np.tile(vis, B), cbk, cbs)
    assert np.array_equal(out.cpu().numpy().reshape(B * S, cbk), ref)


def test_candidate_kernel_prefill_rows(X):
    B, S, ratio, cbs, cbk = 1, 64, 4, 3, 2
    T = S // ratio
    sc = _synthetic_scores(99, S, T, True).view(B, S, T)
    vis = O.visible_lens(0, S, ratio)
    for s in range(S):
        sc[0, s, vis[s]:] = float("-inf")
    d = X.make_dims(n_heads=64, ratio=ratio, index_topk=4, cand_topk_blocks=cbk, cand_block_size=cbs)
    out = torch.empty((B, S, cbk), dtype=torch.int32, device="cuda")
    X.indexer_select_candidate_blocks(d, sc.cuda(), 0, out)
    ref = O.select_candidate_blocks(sc.double().numpy().reshape(S, T), vis, cbk, cbs)
    assert np.array_equal(out.cpu().numpy().reshape(S, cbk), ref)
