"""Shared helpers of the GPU parity tests: seeded inputs for both sides, the
oracle's view of them, and the comparison rules.

Comparison rules (the indexer's stated tolerance):
  * codes, scales, cache rows, RoPE tables and indices: bit-exact;
  * scores: |gpu - oracle| <= 1e-3 + 1e-2 * |oracle|, -inf exactly where the oracle has -inf;
  * a selected set may differ from the oracle's only at entries whose oracle score is
    within that tolerance of the oracle's k-th score (boundary swaps, counted).
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as O
from workloads import ROPE, WORKLOADS, Workload

SCORE_ATOL = 1e-3
SCORE_RTOL = 1e-2

# Boundary swaps per compared case, reported at the end of the session (conftest.py) and
# written to a JSON file: {case: {"swaps": n, "rows": r, "selected": k}}.
SWAPS: dict = {}
# At most this fraction of the selected entries may be boundary swaps.
MAX_SWAP_FRACTION = 1e-3


def record_swaps(case: str, swaps: int, rows: int, selected: int):
    """Records a case's boundary-swap count and asserts it stays a small fraction of the
    entries selected."""
    prev = SWAPS.get(case, {"swaps": 0, "rows": 0, "selected": 0})
    SWAPS[case] = {"swaps": prev["swaps"] + int(swaps), "rows": prev["rows"] + int(rows),
                   "selected": prev["selected"] + int(selected)}
    assert swaps <= max(2, MAX_SWAP_FRACTION * selected), f"{case}: {swaps} boundary swaps in {selected} entries"


def bits(t: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (on the CPU)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def yarn_struct():
    import sparse_attention_top_indexer_gb300 as X
    return X.IndexerYarn(ROPE.theta, ROPE.factor, ROPE.original_seq_len, ROPE.beta_fast, ROPE.beta_slow)


def oracle_table(max_pos: int, rope_dim: int = 64):
    return O.yarn_freqs_cis(rope_dim, max_pos, ROPE.theta, ROPE.factor, ROPE.original_seq_len, ROPE.beta_fast,
                            ROPE.beta_slow)


def gpu_table(max_pos: int, rope_dim: int = 64) -> torch.Tensor:
    import sparse_attention_top_indexer_gb300 as X
    t = torch.empty((max_pos, rope_dim // 2, 2), dtype=torch.float32, device="cuda")
    X.indexer_rope_table(yarn_struct(), rope_dim, max_pos, t)
    return t


def dims_of(wl: Workload, **over):
    import sparse_attention_top_indexer_gb300 as X
    kw = dict(n_heads=wl.H, ratio=wl.ratio, index_topk=wl.topk, offset=wl.offset, rope_dim=wl.rope_dim,
              head_dim=wl.D, cand_topk_blocks=wl.cand_topk_blocks, cand_block_size=wl.cand_block_size,
              norm_eps=wl.norm_eps, key_format=wl.key_format)
    kw.update(over)
    return X.make_dims(**kw)


def publishes_step_key(wl: Workload) -> bool:
    """A decode step publishes the key of the group its token completes."""
    return wl.start_pos > 0 and wl.S == 1 and (wl.start_pos + 1) % wl.ratio == 0


def gpu_cache(wl: Workload, table: torch.Tensor, latent=None, decode_latent=None) -> torch.Tensor:
    """The key cache as the GPU publishes it: prefill keys for slots 0..T-1, then (decode)
    the key of the group completed at start_pos."""
    import sparse_attention_top_indexer_gb300 as X
    lat = wl.latent("cuda") if latent is None else latent
    cache = X.new_key_cache(wl.B, wl.T_cap, key_format=wl.key_format)
    d = dims_of(wl)
    X.indexer_publish_k(d, lat, wl.wk("cuda"), wl.k_norm_w("cuda"), table, 0, cache)
    if publishes_step_key(wl):
        dl = wl.decode_latent("cuda") if decode_latent is None else decode_latent
        X.indexer_publish_k(d, dl, wl.wk("cuda"), wl.k_norm_w("cuda"), table, wl.start_pos, cache)
    return cache


def pages_to_rows(pages) -> np.ndarray:
    """Key pages [..., P, 4352] as 68-byte key rows [..., P*64, 68]: a page is 8 groups of
    544 bytes; in group g, key m = 8g + r has code byte j at (j/16)*128 + r*16 + j%16 and
    its scale word at 512 + r*4 (a pure reordering of bytes)."""
    if isinstance(pages, torch.Tensor):
        pages = pages.cpu().numpy()
    lead, P = pages.shape[:-2], pages.shape[-2]
    g = pages.reshape(-1, P, 8, 544)
    n = g.shape[0]
    codes = g[..., :512].reshape(n, P, 8, 4, 8, 16).transpose(0, 1, 2, 4, 3, 5).reshape(n, P, 64, 64)
    sc = g[..., 512:].reshape(n, P, 64, 4)
    return np.concatenate([codes, sc], axis=-1).reshape(*lead, P * 64, 68)


def fp8_pages_to_rows(pages) -> np.ndarray:
    """FP8 key pages [..., P, 8448] as 132-byte rows [..., P*64, 132]: a page is 8 groups of
    1056 bytes; in group g, key m = 8g + r has code byte j at (j/16)*128 + r*16 + j%16 and
    its f32 scale at 1024 + r*4 (a pure reordering of bytes)."""
    if isinstance(pages, torch.Tensor):
        pages = pages.cpu().numpy()
    lead, P = pages.shape[:-2], pages.shape[-2]
    g = pages.reshape(-1, P, 8, 1056)
    n = g.shape[0]
    codes = g[..., :1024].reshape(n, P, 8, 8, 8, 16).transpose(0, 1, 2, 4, 3, 5).reshape(n, P, 64, 128)
    sc = g[..., 1024:].reshape(n, P, 64, 4)
    return np.concatenate([codes, sc], axis=-1).reshape(*lead, P * 64, 132)


def any_pages_to_rows(pages) -> np.ndarray:
    """Key rows of MXFP4 (4352-byte) or FP8 (8448-byte) pages."""
    return fp8_pages_to_rows(pages) if pages.shape[-1] == 8448 else pages_to_rows(pages)


def pool_to_rows(pool, block_table_row, n_keys: int) -> np.ndarray:
    """The first n_keys key rows [n_keys, 68] of one sequence of a page pool [num_pages, 4352],
    following its block-table row (pool page of each logical page)."""
    if isinstance(pool, torch.Tensor):
        pool = pool.cpu().numpy()
    bt = np.asarray(block_table_row.cpu() if isinstance(block_table_row, torch.Tensor) else block_table_row)
    npages = (n_keys + 63) // 64
    return any_pages_to_rows(pool[bt[:npages]])[:n_keys]


def oracle_cache(wl: Workload, cos, sin, latent=None, decode_latent=None) -> np.ndarray:
    lat = bits(wl.latent() if latent is None else latent)
    wk, knw = bits(wl.wk()), bits(wl.k_norm_w())
    fmt = "fp8" if wl.key_format == 1 else "mxfp4"
    cache = np.zeros((wl.B, wl.T_cap, 132 if fmt == "fp8" else 68), np.uint8)
    for b in range(wl.B):   # one sequence at a time keeps the oracle's temporaries small
        slots, rows, _ = O.publish_keys(lat[b:b + 1], wk, knw, cos, sin, 0, wl.ratio, wl.rope_dim, wl.norm_eps,
                                        fmt=fmt)
        cache[b, slots] = rows[0]
    if publishes_step_key(wl):
        dl = bits(wl.decode_latent() if decode_latent is None else decode_latent)
        slots, rows, _ = O.publish_keys(dl, wk, knw, cos, sin, wl.start_pos, wl.ratio, wl.rope_dim, wl.norm_eps,
                                        fmt=fmt)
        cache[:, slots] = rows
    return cache


def score_tol(ref: np.ndarray) -> np.ndarray:
    return SCORE_ATOL + SCORE_RTOL * np.abs(ref)


def assert_scores_close(gpu: np.ndarray, ref: np.ndarray):
    ninf_r = np.isneginf(ref)
    ninf_g = np.isneginf(gpu)
    assert np.array_equal(ninf_r, ninf_g), f"-inf pattern differs at {np.argwhere(ninf_r != ninf_g)[:5]}"
    fin = ~ninf_r
    err = np.abs(gpu[fin].astype(np.float64) - ref[fin])
    bad = err > score_tol(ref[fin])
    assert not bad.any(), f"{bad.sum()} scores out of tolerance, worst err {err.max():.3e}"
    return float(err.max()) if err.size else 0.0


def compare_topk(gpu: np.ndarray, ref: np.ndarray, ref_scores: np.ndarray, offset: int) -> int:
    """Rows [R, k] of indices (+offset, -1 padded) against the oracle's rows and its f64
    scores [R, T]. Returns the number of boundary swaps; asserts everything else."""
    swaps = 0
    for r in range(gpu.shape[0]):
        g, o = gpu[r], ref[r]
        gv, ov = g[g >= 0], o[o >= 0]
        assert np.all(g[len(gv):] == -1) and np.all(np.diff(gv) > 0), f"row {r}: not ascending / -1 trailing"
        assert len(gv) == len(ov), f"row {r}: {len(gv)} valid vs {len(ov)}"
        if np.array_equal(gv, ov):
            continue
        diff = np.setxor1d(gv, ov) - offset
        sc = ref_scores[r]
        kth = np.min(sc[ov - offset])
        assert np.all(np.isfinite(sc[diff])), f"row {r}: swapped in a masked position"
        assert np.all(np.abs(sc[diff] - kth) <= SCORE_ATOL + SCORE_RTOL * abs(kth)), \
            f"row {r}: selection differs away from the k-th score"
        swaps += len(diff) // 2
    return swaps
