"""Host-side checks of the C ABI: the library loads, exports every function that
include/indexer.h declares, and rejects bad arguments before touching a GPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def X():
    import sparse_attention_top_indexer_gb300 as X
    if not os.path.exists(X.LIB_PATH):
        from sparse_attention_top_indexer_gb300.build import build
        build()
    X.load_library()
    return X


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^\s*(?:int|size_t|const char\*)\s+(indexer_\w+)\s*\(", text, re.M))
    return names


def test_every_declared_symbol_is_exported(X):
    names = _declared()
    assert {"indexer_publish_k", "indexer_scores", "indexer_topk", "indexer_forward"} <= names
    lib = X.load_library()
    for n in names:
        assert hasattr(lib, n), f"{n} declared but not exported"


def test_struct_layouts_match_header(X):
    assert ctypes.sizeof(X.IndexerDims) == 44
    assert X.IndexerYarn.beta_slow.offset == 32


def test_abi_version(X):
    assert X.indexer_abi_version() == 405   # + indexer_compress_weights (upstream producers)


def test_workspace_size_host_only(X):
    d = X.make_dims(n_heads=64, ratio=4, index_topk=2048)
    n = X.indexer_workspace_size(d, 32, 1, 32767)
    # status + q rows + w' + scores, each rounded to 256 bytes
    assert n == 256 + 32 * 64 * 68 + 32 * 64 * 4 + 32 * 8192 * 4
    bad = X.make_dims(n_heads=48, ratio=4, index_topk=2048)
    assert X.indexer_workspace_size(bad, 32, 1, 32767) == 0


def test_validation_rejects_without_launch(X):
    lib = X.load_library()
    d = X.make_dims(n_heads=64, ratio=4, index_topk=16)
    # NULL dims
    rc = lib.indexer_topk(None, None, 1, 1, 0, 0, None, None)
    assert rc == -1 and b"dims" in lib.indexer_last_error()
    # bad head_dim
    d2 = X.make_dims(n_heads=64, ratio=4, index_topk=16, head_dim=96)
    assert lib.indexer_topk(ctypes.byref(d2), 1, 1, 1, 0, 0, 1, None) == -3
    # T inconsistent with start_pos / S / ratio
    assert lib.indexer_topk(ctypes.byref(d), 16, 1, 8, 0, 5, 16, None) == -4
    # misaligned q in forward
    assert lib.indexer_forward(ctypes.byref(d), 0x1001, 0x2000, 1, 8, 0, 0x3000, 64, 0x4000, 64, None, None,
                               0x5000, None, 0x6000, 1 << 20, None) == -2
    # T beyond the cache
    assert lib.indexer_forward(ctypes.byref(d), 0x1000, 0x2000, 1, 1000, 0, 0x3000, 1000, 0x4000, 128, None, None,
                               0x5000, None, 0x6000, 1 << 20, None) == -4
    # cache capacity that is not a whole number of 64-key pages
    assert lib.indexer_forward(ctypes.byref(d), 0x1000, 0x2000, 1, 8, 0, 0x3000, 64, 0x4000, 96, None, None,
                               0x5000, None, 0x6000, 1 << 20, None) == -2
    # workspace too small
    assert lib.indexer_forward(ctypes.byref(d), 0x1000, 0x2000, 1, 8, 0, 0x3000, 64, 0x4000, 128, None, None,
                               0x5000, None, 0x6000, 16, None) == -5
    # decode publish on a token that does not complete a group
    assert lib.indexer_publish_k(ctypes.byref(d), 0x1000, 1, 1, 128, 0x2000, 0x3000, 0x4000, 100, 10, 0x5000, 128,
                                 None) == -4
    # RoPE positions beyond the table
    assert lib.indexer_prep_q(ctypes.byref(d), 0x1000, 0x2000, 1, 8, 0, 0x3000, 4, 0x4000, 0x5000, None) == -4
    # rope_dim odd
    d3 = X.make_dims(n_heads=64, ratio=4, index_topk=16, rope_dim=63)
    assert lib.indexer_prep_q(ctypes.byref(d3), 0x1000, 0x2000, 1, 8, 0, 0x3000, 64, 0x4000, 0x5000, None) == -3
    # candidate filter with too many blocks
    d4 = X.make_dims(n_heads=64, ratio=1, index_topk=16, cand_topk_blocks=4, cand_block_size=1)
    assert lib.indexer_select_candidate_blocks(ctypes.byref(d4), 0x1000, 1, 1, 9999, 10000, 0x2000, None) == -3


def test_paged_workspace_size_host_only(X):
    d = X.make_dims(n_heads=64, ratio=4, index_topk=2048)
    r = lambda x: (x + 255) // 256 * 256
    # 40 rows of 8 sequences (a prefill chunk and decode rows), T_max 8192: status, q rows,
    # w', scores, row metadata (16 B), row groups (32 B; at most ceil(40 / 2) + 8 = 28)
    n = X.indexer_workspace_size_paged(d, 40, 8, 8192)
    assert n == 256 + r(40 * 64 * 68) + r(40 * 64 * 4) + r(40 * 8192 * 4) + r(40 * 16) + r(28 * 32)
    # decode only (one row per sequence): one group per row
    n1 = X.indexer_workspace_size_paged(d, 8, 8, 8192)
    assert n1 == 256 + r(8 * 64 * 68) + r(8 * 64 * 4) + r(8 * 8192 * 4) + r(8 * 16) + r(8 * 32)
    assert X.indexer_workspace_size_paged(d, 8, 4097, 8192) == 0     # too many sequences
    assert X.indexer_workspace_size_paged(d, 8, 8, 40000) == 0       # beyond the top-k width


def test_paged_validation_rejects_without_launch(X):
    lib = X.load_library()
    d = X.make_dims(n_heads=64, ratio=4, index_topk=16)
    ws = 1 << 24
    args = dict(q=0x1000, w=0x2000, Q=8, n_seq=2, seq_pos=0x3000, q_start=0x3100, T_max=1024, rope=0x4000,
                max_pos=4096, pool=0x5000, num_pages=64, bt=0x6000, bt_stride=16, topk=0x7000, ws=0x8000)

    def fwd(**kw):
        a = dict(args, **kw)
        return lib.indexer_forward_paged(ctypes.byref(d), a["q"], a["w"], a["Q"], a["n_seq"], a["seq_pos"],
                                         a["q_start"], a["T_max"], a["rope"], a["max_pos"], a["pool"],
                                         a["num_pages"], a["bt"], a["bt_stride"], None, None, a["topk"], None,
                                         a["ws"], ws, None)
    assert fwd(bt=None) == -1                        # block table required
    assert fwd(pool=0x5008) == -2                    # pool not 16-byte aligned
    assert fwd(bt_stride=15) == -3                   # fewer table columns than pages of T_max
    assert fwd(n_seq=5000) == -3                     # too many sequences
    assert fwd(T_max=40000) == -3                    # beyond the top-k width
    # paged publish: a status workspace is required, the pool must be aligned
    assert lib.indexer_publish_k_paged(ctypes.byref(d), 0x1000, 4, 128, 0x2000, 0x3000, 0x4000, 100, 0x5000,
                                       0x6000, 0x7000, 8, None, 0, None) == -1
    assert lib.indexer_publish_k_paged(ctypes.byref(d), 0x1000, 4, 128, 0x2000, 0x3000, 0x4000, 100, 0x5000,
                                       0x6000, 0x7008, 8, 0x8000, 256, None) == -2


def test_qproj_and_host_step_validation_without_launch(X):
    lib = X.load_library()
    d = X.make_dims(n_heads=64, ratio=4, index_topk=16)
    d8 = X.make_dims(n_heads=64, ratio=4, index_topk=16, key_format=1)

    def qp(dd, Kq=1280, qr=0x1000, wq=0x2000, q_out=None, ws=0x9000, wsb=256):
        return lib.indexer_prep_q_proj(ctypes.byref(dd), qr, Kq, wq, 0x3000, 1, 8, 0, 0x4000, 64, 0x5000, 0x6000,
                                       q_out, ws, wsb, None)
    assert qp(d8) == -3                      # the fused projection writes MXFP4 rows only
    assert qp(d, Kq=96) == -3                # q_lora_rank not a multiple of 64
    assert qp(d, wq=None) == -1
    assert qp(d, wq=0x2008) == -2            # wq_b not 16-byte aligned
    assert qp(d, qr=0x1008) == -2
    assert qp(d, q_out=0x7008) == -2
    assert qp(d, wsb=16) == -5               # no room for the status word

    # the host-buffer step: staging for latent, q, w and the indices after the forward's workspace
    r = lambda x: (x + 255) // 256 * 256
    n = X.indexer_workspace_size_host(d, 32, 1, 32767, 1, 128)
    assert n == (r(X.indexer_workspace_size(d, 32, 1, 32767)) + r(32 * 128 * 2) + r(32 * 64 * 128 * 2) + r(32 * 64 * 2)
                 + r(32 * 16 * 4))

    def fh(topk_h=0x8000, ws=0x10000, ws_bytes=n):
        return lib.indexer_forward_publish_host(ctypes.byref(d), 0x1000, 1, 128, 0x2000, 0x3000, 0x4000, 0x5000, 32, 1,
                                                32767, 0x6000, 32768, 0x7000, 8192, topk_h, ws, ws_bytes, None)
    assert fh(topk_h=None) == -1
    assert fh(ws_bytes=n - 1) == -5
    assert fh(ws=0x10010) == -2              # the staging is carved at 256-byte offsets

    # the step's own checks (cache alignment, T_cap, positions) run before any copy is enqueued
    def fh2(G=1, Din=128, lat=0x1000, cache=0x7000, T_cap=8192, max_pos=32768, ws_bytes=None):
        nb = X.indexer_workspace_size_host(d, 32, 1, 32767, G, Din)
        return lib.indexer_forward_publish_host(ctypes.byref(d), lat, G, Din, 0x2000, 0x3000, 0x4000, 0x5000, 32, 1,
                                                32767, 0x6000, max_pos, cache, T_cap, 0x8000, 0x10000,
                                                nb if ws_bytes is None else ws_bytes, None)
    assert fh2(cache=0x7008) == -2
    assert fh2(T_cap=8128) == -4             # 8192 keys do not fit
    assert fh2(max_pos=32000) == -4          # query position beyond the table
    # no key completes this step: no latent, and Din is not read
    assert X.indexer_workspace_size_host(d, 32, 1, 32767, 0, 0) > 0
    assert fh2(G=0, Din=0, lat=None) not in (-1, -2, -3, -4, -5)   # passes every argument check


def test_row_layout_validation_without_launch(X):
    lib = X.load_library()
    d = X.make_dims(n_heads=64, ratio=4, index_topk=16)
    to_pages = lambda rows=0x1000, n_seq=2, n_keys=100, ld=128, cache=0x2000, T_cap=128: \
        lib.indexer_cache_from_rows(ctypes.byref(d), rows, n_seq, n_keys, ld, cache, T_cap, None)
    to_rows = lambda cache=0x2000, T_cap=128, n_seq=2, n_keys=100, rows=0x1000, ld=128: \
        lib.indexer_cache_to_rows(ctypes.byref(d), cache, T_cap, n_seq, n_keys, rows, ld, None)
    assert to_pages(rows=None) == -1 and to_rows(rows=None) == -1
    assert to_pages(cache=None) == -1 and to_rows(cache=None) == -1
    assert to_pages(T_cap=96) == -2                 # not a whole number of pages
    assert to_pages(n_keys=200) == -4               # beyond T_cap
    assert to_rows(n_keys=129, T_cap=192) == -4     # beyond ld_rows
    assert to_pages(rows=0x1002) == -2              # rows are moved as 4-byte words
    assert to_rows(cache=0x2008) == -2
    assert to_pages(n_seq=0) == -3


def test_missing_library_fails_loudly(tmp_path):
    import sparse_attention_top_indexer_gb300 as X
    saved = X._lib
    X._lib = None
    try:
        with pytest.raises(RuntimeError):
            X.load_library(str(tmp_path / "nope.so"))
    finally:
        X._lib = saved
