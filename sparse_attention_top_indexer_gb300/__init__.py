"""Python binding of the indexer C ABI (include/indexer.h).

Argument marshalling only: every function takes torch tensors that already live
on the GPU, checks dtype / shape / contiguity, and passes raw pointers and the
current CUDA stream to the function of the same name in libindexer.so. All
computation happens in the library's kernels; there is no fallback. If the
library has not been built, loading it raises.
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = [
    "IndexerDims", "IndexerYarn", "IndexerError", "load_library", "KEY_ROW_BYTES", "STATUS_BYTES", "PAGE_KEYS",
    "PAGE_BYTES", "KEY_MXFP4", "KEY_FP8", "ROW_BYTES_FP8", "PAGE_BYTES_FP8", "row_bytes", "page_bytes",
    "new_key_cache", "new_key_pool", "indexer_publish_k_paged", "indexer_forward_paged",
    "indexer_workspace_size_paged", "indexer_forward_publish",
    "indexer_rope_table", "indexer_publish_k", "indexer_prep_q", "indexer_prep_q_proj", "indexer_scores",
    "indexer_select_candidate_blocks", "indexer_topk", "indexer_forward", "indexer_workspace_size",
    "indexer_workspace_init", "indexer_status", "indexer_abi_version", "indexer_forward_publish_host",
    "indexer_workspace_size_host", "make_dims", "indexer_forward_noalloc",
    "NOALLOC_SCRATCH_BYTES", "indexer_noalloc_status", "indexer_cache_from_rows", "indexer_cache_to_rows",
    "indexer_scores_hold_test", "indexer_compress_weights",
]

KEY_ROW_BYTES = 68
PAGE_KEYS = 64
PAGE_BYTES = PAGE_KEYS * KEY_ROW_BYTES    # 4352
KEY_MXFP4, KEY_FP8 = 0, 1
ROW_BYTES_FP8 = 132
PAGE_BYTES_FP8 = PAGE_KEYS * ROW_BYTES_FP8   # 8448
STATUS_BYTES = 256
NOALLOC_SCRATCH_BYTES = 8 * 1024 * 1024
_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libindexer.so")


class IndexerDims(ctypes.Structure):
    _fields_ = [
        ("n_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("rope_dim", ctypes.c_int32),
        ("ratio", ctypes.c_int32), ("index_topk", ctypes.c_int32), ("offset", ctypes.c_int32),
        ("cand_topk_blocks", ctypes.c_int32), ("cand_block_size", ctypes.c_int32), ("norm_eps", ctypes.c_float),
        ("key_format", ctypes.c_int32), ("n_heads_total", ctypes.c_int32),
    ]


class IndexerYarn(ctypes.Structure):
    _fields_ = [
        ("theta", ctypes.c_double), ("factor", ctypes.c_double), ("original_seq_len", ctypes.c_int32),
        ("beta_fast", ctypes.c_double), ("beta_slow", ctypes.c_double),
    ]


class IndexerError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"indexer error {code}: {msg}")
        self.code = code


_lib: Optional[ctypes.CDLL] = None

_P = ctypes.c_void_p
_I = ctypes.c_int
_SIGS = {
    "indexer_rope_table": [ctypes.POINTER(IndexerYarn), _I, _I, _P, _P],
    "indexer_publish_k": [ctypes.POINTER(IndexerDims), _P, _I, _I, _I, _P, _P, _P, _I, _I, _P, _I, _P],
    "indexer_prep_q": [ctypes.POINTER(IndexerDims), _P, _P, _I, _I, _I, _P, _I, _P, _P, _P],
    "indexer_prep_q_proj": [ctypes.POINTER(IndexerDims), _P, _I, _P, _P, _I, _I, _I, _P, _I, _P, _P, _P, _P,
                            ctypes.c_size_t, _P],
    "indexer_scores": [ctypes.POINTER(IndexerDims), _P, _P, _I, _I, _I, _P, _I, _P, _P, _P, ctypes.c_size_t, _P],
    "indexer_select_candidate_blocks": [ctypes.POINTER(IndexerDims), _P, _I, _I, _I, _I, _P, _P],
    "indexer_topk": [ctypes.POINTER(IndexerDims), _P, _I, _I, _I, _I, _P, _P],
    "indexer_forward": [ctypes.POINTER(IndexerDims), _P, _P, _I, _I, _I, _P, _I, _P, _I, _P, _P, _P, _P, _P,
                        ctypes.c_size_t, _P],
    "indexer_forward_noalloc": [ctypes.POINTER(IndexerDims), _P, _P, _I, _I, _I, _P, _I, _P, _I, _P, _P, _P, _P,
                                _P],
    "indexer_forward_publish": [ctypes.POINTER(IndexerDims), _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _P, _I, _P, _I,
                                _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "indexer_forward_publish_host": [ctypes.POINTER(IndexerDims), _P, _I, _I, _P, _P, _P, _P, _I, _I, _I, _P, _I,
                                     _P, _I, _P, _P, ctypes.c_size_t, _P],
    "indexer_workspace_init": [_P, ctypes.c_size_t, _P],
    "indexer_publish_k_paged": [ctypes.POINTER(IndexerDims), _P, _I, _I, _P, _P, _P, _I, _P, _P, _P, _I, _P,
                                ctypes.c_size_t, _P],
    "indexer_forward_paged": [ctypes.POINTER(IndexerDims), _P, _P, _I, _I, _P, _P, _I, _P, _I, _P, _I, _P, _I,
                              _P, _P, _P, _P, _P, ctypes.c_size_t, _P],
    "indexer_status": [_P, _P],
    "indexer_noalloc_status": [_P],
    "indexer_compress_weights": [ctypes.POINTER(IndexerDims), _P, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P,
                                 ctypes.c_size_t, _P],
    "indexer_scores_hold_test": [ctypes.POINTER(IndexerDims), _P, _P, _I, _I, _I, _P, _I, _P, _P, ctypes.c_size_t,
                                 ctypes.c_uint64, _P],
    "indexer_cache_from_rows": [ctypes.POINTER(IndexerDims), _P, _I, _I, _I, _P, _I, _P],
    "indexer_cache_to_rows": [ctypes.POINTER(IndexerDims), _P, _I, _I, _I, _P, _I, _P],
}


def load_library(path: str = LIB_PATH) -> ctypes.CDLL:
    """Load libindexer.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -c 'import __graft_entry__ as g; g.build()'`")
    lib = ctypes.CDLL(path)
    for name, args in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = ctypes.c_int
    lib.indexer_workspace_size.argtypes = [ctypes.POINTER(IndexerDims), _I, _I, _I]
    lib.indexer_workspace_size.restype = ctypes.c_size_t
    lib.indexer_workspace_size_paged.argtypes = [ctypes.POINTER(IndexerDims), _I, _I, _I]
    lib.indexer_workspace_size_host.argtypes = [ctypes.POINTER(IndexerDims), _I, _I, _I, _I, _I]
    lib.indexer_workspace_size_host.restype = ctypes.c_size_t
    lib.indexer_workspace_size_paged.restype = ctypes.c_size_t
    lib.indexer_last_error.argtypes = []
    lib.indexer_last_error.restype = ctypes.c_char_p
    lib.indexer_abi_version.argtypes = []
    lib.indexer_abi_version.restype = ctypes.c_int
    _lib = lib
    return lib


def make_dims(n_heads: int, ratio: int, index_topk: int, offset: int = 0, rope_dim: int = 64,
              head_dim: int = 128, cand_topk_blocks: int = 0, cand_block_size: int = 0,
              norm_eps: float = 1e-6, key_format: int = KEY_MXFP4, n_heads_total: int = 0) -> IndexerDims:
    """n_heads_total: 0, or the model's index head count when this call holds a shard of
    n_heads of them (head-parallel scoring)."""
    return IndexerDims(n_heads, head_dim, rope_dim, ratio, index_topk, offset, cand_topk_blocks, cand_block_size,
                       norm_eps, key_format, n_heads_total)


def row_bytes(key_format: int = KEY_MXFP4) -> int:
    """Bytes of one quantised key or query-head row: 68 (MXFP4) or 132 (FP8)."""
    return ROW_BYTES_FP8 if key_format == KEY_FP8 else KEY_ROW_BYTES


def page_bytes(key_format: int = KEY_MXFP4) -> int:
    """Bytes of one 64-key page: 4352 (MXFP4) or 8448 (FP8)."""
    return PAGE_BYTES_FP8 if key_format == KEY_FP8 else PAGE_BYTES


def new_key_cache(B: int, T_cap: int, device="cuda", key_format: int = KEY_MXFP4) -> torch.Tensor:
    """A zeroed sequence-major key cache: uint8 [B, T_cap / 64, page bytes] (T_cap a multiple of 64)."""
    if T_cap % PAGE_KEYS:
        raise ValueError("T_cap must be a multiple of 64")
    return torch.zeros((B, T_cap // PAGE_KEYS, page_bytes(key_format)), dtype=torch.uint8, device=device)


def new_key_pool(num_pages: int, device="cuda", key_format: int = KEY_MXFP4) -> torch.Tensor:
    """A zeroed page pool: uint8 [num_pages, page bytes], 64 keys per page."""
    return torch.zeros((num_pages, page_bytes(key_format)), dtype=torch.uint8, device=device)


def _cache_tcap(k_cache: torch.Tensor, dims: Optional[IndexerDims] = None) -> int:
    pb = page_bytes(dims.key_format) if dims is not None else k_cache.shape[-1]
    if k_cache.dim() != 3 or k_cache.shape[2] != pb or pb not in (PAGE_BYTES, PAGE_BYTES_FP8):
        raise ValueError(f"k_cache must be the sequence-major uint8 [B, T_cap / 64, {pb}] cache of the dims' format")
    return k_cache.shape[1] * PAGE_KEYS


def _pool_pages(k_pool: torch.Tensor, dims: Optional[IndexerDims] = None) -> int:
    pb = page_bytes(dims.key_format) if dims is not None else k_pool.shape[-1]
    if k_pool.dim() != 2 or k_pool.shape[1] != pb or pb not in (PAGE_BYTES, PAGE_BYTES_FP8):
        raise ValueError(f"k_pool must be the uint8 [num_pages, {pb}] page pool of the dims' format")
    return k_pool.shape[0]


def _check(rc: int):
    if rc != 0:
        raise IndexerError(rc, load_library().indexer_last_error().decode())


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t: Optional[torch.Tensor], dtype=None, name: str = "tensor") -> Optional[int]:
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def _hptr(t: torch.Tensor, dtype, name: str) -> int:
    """Address of a contiguous host tensor (pinned memory lets the library's copies run
    asynchronously)."""
    if t.is_cuda:
        raise ValueError(f"{name} must be a host (CPU) tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t.data_ptr()


def indexer_abi_version() -> int:
    return load_library().indexer_abi_version()


def indexer_rope_table(yarn: IndexerYarn, rope_dim: int, max_pos: int, table: torch.Tensor, stream=None):
    """table: float32 [max_pos, rope_dim // 2, 2] (cos, sin)."""
    if tuple(table.shape) != (max_pos, rope_dim // 2, 2):
        raise ValueError("table must be [max_pos, rope_dim // 2, 2]")
    _check(load_library().indexer_rope_table(ctypes.byref(yarn), rope_dim, max_pos,
                                             _ptr(table, torch.float32, "table"), _stream(stream)))


def indexer_publish_k(dims: IndexerDims, latent: torch.Tensor, wk: torch.Tensor, k_norm_w: torch.Tensor,
                      rope_cs: torch.Tensor, start_pos: int, k_cache: torch.Tensor, stream=None):
    """latent bf16 [B, G, Din]; wk bf16 [128, Din]; k_norm_w bf16 [128]; k_cache uint8 [B, T_cap/64, 4352]."""
    B, G, Din = latent.shape
    T_cap = _cache_tcap(k_cache, dims)
    if k_cache.shape[0] != B:
        raise ValueError("k_cache batch differs from latent")
    _check(load_library().indexer_publish_k(
        ctypes.byref(dims), _ptr(latent, torch.bfloat16, "latent"), B, G, Din, _ptr(wk, torch.bfloat16, "wk"),
        _ptr(k_norm_w, torch.bfloat16, "k_norm_w"), _ptr(rope_cs, torch.float32, "rope_cs"), rope_cs.shape[0],
        start_pos, _ptr(k_cache, torch.uint8, "k_cache"), T_cap, _stream(stream)))


def indexer_prep_q(dims: IndexerDims, q: torch.Tensor, w: torch.Tensor, start_pos: int, rope_cs: torch.Tensor,
                   q_rows: torch.Tensor, w_prime: torch.Tensor, stream=None):
    """q bf16 [B, S, H, 128]; w bf16 [B, S, H]; q_rows uint8 [B, S, H, 68]; w_prime f32 [B, S, H]."""
    B, S, H, _ = q.shape
    _check(load_library().indexer_prep_q(
        ctypes.byref(dims), _ptr(q, torch.bfloat16, "q"), _ptr(w, torch.bfloat16, "w"), B, S, start_pos,
        _ptr(rope_cs, torch.float32, "rope_cs"), rope_cs.shape[0], _ptr(q_rows, torch.uint8, "q_rows"),
        _ptr(w_prime, torch.float32, "w_prime"), _stream(stream)))


def indexer_prep_q_proj(dims: IndexerDims, qr: torch.Tensor, wq_b: torch.Tensor, w: torch.Tensor, start_pos: int,
                        rope_cs: torch.Tensor, q_rows: torch.Tensor, w_prime: torch.Tensor, ws: torch.Tensor,
                        q_out: Optional[torch.Tensor] = None, stream=None):
    """qr bf16 [B, S, Kq]; wq_b bf16 [H * 128, Kq]; w bf16 [B, S, H]; q_rows uint8 [B, S, H, 68];
    w_prime f32 [B, S, H]; ws the status workspace; q_out bf16 [B, S, H, 128] or None."""
    B, S, Kq = qr.shape
    _check(load_library().indexer_prep_q_proj(
        ctypes.byref(dims), _ptr(qr, torch.bfloat16, "qr"), Kq, _ptr(wq_b, torch.bfloat16, "wq_b"),
        _ptr(w, torch.bfloat16, "w"), B, S, start_pos, _ptr(rope_cs, torch.float32, "rope_cs"), rope_cs.shape[0],
        _ptr(q_rows, torch.uint8, "q_rows"), _ptr(w_prime, torch.float32, "w_prime"),
        _ptr(q_out, torch.bfloat16, "q_out"), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
        _stream(stream)))


def indexer_compress_weights(dims: IndexerDims, x: torch.Tensor, wkv: torch.Tensor, wgate: torch.Tensor,
                             norm_w: torch.Tensor, wproj: torch.Tensor, latent: torch.Tensor, w_out: torch.Tensor,
                             ws: torch.Tensor, latent_q: Optional[torch.Tensor] = None, stream=None):
    """x bf16 [B, S, dim]; wkv, wgate bf16 [128, dim]; norm_w bf16 [128]; wproj bf16 [H, dim];
    latent (and latent_q) bf16 [B, S / ratio, 128]; w_out bf16 [B, S, H]; ws the status workspace.
    The Compressor's latent, its fp4/e4m3 quantised copy and weights_proj(x); see include/indexer.h."""
    B, S, dim = x.shape
    _check(load_library().indexer_compress_weights(
        ctypes.byref(dims), _ptr(x, torch.bfloat16, "x"), B, S, dim, _ptr(wkv, torch.bfloat16, "wkv"),
        _ptr(wgate, torch.bfloat16, "wgate"), _ptr(norm_w, torch.bfloat16, "norm_w"),
        _ptr(wproj, torch.bfloat16, "wproj"), _ptr(latent, torch.bfloat16, "latent"),
        _ptr(latent_q, torch.bfloat16, "latent_q"), _ptr(w_out, torch.bfloat16, "w_out"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)))


def indexer_scores(dims: IndexerDims, q_rows: torch.Tensor, w_prime: torch.Tensor, start_pos: int,
                   k_cache: torch.Tensor, scores: torch.Tensor, ws: torch.Tensor,
                   cand_blocks: Optional[torch.Tensor] = None, stream=None):
    """scores f32 [B, S, T]; ws uint8 workspace (>= 256 bytes, status word zeroed once)."""
    B, S = q_rows.shape[:2]
    _check(load_library().indexer_scores(
        ctypes.byref(dims), _ptr(q_rows, torch.uint8, "q_rows"), _ptr(w_prime, torch.float32, "w_prime"), B, S,
        start_pos, _ptr(k_cache, torch.uint8, "k_cache"), _cache_tcap(k_cache, dims),
        _ptr(cand_blocks, torch.int32, "cand_blocks"), _ptr(scores, torch.float32, "scores"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def indexer_scores_hold_test(dims: IndexerDims, q_rows: torch.Tensor, w_prime: torch.Tensor, start_pos: int,
                             k_cache: torch.Tensor, scores: torch.Tensor, ws: torch.Tensor, wait_ns: int, stream=None):
    """Test of the bounded device waits: the several-row score kernel with its producer held
    back, so its other roles' waits run out after wait_ns; indexer_status(ws) then raises
    INDEXER_ERR_DEVICE_TIMEOUT. See include/indexer.h."""
    B, S = q_rows.shape[:2]
    _check(load_library().indexer_scores_hold_test(
        ctypes.byref(dims), _ptr(q_rows, torch.uint8, "q_rows"), _ptr(w_prime, torch.float32, "w_prime"), B, S,
        start_pos, _ptr(k_cache, torch.uint8, "k_cache"), _cache_tcap(k_cache, dims),
        _ptr(scores, torch.float32, "scores"), _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), int(wait_ns),
        _stream(stream)))


def indexer_select_candidate_blocks(dims: IndexerDims, scores: torch.Tensor, start_pos: int,
                                    blocks_out: torch.Tensor, stream=None):
    """scores f32 [B, S, T]; blocks_out int32 [B, S, cand_topk_blocks]."""
    B, S, T = scores.shape
    _check(load_library().indexer_select_candidate_blocks(
        ctypes.byref(dims), _ptr(scores, torch.float32, "scores"), B, S, start_pos, T,
        _ptr(blocks_out, torch.int32, "blocks_out"), _stream(stream)))


def indexer_topk(dims: IndexerDims, scores: torch.Tensor, start_pos: int, out: torch.Tensor, stream=None):
    """scores f32 [B, S, T]; out int32 [B, S, index_topk]."""
    B, S, T = scores.shape
    _check(load_library().indexer_topk(ctypes.byref(dims), _ptr(scores, torch.float32, "scores"), B, S, start_pos,
                                       T, _ptr(out, torch.int32, "out"), _stream(stream)))


def indexer_workspace_size(dims: IndexerDims, B: int, S: int, start_pos: int) -> int:
    return int(load_library().indexer_workspace_size(ctypes.byref(dims), B, S, start_pos))


def indexer_workspace_init(ws: torch.Tensor, stream=None):
    _check(load_library().indexer_workspace_init(_ptr(ws, None, "ws"), ws.numel() * ws.element_size(),
                                                 _stream(stream)))


def indexer_status(ws: torch.Tensor, stream=None):
    """Synchronises the stream; raises IndexerError if a device wait ran out."""
    _check(load_library().indexer_status(_ptr(ws, None, "ws"), _stream(stream)))


def indexer_forward(dims: IndexerDims, q: torch.Tensor, w: torch.Tensor, start_pos: int, rope_cs: torch.Tensor,
                    k_cache: torch.Tensor, topk_out: torch.Tensor, ws: torch.Tensor,
                    cand_in: Optional[torch.Tensor] = None, cand_out: Optional[torch.Tensor] = None,
                    scores_out: Optional[torch.Tensor] = None, stream=None):
    """The whole path after the key publish; see include/indexer.h."""
    B, S = q.shape[:2]
    _check(load_library().indexer_forward(
        ctypes.byref(dims), _ptr(q, torch.bfloat16, "q"), _ptr(w, torch.bfloat16, "w"), B, S, start_pos,
        _ptr(rope_cs, torch.float32, "rope_cs"), rope_cs.shape[0], _ptr(k_cache, torch.uint8, "k_cache"),
        _cache_tcap(k_cache, dims), _ptr(cand_in, torch.int32, "cand_in"), _ptr(cand_out, torch.int32, "cand_out"),
        _ptr(topk_out, torch.int32, "topk_out"), _ptr(scores_out, torch.float32, "scores_out"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def indexer_forward_noalloc(dims: IndexerDims, q: torch.Tensor, w: torch.Tensor, start_pos: int,
                            rope_cs: torch.Tensor, k_cache: torch.Tensor, topk_out: torch.Tensor,
                            cand_in: Optional[torch.Tensor] = None, cand_out: Optional[torch.Tensor] = None,
                            scores_out: Optional[torch.Tensor] = None, stream=None):
    """indexer_forward without a workspace, for callers that cannot allocate device
    memory when they call it (a plugin inside a runtime that owns the device's memory,
    a server with a memory budget fixed at start-up). The library's fixed static
    scratch is used instead; include/indexer.h states its size limit and why calls
    that overlap on the GPU must not be issued."""
    B, S = q.shape[:2]
    _check(load_library().indexer_forward_noalloc(
        ctypes.byref(dims), _ptr(q, torch.bfloat16, "q"), _ptr(w, torch.bfloat16, "w"), B, S, start_pos,
        _ptr(rope_cs, torch.float32, "rope_cs"), rope_cs.shape[0], _ptr(k_cache, torch.uint8, "k_cache"),
        _cache_tcap(k_cache, dims), _ptr(cand_in, torch.int32, "cand_in"), _ptr(cand_out, torch.int32, "cand_out"),
        _ptr(topk_out, torch.int32, "topk_out"), _ptr(scores_out, torch.float32, "scores_out"), _stream(stream)))


def indexer_noalloc_status(stream=None):
    """Synchronises the stream, reads and clears the status word of the no-alloc entry
    point's static scratch on the current device; raises IndexerError if a device wait of
    the last indexer_forward_noalloc call ran out."""
    _check(load_library().indexer_noalloc_status(_stream(stream)))


def indexer_cache_from_rows(dims: IndexerDims, rows: torch.Tensor, k_cache: torch.Tensor, n_keys: Optional[int] = None,
                            stream=None):
    """Keys given as row-major rows uint8 [n_seq, ld_rows, row bytes] (the pages' indexer-cache
    layout) into pages k_cache uint8 [n_seq, T_cap / 64, page bytes]; keys 0 .. n_keys-1 of every
    sequence (default: all rows that fit)."""
    n_seq, ld_rows, rb = rows.shape
    T_cap = _cache_tcap(k_cache, dims)
    if rb != row_bytes(dims.key_format) or k_cache.shape[0] != n_seq:
        raise ValueError("rows must be [n_seq, ld_rows, row bytes of the dims' format] and match k_cache's batch")
    n = min(ld_rows, T_cap) if n_keys is None else n_keys
    _check(load_library().indexer_cache_from_rows(ctypes.byref(dims), _ptr(rows, torch.uint8, "rows"), n_seq, n,
                                                  ld_rows, _ptr(k_cache, torch.uint8, "k_cache"), T_cap,
                                                  _stream(stream)))


def indexer_cache_to_rows(dims: IndexerDims, k_cache: torch.Tensor, rows: torch.Tensor, n_keys: Optional[int] = None,
                          stream=None):
    """Pages k_cache uint8 [n_seq, T_cap / 64, page bytes] into row-major rows uint8
    [n_seq, ld_rows, row bytes]; keys 0 .. n_keys-1 of every sequence (default: all that fit)."""
    n_seq, ld_rows, rb = rows.shape
    T_cap = _cache_tcap(k_cache, dims)
    if rb != row_bytes(dims.key_format) or k_cache.shape[0] != n_seq:
        raise ValueError("rows must be [n_seq, ld_rows, row bytes of the dims' format] and match k_cache's batch")
    n = min(ld_rows, T_cap) if n_keys is None else n_keys
    _check(load_library().indexer_cache_to_rows(ctypes.byref(dims), _ptr(k_cache, torch.uint8, "k_cache"), T_cap,
                                                n_seq, n, _ptr(rows, torch.uint8, "rows"), ld_rows, _stream(stream)))


def indexer_publish_k_paged(dims: IndexerDims, latent: torch.Tensor, wk: torch.Tensor, k_norm_w: torch.Tensor,
                            rope_cs: torch.Tensor, positions: torch.Tensor, slot_mapping: torch.Tensor,
                            k_pool: torch.Tensor, ws: torch.Tensor, stream=None):
    """latent bf16 [N, Din]; positions int32 [N] (RoPE position of each key); slot_mapping
    int32 [N] (pool slot = page * 64 + key in page, < 0 skipped); k_pool uint8 [num_pages, 4352];
    ws holds the status word."""
    N, Din = latent.shape
    if tuple(positions.shape) != (N,) or tuple(slot_mapping.shape) != (N,):
        raise ValueError("positions and slot_mapping must be [N]")
    _check(load_library().indexer_publish_k_paged(
        ctypes.byref(dims), _ptr(latent, torch.bfloat16, "latent"), N, Din, _ptr(wk, torch.bfloat16, "wk"),
        _ptr(k_norm_w, torch.bfloat16, "k_norm_w"), _ptr(rope_cs, torch.float32, "rope_cs"), rope_cs.shape[0],
        _ptr(positions, torch.int32, "positions"), _ptr(slot_mapping, torch.int32, "slot_mapping"),
        _ptr(k_pool, torch.uint8, "k_pool"), _pool_pages(k_pool, dims), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)))


def indexer_workspace_size_paged(dims: IndexerDims, Q: int, n_seq: int, T_max: int) -> int:
    return int(load_library().indexer_workspace_size_paged(ctypes.byref(dims), Q, n_seq, T_max))


def indexer_forward_paged(dims: IndexerDims, q: torch.Tensor, w: torch.Tensor, seq_pos: torch.Tensor,
                          q_start: torch.Tensor, T_max: int, rope_cs: torch.Tensor, k_pool: torch.Tensor,
                          block_table: torch.Tensor, topk_out: torch.Tensor, ws: torch.Tensor,
                          cand_in: Optional[torch.Tensor] = None, cand_out: Optional[torch.Tensor] = None,
                          scores_out: Optional[torch.Tensor] = None, stream=None):
    """A batch of sequences with their own start positions and query rows, keys in a page
    pool: q bf16 [Q, H, 128]; w bf16 [Q, H]; seq_pos int32 [n_seq]; q_start int32 [n_seq + 1];
    block_table int32 [n_seq, bt_stride]; topk_out int32 [Q, index_topk]; scores_out f32
    [Q, T_max]; see include/indexer.h."""
    Q = q.shape[0]
    n_seq = seq_pos.shape[0]
    if tuple(q_start.shape) != (n_seq + 1,) or block_table.dim() != 2 or block_table.shape[0] != n_seq:
        raise ValueError("q_start must be [n_seq + 1] and block_table [n_seq, bt_stride]")
    _check(load_library().indexer_forward_paged(
        ctypes.byref(dims), _ptr(q, torch.bfloat16, "q"), _ptr(w, torch.bfloat16, "w"), Q, n_seq,
        _ptr(seq_pos, torch.int32, "seq_pos"), _ptr(q_start, torch.int32, "q_start"), T_max,
        _ptr(rope_cs, torch.float32, "rope_cs"), rope_cs.shape[0], _ptr(k_pool, torch.uint8, "k_pool"),
        _pool_pages(k_pool, dims), _ptr(block_table, torch.int32, "block_table"), block_table.shape[1],
        _ptr(cand_in, torch.int32, "cand_in"), _ptr(cand_out, torch.int32, "cand_out"),
        _ptr(topk_out, torch.int32, "topk_out"), _ptr(scores_out, torch.float32, "scores_out"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)))


def indexer_workspace_size_host(dims: IndexerDims, B: int, S: int, start_pos: int, G: int, Din: int) -> int:
    return int(load_library().indexer_workspace_size_host(ctypes.byref(dims), B, S, start_pos, G, Din))


def indexer_forward_publish_host(dims: IndexerDims, latent_h: torch.Tensor, wk: torch.Tensor, k_norm_w: torch.Tensor,
                                 q_h: torch.Tensor, w_h: torch.Tensor, start_pos: int, rope_cs: torch.Tensor,
                                 k_cache: torch.Tensor, topk_out_h: torch.Tensor, ws: torch.Tensor, stream=None):
    """indexer_forward_publish with latent_h [B, G, Din], q_h [B, S, H, 128], w_h [B, S, H] and
    topk_out_h [B, S, index_topk] in host memory; ws of indexer_workspace_size_host bytes. The
    indices are in topk_out_h once the stream has passed the call."""
    B, G, Din = latent_h.shape
    S = q_h.shape[1]
    if q_h.shape[0] != B or k_cache.shape[0] != B:
        raise ValueError("latent_h, q_h and k_cache must share the batch")
    lat = _hptr(latent_h, torch.bfloat16, "latent_h") if G > 0 else None   # G == 0: no key this step
    _check(load_library().indexer_forward_publish_host(
        ctypes.byref(dims), lat, G, Din, _ptr(wk, torch.bfloat16, "wk"),
        _ptr(k_norm_w, torch.bfloat16, "k_norm_w"), _hptr(q_h, torch.bfloat16, "q_h"), _hptr(w_h, torch.bfloat16, "w_h"),
        B, S, start_pos, _ptr(rope_cs, torch.float32, "rope_cs"), rope_cs.shape[0], _ptr(k_cache, torch.uint8, "k_cache"),
        _cache_tcap(k_cache, dims), _hptr(topk_out_h, torch.int32, "topk_out_h"), _ptr(ws, None, "ws"),
        ws.numel() * ws.element_size(), _stream(stream)))


def indexer_forward_publish(dims: IndexerDims, latent: torch.Tensor, wk: torch.Tensor, k_norm_w: torch.Tensor,
                            q: torch.Tensor, w: torch.Tensor, start_pos: int, rope_cs: torch.Tensor,
                            k_cache: torch.Tensor, topk_out: torch.Tensor, ws: torch.Tensor,
                            cand_in: Optional[torch.Tensor] = None, cand_out: Optional[torch.Tensor] = None,
                            scores_out: Optional[torch.Tensor] = None, stream=None):
    """indexer_publish_k(latent [B, G, Din]) then indexer_forward(q [B, S, H, 128]) in one call."""
    B, G, Din = latent.shape
    S = q.shape[1]
    if q.shape[0] != B or k_cache.shape[0] != B:
        raise ValueError("latent, q and k_cache must share the batch")
    _check(load_library().indexer_forward_publish(
        ctypes.byref(dims), _ptr(latent, torch.bfloat16, "latent"), G, Din, _ptr(wk, torch.bfloat16, "wk"),
        _ptr(k_norm_w, torch.bfloat16, "k_norm_w"), _ptr(q, torch.bfloat16, "q"), _ptr(w, torch.bfloat16, "w"), B, S,
        start_pos, _ptr(rope_cs, torch.float32, "rope_cs"), rope_cs.shape[0], _ptr(k_cache, torch.uint8, "k_cache"),
        _cache_tcap(k_cache, dims), _ptr(cand_in, torch.int32, "cand_in"), _ptr(cand_out, torch.int32, "cand_out"),
        _ptr(topk_out, torch.int32, "topk_out"), _ptr(scores_out, torch.float32, "scores_out"),
        _ptr(ws, None, "ws"), ws.numel() * ws.element_size(), _stream(stream)))
