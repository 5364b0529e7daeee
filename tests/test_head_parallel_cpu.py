"""Head-parallel scoring on CPU ranks (gloo, world size 2): each rank takes its shard of
the index heads (head_range), computes the oracle's partial scores with the model's head
factor, and the all-reduce of the partials must give the full oracle scores and the same
top-k ("DeepSeek V4.1" index-keys page: Indexer.__init__ n_local_heads, Indexer.forward
dist.all_reduce(index_score)). No GPU: the ranks run the oracle, which shares no code with
the kernels; this covers the split, the head factor and the reduction."""
import json
import os
import socket
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = r"""
import json, os, sys
sys.path.insert(0, {root!r})
import numpy as np
import torch
import torch.distributed as dist
import oracle as O
from sparse_attention_top_indexer_gb300.head_parallel import head_range, shard_dims
from sparse_attention_top_indexer_gb300 import make_dims
from tests import cases as C
from workloads import WORKLOADS
import dataclasses

dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
out = {{"rank": rank}}
for name, over in (("tiny_prefill", dict()), ("decode", dict(B=2, start_pos=4095, H=16))):
    wl = dataclasses.replace(WORKLOADS[name], **over)
    cos, sin = C.oracle_table(wl.max_pos)
    cache = C.oracle_cache(wl, cos, sin)
    q, w = C.bits(wl.q()), C.bits(wl.w())
    vis = O.visible_lens(wl.start_pos, wl.S, wl.ratio)
    h0, h1 = head_range(wl.H, world, rank)
    rows, wp, _ = O.prep_queries(q[:, :, h0:h1], w[:, :, h0:h1], cos, sin, wl.start_pos, wl.rope_dim, wl.H)
    part = torch.from_numpy(O.index_scores(rows, wp, cache, wl.T, vis))
    dist.all_reduce(part, op=dist.ReduceOp.SUM)
    full_rows, full_wp, _ = O.prep_queries(q, w, cos, sin, wl.start_pos, wl.rope_dim, wl.H)
    full = O.index_scores(full_rows, full_wp, cache, wl.T, vis)
    got = part.numpy()
    fin = np.isfinite(full)
    same_mask = bool(np.array_equal(np.isneginf(got), np.isneginf(full)))
    err = float(np.max(np.abs(got[fin] - full[fin]) / (np.abs(full[fin]) + 1e-30))) if fin.any() else 0.0
    top_p = O.topk_positions(got.reshape(-1, wl.T), np.tile(vis, wl.B), wl.topk, wl.offset, wl.T)
    top_f = O.topk_positions(full.reshape(-1, wl.T), np.tile(vis, wl.B), wl.topk, wl.offset, wl.T)
    sd = shard_dims(make_dims(n_heads=wl.H, ratio=wl.ratio, index_topk=wl.topk), world)
    out[name] = {{"heads": [h0, h1], "same_mask": same_mask, "max_rel_err": err,
                 "topk_equal": bool(np.array_equal(top_p, top_f)),
                 "shard_dims": [sd.n_heads, sd.n_heads_total]}}
print(json.dumps(out), flush=True)
dist.destroy_process_group()
"""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def test_partial_scores_all_reduce_to_the_full_scores():
    port = _free_port()
    procs = []
    for rank in range(2):
        env = dict(os.environ, MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE="2",
                   LOCAL_RANK=str(rank), CUDA_VISIBLE_DEVICES="", OMP_NUM_THREADS="1")
        procs.append(subprocess.Popen([sys.executable, "-c", _CHILD.format(root=ROOT)], env=env, cwd=ROOT,
                                      stdout=subprocess.PIPE, stderr=subprocess.PIPE, text=True))
    outs = []
    for p in procs:
        o, e = p.communicate(timeout=600)
        assert p.returncode == 0, e[-3000:]
        outs.append(json.loads(o.strip().splitlines()[-1]))
    outs.sort(key=lambda o: o["rank"])
    for name, H in (("tiny_prefill", 8), ("decode", 16)):
        assert [o[name]["heads"] for o in outs] == [[0, H // 2], [H // 2, H]]
        for o in outs:
            r = o[name]
            assert r["same_mask"] and r["topk_equal"], r
            assert r["max_rel_err"] <= 1e-12, r
            assert r["shard_dims"] == [H // 2, H]


def test_head_range_and_shard_dims_host_logic():
    from sparse_attention_top_indexer_gb300 import make_dims
    from sparse_attention_top_indexer_gb300.head_parallel import head_range, shard_dims
    assert [head_range(64, 4, r) for r in range(4)] == [(0, 16), (16, 32), (32, 48), (48, 64)]
    d = shard_dims(make_dims(n_heads=64, ratio=4, index_topk=2048, offset=7, cand_topk_blocks=3,
                             cand_block_size=64), 8)
    assert (d.n_heads, d.n_heads_total, d.index_topk, d.offset, d.cand_topk_blocks) == (8, 64, 2048, 7, 3)
    import pytest
    with pytest.raises(ValueError):
        head_range(64, 3, 0)
