"""Head-parallel indexer scoring across ranks (the index heads split over GPUs).

The "DeepSeek V4.1" index-keys page runs the indexer tensor-parallel over its heads:
Indexer.__init__ gives each rank n_local_heads = index_n_heads // world_size of the query
heads (wq_b and weights_proj are column-parallel), the head weights keep the factor
softmax_scale * index_n_heads^-0.5 of the whole model, and Indexer.forward sums the
ranks' partial scores with dist.all_reduce before the causal mask and the top-k. The
ReLU acts per head and the head sum is linear, so the partial sums add up to the full
score exactly up to f32 rounding order.

Here each rank's part runs in the library's kernels (indexer_prep_q with
dims.n_heads_total set, indexer_scores, indexer_topk); the exchange is one
torch.distributed all-reduce (NCCL between GPUs) of the f32 score tensor. Masked
entries are -inf in every partial, so they stay -inf in the sum. This module only
orders the calls and the collective; it does no arithmetic of its own.
"""
from __future__ import annotations

from typing import Callable, Optional

import torch

from . import IndexerDims, indexer_prep_q, indexer_scores, indexer_select_candidate_blocks, indexer_topk, make_dims

__all__ = ["head_range", "shard_dims", "partial_scores", "forward_head_parallel"]


def head_range(n_heads: int, world: int, rank: int) -> tuple:
    """The heads [h0, h1) of rank `rank` out of `world` (n_heads // world each, in rank order,
    the column-parallel split of wq_b and weights_proj)."""
    if world < 1 or not 0 <= rank < world or n_heads % world:
        raise ValueError(f"{n_heads} heads do not split over {world} ranks (rank {rank})")
    n = n_heads // world
    return rank * n, (rank + 1) * n


def shard_dims(dims: IndexerDims, world: int) -> IndexerDims:
    """The dims of one rank's shard: n_heads // world heads, n_heads_total the model's."""
    total = dims.n_heads_total or dims.n_heads
    if dims.n_heads % world:
        raise ValueError(f"{dims.n_heads} heads do not split over {world} ranks")
    return make_dims(n_heads=dims.n_heads // world, ratio=dims.ratio, index_topk=dims.index_topk,
                     offset=dims.offset, rope_dim=dims.rope_dim, head_dim=dims.head_dim,
                     cand_topk_blocks=dims.cand_topk_blocks, cand_block_size=dims.cand_block_size,
                     norm_eps=dims.norm_eps, key_format=dims.key_format, n_heads_total=total)


def partial_scores(sdims: IndexerDims, q_local: torch.Tensor, w_local: torch.Tensor, start_pos: int,
                   rope_cs: torch.Tensor, k_cache: torch.Tensor, scores: torch.Tensor, ws: torch.Tensor,
                   q_rows: Optional[torch.Tensor] = None, w_prime: Optional[torch.Tensor] = None,
                   cand_in: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """This shard's part of the scores: query prep of its heads (the model's head factor),
    then the score kernel over them; -inf where masked (causal, and outside cand_in's
    blocks when given). scores f32 [B, S, T] is written and returned."""
    from . import row_bytes
    B, S, H, D = q_local.shape
    if q_rows is None:
        q_rows = torch.empty((B, S, H, row_bytes(sdims.key_format)), dtype=torch.uint8, device=q_local.device)
    if w_prime is None:
        w_prime = torch.empty((B, S, H), dtype=torch.float32, device=q_local.device)
    indexer_prep_q(sdims, q_local, w_local, start_pos, rope_cs, q_rows, w_prime, stream=stream)
    indexer_scores(sdims, q_rows, w_prime, start_pos, k_cache, scores, ws, cand_blocks=cand_in, stream=stream)
    return scores


def forward_head_parallel(dims: IndexerDims, q_local: torch.Tensor, w_local: torch.Tensor, start_pos: int,
                          rope_cs: torch.Tensor, k_cache: torch.Tensor, topk_out: torch.Tensor, ws: torch.Tensor,
                          scores: torch.Tensor, world: int, cand_in: Optional[torch.Tensor] = None,
                          cand_out: Optional[torch.Tensor] = None,
                          all_reduce: Optional[Callable[[torch.Tensor], None]] = None, group=None, stream=None):
    """One rank of the head-parallel forward: dims are the model's (all heads); q_local
    [B, S, n_heads/world, 128] and w_local [B, S, n_heads/world] are this rank's heads
    (head_range). The partial scores are summed over the ranks by `all_reduce` (default:
    torch.distributed.all_reduce on `group`), then the candidate blocks (cand_out) and the
    top-k run on the full scores, identically on every rank."""
    sdims = shard_dims(dims, world)
    partial_scores(sdims, q_local, w_local, start_pos, rope_cs, k_cache, scores, ws, cand_in=cand_in, stream=stream)
    if all_reduce is None:
        import torch.distributed as dist
        dist.all_reduce(scores, op=dist.ReduceOp.SUM, group=group)
    else:
        all_reduce(scores)
    if cand_out is not None:
        indexer_select_candidate_blocks(dims, scores, start_pos, cand_out, stream=stream)
    indexer_topk(dims, scores, start_pos, topk_out, stream=stream)
    return topk_out
