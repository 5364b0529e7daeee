"""CPU oracle for the DeepSeek-V4.1 compressed-attention indexer.

TEST INFRASTRUCTURE ONLY. Nothing in the product path imports this package:
only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
leg may import or call it. It shares no code with the CUDA library.

Sources (cited by page title and section throughout):
  * "index-keys page"  -- DeepSeek V4.1, blocks / last-pooled-group / source-layer /
    attention / indexer / index-keys (atlas.klimoza.dev): the PyTorch
    `class Indexer` and `SharedAttentionRuntime`.
  * "compress module page" -- "Module compress", spark_model::layers::
    deepseek_v41_ref::compress API docs (docs.atlascybernetics.ai): quantiser,
    YaRN and select_candidate_blocks one-line definitions, precision policy.
  * "attention.py patch page" -- launcher/docker-images/dsv41-flash/patches/
    attention.py (git.kilork.org): the 68-byte MXFP4 key row
    (_indexer_k_cache_head_dim) and the short-context top-k fill
    (_fill_short_context_topk_indices, DeepseekV4Indexer.forward).

Parity status: every function below is pinned by tests/test_oracle_pins.py,
except select_candidate_blocks, whose body the pages do not give: its
implementation is pinned against brute force and invariants, but the reading
itself (block score = max) is a reading, not a fact the pages fix -- "parity
unpinned" for that reading.
"""
from .indexer_oracle import *  # noqa: F401,F403
from .indexer_oracle import __all__  # noqa: F401
