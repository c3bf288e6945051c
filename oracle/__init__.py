"""CPU oracle for paged top-k sparse MLA (test infrastructure only).

This package is the slow, plain, obviously-correct statement of what the hot
path computes.  It exists to check the CUDA library; it is NOT part of the
product.  Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline``
/ ``--impl reference`` legs of ``bench.py`` may import it.  It shares no code
with the CUDA path (``paged_sparse_mla_gb300``) and imports nothing from it.

Everything is numpy, evaluated in float64 unless a step is defined in another
precision (the FP8 store is defined in fp32 arithmetic; final indexer scores
are fp32).

Sources, abbreviated in the docstrings below:

* [AgentX]  -- "vLLM、エージェント型ワークロード向け最適化技術「AgentX」を公開"
  (news.ainew.jp rendering of the vLLM AgentX blog post).  Sections cited by
  their topic: "Hybrid KV cache management" (shared block pool, packed KV
  layout), "Kimi K3" (MLA latent shared by all heads; DCP with LSE merge),
  "DeepSeek V4" (64-head indexer producing one global top-k per token;
  sparse-MLA scan/gather dominates).
* [GLM-5.3] -- aisoku.org article on vLLM serving GLM-5.3 on 16xH200 with
  PCP8xDCP8 prefill and Hybrid HiSparse decode.  Sections "What is new"
  (MLA latent KV shared by 64 heads; indexer picking 2,048 tokens),
  "Config and numbers" (MTP3; FP8 KV), "How to try" (sparse_mla_force_mqa:
  prompts inside the top-k still take the sparse MQA kernel; FP8 KV cache).
* [OCP-FP8] -- the OCP 8-bit floating point specification (E4M3 format).
* [OCP-MX]  -- the OCP Microscaling Formats (MX) specification, for its FP4
  E2M1 element type, the reading taken for FP4 indexer keys ([AgentX "Hybrid
  KV cache management"] names an FP4 indexer but no format).

``oracle.dcp`` states the split-context form (token shards, candidate merge,
log-sum-exp merge of partial outputs) of [AgentX "Kimi K3"] DCP.

The pages give no formulas.  Where a step is not fixed by them, the reading
taken here is the plainest one consistent with the rest (score function
sum_h w_h * ReLU(q_h . k) * s_k, per-tile amax/448 quantisation, ties to the
lower token index); each such reading is marked "reading:" in the docstring.

Pins (tests that tie this oracle to something other than itself) live in
``tests/test_oracle_*.py``.
"""

from .fp8 import e4m3_decode, e4m3_encode, E4M3_MAX
from .fp4 import e2m1_decode, e2m1_encode, e2m1_pack, e2m1_unpack, E2M1_MAX
from .layout import PoolLayout
from .store import kvpack_store, read_record, read_index_key
from .indexer import index_scores, index_scores_row, query_positions, context_slots
from .topk import topk_select
from .attention import attend, sparse_attend, dense_attend
from .pipeline import decode_step
from .store import bf16_bits_to_f64, quantize_latent
from . import dcp

__all__ = [
    "e4m3_decode", "e4m3_encode", "E4M3_MAX", "e2m1_decode", "e2m1_encode", "e2m1_pack", "e2m1_unpack",
    "E2M1_MAX", "PoolLayout", "kvpack_store",
    "read_record", "read_index_key", "index_scores", "index_scores_row",
    "query_positions", "context_slots", "topk_select", "attend", "sparse_attend",
    "dense_attend", "decode_step", "bf16_bits_to_f64", "quantize_latent", "dcp",
]
