"""Plain CPU oracle for split-KV attention with a cost-aware LPT planner.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path (the CUDA library in
``context_long_attention_lpt_gb300`` and its Python binding) imports, calls or
links anything here.  The only callers are ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline / reference legs of ``bench.py``.

What it computes, with the passage each part follows (page: "Split-KV"
knowledge card, kongchang.com):

* ``attention``  - unsharded softmax attention in fp64 over paged K/V with
  grouped query heads.  The card's closing fact ("All Facts": Split-KV is exact,
  its results are strictly consistent with the non-sharded case) makes this the
  single correct answer every sharded computation must reproduce.
* ``partial`` / ``merge`` - one shard's attention over only its local KV blocks,
  emitting a query-sized output and its log-sum-exp, and the exact combination
  of such partials (card intro and "Timeline": each device keeps its K/V shard
  local and only tensors the size of the queries are exchanged).  The pages do
  not print the combination rule; the log-sum-exp weighted merge is the
  plainest exact reading (see ``merge``).
* ``block_costs`` / ``lpt_assign`` / ``imbalance`` - the cost-aware
  longest-processing-time-first allocation of context KV blocks to shards and
  its load-imbalance rate ("Timeline" / "All Facts": cost-aware LPT, load
  imbalance below 1%).
* ``attention_backward`` / ``partial_backward`` / ``delta`` - fp64 gradients
  dQ, dK, dV of the same attention, unsharded and restricted to one shard's
  keys (card intro: a training method; "All Facts": exact), from the merged
  forward's L and D = rowsum(dO * O).
* ``dcp_select`` - split selection that models attention completion together
  with the dependent reduction (LiquidCP abstract, PaperTrail: MegaDCP), built
  on the same LPT plans.

Everything is written for readability, not speed: fp64 throughout, a library
matmul / sort as the only primitives, no blocking or fusion beyond what the
definitions state.
"""

from .attn import attention, attention_rows, partial, merge, visible_keys, gather_sequence
from .backward import attention_backward, partial_backward, delta, backward_rows, backward_keys
from .lpt import block_costs, lpt_assign, imbalance, shard_key_sets, partial_rows, dcp_select

__all__ = [
    "attention_backward",
    "partial_backward",
    "delta",
    "backward_rows",
    "backward_keys",
    "attention",
    "attention_rows",
    "partial",
    "merge",
    "visible_keys",
    "gather_sequence",
    "block_costs",
    "lpt_assign",
    "imbalance",
    "shard_key_sets",
    "partial_rows",
    "dcp_select",
]
