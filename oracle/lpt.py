"""Cost-aware longest-processing-time-first (LPT) allocation of KV blocks to shards.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Follows the Split-KV knowledge card (kongchang.com), "Timeline" and "All
Facts": context KV blocks are allocated to CP ranks by a cost-aware LPT rule,
with a load imbalance below 1%.  The card defines neither the cost, the tie
order nor the imbalance rate; the readings taken here are:

* cost of a block = number of (query, key) pairs inside it that the attention
  mask leaves visible.  For a fully visible block that is q_len x tokens in the
  block; for the block holding a causal tail it counts the triangle.
* blocks are numbered globally, sequence after sequence, logical block order
  within a sequence.  LPT takes them by cost, largest first, equal costs by
  lower global number, and puts each on the shard with the smallest load so
  far, equal loads going to the lower shard id.  Loads are integers, so no
  floating-point tie can arise.
* imbalance rate = max load / mean load - 1.
"""

import numpy as np

from .attn import visible_keys


def block_costs(q_len, kv_len, block_len, causal):
    """Cost of every KV block, in global block order.

    Block j of sequence b holds keys [j*block_len, min((j+1)*block_len, kv_len)).
    Its cost is the number of (query t, key k) pairs with k in the block and k
    visible to t.
    """
    costs = []
    for lq, lk in zip(q_len, kv_len):
        lq, lk = int(lq), int(lk)
        vis = np.array([visible_keys(lq, lk, t, causal) for t in range(lq)], dtype=np.int64)
        n_blocks = -(-lk // block_len)
        for j in range(n_blocks):
            lo = j * block_len
            hi = min(lk, lo + block_len)
            seen = np.clip(np.minimum(vis, hi) - lo, 0, None)
            costs.append(int(seen.sum()))
    return costs


def lpt_assign(costs, n_shards):
    """LPT: largest block first, each onto the currently least-loaded shard.

    Returns (shard_of_block list[int], load list[int]).
    """
    order = sorted(range(len(costs)), key=lambda g: (-int(costs[g]), g))
    load = [0] * n_shards
    shard_of_block = [-1] * len(costs)
    for g in order:
        best = least_loaded(load)
        shard_of_block[g] = best
        load[best] += int(costs[g])
    return shard_of_block, load


def least_loaded(load):
    """Index of the smallest load; equal loads go to the lower shard id."""
    best = 0
    for s in range(1, len(load)):
        if load[s] < load[best]:
            best = s
    return best


def imbalance(load):
    """max / mean - 1 of the shard loads (0 for a perfectly even plan)."""
    mean = sum(load) / len(load)
    if mean == 0:
        return 0.0
    return max(load) / mean - 1.0


def shard_key_sets(shard_of_block, kv_len, block_len, n_shards):
    """Per shard, per sequence: the logical blocks the plan put on that shard.

    Returns key_sets[s][b] = sorted list of logical block indices.
    """
    sets = [[[] for _ in kv_len] for _ in range(n_shards)]
    g = 0
    for b, lk in enumerate(kv_len):
        for j in range(-(-int(lk) // block_len)):
            sets[shard_of_block[g]][b].append(j)
            g += 1
    return sets


def partial_rows(shard_of_block, q_len, kv_len, block_len):
    """Rows the merge has to reduce: sum over distinct (shard, sequence) pairs of q_len."""
    pairs = set()
    g = 0
    for b, lk in enumerate(kv_len):
        for _ in range(-(-int(lk) // block_len)):
            pairs.add((shard_of_block[g], b))
            g += 1
    return sum(int(q_len[b]) for _, b in pairs)


def shard_tokens(shard_of_block, kv_len, block_len, n_shards):
    """K/V tokens each shard streams (the keys of its blocks)."""
    tok = [0] * n_shards
    g = 0
    for lk in kv_len:
        for j in range(-(-int(lk) // block_len)):
            tok[shard_of_block[g]] += min(block_len, int(lk) - j * block_len)
            g += 1
    return tok


def dcp_select(q_len, kv_len, block_len, causal, max_shards, alpha, beta, gamma=0.0):
    """Split selection that models attention completion together with its reduction.

    After the LiquidCP abstract (PaperTrail, arXiv 2611.04401): MegaDCP picks
    history-KV splits by jointly modelling the completion of attention and of the
    reductions that depend on it.  The abstract gives no formula; the reading
    taken here: for every shard count s in 1..max_shards, plan the blocks with
    the cost-aware LPT rule onto s shards; the shards run concurrently, so
    attention completes with the slowest shard - its compute (alpha per unit
    of block cost) plus its K/V streaming (gamma per token) - and the reduction
    then combines one partial row per (shard, sequence) pair and query token:
        T(s) = max_k (alpha * load_k + gamma * tokens_k) + beta * partial_rows(s)
    (IEEE double, each product rounded, in exactly this order).  The smallest s
    reaching the least T wins.  Returns (s, shard_of_block, load, T(s)).
    """
    costs = block_costs(q_len, kv_len, block_len, causal)
    best = None
    for s in range(1, max_shards + 1):
        sob, load = lpt_assign(costs, s)
        tok = shard_tokens(sob, kv_len, block_len, s)
        t_att = max(float(alpha) * float(load[k]) + float(gamma) * float(tok[k]) for k in range(s))
        t = t_att + float(beta) * float(partial_rows(sob, q_len, kv_len, block_len))
        if best is None or t < best[3]:
            best = (s, sob, load, t)
    return best
