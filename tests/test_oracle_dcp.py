"""Pins for the oracle's split-selection model (dcp_select) and its helpers.

The model: plan s shards with the cost-aware LPT rule, then
    T(s) = max_k (alpha * load_k + gamma * tokens_k) + beta * partial_rows(s)
and take the smallest s reaching the least T.  Each expected value below is
worked out by hand from the definitions (LPT: largest cost first, ties by
block index, onto the least-loaded shard, ties by shard id), not by calling
the oracle.
"""

import itertools

import pytest

import oracle
from oracle.lpt import shard_tokens

# One decode query against 1000 keys in 256-key blocks (non-causal):
# block tokens = costs = [256, 256, 256, 232].
#   s=1: loads [1000]            rows 1
#   s=2: 0->0, 1->1, 2->0, 3->1  loads [512, 488]       rows 2
#   s=3: 0,1,2 -> 0,1,2; 3->0    loads [488, 256, 256]  rows 3
#   s=4: one block each          loads [256,256,256,232] rows 4
DECODE = dict(q_len=[1], kv_len=[1000], block_len=256, causal=False, max_shards=4)


@pytest.mark.parametrize("alpha,beta,gamma,s,t", [
    (1.0, 100.0, 0.0, 4, 656.0),     # 1100, 712, 788, 656
    (1.0, 200.0, 0.0, 2, 912.0),     # 1200, 912, 1088, 1056
    (0.0, 0.0, 1.0, 4, 256.0),       # max tokens 1000, 512, 488, 256
    (1.0, 300.0, 1.0, 2, 1624.0),    # 2300, 1624, 1876, 1712
    (0.0, 5.0, 0.0, 1, 5.0),         # only the reduction counts: one shard
])
def test_dcp_decode_worked_example(alpha, beta, gamma, s, t):
    got = oracle.dcp_select(alpha=alpha, beta=beta, gamma=gamma, **DECODE)
    assert got[0] == s and got[3] == t


# Causal: 4 query tokens at positions 4..7 against 8 keys in 4-key blocks.
# Block 0 (keys 0-3) is seen whole by every row: cost 16.  Block 1 (keys 4-7)
# is seen by 1, 2, 3, 4 keys: cost 10.  Each block holds 4 tokens; each
# (shard, sequence) pair adds q_len = 4 partial rows.
#   s=1: load 26, tokens 8, rows 4      s=2: loads [16, 10], tokens [4, 4], rows 8
CAUSAL = dict(q_len=[4], kv_len=[8], block_len=4, causal=True, max_shards=2)


@pytest.mark.parametrize("alpha,beta,gamma,s,t", [
    (1.0, 2.0, 0.0, 2, 32.0),        # 34 vs 32
    (1.0, 3.0, 0.0, 1, 38.0),        # 38 vs 40
    (1.0, 3.0, 2.0, 2, 48.0),        # 26+16+12 = 54 vs max(16+8, 10+8) + 24 = 48
])
def test_dcp_causal_worked_example(alpha, beta, gamma, s, t):
    got = oracle.dcp_select(alpha=alpha, beta=beta, gamma=gamma, **CAUSAL)
    assert got[0] == s and got[3] == t


def test_dcp_ties_take_fewest_shards():
    # Equal non-causal blocks, 6 of them: max load ceil(6/s) blocks, rows s.
    # alpha=1 (per cost unit of 1 key x 1 query), beta chosen so s=2 and s=3 tie:
    # s=2: 3*10 + 2*beta ; s=3: 2*10 + 3*beta  -> equal at beta=10.
    got = oracle.dcp_select([1], [60], 10, False, 6, 1.0, 10.0)
    assert got[0] == 2 and got[3] == 50.0


def test_dcp_without_reduction_cost_is_min_max_load():
    # beta = gamma = 0: the least T is the LPT makespan over all s; with equal
    # blocks the makespan is ceil(n/s) blocks, first reached at s = n.
    for n in (1, 5, 8):
        got = oracle.dcp_select([1], [7 * n], 7, False, 12, 1.0, 0.0)
        assert got[0] == n and got[3] == 7.0


def test_partial_rows_and_tokens_by_enumeration():
    # Brute force over every assignment of 5 blocks (two sequences) to 3 shards.
    q_len, kv_len, bl = [3, 2], [20, 11], 8      # blocks: 8,8,4 | 8,3
    toks = [8, 8, 4, 8, 3]
    seq = [0, 0, 0, 1, 1]
    for sob in itertools.product(range(3), repeat=5):
        pairs = {(sob[g], seq[g]) for g in range(5)}
        assert oracle.partial_rows(list(sob), q_len, kv_len, bl) == sum(q_len[b] for _, b in pairs)
        want = [sum(t for g, t in enumerate(toks) if sob[g] == k) for k in range(3)]
        assert shard_tokens(list(sob), kv_len, bl, 3) == want


def test_dcp_matches_exhaustive_model():
    # The selection equals the argmin of T(s) evaluated from the plan of each s
    # with shard loads / tokens / rows counted directly (mixed causal lengths).
    q_len, kv_len, bl = [3, 1, 5], [37, 9, 64], 8
    costs = oracle.block_costs(q_len, kv_len, bl, True)
    tokens = [min(bl, lk - j * bl) for lk in kv_len for j in range(-(-lk // bl))]
    seq = [b for b, lk in enumerate(kv_len) for _ in range(-(-lk // bl))]
    a, bt, gm = 0.5, 9.0, 0.25
    best = None
    for s in range(1, 9):
        sob, _ = oracle.lpt_assign(costs, s)
        per = [a * sum(c for g, c in enumerate(costs) if sob[g] == k)
               + gm * sum(t for g, t in enumerate(tokens) if sob[g] == k) for k in range(s)]
        rows = sum(q_len[b] for b in {seq[g] for g in range(len(sob))}
                   for _ in range(len({sob[g] for g in range(len(sob)) if seq[g] == b})))
        t = max(per) + bt * rows
        if best is None or t < best[1]:
            best = (s, t)
    got = oracle.dcp_select(q_len, kv_len, bl, True, 8, a, bt, gm)
    assert got[0] == best[0] and got[3] == pytest.approx(best[1], rel=1e-12)
