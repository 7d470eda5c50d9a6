"""Pins for the CPU oracle: closed forms, library cross-checks, invariants, brute force.

The pages print no worked example for split-KV attention, so the oracle is
pinned by what mathematics fixes:
* hand-derived values (tests/golden/closed_forms.json);
* torch's own scaled_dot_product_attention in fp64 on small shapes;
* the exactness fact of the Split-KV card ("All Facts": results strictly
  consistent with the non-sharded case): merging any split of the keys must
  reproduce the unsharded result;
* Graham's bound for LPT, against brute-force optimal makespans on tiny inputs.
The last group plants plausible mistakes in the oracle and checks that a pin
catches each one.
"""

import itertools
import math
import random

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import attn as oatt
from oracle import lpt as olpt

pytestmark = pytest.mark.filterwarnings("ignore")


def _paged(k_seq, v_seq, block_len, perm_seed=None):
    """Lay a contiguous [n, Hkv, d] K/V sequence out as a paged pool + table row."""
    n = k_seq.shape[0]
    nb = -(-n // block_len)
    pool_k = torch.zeros((nb, block_len) + tuple(k_seq.shape[1:]), dtype=k_seq.dtype)
    pool_v = torch.zeros((nb, block_len) + tuple(v_seq.shape[1:]), dtype=v_seq.dtype)
    phys = list(range(nb))
    if perm_seed is not None:
        random.Random(perm_seed).shuffle(phys)
    for j in range(nb):
        lo, hi = j * block_len, min(n, (j + 1) * block_len)
        pool_k[phys[j], : hi - lo] = k_seq[lo:hi]
        pool_v[phys[j], : hi - lo] = v_seq[lo:hi]
    return pool_k, pool_v, phys


def _random_batch(seed, B=3, Hq=4, Hkv=2, d=8, block_len=4, causal=True, max_ctx=13, max_q=5):
    g = torch.Generator().manual_seed(seed)
    rng = random.Random(seed)
    q_len = [rng.randint(1, max_q) for _ in range(B)]
    kv_len = [rng.randint(0, max_ctx) + (q if causal else 0) for q in q_len]
    if not causal:
        kv_len = [max(1, n) for n in kv_len]
    nblk = [-(-n // block_len) for n in kv_len]
    n_pool = sum(nblk) + 2
    phys = list(range(n_pool))
    rng.shuffle(phys)
    table = torch.zeros((B, max(nblk)), dtype=torch.int32)
    i = 0
    for b in range(B):
        for j in range(nblk[b]):
            table[b, j] = phys[i]
            i += 1
    q = torch.randn((sum(q_len), Hq, d), generator=g, dtype=torch.float64)
    kp = torch.randn((n_pool, block_len, Hkv, d), generator=g, dtype=torch.float64)
    vp = torch.randn((n_pool, block_len, Hkv, d), generator=g, dtype=torch.float64)
    return dict(q=q, k_pool=kp, v_pool=vp, block_table=table, q_len=q_len, kv_len=kv_len,
                block_len=block_len, causal=causal, scale=1.0 / math.sqrt(d))


# ---------------------------------------------------------------- closed forms


def test_two_keys_closed_form(golden):
    c = golden["two_keys"]
    k = torch.tensor(c["k"], dtype=torch.float64)[:, None, :]
    v = torch.tensor(c["v"], dtype=torch.float64)[:, None, :]
    kp, vp, phys = _paged(k, v, block_len=2)
    q = torch.tensor(c["q"], dtype=torch.float64)[None, None, :]
    o, l = oracle.attention(q, kp, vp, torch.tensor([phys]), [1], [2], 2, False, c["scale"])
    assert torch.allclose(o[0, 0], torch.tensor(c["O"], dtype=torch.float64), atol=1e-15, rtol=0)
    assert abs(l[0, 0].item() - c["L"]) < 1e-15


def test_causal_tail_zero_keys(golden):
    c = golden["causal_tail_zero_keys"]
    g = torch.Generator().manual_seed(0)
    n = c["kv_len"]
    k = torch.zeros((n, 1, 8), dtype=torch.float64)
    v = torch.randn((n, 1, 8), generator=g, dtype=torch.float64)
    kp, vp, phys = _paged(k, v, block_len=2, perm_seed=1)
    q = torch.randn((c["q_len"], 1, 8), generator=g, dtype=torch.float64)
    o, l = oracle.attention(q, kp, vp, torch.tensor([phys]), [c["q_len"]], [n], 2, True, 0.3)
    for t in range(c["q_len"]):
        nv = c["visible"][t]
        assert oracle.visible_keys(c["q_len"], n, t, True) == nv
        assert abs(l[t, 0].item() - c["L"][t]) < 1e-14
        assert torch.allclose(o[t, 0], v[:nv, 0].mean(0), atol=1e-14, rtol=0)


def test_constant_values_give_that_value():
    b = _random_batch(3)
    c = torch.linspace(-2, 3, b["v_pool"].shape[-1], dtype=torch.float64)
    b["v_pool"] = torch.zeros_like(b["v_pool"]) + c
    o, _ = oracle.attention(**b)
    assert torch.allclose(o, c.expand_as(o), atol=1e-13, rtol=0)


def test_softmax_weights_via_identity_values():
    """With V = I the output row is the softmax row itself: it sums to 1 and
    P_j = exp(s_j - L) with s_j = scale * q . k_j."""
    g = torch.Generator().manual_seed(5)
    n, d = 6, 8
    k = torch.randn((n, 1, d), generator=g, dtype=torch.float64)
    v = torch.eye(n, d, dtype=torch.float64)[:, None, :]
    kp, vp, phys = _paged(k, v, block_len=4, perm_seed=2)
    q = torch.randn((2, 1, d), generator=g, dtype=torch.float64)
    o, l = oracle.attention(q, kp, vp, torch.tensor([phys]), [2], [n], 4, False, 0.7)
    for t in range(2):
        p = o[t, 0, :n]
        assert abs(p.sum().item() - 1.0) < 1e-14
        assert torch.all(o[t, 0, n:] == 0)
        for j in range(n):
            s = 0.7 * float(torch.dot(q[t, 0], k[j, 0]))
            assert abs(p[j].item() - math.exp(s - l[t, 0].item())) < 1e-14


def test_gqa_mapping_contiguous():
    """Query head h reads K/V head h // G."""
    g = torch.Generator().manual_seed(7)
    n, d, hq, hkv = 9, 4, 4, 2
    k = torch.randn((n, hkv, d), generator=g, dtype=torch.float64)
    k[:, 1] = 0.0  # kv head 1: uniform weights -> L = ln n
    v = torch.zeros((n, hkv, d), dtype=torch.float64)
    v[:, 0] = 1.0
    v[:, 1] = 2.0
    kp, vp, phys = _paged(k, v, block_len=4)
    q = torch.randn((1, hq, d), generator=g, dtype=torch.float64)
    o, l = oracle.attention(q, kp, vp, torch.tensor([phys]), [1], [n], 4, False, 0.5)
    for h in range(hq):
        assert torch.allclose(o[0, h], torch.full((d,), 1.0 + (h // 2), dtype=torch.float64))
    assert abs(l[0, 2].item() - math.log(n)) < 1e-14
    assert abs(l[0, 3].item() - math.log(n)) < 1e-14
    assert abs(l[0, 0].item() - math.log(n)) > 1e-6


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("causal", [False, True])
def test_matches_torch_sdpa(seed, causal):
    """torch's fp64 scaled_dot_product_attention on the contiguous, mask-explicit form."""
    b = _random_batch(seed, causal=causal)
    o, _ = oracle.attention(**b)
    g = b["q"].shape[1] // b["k_pool"].shape[2]
    cu = 0
    for i, (lq, lk) in enumerate(zip(b["q_len"], b["kv_len"])):
        ks = oatt.gather_sequence(b["k_pool"], b["block_table"][i], lk, b["block_len"])
        vs = oatt.gather_sequence(b["v_pool"], b["block_table"][i], lk, b["block_len"])
        qq = b["q"][cu : cu + lq].permute(1, 0, 2)  # [Hq, Lq, d]
        kk = ks.permute(1, 0, 2).repeat_interleave(g, 0)
        vv = vs.permute(1, 0, 2).repeat_interleave(g, 0)
        pos = torch.arange(lk)
        qpos = torch.arange(lq) + (lk - lq)
        mask = (pos[None, :] <= qpos[:, None]) if causal else torch.ones((lq, lk), dtype=torch.bool)
        ref = F.scaled_dot_product_attention(qq, kk, vv, attn_mask=mask, scale=b["scale"])
        assert torch.allclose(o[cu : cu + lq], ref.permute(1, 0, 2), atol=1e-12, rtol=0)
        cu += lq


def test_paging_permutation_invariance():
    b = _random_batch(11, B=2)
    o1, l1 = oracle.attention(**b)
    # move every block to a new physical slot
    n_pool = b["k_pool"].shape[0]
    perm = torch.randperm(n_pool, generator=torch.Generator().manual_seed(3))
    kp2 = torch.empty_like(b["k_pool"])
    vp2 = torch.empty_like(b["v_pool"])
    kp2[perm] = b["k_pool"]
    vp2[perm] = b["v_pool"]
    b2 = dict(b, k_pool=kp2, v_pool=vp2, block_table=perm[b["block_table"].long()].to(torch.int32))
    o2, l2 = oracle.attention(**b2)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_rows_match_full():
    b = _random_batch(12)
    o, l = oracle.attention(**b)
    rows = [(0, 0, 0), (1, b["q_len"][1] - 1, 3), (2, 0, 2), (0, b["q_len"][0] - 1, 1)]
    cu = [0, b["q_len"][0], b["q_len"][0] + b["q_len"][1]]
    orow, lrow = oracle.attention_rows(**b, rows=rows)
    for i, (bb, t, h) in enumerate(rows):
        assert torch.allclose(orow[i], o[cu[bb] + t, h], atol=1e-14, rtol=0)
        assert abs(lrow[i] - l[cu[bb] + t, h]) < 1e-13


# ------------------------------------------------------------ exactness (merge)


@pytest.mark.parametrize("seed", range(8))
def test_merge_of_any_split_is_exact(seed):
    """Random assignments of blocks to S shards (empty shards included)."""
    rng = random.Random(100 + seed)
    b = _random_batch(seed, causal=bool(seed % 2), block_len=rng.choice([2, 3, 4]))
    o_ref, l_ref = oracle.attention(**b)
    S = rng.randint(1, 6)
    parts = []
    owner = [[rng.randrange(S) for _ in range(-(-n // b["block_len"]))] for n in b["kv_len"]]
    for s in range(S):
        keys = [[j for j, o in enumerate(owner[i]) if o == s] for i in range(len(owner))]
        parts.append(oracle.partial(**b, key_blocks=keys))
    o, l = oracle.merge(parts)
    assert torch.allclose(o, o_ref, atol=1e-12, rtol=0)
    assert torch.allclose(l, l_ref, atol=1e-12, rtol=0)


def test_single_shard_merge_is_identity():
    b = _random_batch(21)
    part = oracle.attention(**b)
    o, l = oracle.merge([part])
    assert torch.allclose(o, part[0], atol=1e-15) and torch.allclose(l, part[1], atol=1e-15)


def test_empty_shard_partial_is_neg_inf_zero():
    b = _random_batch(22)
    o, l = oracle.partial(**b, key_blocks=[[] for _ in b["q_len"]])
    assert torch.all(o == 0) and torch.all(torch.isneginf(l))


def test_invisible_block_partial():
    """A shard holding only keys past a query's causal position gives that row -inf."""
    g = torch.Generator().manual_seed(1)
    lq, lk, bl = 4, 6, 2  # query t at position 2+t
    k = torch.randn((lk, 1, 4), generator=g, dtype=torch.float64)
    v = torch.randn((lk, 1, 4), generator=g, dtype=torch.float64)
    kp, vp, phys = _paged(k, v, bl)
    q = torch.randn((lq, 1, 4), generator=g, dtype=torch.float64)
    o, l = oracle.partial(q, kp, vp, torch.tensor([phys]), [lq], [lk], bl, True, 0.5, [[2]])
    # block 2 = keys {4,5}: invisible to t=0,1 (positions 2,3), visible to t=2 (key 4), t=3
    assert torch.isneginf(l[0, 0]) and torch.isneginf(l[1, 0])
    assert torch.all(o[:2] == 0)
    assert torch.allclose(o[2, 0], v[4, 0], atol=1e-15)


# --------------------------------------------------------------------- LPT


def test_block_costs_golden(golden):
    c = golden["block_costs"]
    assert olpt.block_costs(c["q_len"], c["kv_len"], c["block_len"], True) == c["causal"]
    assert olpt.block_costs(c["q_len"], c["kv_len"], c["block_len"], False) == c["non_causal"]


@pytest.mark.parametrize("seed", range(5))
def test_block_costs_sum_closed_form(seed):
    """Summed over blocks, the causal cost is q_len*context + q_len*(q_len+1)/2."""
    rng = random.Random(seed)
    q = [rng.randint(1, 40) for _ in range(4)]
    ctx = [rng.randint(0, 300) for _ in range(4)]
    kv = [a + b for a, b in zip(q, ctx)]
    bl = rng.choice([7, 16, 32])
    costs = olpt.block_costs(q, kv, bl, True)
    assert sum(costs) == sum(a * c + a * (a + 1) // 2 for a, c in zip(q, ctx))
    assert len(costs) == sum(-(-n // bl) for n in kv)
    costs_nc = olpt.block_costs(q, kv, bl, False)
    assert sum(costs_nc) == sum(a * n for a, n in zip(q, kv))


def test_lpt_ties_golden(golden):
    for c in golden["lpt_ties"]:
        sob, load = olpt.lpt_assign(c["costs"], c["n_shards"])
        assert sob == c["shard_of_block"] and load == c["load"]


def _opt_makespan(costs, S):
    best = None
    for assign in itertools.product(range(S), repeat=len(costs)):
        load = [0] * S
        for c, s in zip(costs, assign):
            load[s] += c
        m = max(load)
        best = m if best is None else min(best, m)
    return best


@pytest.mark.parametrize("seed", range(40))
def test_lpt_graham_bound_vs_brute_force(seed):
    rng = random.Random(seed)
    n = rng.randint(1, 8)
    S = rng.randint(1, 3)
    costs = [rng.randint(0, 20) for _ in range(n)]
    sob, load = olpt.lpt_assign(costs, S)
    assert sorted(range(n), key=lambda g: g) == sorted(range(n))
    assert all(0 <= s < S for s in sob)
    assert sum(load) == sum(costs)
    assert [sum(c for c, s in zip(costs, sob) if s == k) for k in range(S)] == load
    opt = _opt_makespan(costs, S)
    assert max(load) * 3 * S <= (4 * S - 1) * opt  # LPT <= (4/3 - 1/(3S)) OPT
    assert max(load) >= opt


def _plan_for(name):
    from context_long_attention_lpt_gb300 import workloads as wl

    w = wl.WORKLOADS[name]
    q, kv = wl.lengths(w)
    costs = olpt.block_costs(q, kv, w.block_len, w.causal)
    sob, load = olpt.lpt_assign(costs, w.n_shards)
    return w, costs, sob, load


@pytest.mark.parametrize("name", ["shortq", "largest"])
def test_workload_plans_golden(golden, name):
    c = golden["workload_plans"][name]
    w, costs, sob, load = _plan_for(name)
    assert len(costs) == c["n_blocks"]
    assert costs[:-1] == [c["full_cost"]] * (c["n_blocks"] - 1) and costs[-1] == c["tail_cost"]
    assert max(load) == c["max_load"]
    assert sum(load) == c["mean_load"] * w.n_shards
    assert abs(olpt.imbalance(load) - c["imbalance"]) < 1e-15
    assert sob[-1] == 0
    assert sob[:-1] == [g % w.n_shards for g in range(c["n_blocks"] - 1)]


@pytest.mark.parametrize("name", ["decode", "tiny"])
def test_uniform_plans_golden(golden, name):
    c = golden["workload_plans"][name]
    w, costs, sob, load = _plan_for(name)
    assert costs == [c["block_cost"]] * c["n_blocks"]
    assert sob == [g % w.n_shards for g in range(c["n_blocks"])]
    assert load == [c["load_each"]] * w.n_shards


# ------------------------------------------------- planted mistakes are caught


def test_planted_off_by_one_causal_is_caught(golden, monkeypatch):
    c = golden["causal_tail_zero_keys"]
    monkeypatch.setattr(oatt, "visible_keys", lambda ql, kl, t, causal: int(kl) - int(ql) + int(t))
    k = torch.zeros((c["kv_len"], 1, 4), dtype=torch.float64)
    v = torch.ones((c["kv_len"], 1, 4), dtype=torch.float64)
    kp, vp, phys = _paged(k, v, 2)
    q = torch.zeros((c["q_len"], 1, 4), dtype=torch.float64)
    _, l = oatt.attention(q, kp, vp, torch.tensor([phys]), [c["q_len"]], [c["kv_len"]], 2, True, 1.0)
    assert abs(l[0, 0].item() - c["L"][0]) > 0.1


def test_planted_unweighted_merge_is_caught():
    b = _random_batch(30)
    o_ref, _ = oracle.attention(**b)
    nb = [-(-n // b["block_len"]) for n in b["kv_len"]]
    parts = [oracle.partial(**b, key_blocks=[[j for j in range(n) if j % 2 == s] for n in nb])
             for s in range(2)]
    bad = 0.5 * (parts[0][0] + parts[1][0])  # forgets the exp(L_i - L) weights
    assert (bad - o_ref).abs().max() > 1e-3


def test_planted_reversed_tie_break_is_caught(golden, monkeypatch):
    """oracle.lpt_assign with its least-loaded choice sending equal loads to the HIGHEST shard
    id no longer reproduces the hand-worked tie cases."""
    from oracle import lpt as olpt

    def highest_id_on_ties(load):
        return max(range(len(load)), key=lambda s: (-load[s], s))

    for c in golden["lpt_ties"]:
        assert oracle.lpt_assign(c["costs"], c["n_shards"])[0] == c["shard_of_block"]
    monkeypatch.setattr(olpt, "least_loaded", highest_id_on_ties)
    caught = [oracle.lpt_assign(c["costs"], c["n_shards"])[0] != c["shard_of_block"] for c in golden["lpt_ties"]]
    assert any(caught)
    assert caught[0]


def test_planted_dropped_scale_is_caught(golden):
    c = golden["two_keys"]
    k = torch.tensor(c["k"], dtype=torch.float64)[:, None, :]
    v = torch.tensor(c["v"], dtype=torch.float64)[:, None, :]
    kp, vp, phys = _paged(k, v, block_len=2)
    q = torch.tensor(c["q"], dtype=torch.float64)[None, None, :]
    _, l = oracle.attention(q, kp, vp, torch.tensor([phys]), [1], [2], 2, False, 1.0)
    assert abs(l[0, 0].item() - c["L"]) > 0.1
