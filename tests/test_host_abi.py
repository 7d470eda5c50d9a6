"""Host-side checks of the C ABI (no GPU): exports, block costs, LPT plan, work lists, errors.

The C++ planner must reproduce the oracle's LPT plan bit for bit (integer
costs, fixed tie order), on every workload and on random fuzz cases.
"""

import ctypes
import os
import random
import re

import numpy as np
import pytest

import oracle
from context_long_attention_lpt_gb300 import workloads as wl

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def k():
    from context_long_attention_lpt_gb300 import build, splitkv

    if not os.path.exists(splitkv.library_path()):
        build.build()
    splitkv.lib()
    return splitkv


def test_a_missing_library_raises_and_nothing_falls_back(k, monkeypatch, tmp_path):
    """Without the built library every entry point, host planning included, raises: the
    package has no CPU fallback for any step of the path."""
    from context_long_attention_lpt_gb300 import runner

    monkeypatch.setattr(k, "_LIB_PATH", str(tmp_path / "libsplitkv.so"))
    monkeypatch.setattr(k, "_lib", None)
    with pytest.raises(RuntimeError, match="not found"):
        k.splitkv_block_costs([4], [8], 4, True)
    with pytest.raises(RuntimeError, match="not found"):
        runner.SplitKVAttention([4], [8], 4, True, 2, 4, 4, 64, None, device="cpu")


def _header_symbols():
    text = open(os.path.join(ROOT, "include", "splitkv.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(splitkv_\w+)\s*\(", text)))


def test_library_exports_every_declared_symbol(k):
    syms = _header_symbols()
    assert len(syms) >= 10
    L = k.lib()
    for s in syms:
        assert hasattr(L, s), s
    assert set(syms) == set(k.exported_symbols())


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_costs_and_plan_match_oracle_on_workloads(k, name):
    w = wl.WORKLOADS[name]
    q, kv = wl.lengths(w)
    costs = k.splitkv_block_costs(q, kv, w.block_len, w.causal)
    ref_costs = oracle.block_costs(q, kv, w.block_len, w.causal)
    assert costs.tolist() == ref_costs
    sob, load = k.splitkv_plan(costs, w.n_shards)
    ref_sob, ref_load = oracle.lpt_assign(ref_costs, w.n_shards)
    assert sob.tolist() == ref_sob
    assert load.tolist() == ref_load


def test_fuzz_costs_and_plans_bit_exact(k):
    rng = random.Random(1234)
    for case in range(3000):
        B = rng.randint(1, 4)
        causal = rng.random() < 0.6
        q = [rng.randint(0, 40) for _ in range(B)]
        kv = [qq + rng.randint(0 if qq else 1, 200) for qq in q]
        bl = rng.choice([1, 3, 8, 16, 64])
        S = rng.randint(1, 9)
        costs = k.splitkv_block_costs(q, kv, bl, causal)
        ref = oracle.block_costs(q, kv, bl, causal)
        assert costs.tolist() == ref, (case, q, kv, bl, causal)
        sob, load = k.splitkv_plan(costs, S)
        rsob, rload = oracle.lpt_assign(ref, S)
        assert sob.tolist() == rsob and load.tolist() == rload, case


def test_fuzz_plans_with_many_ties(k):
    rng = random.Random(99)
    for case in range(2000):
        n = rng.randint(0, 60)
        costs = [rng.choice([0, 1, 2, 5, 5, 5, 9]) for _ in range(n)]
        S = rng.randint(1, 12)
        sob, load = k.splitkv_plan(np.array(costs, dtype=np.int64), S)
        rsob, rload = oracle.lpt_assign(costs, S)
        assert sob.tolist() == rsob and load.tolist() == rload, case


def test_fuzz_plans_with_costs_across_many_bytes(k):
    """Costs whose differences sit in different bytes (up to 2^50, so every radix digit of
    the LPT order is exercised), with repeated values and zeros: the plan is the oracle's."""
    rng = random.Random(7)
    for case in range(600):
        n = rng.randint(0, 300)
        pool = [rng.randint(0, 1 << rng.choice([4, 12, 20, 33, 50])) for _ in range(rng.randint(1, 12))]
        costs = [rng.choice(pool + [0]) for _ in range(n)]
        S = rng.randint(1, 20)
        sob, load = k.splitkv_plan(np.array(costs, dtype=np.int64), S)
        rsob, rload = oracle.lpt_assign(costs, S)
        assert sob.tolist() == rsob and load.tolist() == rload, case


def test_fuzz_work_lists_launch_order(k):
    """Random batches: the items are the plan's (shard, sequence) pairs, launched by cost
    descending, then shard, then sequence."""
    rng = random.Random(31)
    for case in range(300):
        B = rng.randint(1, 6)
        causal = rng.random() < 0.6
        q = [rng.randint(0, 300) for _ in range(B)]
        kv = [qq + rng.randint(0 if qq else 1, 5000) for qq in q]
        bl = rng.choice([16, 64, 128, 1024])
        S = rng.randint(1, 16)
        costs = k.splitkv_block_costs(q, kv, bl, causal)
        sob, _ = k.splitkv_plan(costs, S)
        work, n_items, _ = k.splitkv_build_work(q, kv, bl, costs, sob, S)
        d = _decode_work(work)
        gbase = np.cumsum([0] + [-(-n // bl) for n in kv])
        pairs = {}
        for g in range(len(costs)):
            b = int(np.searchsorted(gbase, g, side="right") - 1)
            pairs.setdefault((int(sob[g]), b), 0)
            pairs[(int(sob[g]), b)] += int(costs[g])
        want = sorted(((-c, s_, b) for (s_, b), c in pairs.items()))
        got = []
        for it in d["items"]:
            shard, seq, clo, chi = int(it[0]), int(it[1]), int(it[8]), int(it[9])
            got.append((-((clo & 0xFFFFFFFF) | (chi << 32)), shard, seq))
        assert got == want, case


def _decode_work(work):
    hdr = work[:16]
    assert hdr[0] == 0x534B5632
    B, n_items, n_shards, bl, total_q, max_q = hdr[1:7]
    off_seq, off_items, off_blocks, off_seq_items, n_blocks = hdr[7:12]
    # the sections sit where B and n_items place them (the kernels rely on it)
    assert off_seq == 16 and off_items == 16 + 4 * (B + 1) and off_blocks == off_items + 12 * n_items
    assert off_seq_items == off_blocks + n_blocks
    seqs = work[off_seq: off_seq + 4 * (B + 1)].reshape(B + 1, 4)
    items = work[off_items: off_items + 12 * n_items].reshape(n_items, 12)
    blocks = work[off_blocks: off_blocks + n_blocks]
    seq_items = work[off_seq_items: off_seq_items + n_items]
    return dict(B=B, n_items=n_items, total_q=total_q, max_q=max_q, seqs=seqs, items=items,
                blocks=blocks, seq_items=seq_items, n_blocks=n_blocks)


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_work_lists_cover_the_plan(k, name):
    w = wl.WORKLOADS[name]
    q, kv = wl.lengths(w)
    costs = k.splitkv_block_costs(q, kv, w.block_len, w.causal)
    sob, _ = k.splitkv_plan(costs, w.n_shards)
    work, n_items, part_rows = k.splitkv_build_work(q, kv, w.block_len, costs, sob, w.n_shards)
    d = _decode_work(work)
    assert d["n_items"] == n_items and d["total_q"] == sum(q) and d["max_q"] == max(q)
    sets = oracle.shard_key_sets(sob.tolist(), kv, w.block_len, w.n_shards)
    seen = set()
    rows = 0
    item_costs = []
    gbase = np.cumsum([0] + [-(-n // w.block_len) for n in kv])
    for i, it in enumerate(d["items"]):
        shard, seq, off, cnt, prow, iq, ikv, icu, clo, chi, z0, z1 = it.tolist()
        assert (iq, ikv, icu, z0, z1) == (q[seq], kv[seq], sum(q[:seq]), 0, 0)  # the sequence's row, copied
        blks = d["blocks"][off: off + cnt].tolist()
        assert blks == sets[shard][seq] and cnt > 0
        for j in blks:
            assert (seq, j) not in seen
            seen.add((seq, j))
        assert prow == rows
        rows += q[seq]
        cost = (clo & 0xFFFFFFFF) | (chi << 32)
        assert cost == sum(costs[gbase[seq] + j] for j in blks)
        item_costs.append(cost)
    assert len(seen) == len(costs)
    assert rows == part_rows
    assert item_costs == sorted(item_costs, reverse=True)
    # launch order: cost descending, then shard, then sequence
    keys = [(-c, int(it[0]), int(it[1])) for c, it in zip(item_costs, d["items"])]
    assert keys == sorted(keys)
    # per-sequence item lists: every item of the sequence, ascending shard
    for b in range(len(q)):
        p0, p1 = d["seqs"][b, 3], d["seqs"][b + 1, 3]
        its = d["seq_items"][p0:p1].tolist()
        assert all(d["items"][i, 1] == b for i in its)
        assert [d["items"][i, 0] for i in its] == sorted(d["items"][i, 0] for i in its)
        assert sorted(its) == sorted(i for i in range(n_items) if d["items"][i, 1] == b)
        assert d["seqs"][b, 0] == sum(q[:b]) and d["seqs"][b, 1] == q[b] and d["seqs"][b, 2] == kv[b]


@pytest.mark.parametrize("name,max_blocks", [("decode", 2), ("decode", 3), ("varlen", 5), ("shortq", 1),
                                             ("largest", 4), ("tiny", 64)])
def test_split_work_lists_cover_the_plan(k, name, max_blocks):
    """Items cut to at most max_blocks blocks: per (shard, sequence) their blocks, in order, are the
    plan's key set of that shard; partial rows stay contiguous; the per-sequence lists hold every item."""
    w = wl.WORKLOADS[name]
    q, kv = wl.lengths(w)
    costs = k.splitkv_block_costs(q, kv, w.block_len, w.causal)
    sob, _ = k.splitkv_plan(costs, w.n_shards)
    work, n_items, part_rows = k.splitkv_build_work_split(q, kv, w.block_len, costs, sob, w.n_shards, max_blocks)
    d = _decode_work(work)
    assert d["n_items"] == n_items
    sets = oracle.shard_key_sets(sob.tolist(), kv, w.block_len, w.n_shards)
    got = {}
    rows = 0
    gbase = np.cumsum([0] + [-(-n // w.block_len) for n in kv])
    item_costs = []
    for it in d["items"]:
        shard, seq, off, cnt, prow, iq, ikv, icu, clo, chi = it.tolist()[:10]
        assert (iq, ikv, icu) == (q[seq], kv[seq], sum(q[:seq]))
        assert 0 < cnt <= max_blocks
        blks = d["blocks"][off: off + cnt].tolist()
        got.setdefault((shard, seq), []).append(blks)
        assert prow == rows
        rows += q[seq]
        cost = (clo & 0xFFFFFFFF) | (chi << 32)
        assert cost == sum(costs[gbase[seq] + j] for j in blks)
        item_costs.append(cost)
    assert rows == part_rows
    assert item_costs == sorted(item_costs, reverse=True)
    for (shard, seq), runs in got.items():
        # the runs of one (shard, sequence) pair cut its ascending block list in order
        assert sorted(sum(runs, [])) == sets[shard][seq]
        assert all(len(r) == max_blocks for r in sorted(runs, key=lambda r: r[0])[:-1])
    assert sum(len(v) for s in sets for v in s) == sum(len(r) for runs in got.values() for r in runs)
    for b in range(len(q)):
        p0, p1 = d["seqs"][b, 3], d["seqs"][b + 1, 3]
        its = d["seq_items"][p0:p1].tolist()
        assert sorted(its) == sorted(i for i in range(n_items) if d["items"][i, 1] == b)
    # no cut reproduces the plain work lists
    plain = k.splitkv_build_work(q, kv, w.block_len, costs, sob, w.n_shards)
    same = k.splitkv_build_work_split(q, kv, w.block_len, costs, sob, w.n_shards, 0)
    assert np.array_equal(plain[0], same[0]) and plain[1:] == same[1:]


def test_imbalance_on_workloads(k):
    """The library's max/mean - 1 of the LPT loads equals the oracle's bit for bit; the
    hand-derived values for the workloads are pinned in test_oracle."""
    for name in wl.WORKLOADS:
        w = wl.WORKLOADS[name]
        q, kv = wl.lengths(w)
        _, load = k.splitkv_plan(k.splitkv_block_costs(q, kv, w.block_len, w.causal), w.n_shards)
        assert k.splitkv_imbalance(load) == oracle.imbalance(load.tolist())


def test_imbalance_fuzz_and_edges(k):
    rng = np.random.default_rng(17)
    for _ in range(2000):
        n = int(rng.integers(1, 70))
        hi = int(rng.choice([3, 1000, 1 << 40]))
        load = rng.integers(0, hi, size=n).astype(np.int64)
        assert k.splitkv_imbalance(load) == oracle.imbalance(load.tolist())
    assert k.splitkv_imbalance(np.zeros(5, dtype=np.int64)) == 0.0
    assert k.splitkv_imbalance(np.array([7, 7, 7], dtype=np.int64)) == 0.0
    assert k.splitkv_imbalance(np.array([3, 1], dtype=np.int64)) == 0.5
    with pytest.raises(k.SplitKVError):
        k.splitkv_imbalance(np.array([1, -1], dtype=np.int64))
    with pytest.raises(k.SplitKVError):
        k.splitkv_imbalance(np.array([1 << 53, 1], dtype=np.int64))
    with pytest.raises(k.SplitKVError):
        k.splitkv_imbalance(np.zeros(0, dtype=np.int64))


def test_errors_are_statuses_not_crashes(k):
    L = k.lib()
    assert L.splitkv_plan(None, 5, 2, None, None) < 0
    assert "bad block arrays" in k.splitkv_last_error()
    c = np.array([1, 2, 3], dtype=np.int64)
    sob = np.zeros(3, dtype=np.int32)
    load = np.zeros(1, dtype=np.int64)
    assert L.splitkv_plan(c.ctypes.data_as(ctypes.c_void_p), 3, 0, sob.ctypes.data_as(ctypes.c_void_p),
                          load.ctypes.data_as(ctypes.c_void_p)) < 0
    with pytest.raises(k.SplitKVError):
        k.splitkv_block_costs([5], [3], 4, True)  # q_len > kv_len
    with pytest.raises(k.SplitKVError):
        k.splitkv_build_work([1], [4], 2, [1, 1], [0, 7], 2)  # shard id out of range
    with pytest.raises(k.SplitKVError):
        k.splitkv_num_blocks([4], 0)
    # device entry points validate before touching the GPU
    assert L.splitkv_attn_partial(None, None, None, 0, None, 0, None, 1, 1, 1, 1, 4, 3, 128, 128,
                                  1.0, 0, 1, None, None, 0, 0, None) == -1
    assert L.splitkv_attn_partial(None, None, None, 0, None, 0, None, 1, 1, 1, 1, 4, 4, 96, 128,
                                  1.0, 0, 1, None, None, 0, 0, None) == -2
    assert L.splitkv_merge(None, None, 0, None, 1, 4, 4, 128, 5, None, None, None) == -1
    assert L.splitkv_auto_kernel(4, 3, 128, 128, 1, 1) < 0
    assert L.splitkv_backward_kernel(4, 3, 128, 128, 1) < 0
    assert k.splitkv_backward_kernel(32, 8, 128, 256, k.SPLITKV_BF16) == k.KERNEL_TC
    assert k.splitkv_backward_kernel(32, 8, 64, 256, k.SPLITKV_BF16) == k.KERNEL_SIMT
    assert k.splitkv_backward_kernel(4, 4, 128, 128, k.SPLITKV_F32) == k.KERNEL_SIMT


def test_work_buffer_too_small_is_capacity_error(k):
    L = k.lib()
    q = np.array([2], dtype=np.int32)
    kv = np.array([9], dtype=np.int32)
    c = k.splitkv_block_costs(q, kv, 4, True)
    sob, _ = k.splitkv_plan(c, 2)
    work = np.zeros(4, dtype=np.int32)
    n_items = ctypes.c_int32()
    rows = ctypes.c_int64()
    p = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    st = L.splitkv_build_work(p(q), p(kv), 1, 4, p(c), p(sob), len(c), 2, p(work), 4,
                              ctypes.byref(n_items), ctypes.byref(rows))
    assert st == -4


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
@pytest.mark.parametrize("alpha,beta,gamma", [(1.0, 0.0, 0.0), (1.0, 1e9, 0.0), (1.0, 100.0, 0.0),
                                              (0.25, 3.5, 0.0), (0.1, 3.0, 7.3), (1.3e-11, 1.9e-8, 7.2e-10)])
def test_dcp_selection_matches_oracle(k, name, alpha, beta, gamma):
    w = wl.WORKLOADS[name]
    q, kv = wl.lengths(w)
    s, sob, load, t = k.splitkv_plan_dcp(q, kv, w.block_len, w.causal, w.n_shards, alpha, beta, gamma)
    rs, rsob, rload, rt = oracle.dcp_select(q, kv, w.block_len, w.causal, w.n_shards, alpha, beta, gamma)
    assert (s, sob.tolist(), load[:s].tolist(), t) == (rs, rsob, rload, rt)
    assert (load[s:] == 0).all()


def test_fuzz_dcp_selection(k):
    rng = random.Random(77)
    for case in range(300):
        B = rng.randint(1, 4)
        q = [rng.randint(1, 30) for _ in range(B)]
        kv = [qq + rng.randint(0, 200) for qq in q]
        bl = rng.choice([4, 16, 32])
        S = rng.randint(1, 8)
        a, b, c = rng.choice([0.0, 1.0, 2.5]), rng.choice([0.0, 0.5, 7.0, 1e6]), rng.choice([0.0, 0.3, 11.0])
        causal = rng.random() < 0.5
        got = k.splitkv_plan_dcp(q, kv, bl, causal, S, a, b, c)
        ref = oracle.dcp_select(q, kv, bl, causal, S, a, b, c)
        assert (got[0], got[1].tolist(), got[3]) == (ref[0], ref[1], ref[3]), case


def test_dcp_extremes(k):
    """No reduction cost: the least makespan wins; prohibitive reduction cost: one shard."""
    w = wl.WORKLOADS["varlen"]
    q, kv = wl.lengths(w)
    costs = oracle.block_costs(q, kv, w.block_len, w.causal)
    s, _, load, t = k.splitkv_plan_dcp(q, kv, w.block_len, w.causal, w.n_shards, 1.0, 0.0)
    best = min(max(oracle.lpt_assign(costs, m)[1]) for m in range(1, w.n_shards + 1))
    assert t == best and max(load) == best
    s1, sob1, _, _ = k.splitkv_plan_dcp(q, kv, w.block_len, w.causal, w.n_shards, 1.0, 1e12)
    assert s1 == 1 and set(sob1.tolist()) == {0}


def test_fused_launch_count_by_kernel(k):
    """splitkv_attn_fused merges inside the launch for the decode and tensor-core kernels."""
    BF, F32 = k.SPLITKV_BF16, k.SPLITKV_F32
    assert k.splitkv_fused_launches(32, 8, 128, 256, 1, 128, BF) == 1          # decode kernel
    assert k.splitkv_fused_launches(32, 8, 128, 256, 1, 5000, BF) == 2         # decode, too many items
    assert k.splitkv_fused_launches(32, 8, 128, 1024, 512, 64, BF) == 1        # tensor cores
    assert k.splitkv_fused_launches(4, 4, 64, 128, 16, 4, F32) == 2            # CUDA-core kernel
    assert k.splitkv_fused_launches(32, 8, 128, 1024, 512, 64, BF, k.KERNEL_SIMT) == 2
    with pytest.raises(k.SplitKVError):
        k.splitkv_fused_launches(30, 8, 128, 1024, 512, 64, BF)


def _tail_expected(k, q, kv, w, costs, sob, upi, slots, pieces):
    """The tail cut written out from the plain work lists: the last ceil((units mod slots) /
    upi) items in launch order, each cut into min(pieces, blocks) runs of consecutive blocks."""
    plain = _decode_work(k.splitkv_build_work(q, kv, w.block_len, costs, sob, w.n_shards)[0])
    runs = []
    for it in plain["items"]:
        shard, seq, off, cnt = it[:4].tolist()
        runs.append((shard, seq, plain["blocks"][off: off + cnt].tolist()))
    n0 = len(runs)
    units = n0 * upi
    if upi <= 0 or slots <= 0 or pieces <= 1 or units <= slots or units % slots == 0:
        return runs
    tail = -(-(units % slots) // upi)
    out = runs[: n0 - tail]
    for shard, seq, blks in runs[n0 - tail:]:
        p = min(pieces, len(blks))
        at = 0
        for j in range(p):
            c = len(blks) // p + (1 if j < len(blks) % p else 0)
            out.append((shard, seq, blks[at: at + c]))
            at += c
    return out


@pytest.mark.parametrize("name,upi,slots,pieces", [("decode", 8, 304, 4), ("decode", 8, 304, 3), ("decode", 8, 1000, 4),
                                                   ("decode", 8, 256, 4), ("decode", 8, 2048, 4), ("varlen", 40, 152, 4),
                                                   ("shortq", 64, 152, 8), ("specdec", 8, 152, 2), ("tiny", 4, 3, 4),
                                                   ("decode", 8, 304, 1), ("decode", 8, 304, 100)])
def test_tail_work_lists(k, name, upi, slots, pieces):
    """splitkv_build_work_tail: the items of the last partial wave are cut into runs of
    consecutive blocks and launched last, the rest is the plain descriptor; every (shard,
    sequence) pair still holds exactly the plan's key set and the partial rows stay contiguous."""
    w = wl.WORKLOADS[name]
    q, kv = wl.lengths(w)
    costs = k.splitkv_block_costs(q, kv, w.block_len, w.causal)
    sob, _ = k.splitkv_plan(costs, w.n_shards)
    work, n_items, part_rows = k.splitkv_build_work_tail(q, kv, w.block_len, costs, sob, w.n_shards, upi, slots,
                                                         pieces)
    d = _decode_work(work)
    want = _tail_expected(k, q, kv, w, costs, sob, upi, slots, pieces)
    assert n_items == d["n_items"] == len(want)
    rows = 0
    gbase = np.cumsum([0] + [-(-n // w.block_len) for n in kv])
    got = {}
    for it, (shard, seq, blks) in zip(d["items"], want):
        s_, b_, off, cnt, prow, iq, ikv, icu, clo, chi = it.tolist()[:10]
        assert (iq, ikv, icu) == (q[seq], kv[seq], sum(q[:seq]))
        assert (s_, b_) == (shard, seq) and d["blocks"][off: off + cnt].tolist() == blks
        assert prow == rows
        rows += q[seq]
        assert ((clo & 0xFFFFFFFF) | (chi << 32)) == sum(costs[gbase[seq] + j] for j in blks)
        got.setdefault((shard, seq), []).extend(blks)
    assert rows == part_rows
    sets = oracle.shard_key_sets(sob.tolist(), kv, w.block_len, w.n_shards)
    for (shard, seq), blks in got.items():
        assert sorted(blks) == sets[shard][seq]
    assert sum(len(v) for s in sets for v in s) == sum(len(v) for v in got.values())
    for b in range(len(q)):
        p0, p1 = d["seqs"][b, 3], d["seqs"][b + 1, 3]
        its = d["seq_items"][p0:p1].tolist()
        assert sorted(its) == sorted(i for i in range(n_items) if d["items"][i, 1] == b)
        assert [d["items"][i, 0] for i in its] == sorted(d["items"][i, 0] for i in its)


def test_tail_cut_rejects_negative_arguments(k):
    w = wl.WORKLOADS["decode"]
    q, kv = wl.lengths(w)
    costs = k.splitkv_block_costs(q, kv, w.block_len, w.causal)
    sob, _ = k.splitkv_plan(costs, w.n_shards)
    for bad in ((-1, 304, 4), (8, -1, 4), (8, 304, -2)):
        with pytest.raises(k.SplitKVError):
            k.splitkv_build_work_tail(q, kv, w.block_len, costs, sob, w.n_shards, *bad)


def _plan_batch(k, q, kv, bl, causal, S, words=None, cut=(0, 0, 0)):
    n = k.splitkv_num_blocks(kv, bl)
    cost, sob, load = np.zeros(n, np.int64), np.zeros(n, np.int32), np.zeros(S, np.int64)
    work = np.zeros(words if words is not None else k.splitkv_work_words(n, len(q)), np.int32)
    upi, slots, pieces = cut
    n_items, part_rows = k.splitkv_plan_batch(q, kv, bl, causal, S, cost, sob, load, work, units_per_item=upi,
                                              slots=slots, pieces=pieces)
    return cost, sob, load, work, n_items, part_rows


def test_plan_batch_is_the_three_calls(k):
    """The one-call plan gives the oracle's costs and LPT plan and the same descriptor as
    splitkv_build_work (splitkv_build_work_tail with a tail cut), on every workload and on fuzz
    cases."""
    rng = random.Random(77)
    cases = [(*wl.lengths(w), w.block_len, w.causal, w.n_shards) for w in wl.WORKLOADS.values()]
    for _ in range(300):
        B = rng.randint(1, 5)
        q = [rng.randint(0, 40) for _ in range(B)]
        kv = [qq + rng.randint(0 if qq else 1, 300) for qq in q]
        cases.append((q, kv, rng.choice([1, 4, 16, 64]), rng.random() < 0.6, rng.randint(1, 9)))
    for q, kv, bl, causal, S in cases:
        cost, sob, load, work, n_items, part_rows = _plan_batch(k, q, kv, bl, causal, S)
        ref_cost = oracle.block_costs(q, kv, bl, causal)
        ref_sob, ref_load = oracle.lpt_assign(ref_cost, S)
        assert cost.tolist() == ref_cost and sob.tolist() == ref_sob and load.tolist() == ref_load
        ref_work, ref_items, ref_rows = k.splitkv_build_work(q, kv, bl, cost, sob, S)
        assert np.array_equal(work, ref_work) and (n_items, part_rows) == (ref_items, ref_rows)
        cut = (rng.randint(1, 8), rng.randint(1, 40), rng.randint(2, 5))
        *_, work, n_items, part_rows = _plan_batch(k, q, kv, bl, causal, S, cut=cut)
        ref_work, ref_items, ref_rows = k.splitkv_build_work_tail(q, kv, bl, cost, sob, S, *cut)
        assert np.array_equal(work, ref_work) and (n_items, part_rows) == (ref_items, ref_rows)


def test_plan_batch_errors(k):
    w = wl.WORKLOADS["shortq"]
    q, kv = wl.lengths(w)
    n = k.splitkv_num_blocks(kv, w.block_len)
    words = k.splitkv_work_words(n, len(q))
    with pytest.raises(k.SplitKVError) as e:
        _plan_batch(k, q, kv, w.block_len, w.causal, w.n_shards, words=words - 1)
    assert e.value.status == -4
    cost, sob, load = np.zeros(n + 1, np.int64), np.zeros(n + 1, np.int32), np.zeros(w.n_shards, np.int64)
    with pytest.raises(k.SplitKVError):  # n_blocks does not match the batch
        k.splitkv_plan_batch(q, kv, w.block_len, w.causal, w.n_shards, cost, sob, load, np.zeros(words + 8, np.int32))
    with pytest.raises(TypeError):  # outputs of the wrong type are refused before the call
        k.splitkv_plan_batch(q, kv, w.block_len, w.causal, w.n_shards, cost[:n].astype(np.int32), sob[:n], load,
                             np.zeros(words, np.int32))
    with pytest.raises(k.SplitKVError):
        k.splitkv_plan_batch(q, kv, w.block_len, w.causal, 0, cost[:n], sob[:n], load[:0], np.zeros(words, np.int32))
