"""GPU parity: the CUDA path (through the C ABI) against the fp64 CPU oracle.

Small cases compare every output element; the full-size workloads compare
sampled rows the oracle computes one by one.  Every case poisons the K/V slots
past each sequence's end with NaN, so a kernel that reads them fails.
"""

import numpy as np
import pytest
import torch

import oracle
from context_long_attention_lpt_gb300 import splitkv as K
from context_long_attention_lpt_gb300 import workloads as wl
from context_long_attention_lpt_gb300.runner import SplitKVAttention
from tests.parity_helpers import (SMALL, TOL_L, TOL_O, assert_close, compare_rows, full_reference,  # noqa: F401
                                  max_errors, run_cuda, sample_rows)

pytestmark = pytest.mark.gpu



@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    K.lib()


@pytest.mark.parametrize("kernel", [K.KERNEL_AUTO, K.KERNEL_SIMT])
@pytest.mark.parametrize("name", list(SMALL))
def test_small_cases_every_element(name, kernel):
    w = SMALL[name]
    inp, run, out, lse = run_cuda(w, kernel=kernel)
    o_ref, l_ref = full_reference(inp)
    eo, el = max_errors(out, lse, o_ref, l_ref)
    assert_close(w, eo, el, f"{name}/{K.KERNEL_NAMES.get(run.kernel_used())}")
    assert K.splitkv_device_status(clear=True) == 0


@pytest.mark.parametrize("seed", range(6))
def test_tensor_core_few_tile_items(seed):
    """Items of one or two 128-key tiles, partial query tiles and a ragged last block:
    the pipeline's start-up and drain paths of the tensor-core kernel, repeated."""
    rng = np.random.default_rng(seed)
    w = wl.custom("shortq", causal=bool(seed % 2), q_len=int(rng.integers(1, 70)),
                  context=int(rng.integers(200, 1500)), block_len=128, n_shards=int(rng.integers(2, 9)),
                  seed=100 + seed)
    inp, run, out, lse = run_cuda(w, kernel=K.KERNEL_TC)
    eo, el = max_errors(out, lse, *full_reference(inp))
    assert_close(w, eo, el, f"seed {seed}")
    assert K.splitkv_device_status(clear=True) == 0


@pytest.mark.parametrize("kernel", [K.KERNEL_AUTO, K.KERNEL_SIMT])
@pytest.mark.parametrize("name", ["decode_small", "shortq_small", "varlen_small", "tiny", "causal_empty_units"])
def test_partials_match_oracle_partials(name, kernel):
    """Each work item's (O_i, L_i) equals the oracle's partial over the oracle's own shard
    (items uncut, so each item is a whole (shard, sequence) pair)."""
    w = SMALL[name]
    inp, run, _, _ = run_cuda(w, kernel=kernel, tail_pieces=0)
    costs = oracle.block_costs(inp.q_len, inp.kv_len, w.block_len, w.causal)
    sob, _ = oracle.lpt_assign(costs, w.n_shards)
    sets = oracle.shard_key_sets(sob, inp.kv_len, w.block_len, w.n_shards)
    work = run.work_host
    off_items, n_items = work[8], work[2]
    o_part = run.o_part.cpu().double()
    l_part = run.lse_part.cpu().double()
    cu = np.concatenate([[0], np.cumsum(inp.q_len)])
    args = (inp.q.cpu(), inp.k_pool.cpu(), inp.v_pool.cpu(), inp.block_table.cpu(), inp.q_len,
            inp.kv_len, w.block_len, w.causal, w.scale)
    cache = {}
    for i in range(n_items):
        shard, seq, _, _, prow = work[off_items + 12 * i: off_items + 12 * i + 5].tolist()
        if shard not in cache:
            cache[shard] = oracle.partial(*args, key_blocks=sets[shard])
        o_ref, l_ref = cache[shard]
        lq = inp.q_len[seq]
        sl = slice(int(cu[seq]), int(cu[seq]) + lq)
        eo, el = max_errors(o_part[prow: prow + lq], l_part[prow: prow + lq], o_ref[sl], l_ref[sl])
        assert_close(w, eo, el, f"{name} item {i} (shard {shard}, seq {seq})")


@pytest.mark.parametrize("name", list(wl.WORKLOADS))
def test_full_size_workloads_sampled_rows(name):
    """Every workload at full size, auto kernel (what the benchmark runs), sampled rows."""
    w = wl.WORKLOADS[name]
    inp, run, out, lse = run_cuda(w, kernel=K.KERNEL_AUTO)
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    rows = sample_rows(inp, 48 if name != "tiny" else 64, seed=7)
    eo, el = compare_rows(inp, out, lse, rows)
    assert_close(w, eo, el, f"{name}/{K.KERNEL_NAMES.get(run.kernel_used())}")
    assert K.splitkv_device_status() == 0


def test_more_shards_than_blocks():
    w = wl.custom("decode", B=1, context=700, n_shards=9)  # 3 blocks, 6 empty shards
    inp, run, out, lse = run_cuda(w)
    assert (run.shard_load == 0).sum() == 6
    eo, el = max_errors(out, lse, *full_reference(inp))
    assert_close(w, eo, el)


def test_single_shard():
    w = wl.custom("shortq", q_len=33, context=1200, block_len=256, n_shards=1)
    inp, run, out, lse = run_cuda(w)
    assert run.n_items == 1
    eo, el = max_errors(out, lse, *full_reference(inp))
    assert_close(w, eo, el)


@pytest.mark.parametrize("kernel", [K.KERNEL_AUTO, K.KERNEL_SIMT])
def test_ragged_batch_with_empty_and_single_key_sequences(kernel):
    w = wl.custom("varlen", B=4, block_len=128, n_shards=5)
    lens = ([0, 1, 130, 7], [5, 1, 400, 7])  # no queries; one key; several tiles; one short block
    inp, run, out, lse = run_cuda(w, kernel=kernel, lens=lens)
    eo, el = max_errors(out, lse, *full_reference(inp))
    assert_close(w, eo, el)


def test_runs_are_deterministic():
    w = SMALL["varlen_small"]
    _, _, out1, lse1 = run_cuda(w)
    _, _, out2, lse2 = run_cuda(w)
    assert torch.equal(out1, out2) and torch.equal(lse1, lse2)


def test_out_of_range_block_is_reported_not_read():
    w = wl.custom("decode", B=2, context=1000, n_shards=3)
    inp = wl.make_inputs(w, device="cuda")
    K.splitkv_device_status(clear=True)
    bad = inp.block_table.clone()
    bad[1, 2] = inp.n_pool_blocks + 5
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype)
    run(inp.q, inp.k_pool, inp.v_pool, bad, w.scale)
    torch.cuda.synchronize()
    assert K.splitkv_device_status(clear=True) & 1
    assert K.splitkv_device_status() == 0
    out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    torch.cuda.synchronize()
    eo, el = max_errors(out, lse, *full_reference(inp))
    assert_close(w, eo, el)


@pytest.mark.parametrize("name,kernel", [("decode_small", K.KERNEL_AUTO), ("decode_small", K.KERNEL_SIMT),
                                         ("varlen_small", K.KERNEL_AUTO), ("shortq_small", K.KERNEL_AUTO),
                                         ("tiny", K.KERNEL_AUTO)])
def test_descriptor_of_another_launch_is_reported_not_used(name, kernel):
    """A launch told fewer items or sequences than its descriptor was built for finds the rows
    where its own arguments place them, sees the header disagree, writes nothing and sets bit 3
    of the status word (forward and backward kernels)."""
    w = SMALL[name]
    inp = wl.make_inputs(w, device="cuda")
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, kernel=kernel, tail_pieces=0)
    out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    torch.cuda.synchronize()
    assert K.splitkv_device_status(clear=True) == 0 and run.n_items >= 2
    dout = torch.ones_like(out)
    delta = torch.zeros((run.total_q, w.Hq), dtype=torch.float32, device="cuda")
    cases = [(run.n_items - 1, run.B)] + ([(run.n_items, run.B - 1)] if run.B > 1 else [])
    for n_items, B in cases:
        run._o_part.fill_(7.0)
        K.splitkv_attn_partial(inp.q, inp.k_pool, inp.v_pool, inp.block_table, run.work_device, n_items, B,
                               run.total_q, run.max_q_len, w.block_len, w.scale, w.causal, run._o_part,
                               run._lse_part, kernel=kernel)
        torch.cuda.synchronize()
        assert K.splitkv_device_status(clear=True) == 8, (n_items, B)
        assert bool((run._o_part == 7.0).all())
        dq_part = torch.full((max(run.part_rows, 1), w.Hq, w.d), 7.0, dtype=torch.float32, device="cuda")
        dk = torch.full(tuple(inp.k_pool.shape), 7.0, dtype=torch.float32, device="cuda")
        dv = torch.full(tuple(inp.v_pool.shape), 7.0, dtype=torch.float32, device="cuda")
        K.splitkv_attn_backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, run.work_device, n_items, B,
                                run.total_q, run.max_q_len, w.block_len, w.scale, w.causal, dout, lse, delta,
                                dq_part, dk, dv)
        torch.cuda.synchronize()
        assert K.splitkv_device_status(clear=True) == 8, (n_items, B)
        assert bool((dk == 7.0).all()) and bool((dv == 7.0).all())
        # the CUDA-core backward clears the partial dQ rows before its atomic adds
        code = K.SPLITKV_F32 if w.dtype == "f32" else K.SPLITKV_BF16
        tc = K.splitkv_backward_kernel(w.Hq, w.Hkv, w.d, w.block_len, code) == K.KERNEL_TC
        assert bool((dq_part == (7.0 if tc else 0.0)).all())


def test_bad_arguments_raise_before_launch():
    w = SMALL["decode_small"]
    inp = wl.make_inputs(w, device="cuda")
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype)
    with pytest.raises(K.SplitKVError):
        K.splitkv_attn_partial(inp.q, inp.k_pool, inp.v_pool, inp.block_table, run.work_device,
                               run.n_items, run.B, run.total_q, run.max_q_len, w.block_len, float("nan"),
                               w.causal, run._o_part, run._lse_part)
    with pytest.raises(K.SplitKVError):  # tensor-core kernel does not take block_len % 128 != 0
        w2 = wl.custom("shortq", q_len=40, context=1000, block_len=200, n_shards=2)
        run_cuda(w2, kernel=K.KERNEL_TC)


@pytest.mark.parametrize("name", ["decode_small", "decode_gqa8", "shortq_small", "varlen_small", "largest_small",
                                  "causal_empty_units", "tiny"])
def test_fused_single_launch_matches_oracle(name):
    """splitkv_attn_fused: the decode and tensor-core kernels merge in their own launch (the
    last CTA per group); the CUDA-core kernel falls back to two launches.  Two calls in a row:
    the tickets return to zero."""
    w = SMALL[name]
    inp = wl.make_inputs(w, device="cuda", poison_tail=True)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, fused=True)
    o_ref, l_ref = full_reference(inp)
    for _ in range(2):
        out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
        torch.cuda.synchronize()
        eo, el = max_errors(out, lse, o_ref, l_ref)
        assert_close(w, eo, el, f"fused {name}")
        assert int(run.tickets.abs().sum()) == 0
    assert K.splitkv_device_status() == 0


def test_fused_decode_full_size_and_ragged():
    w = wl.WORKLOADS["decode"]
    inp = wl.make_inputs(w, device="cuda")
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, fused=True)
    out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    torch.cuda.synchronize()
    eo, el = compare_rows(inp, out, lse, sample_rows(inp, 64, seed=3))
    assert_close(w, eo, el, "fused decode full size")
    # ragged batch with an empty sequence and a single-key sequence
    w2 = wl.custom("decode", B=4, n_shards=5)
    lens = ([1, 0, 1, 1], [1, 0, 777, 300])
    inp2 = wl.make_inputs(w2, device="cuda", poison_tail=True, lens=lens)
    run2 = SplitKVAttention(inp2.q_len, inp2.kv_len, w2.block_len, w2.causal, w2.n_shards, w2.Hq, w2.Hkv,
                            w2.d, inp2.q.dtype, fused=True)
    out2, lse2 = run2(inp2.q, inp2.k_pool, inp2.v_pool, inp2.block_table, w2.scale)
    torch.cuda.synchronize()
    eo, el = max_errors(out2, lse2, *full_reference(inp2))
    assert_close(w2, eo, el, "fused ragged")
    assert int(run2.tickets.abs().sum()) == 0


@pytest.mark.parametrize("name,beta,gamma", [("varlen_small", 50.0, 0.0), ("decode_small", 1e9, 0.0),
                                             ("shortq_small", 3.0, 0.0), ("varlen_small", 40.0, 0.5)])
def test_dcp_plan_through_the_kernels(name, beta, gamma):
    """The split-selection planner's plan (fewer shards than offered) runs through the same kernels."""
    w = SMALL[name]
    inp = wl.make_inputs(w, device="cuda", poison_tail=True)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, planner="dcp", dcp_alpha=1.0, dcp_beta=beta, dcp_gamma=gamma)
    ref = oracle.dcp_select(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, 1.0, beta, gamma)
    assert run.n_shards_used == ref[0] and run.shard_of_block.tolist() == ref[1]
    out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    torch.cuda.synchronize()
    eo, el = max_errors(out, lse, *full_reference(inp))
    assert_close(w, eo, el, f"dcp {name}")


def test_runner_on_a_side_stream():
    """Plans uploaded on one stream and device calls on another: the runner orders the
    work upload before the calls and the next upload after them."""
    w = SMALL["shortq_small"]
    inp = wl.make_inputs(w, device="cuda", poison_tail=True)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, device="cuda")
    side = torch.cuda.Stream()
    o_ref, l_ref = full_reference(inp)
    for plan_stream in (side, None):  # upload on the side stream, then on the current one
        for _ in range(3):
            run.plan(stream=plan_stream)
            with torch.cuda.stream(side):
                out = torch.empty((run.total_q, w.Hq, w.d), dtype=inp.q.dtype, device="cuda")
                lse = torch.empty((run.total_q, w.Hq), dtype=torch.float32, device="cuda")
            run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, stream=side)
        side.synchronize()
        eo, el = max_errors(out, lse, o_ref, l_ref)
        assert_close(w, eo, el, f"side stream, plan on {'side' if plan_stream else 'current'}")
    dq, dk, dv = run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse,
                              torch.ones_like(out), stream=side)
    side.synchronize()
    assert torch.isfinite(dq).all()
    assert K.splitkv_device_status(clear=True) == 0


@pytest.mark.parametrize("name", ["decode_small", "shortq_small"])
def test_next_plan_uploads_while_the_previous_batch_runs(name):
    """Each plan goes to a copy stream into the descriptor buffer the running batch does not
    read; plans alternate between two different cuts (different item counts and partial
    rows), so a batch that read the other buffer, or a buffer still being written, fails."""
    w = SMALL[name]
    inp = wl.make_inputs(w, device="cuda", poison_tail=True)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, device="cuda", tail_pieces=0)
    up = torch.cuda.Stream()
    o_ref, l_ref = full_reference(inp)
    results = []
    for i in range(8):
        run.item_blocks = 1 if i % 2 else 0
        run.plan(stream=up)
        results.append((run.n_items,) + run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale))
    torch.cuda.synchronize()
    assert len({r[0] for r in results}) == 2
    for n_items, out, lse in results:
        eo, el = max_errors(out, lse, o_ref, l_ref)
        assert_close(w, eo, el, f"{name}, plan of {n_items} items uploaded on a copy stream")
    assert K.splitkv_device_status(clear=True) == 0


@pytest.mark.parametrize("name", ["shortq_small", "varlen_small", "largest_small", "causal_empty_units"])
def test_fused_tensor_core_equals_two_launches_bit_for_bit(name):
    """The tensor-core kernel's in-launch merge computes every row as the merge kernel does."""
    w = SMALL[name]
    inp = wl.make_inputs(w, device="cuda", poison_tail=True)
    two = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype)
    one = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, fused=True)
    assert one.kernel_used() == K.KERNEL_TC and one.fuses_in_one_launch()
    o2, l2 = two(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    o1, l1 = one(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert int(one.tickets.abs().sum()) == 0
    assert K.splitkv_device_status() == 0


@pytest.mark.parametrize("name", ["largest", "varlen"])
def test_fused_tensor_core_full_size(name):
    """Full-size tensor-core workloads through the one-launch path: sampled rows against the
    oracle, tickets back to zero after two calls."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, device="cuda")
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, fused=True)
    assert run.fuses_in_one_launch()
    for _ in range(2):
        out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    torch.cuda.synchronize()
    assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
    eo, el = compare_rows(inp, out, lse, sample_rows(inp, 48, seed=9))
    assert_close(w, eo, el, f"fused {name}")
    assert int(run.tickets.abs().sum()) == 0
    assert K.splitkv_device_status() == 0


@pytest.mark.parametrize("name,max_blocks", [("decode_small", 2), ("decode_gqa8", 1), ("shortq_small", 1),
                                             ("varlen_small", 2)])
@pytest.mark.parametrize("fused", [False, True])
def test_split_items_merge_to_the_unsharded_result(name, max_blocks, fused):
    """Work items cut into runs of a few blocks (more partial rows per sequence) give the
    oracle's unsharded attention, two launches and one."""
    w = SMALL[name]
    inp = wl.make_inputs(w, device="cuda", poison_tail=True)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, fused=fused, item_blocks=max_blocks)
    whole = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                             inp.q.dtype)
    assert run.n_items > whole.n_items
    o_ref, l_ref = full_reference(inp)
    for _ in range(2):
        out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
        torch.cuda.synchronize()
        eo, el = max_errors(out, lse, o_ref, l_ref)
        assert_close(w, eo, el, f"{name} items of {max_blocks} blocks, fused={fused}")
    if fused and run.fuses_in_one_launch():
        assert int(run.tickets.abs().sum()) == 0
    assert K.splitkv_device_status() == 0


def test_split_items_decode_full_size():
    w = wl.WORKLOADS["decode"]
    inp = wl.make_inputs(w, device="cuda")
    for fused in (False, True):
        run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                               inp.q.dtype, fused=fused, item_blocks=2)
        out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
        torch.cuda.synchronize()
        eo, el = compare_rows(inp, out, lse, sample_rows(inp, 64, seed=5))
        assert_close(w, eo, el, f"decode, items of 2 blocks, fused={fused}")
    assert K.splitkv_device_status() == 0


@pytest.mark.parametrize("name,slots", [("decode_small", 7), ("shortq_small", 57), ("varlen_small", 11),
                                        ("specdec_small", 9)])
@pytest.mark.parametrize("fused", [False, True])
def test_tail_cut_merges_to_the_unsharded_result(name, slots, fused):
    """The last partial wave's items cut into pieces (a small resident-CTA count stands in for
    the device's, so that the small cases have a tail) give the oracle's unsharded attention."""
    w = SMALL[name]
    inp = wl.make_inputs(w, device="cuda", poison_tail=True)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, fused=fused, tail_pieces=3, tail_slots=slots)
    whole = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                             inp.q.dtype)
    assert run.n_items > whole.n_items
    o_ref, l_ref = full_reference(inp)
    for _ in range(2):
        out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
        torch.cuda.synchronize()
        eo, el = max_errors(out, lse, o_ref, l_ref)
        assert_close(w, eo, el, f"{name} tail cut over {slots} slots, fused={fused}")
    if fused and run.fuses_in_one_launch():
        assert int(run.tickets.abs().sum()) == 0
    assert K.splitkv_device_status() == 0


@pytest.mark.parametrize("name", ["decode", "specdec"])
def test_tail_cut_full_size_on_the_device_slot_count(name):
    """Full size, with the resident-CTA count of the device: decode launches 1024 units, which
    leaves a partial last wave on any GB300 occupancy of 1 or 2 CTAs per SM."""
    w = wl.WORKLOADS[name]
    inp = wl.make_inputs(w, device="cuda")
    code = K.SPLITKV_BF16
    slots, per_item = K.splitkv_partial_slots(w.Hq, w.Hkv, w.d, w.block_len, max(inp.q_len), code)
    assert slots > 0 and per_item >= w.Hkv
    for fused in (False, True):
        run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                               inp.q.dtype, fused=fused, tail_pieces=4)
        out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
        torch.cuda.synchronize()
        eo, el = compare_rows(inp, out, lse, sample_rows(inp, 64, seed=7))
        assert_close(w, eo, el, f"{name}, tail cut, fused={fused}")
    assert K.splitkv_device_status() == 0
