"""splitkv_attention_noalloc: the device path with no allocation, against the caller-buffer path.

Callers that cannot allocate device memory (a plugin inside a host that owns all
device memory, a loop that must not stall or fail on an allocation) get one entry
point whose intermediate buffers live in a fixed array inside the library.  Its
results must equal those of splitkv_attn_partial + splitkv_merge with caller
buffers, call after call, although every call reuses the same array.
"""

import pytest
import torch

from context_long_attention_lpt_gb300 import splitkv as K
from context_long_attention_lpt_gb300 import workloads as wl
from context_long_attention_lpt_gb300.runner import SplitKVAttention
from tests.parity_helpers import TOL_L, TOL_O

pytestmark = pytest.mark.gpu

CASES = [
    wl.custom("shortq", q_len=77, context=2500, block_len=256, n_shards=7),  # tensor-core kernel
    wl.custom("decode", B=4, context=5000, n_shards=6),                      # decode kernel
]


def _both_paths(w):
    inp = wl.make_inputs(w, device="cuda", poison_tail=True)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype)
    ref_out, ref_lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    out = torch.full_like(ref_out, float("nan"))
    lse = torch.full_like(ref_lse, float("nan"))
    K.splitkv_attention_noalloc(inp.q, inp.k_pool, inp.v_pool, inp.block_table, run.work_host, run.n_items,
                                run.B, run.total_q, run.max_q_len, w.block_len, w.scale, w.causal,
                                run.part_rows, out, lse)
    torch.cuda.synchronize()
    return w, ref_out, ref_lse, out, lse


def test_noalloc_equals_caller_buffer_path_on_two_calls_in_a_row():
    assert torch.cuda.is_available()
    for w in CASES:  # second call reuses the array the first one left behind
        w, ref_out, ref_lse, out, lse = _both_paths(w)
        assert torch.isfinite(out.float()).all() and torch.isfinite(lse).all()
        assert (out.float() - ref_out.float()).abs().max().item() <= TOL_O[w.dtype]
        assert (lse - ref_lse).abs().max().item() <= TOL_L
        # same plan, same kernels, same arithmetic: the results are identical bit for bit
        assert torch.equal(out, ref_out) and torch.equal(lse, ref_lse)


def test_noalloc_repeated_calls_take_no_device_memory():
    """After the first call on the device, further calls leave torch's allocator and the
    device's free memory where they were."""
    w = CASES[0]
    inp = wl.make_inputs(w, device="cuda")
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype)
    out = torch.empty((run.total_q, w.Hq, w.d), dtype=inp.q.dtype, device="cuda")
    lse = torch.empty((run.total_q, w.Hq), dtype=torch.float32, device="cuda")

    def call():
        K.splitkv_attention_noalloc(inp.q, inp.k_pool, inp.v_pool, inp.block_table, run.work_host, run.n_items,
                                    run.B, run.total_q, run.max_q_len, w.block_len, w.scale, w.causal,
                                    run.part_rows, out, lse)

    call()
    torch.cuda.synchronize()
    free0, allocated0, reserved0 = torch.cuda.mem_get_info()[0], torch.cuda.memory_allocated(), \
        torch.cuda.memory_reserved()
    for _ in range(5):
        call()
    torch.cuda.synchronize()
    assert torch.cuda.memory_allocated() == allocated0
    assert torch.cuda.memory_reserved() == reserved0
    assert torch.cuda.mem_get_info()[0] == free0


def test_noalloc_rejects_problems_larger_than_its_array():
    w = wl.custom("shortq", q_len=512, context=131072, n_shards=64)  # 64 x 512 partial rows: > 64 MiB
    q_len, kv_len = wl.lengths(w)
    costs = K.splitkv_block_costs(q_len, kv_len, w.block_len, w.causal)
    sob, _ = K.splitkv_plan(costs, w.n_shards)
    work, n_items, part_rows = K.splitkv_build_work(q_len, kv_len, w.block_len, costs, sob, w.n_shards)
    q = torch.zeros((sum(q_len), w.Hq, w.d), dtype=torch.bfloat16, device="cuda")
    pool = torch.zeros((1, w.block_len, w.Hkv, w.d), dtype=torch.bfloat16, device="cuda")
    table = torch.zeros((1, 1), dtype=torch.int32, device="cuda")
    out = torch.empty_like(q)
    lse = torch.empty((sum(q_len), w.Hq), dtype=torch.float32, device="cuda")
    with pytest.raises(K.SplitKVError) as e:
        K.splitkv_attention_noalloc(q, pool, pool, table, work, n_items, 1, sum(q_len), max(q_len),
                                    w.block_len, w.scale, w.causal, part_rows, out, lse)
    assert e.value.status == -4 and "scratch" in str(e.value)


def test_noalloc_rejects_sizes_that_do_not_match_the_descriptor():
    """part_rows, total_q and max_q_len are checked against the host descriptor before any
    work, so a wrong row count cannot make the kernels write past the fixed array."""
    w = CASES[0]
    inp = wl.make_inputs(w, device="cuda")
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype)
    out = torch.empty((run.total_q, w.Hq, w.d), dtype=inp.q.dtype, device="cuda")
    lse = torch.empty((run.total_q, w.Hq), dtype=torch.float32, device="cuda")
    good = dict(n_items=run.n_items, B=run.B, total_q=run.total_q, max_q_len=run.max_q_len,
                part_rows=run.part_rows)
    for bad in ({"part_rows": run.part_rows - 1}, {"part_rows": run.part_rows + 1}, {"part_rows": 1 << 60},
                {"total_q": run.total_q + 1}, {"max_q_len": run.max_q_len + 1}):
        a = dict(good, **bad)
        with pytest.raises(K.SplitKVError) as e:
            K.splitkv_attention_noalloc(inp.q, inp.k_pool, inp.v_pool, inp.block_table, run.work_host,
                                        a["n_items"], a["B"], a["total_q"], a["max_q_len"], w.block_len, w.scale,
                                        w.causal, a["part_rows"], out, lse)
        assert e.value.status == -1, bad
    torch.cuda.synchronize()
    assert K.splitkv_device_status() == 0
