"""GPU parity of the split-KV backward pass against the fp64 oracle.

The CUDA path computes per-shard dK / dV and partial dQ over the LPT plan's work
items, then sums the partial dQ; the oracle differentiates the unsharded
attention.  Each gradient tensor must meet the scale-relative criterion of
``parity_helpers.grad_close`` (normwise and max-wise error relative to the
tensor's own size): the gradients here are far below 1, so an absolute bound
would accept a kernel that wrote zeros.  The bf16 d=128 cases run the
tensor-core kernels (bf16 P and dS feed the MMAs); fp32 and d=64 the CUDA-core
kernel."""

import random

import pytest
import torch

import oracle
from context_long_attention_lpt_gb300 import splitkv as K
from context_long_attention_lpt_gb300 import workloads as wl
from tests.parity_helpers import SMALL, assert_grad_close, run_cuda

pytestmark = pytest.mark.gpu


def _valid_key_slots(inp, w):
    """Pool slots that hold a sequence key: only they carry gradients."""
    valid = torch.zeros(inp.k_pool.shape[:2], dtype=torch.bool)
    table = inp.block_table.cpu()
    for b, n in enumerate(inp.kv_len):
        for j in range(-(-n // w.block_len)):
            valid[int(table[b, j]), : min(w.block_len, n - j * w.block_len)] = True
    return valid


def _check_every_element(w, inp, out, lse, dout, dq, dk, dv, what):
    args = (inp.q.cpu(), inp.k_pool.cpu(), inp.v_pool.cpu(), inp.block_table.cpu(), inp.q_len, inp.kv_len,
            w.block_len, w.causal, w.scale)
    o_ref, l_ref = oracle.attention(*args)
    do64 = dout.cpu().double()
    rdq, rdk, rdv = oracle.attention_backward(*args, do=do64, lse=l_ref, dlt=oracle.delta(o_ref, do64))
    valid = _valid_key_slots(inp, w)
    for nm, got, ref in (("dq", dq.cpu(), rdq), ("dk", dk.cpu()[valid], rdk[valid]),
                         ("dv", dv.cpu()[valid], rdv[valid])):
        assert_grad_close(w.dtype, got, ref, f"{what} {nm}")


@pytest.mark.parametrize("name", ["tiny", "decode_small", "shortq_small", "varlen_small", "noncausal_multi_q",
                                  "bf16_d64", "largest_small", "causal_empty_units", "many_key_tiles",
                                  "gqa16_tc", "gqa2_tc"])
def test_backward_matches_oracle(name):
    w = SMALL[name]
    inp, run, out, lse = run_cuda(w)
    g = torch.Generator(device="cuda").manual_seed(11)
    dout = torch.randn(out.shape, generator=g, device="cuda", dtype=torch.float32).to(out.dtype)
    dq, dk, dv = run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)
    torch.cuda.synchronize()
    assert K.splitkv_device_status() == 0
    _check_every_element(w, inp, out, lse, dout, dq, dk, dv, name)


def test_backward_ragged_batch_with_empty_and_single_key_sequences():
    """A sequence with no queries (no gradient anywhere), one with a single key, one over
    several tiles and one short block, through the tensor-core backward."""
    w = wl.custom("varlen", B=4, block_len=128, n_shards=5)
    lens = ([0, 1, 130, 7], [5, 1, 400, 7])
    inp, run, out, lse = run_cuda(w, lens=lens)
    assert K.splitkv_backward_kernel(w.Hq, w.Hkv, w.d, w.block_len, K.SPLITKV_BF16) == K.KERNEL_TC
    g = torch.Generator(device="cuda").manual_seed(5)
    dout = torch.randn(out.shape, generator=g, device="cuda", dtype=torch.float32).to(out.dtype)
    dq, dk, dv = run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)
    torch.cuda.synchronize()
    assert K.splitkv_device_status() == 0
    _check_every_element(w, inp, out, lse, dout, dq, dk, dv, "ragged")
    # the sequence without queries has no gradient on its keys
    table = inp.block_table.cpu()
    b0 = [int(table[0, j]) for j in range(-(-inp.kv_len[0] // w.block_len))]
    assert (dk[b0, : inp.kv_len[0]] == 0).all() and (dv[b0, : inp.kv_len[0]] == 0).all()


def test_backward_is_deterministic_in_dk_dv_and_close_in_dq():
    w = SMALL["varlen_small"]
    inp, run, out, lse = run_cuda(w)
    dout = torch.ones_like(out)
    a = [x.clone() for x in run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)]
    b = run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)
    torch.cuda.synchronize()
    assert torch.equal(a[1], b[1]) and torch.equal(a[2], b[2])  # dK / dV: no atomics
    assert (a[0] - b[0]).abs().max().item() < 1e-4  # dQ: fp32 atomics on the CUDA-core path


@pytest.mark.parametrize("name", ["shortq", "largest", "varlen", "decode"])
def test_backward_full_size_sampled(name):
    """Full-size workloads: sampled dQ rows and sampled dK / dV keys against the oracle,
    which computes each from its own forward (L, D) over all keys.  The samples of each
    gradient are checked together with the scale-relative criterion."""
    w = wl.WORKLOADS[name]
    inp, run, out, lse = run_cuda(w)
    g = torch.Generator(device="cuda").manual_seed(21)
    dout = torch.randn(out.shape, generator=g, device="cuda", dtype=torch.float32).to(out.dtype)
    dq, dk, dv = run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)
    torch.cuda.synchronize()
    assert K.splitkv_device_status() == 0
    rng = random.Random(3)
    qc, kc, vc, tc, doc = inp.q.cpu(), inp.k_pool.cpu(), inp.v_pool.cpu(), inp.block_table.cpu(), dout.cpu()
    args = (qc, kc, vc, tc, inp.q_len, inp.kv_len, w.block_len, w.causal, w.scale, doc)
    rows = sorted({(b, rng.randrange(inp.q_len[b]), rng.randrange(w.Hq)) for b in rng.sample(range(w.B), min(w.B, 3))
                   for _ in range(8)})
    ref_dq = oracle.backward_rows(*args, rows=rows)
    cu = [0]
    for n in inp.q_len:
        cu.append(cu[-1] + n)
    got_dq = torch.stack([dq[cu[b] + t, h].cpu() for b, t, h in rows])
    assert_grad_close(w.dtype, got_dq, ref_dq, f"{name} sampled dq rows")
    # keys of the sequence with the shortest context (the oracle's cost grows with q_len x kv_len)
    b0 = min(range(w.B), key=lambda b: (inp.kv_len[b], b))
    kv = inp.kv_len[b0]
    keys = [(b0, kvh, p) for kvh in (0, w.Hkv - 1)
            for p in (0, kv - 1, rng.randrange(kv), rng.randrange(kv), rng.randrange(kv))]
    ref_dk, ref_dv = oracle.backward_keys(*args, keys=keys)
    got_dk = torch.stack([dk[int(tc[b, p // w.block_len]), p % w.block_len, kvh].cpu() for b, kvh, p in keys])
    got_dv = torch.stack([dv[int(tc[b, p // w.block_len]), p % w.block_len, kvh].cpu() for b, kvh, p in keys])
    assert_grad_close(w.dtype, got_dk, ref_dk, f"{name} sampled dk keys")
    assert_grad_close(w.dtype, got_dv, ref_dv, f"{name} sampled dv keys")


REPEAT_CASES = {name: wl.WORKLOADS[name] for name in ("decode", "shortq", "largest", "varlen")}
# three 64-row tiles per sequence and ~49 key tiles per dK/dV CTA: K and V are reloaded
# every third row tile while the next loads are in flight
REPEAT_CASES["reload_kv"] = wl.custom("shortq", q_len=48, context=200000, block_len=1024, n_shards=2)


@pytest.mark.parametrize("name", list(REPEAT_CASES))
def test_tensor_core_backward_is_bitwise_repeatable_at_full_size(name):
    """The tensor-core backward has no atomics: repeated runs give the same bits.  A hand-off
    race between the elementwise warps and the MMA lane, or a K/V reload over a tile still in
    use, would show up as differing runs."""
    w = REPEAT_CASES[name]
    assert K.splitkv_backward_kernel(w.Hq, w.Hkv, w.d, w.block_len, K.SPLITKV_BF16) == K.KERNEL_TC
    inp, run, out, lse = run_cuda(w)
    g = torch.Generator(device="cuda").manual_seed(31)
    dout = torch.randn(out.shape, generator=g, device="cuda", dtype=torch.float32).to(out.dtype)
    first = [x.clone() for x in run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)]
    for _ in range(4):
        again = run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)
        torch.cuda.synchronize()
        for a_, b_ in zip(first, again):
            assert torch.equal(a_, b_)
    assert K.splitkv_device_status() == 0
