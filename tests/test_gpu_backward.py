"""GPU parity of the split-KV backward pass against the fp64 oracle.

The CUDA path computes per-shard dK / dV and partial dQ over the LPT plan's work
items, then sums the partial dQ; the oracle differentiates the unsharded
attention.  Gradients are compared element by element.  The bf16 d=128 cases run
the tensor-core kernels (bf16 P and dS feed the MMAs); fp32 and d=64 the CUDA-core
kernel."""

import pytest
import torch

import oracle
from context_long_attention_lpt_gb300 import splitkv as K
from context_long_attention_lpt_gb300 import workloads as wl
from tests.parity_helpers import run_cuda
from tests.test_gpu_parity import SMALL

pytestmark = pytest.mark.gpu

TOL = {"f32": 2e-4, "bf16": 2e-2}


@pytest.mark.parametrize("name", ["tiny", "decode_small", "shortq_small", "varlen_small", "noncausal_multi_q",
                                  "bf16_d64", "largest_small", "causal_empty_units"])
def test_backward_matches_oracle(name):
    w = SMALL[name]
    inp, run, out, lse = run_cuda(w)
    g = torch.Generator(device="cuda").manual_seed(11)
    dout = torch.randn(out.shape, generator=g, device="cuda", dtype=torch.float32).to(out.dtype)
    dq, dk, dv = run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)
    torch.cuda.synchronize()
    assert K.splitkv_device_status() == 0
    args = (inp.q.cpu(), inp.k_pool.cpu(), inp.v_pool.cpu(), inp.block_table.cpu(), inp.q_len, inp.kv_len,
            w.block_len, w.causal, w.scale)
    o_ref, l_ref = oracle.attention(*args)
    do64 = dout.cpu().double()
    rdq, rdk, rdv = oracle.attention_backward(*args, do=do64, lse=l_ref, dlt=oracle.delta(o_ref, do64))
    # only key slots that hold sequence keys carry gradients
    valid = torch.zeros(inp.k_pool.shape[:2], dtype=torch.bool)
    table = inp.block_table.cpu()
    for b, n in enumerate(inp.kv_len):
        for j in range(-(-n // w.block_len)):
            valid[int(table[b, j]), : min(w.block_len, n - j * w.block_len)] = True
    tol = TOL[w.dtype]
    for nm, got, ref in (("dq", dq.cpu().double(), rdq), ("dk", dk.cpu().double()[valid], rdk[valid]),
                         ("dv", dv.cpu().double()[valid], rdv[valid])):
        err = (got - ref).abs().max().item()
        assert err <= tol, f"{name} {nm}: max err {err:.3e} > {tol}"


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
    args = (inp.q.cpu(), inp.k_pool.cpu(), inp.v_pool.cpu(), inp.block_table.cpu(), inp.q_len, inp.kv_len,
            w.block_len, w.causal, w.scale)
    o_ref, l_ref = oracle.attention(*args)
    do64 = dout.cpu().double()
    rdq, rdk, rdv = oracle.attention_backward(*args, do=do64, lse=l_ref, dlt=oracle.delta(o_ref, do64))
    valid = torch.zeros(inp.k_pool.shape[:2], dtype=torch.bool)
    table = inp.block_table.cpu()
    for b, n in enumerate(inp.kv_len):
        for j in range(-(-n // w.block_len)):
            valid[int(table[b, j]), : min(w.block_len, n - j * w.block_len)] = True
    for nm, got, ref in (("dq", dq.cpu().double(), rdq), ("dk", dk.cpu().double()[valid], rdk[valid]),
                         ("dv", dv.cpu().double()[valid], rdv[valid])):
        err = (got - ref).abs().max().item()
        assert err <= TOL[w.dtype], f"{nm}: max err {err:.3e}"
    # the sequence without queries has no gradient on its keys
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


@pytest.mark.parametrize("name", ["shortq", "largest", "decode"])
def test_backward_full_size_sampled(name):
    """Full-size workloads: sampled dQ rows and sampled dK / dV keys against the oracle,
    which computes each from its own forward (L, D) over all keys."""
    import random

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
                   for _ in range(6)})
    ref_dq = oracle.backward_rows(*args, rows=rows)
    cu = [0]
    for n in inp.q_len:
        cu.append(cu[-1] + n)
    got_dq = torch.stack([dq[cu[b] + t, h].cpu().double() for b, t, h in rows])
    assert (got_dq - ref_dq).abs().max().item() <= TOL[w.dtype]
    b0 = 0
    kv = inp.kv_len[b0]
    keys = [(b0, kvh, p) for kvh in (0, w.Hkv - 1) for p in (0, kv - 1, rng.randrange(kv), rng.randrange(kv))]
    ref_dk, ref_dv = oracle.backward_keys(*args, keys=keys)
    for i, (b, kvh, p) in enumerate(keys):
        phys = int(tc[b, p // w.block_len])
        off = p % w.block_len
        assert (dk[phys, off, kvh].cpu().double() - ref_dk[i]).abs().max().item() <= TOL[w.dtype], ("dk", keys[i])
        assert (dv[phys, off, kvh].cpu().double() - ref_dv[i]).abs().max().item() <= TOL[w.dtype], ("dv", keys[i])
