"""Seeded random shapes through the whole path, every output element against the oracle.

Each seed draws one small problem: batch size, ragged query and context lengths
(sequences without queries included), GQA group size 1-16, head dim 64 or 128,
fp32 or bf16, block length 64-512, causal or not, 1-12 shards, and a launch mode
(two launches or the fused one; whole items, items cut into runs of blocks, or the
last partial wave cut into pieces over a small resident-CTA count).  The kernel is
the library's own choice for the shape, so the draws reach the decode, tensor-core
and CUDA-core kernels and every launch mode of each.  The backward pass runs on
the same draw and must meet the scale-relative gradient criterion.  K/V slots past
each sequence's end hold NaN.
"""

import numpy as np
import pytest
import torch

import oracle
from context_long_attention_lpt_gb300 import splitkv as K
from context_long_attention_lpt_gb300 import workloads as wl
from tests.parity_helpers import assert_close, assert_grad_close, full_reference, max_errors, run_cuda

pytestmark = pytest.mark.gpu

N_SEEDS = 150


@pytest.fixture(scope="module", autouse=True)
def _lib():
    assert torch.cuda.is_available()
    K.lib()


def _draw(seed):
    """(workload, (q_len, kv_len), runner keywords) of one seed."""
    rng = np.random.default_rng(7000 + seed)
    hkv = int(rng.choice([1, 2, 4]))
    g = int(rng.choice([1, 2, 4, 8, 16]))
    dtype = "f32" if rng.random() < 0.1 else "bf16"
    d = 64 if rng.random() < 0.1 else 128
    block_len = int(rng.choice([64, 128, 128, 256, 256, 512]))
    causal = bool(rng.random() < 0.7)
    B = int(rng.integers(1, 6))
    if rng.random() < 0.5:  # decode-like: the same few query tokens per sequence
        q_len = [int(rng.choice([1, 2, 3, 4, 8]))] * B
    else:
        q_len = [int(rng.integers(0, 200)) for _ in range(B)]
        if not any(q_len):
            q_len[0] = 1
    ctx = [int(rng.integers(0, 4000)) for _ in range(B)]
    kv_len = [c + q if causal else max(c, q, 1) for c, q in zip(ctx, q_len)]
    w = wl.Workload(f"fuzz{seed}", B=B, Hq=hkv * g, Hkv=hkv, d=d, block_len=block_len,
                    n_shards=int(rng.integers(1, 13)), causal=causal, dtype=dtype, varlen=True,
                    seed=500 + seed)
    kw = {"fused": bool(rng.random() < 0.35)}
    mode = rng.random()
    if mode < 0.25:
        kw.update(tail_pieces=int(rng.integers(2, 6)), tail_slots=int(rng.integers(1, 24)))
    elif mode < 0.4:
        kw.update(item_blocks=int(rng.integers(1, 4)))
    else:
        kw.update(tail_pieces=0)
    return w, (q_len, kv_len), kw


def _valid_key_slots(inp, w):
    valid = torch.zeros(inp.k_pool.shape[:2], dtype=torch.bool)
    table = inp.block_table.cpu()
    for b, n in enumerate(inp.kv_len):
        for j in range(-(-n // w.block_len)):
            valid[int(table[b, j]), : min(w.block_len, n - j * w.block_len)] = True
    return valid


@pytest.mark.parametrize("seed", range(N_SEEDS))
def test_random_shape_forward_and_backward(seed):
    w, lens, kw = _draw(seed)
    code = K.SPLITKV_F32 if w.dtype == "f32" else K.SPLITKV_BF16
    if kw.get("tail_pieces", 0) > 1 and K.splitkv_auto_kernel(w.Hq, w.Hkv, w.d, w.block_len, max(lens[0]),
                                                              code) == K.KERNEL_SIMT:
        kw.update(tail_pieces=0, tail_slots=None)  # the tail cut is defined for the CTA-unit kernels only
    inp, run, out, lse = run_cuda(w, lens=lens, **kw)
    what = f"seed {seed}: {w.B} seqs q{lens[0]} kv{lens[1]} Hq{w.Hq}/Hkv{w.Hkv} d{w.d} {w.dtype} " \
           f"block {w.block_len} S{w.n_shards} causal={w.causal} {kw} " \
           f"kernel {K.KERNEL_NAMES.get(run.kernel_used())}"
    o_ref, l_ref = full_reference(inp)
    eo, el = max_errors(out, lse, o_ref, l_ref)
    assert_close(w, eo, el, what)
    assert K.splitkv_device_status(clear=True) == 0, what
    if kw.get("fused") and run.fuses_in_one_launch():
        assert int(run.tickets.abs().sum()) == 0, what

    gen = torch.Generator(device="cuda").manual_seed(seed)
    dout = torch.randn(out.shape, generator=gen, device="cuda", dtype=torch.float32).to(out.dtype)
    dq, dk, dv = run.backward(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale, out, lse, dout)
    torch.cuda.synchronize()
    assert K.splitkv_device_status(clear=True) == 0, what
    args = (inp.q.cpu(), inp.k_pool.cpu(), inp.v_pool.cpu(), inp.block_table.cpu(), inp.q_len, inp.kv_len,
            w.block_len, w.causal, w.scale)
    do64 = dout.cpu().double()
    rdq, rdk, rdv = oracle.attention_backward(*args, do=do64, lse=l_ref, dlt=oracle.delta(o_ref, do64))
    valid = _valid_key_slots(inp, w)
    for nm, got, ref in (("dq", dq.cpu(), rdq), ("dk", dk.cpu()[valid], rdk[valid]),
                         ("dv", dv.cpu()[valid], rdv[valid])):
        assert_grad_close(w.dtype, got, ref, f"{what} {nm}")
