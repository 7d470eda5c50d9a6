"""Pins for the oracle's backward pass: finite differences, torch autograd through
scaled_dot_product_attention, and the exactness of the split (partial dQ sum to
dQ; each shard's dK / dV are the unsharded ones on its keys)."""

import math
import random

import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import attn as oatt
from tests.test_oracle import _random_batch


def _grads(b, seed=0):
    g = torch.Generator().manual_seed(seed)
    o, lse = oracle.attention(**b)
    do = torch.randn(o.shape, generator=g, dtype=torch.float64)
    dlt = oracle.delta(o, do)
    return do, oracle.attention_backward(**b, do=do, lse=lse, dlt=dlt), lse, dlt


def _loss(b, w):
    o, _ = oracle.attention(**b)
    return float((o * w).sum())


@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_finite_differences(causal):
    b = _random_batch(4, B=2, Hq=4, Hkv=2, d=4, block_len=3, causal=causal, max_ctx=6, max_q=3)
    do, (dq, dk, dv), _, _ = _grads(b, seed=1)
    rng = random.Random(0)
    eps = 1e-6
    checks = 0
    for name, grad in (("q", dq), ("k_pool", dk), ("v_pool", dv)):
        t = b[name]
        for _ in range(12):
            idx = tuple(rng.randrange(n) for n in t.shape)
            orig = t[idx].item()
            t[idx] = orig + eps
            up = _loss(b, do)
            t[idx] = orig - eps
            down = _loss(b, do)
            t[idx] = orig
            fd = (up - down) / (2 * eps)
            assert abs(fd - grad[idx].item()) < 1e-6, (name, idx, fd, grad[idx].item())
            checks += 1
    assert checks == 36


@pytest.mark.parametrize("seed", range(4))
@pytest.mark.parametrize("causal", [False, True])
def test_backward_matches_autograd_through_sdpa(seed, causal):
    b = _random_batch(seed, causal=causal)
    do, (dq, dk, dv), _, _ = _grads(b, seed=seed)
    gsz = b["q"].shape[1] // b["k_pool"].shape[2]
    cu = 0
    for i, (lq, lk) in enumerate(zip(b["q_len"], b["kv_len"])):
        ks = oatt.gather_sequence(b["k_pool"], b["block_table"][i], lk, b["block_len"]).clone().requires_grad_(True)
        vs = oatt.gather_sequence(b["v_pool"], b["block_table"][i], lk, b["block_len"]).clone().requires_grad_(True)
        qq = b["q"][cu: cu + lq].clone().requires_grad_(True)
        pos = torch.arange(lk)
        qpos = torch.arange(lq) + (lk - lq)
        mask = (pos[None, :] <= qpos[:, None]) if causal else torch.ones((lq, lk), dtype=torch.bool)
        out = F.scaled_dot_product_attention(qq.permute(1, 0, 2), ks.permute(1, 0, 2).repeat_interleave(gsz, 0),
                                             vs.permute(1, 0, 2).repeat_interleave(gsz, 0), attn_mask=mask,
                                             scale=b["scale"])
        out.permute(1, 0, 2).backward(do[cu: cu + lq])
        assert torch.allclose(dq[cu: cu + lq], qq.grad, atol=1e-11, rtol=0)
        # gather the pool gradients of this sequence
        dk_seq = oatt.gather_sequence(dk, b["block_table"][i], lk, b["block_len"])
        dv_seq = oatt.gather_sequence(dv, b["block_table"][i], lk, b["block_len"])
        assert torch.allclose(dk_seq, ks.grad, atol=1e-11, rtol=0)
        assert torch.allclose(dv_seq, vs.grad, atol=1e-11, rtol=0)
        cu += lq


@pytest.mark.parametrize("seed", range(5))
def test_split_backward_is_exact(seed):
    rng = random.Random(seed)
    b = _random_batch(seed, causal=bool(seed % 2), block_len=rng.choice([2, 3, 4]))
    do, (dq, dk, dv), lse, dlt = _grads(b, seed=seed)
    S = rng.randint(1, 5)
    owner = [[rng.randrange(S) for _ in range(-(-n // b["block_len"]))] for n in b["kv_len"]]
    dq_sum = torch.zeros_like(dq)
    dk_sum = torch.zeros_like(dk)
    dv_sum = torch.zeros_like(dv)
    for s in range(S):
        keys = [[j for j, o in enumerate(owner[i]) if o == s] for i in range(len(owner))]
        dqs, dks, dvs = oracle.partial_backward(**b, do=do, lse=lse, dlt=dlt, key_blocks=keys)
        dq_sum += dqs
        dk_sum += dks
        dv_sum += dvs
    assert torch.allclose(dq_sum, dq, atol=1e-12, rtol=0)
    assert torch.allclose(dk_sum, dk, atol=1e-12, rtol=0)
    assert torch.allclose(dv_sum, dv, atol=1e-12, rtol=0)


def test_planted_missing_delta_is_caught():
    b = _random_batch(9, causal=True)
    o, lse = oracle.attention(**b)
    do = torch.randn(o.shape, generator=torch.Generator().manual_seed(2), dtype=torch.float64)
    good = oracle.attention_backward(**b, do=do, lse=lse, dlt=oracle.delta(o, do))
    bad = oracle.attention_backward(**b, do=do, lse=lse, dlt=torch.zeros_like(lse))
    assert (good[0] - bad[0]).abs().max() > 1e-3  # dQ changes when D is dropped


@pytest.mark.parametrize("causal", [False, True])
def test_sampled_row_and_key_gradients_match_full(causal):
    b = _random_batch(13, causal=causal, B=2)
    do, (dq, dk, dv), _, _ = _grads(b, seed=5)
    cu = [0, b["q_len"][0]]
    rows = [(0, 0, 1), (1, b["q_len"][1] - 1, 3), (0, b["q_len"][0] - 1, 0)]
    got = oracle.backward_rows(**b, do=do, rows=rows)
    for i, (bb, t, h) in enumerate(rows):
        assert torch.allclose(got[i], dq[cu[bb] + t, h], atol=1e-12, rtol=0)
    keys = [(0, 0, 0), (1, 1, b["kv_len"][1] - 1), (1, 0, 2)]
    gk, gv = oracle.backward_keys(**b, do=do, keys=keys, row_chunk=2)
    for i, (bb, kvh, pos) in enumerate(keys):
        blk, off = pos // b["block_len"], pos % b["block_len"]
        phys = int(b["block_table"][bb, blk])
        assert torch.allclose(gk[i], dk[phys, off, kvh], atol=1e-12, rtol=0)
        assert torch.allclose(gv[i], dv[phys, off, kvh], atol=1e-12, rtol=0)
