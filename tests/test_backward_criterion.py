"""The backward parity criterion can fail: planted mistakes (on the CPU, in the
oracle's output) are rejected, and a model of the tensor-core kernel's own
rounding is accepted.

The criterion (``parity_helpers.grad_close``) bounds each gradient tensor's error
relative to that tensor's size.  Three planted mistakes must fail it on the small
parity cases: a backward that writes zeros for dK / dV, and one that drops the
D = rowsum(dO * O) term of dS = P (dP - D), which changes dQ and dK.  The bf16
model rounds what the tensor-core kernels round (P and dS to bf16 before their
MMAs, the output O to bf16 before D) and must pass, so the limits sit above the
arithmetic the kernels actually do."""

import pytest
import torch

import oracle
from oracle import attn as oatt
from context_long_attention_lpt_gb300 import workloads as wl
from tests.parity_helpers import GRAD_MAX, GRAD_REL, SMALL, grad_close, grad_errors

CASES = ["decode_small", "shortq_small", "varlen_small", "largest_small", "causal_empty_units"]


def _bf16(x):
    return x.to(torch.bfloat16).to(torch.float64)


def _reference(w, seed=11):
    inp = wl.make_inputs(w, device="cpu")
    args = (inp.q, inp.k_pool, inp.v_pool, inp.block_table, inp.q_len, inp.kv_len, w.block_len, w.causal,
            w.scale)
    o, lse = oracle.attention(*args)
    g = torch.Generator().manual_seed(seed)
    do = torch.randn(o.shape, generator=g).to(inp.q.dtype).double()
    dlt = oracle.delta(o, do)
    return inp, args, o, lse, do, dlt, oracle.attention_backward(*args, do=do, lse=lse, dlt=dlt)


def _bf16_kernel_model(w, inp, o, lse, do):
    """The gradients with the tensor-core kernels' roundings: D from the bf16 output,
    P and dS rounded to bf16 before the products that use them (fp64 elsewhere)."""
    hq, d = inp.q.shape[1], inp.q.shape[2]
    g = hq // inp.k_pool.shape[2]
    dlt = (do * _bf16(o)).sum(-1)
    dq = torch.zeros((inp.total_q, hq, d), dtype=torch.float64)
    dk = torch.zeros(inp.k_pool.shape, dtype=torch.float64)
    dv = torch.zeros(inp.v_pool.shape, dtype=torch.float64)
    cu = 0
    for b, (lq, lk) in enumerate(zip(inp.q_len, inp.kv_len)):
        if lq == 0:
            continue
        ks = oatt.gather_sequence(inp.k_pool, inp.block_table[b], lk, w.block_len).double()
        vs = oatt.gather_sequence(inp.v_pool, inp.block_table[b], lk, w.block_len).double()
        vis = torch.tensor([oatt.visible_keys(lq, lk, t, w.causal) for t in range(lq)])
        mask = torch.arange(lk)[None, :] < vis[:, None]
        dks = torch.zeros((lk, ks.shape[1], d), dtype=torch.float64)
        dvs = torch.zeros_like(dks)
        for h in range(hq):
            qh = inp.q[cu: cu + lq, h].double()
            doh = do[cu: cu + lq, h]
            kh, vh = ks[:, h // g], vs[:, h // g]
            p = torch.where(mask, torch.exp(w.scale * (qh @ kh.T) - lse[cu: cu + lq, h, None]), 0.0)
            dvs[:, h // g] += _bf16(p).T @ doh
            ds = _bf16(p * (doh @ vh.T - dlt[cu: cu + lq, h, None]))
            dq[cu: cu + lq, h] = w.scale * (ds @ kh)
            dks[:, h // g] += w.scale * (ds.T @ qh)
        for j in range(-(-lk // w.block_len)):
            lo, hi = j * w.block_len, min(lk, (j + 1) * w.block_len)
            pb = int(inp.block_table[b, j])
            dk[pb, : hi - lo] = dks[lo:hi]
            dv[pb, : hi - lo] = dvs[lo:hi]
        cu += lq
    return dq, dk, dv


def _valid(inp, w):
    valid = torch.zeros(inp.k_pool.shape[:2], dtype=torch.bool)
    for b, n in enumerate(inp.kv_len):
        for j in range(-(-n // w.block_len)):
            valid[int(inp.block_table[b, j]), : min(w.block_len, n - j * w.block_len)] = True
    return valid


@pytest.mark.parametrize("name", CASES)
def test_planted_zero_gradients_fail(name):
    w = SMALL[name]
    inp, _, _, _, _, _, (dq, dk, dv) = _reference(w)
    valid = _valid(inp, w)
    for ref in (dq, dk[valid], dv[valid]):
        assert ref.abs().max() > 0
        assert not grad_close(w.dtype, torch.zeros_like(ref), ref)
        assert not grad_close("f32", torch.zeros_like(ref), ref)


@pytest.mark.parametrize("name", CASES)
def test_planted_dropped_delta_fails(name):
    """dS = P dP instead of P (dP - D): dQ and dK must both fail the criterion."""
    w = SMALL[name]
    inp, args, _, lse, do, dlt, (dq, dk, _) = _reference(w)
    bq, bk, _ = oracle.attention_backward(*args, do=do, lse=lse, dlt=torch.zeros_like(dlt))
    valid = _valid(inp, w)
    assert not grad_close(w.dtype, bq, dq)
    assert not grad_close(w.dtype, bk[valid], dk[valid])


def test_planted_dropped_scale_and_sign_fail():
    """A missing softmax scale on dQ and a flipped sign of dV fail as well."""
    w = SMALL["shortq_small"]
    inp, _, _, _, _, _, (dq, _, dv) = _reference(w)
    assert not grad_close(w.dtype, dq / w.scale, dq)
    valid = _valid(inp, w)
    assert not grad_close(w.dtype, -dv[valid], dv[valid])


@pytest.mark.parametrize("name", ["decode_small", "shortq_small", "largest_small", "causal_empty_units"])
def test_bf16_kernel_rounding_model_passes(name):
    """The kernels' bf16 roundings stay well inside the bf16 limits (by a factor >= 3)."""
    w = SMALL[name]
    inp, _, o, lse, do, _, (dq, dk, dv) = _reference(w)
    mq, mk, mv = _bf16_kernel_model(w, inp, o, lse, do)
    valid = _valid(inp, w)
    for got, ref in ((mq, dq), (mk[valid], dk[valid]), (mv[valid], dv[valid])):
        rel, relmax = grad_errors(got, ref)
        assert rel <= GRAD_REL["bf16"] / 3 and relmax <= GRAD_MAX["bf16"] / 3, (rel, relmax)
        assert rel > 0  # the model does round
