"""Shared helpers of the GPU parity tests: run the CUDA path, sample rows, compare with the oracle."""

import math
import random

import numpy as np
import torch

import oracle
from context_long_attention_lpt_gb300 import workloads as wl
from context_long_attention_lpt_gb300.runner import SplitKVAttention

# Tolerances (max abs error vs the fp64 oracle): bf16 inputs 2e-2 on O, fp32
# inputs 1e-4 on O, LSE 1e-3 for both.
TOL_O = {"f32": 1e-4, "bf16": 2e-2}
TOL_L = 1e-3


def run_cuda(w, kernel=0, poison=True, device="cuda", spare_blocks=0, lens=None):
    inp = wl.make_inputs(w, device=device, poison_tail=poison, spare_blocks=spare_blocks, lens=lens)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, device=device, kernel=kernel)
    out, lse = run(inp.q, inp.k_pool, inp.v_pool, inp.block_table, w.scale)
    torch.cuda.synchronize()
    return inp, run, out, lse


def full_reference(inp):
    w = inp.w
    return oracle.attention(inp.q.cpu(), inp.k_pool.cpu(), inp.v_pool.cpu(), inp.block_table.cpu(),
                            inp.q_len, inp.kv_len, w.block_len, w.causal, w.scale)


def sample_rows(inp, n, seed=0):
    """(b, t, h) rows: the first and last token of every sequence plus random ones."""
    rng = random.Random(seed)
    rows = set()
    for b, lq in enumerate(inp.q_len):
        if lq == 0:
            continue
        rows.add((b, 0, rng.randrange(inp.w.Hq)))
        rows.add((b, lq - 1, rng.randrange(inp.w.Hq)))
    live = [b for b, lq in enumerate(inp.q_len) if lq > 0]
    while len(rows) < n:
        b = rng.choice(live)
        rows.add((b, rng.randrange(inp.q_len[b]), rng.randrange(inp.w.Hq)))
    return sorted(rows, key=lambda r: (r[0], r[2] // inp.w.G, r[1], r[2]))


def compare_rows(inp, out, lse, rows):
    w = inp.w
    o_ref, l_ref = oracle.attention_rows(inp.q.cpu(), inp.k_pool.cpu(), inp.v_pool.cpu(),
                                         inp.block_table.cpu(), inp.q_len, inp.kv_len, w.block_len,
                                         w.causal, w.scale, rows)
    cu = np.concatenate([[0], np.cumsum(inp.q_len)])
    idx_row = torch.tensor([int(cu[b] + t) for b, t, _ in rows])
    idx_h = torch.tensor([h for _, _, h in rows])
    o = out.cpu()[idx_row, idx_h].double()
    l = lse.cpu()[idx_row, idx_h].double()
    return (o - o_ref).abs().max().item(), (l - l_ref).abs().max().item()


def max_errors(out, lse, o_ref, l_ref):
    eo = (out.double().cpu() - o_ref).abs().max().item()
    el = (lse.double().cpu() - l_ref)
    finite = torch.isfinite(l_ref)
    assert torch.equal(torch.isfinite(lse.cpu()), finite), "-inf pattern of LSE differs"
    el = el[finite].abs().max().item() if finite.any() else 0.0
    return eo, el


def assert_close(w, eo, el, what=""):
    assert not math.isnan(eo) and not math.isnan(el), f"{what}: NaN in output"
    assert eo <= TOL_O[w.dtype], f"{what}: max|dO| = {eo:.3e} > {TOL_O[w.dtype]}"
    assert el <= TOL_L, f"{what}: max|dL| = {el:.3e} > {TOL_L}"
