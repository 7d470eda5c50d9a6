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

# Backward criterion, relative to the size of each gradient tensor (the gradients of
# these workloads are far smaller than 1, so an absolute 2e-2 would accept zeros).
# The bf16 tensor-core backward rounds P and dS to bf16 (unit roundoff u = 2^-9)
# before the MMAs that use them, and D comes from the bf16-rounded output; with
# errors of random sign each gradient's normwise relative error is about
# u / sqrt(3) ~ 1.1e-3.  The fp32 CUDA-core backward accumulates in fp32.
#   normwise:  ||got - ref||_F  <= GRAD_REL[dtype] * ||ref||_F
#   max-wise:  max|got - ref|   <= GRAD_MAX[dtype] * max|ref|
# plus an absolute floor GRAD_FLOOR for tensors whose reference is (near) zero.
GRAD_REL = {"f32": 1e-4, "bf16": 1e-2}
GRAD_MAX = {"f32": 1e-3, "bf16": 2e-2}
GRAD_FLOOR = 1e-7

# The small parity cases: reduced copies of the workloads (ragged lengths, several
# shards, GQA 8:1, d = 64, non-causal, causal units without keys).
SMALL = {
    "tiny": wl.WORKLOADS["tiny"],
    "decode_small": wl.custom("decode", B=3, context=3000, n_shards=5),
    "decode_gqa8": wl.custom("decode", B=2, Hq=64, Hkv=8, context=1500, n_shards=4),
    "shortq_small": wl.custom("shortq", q_len=77, context=2500, block_len=256, n_shards=7),
    "varlen_small": wl.custom("varlen", B=4, ctx_range=(100, 3000), q_range=(1, 300), block_len=128,
                              n_shards=6),
    "largest_small": wl.custom("largest", q_len=64, context=5000, block_len=512, n_shards=3),
    "noncausal_multi_q": wl.custom("shortq", causal=False, q_len=9, context=1000, block_len=128,
                                   n_shards=4),
    "bf16_d64": wl.custom("shortq", d=64, q_len=20, context=900, block_len=128, n_shards=3),
    # causal queries longer than the context, one block per shard: the first query rows see
    # none of the last blocks, so many (item, head, row tile) units have no key tile at all
    "causal_empty_units": wl.custom("shortq", q_len=600, context=100, block_len=128, n_shards=6),
    # one 64-row tile per sequence and ~12 key tiles per dK/dV CTA: K and V are reloaded
    # after every row tile
    "specdec_small": wl.custom("specdec", B=3, context=3000, n_shards=5),
    # group sizes other than 4 on the tensor-core path: 16 query heads per K/V head
    # (8 tokens per 128-row tile) and 2
    "gqa16_tc": wl.custom("shortq", Hq=64, Hkv=4, q_len=20, context=1500, block_len=128, n_shards=3),
    "gqa2_tc": wl.custom("shortq", Hq=16, Hkv=8, q_len=90, context=1100, block_len=256, n_shards=4),
    "many_key_tiles": wl.custom("shortq", q_len=16, context=24000, block_len=128, n_shards=1),
}


def run_cuda(w, kernel=0, poison=True, device="cuda", spare_blocks=0, lens=None, **runner_kw):
    inp = wl.make_inputs(w, device=device, poison_tail=poison, spare_blocks=spare_blocks, lens=lens)
    run = SplitKVAttention(inp.q_len, inp.kv_len, w.block_len, w.causal, w.n_shards, w.Hq, w.Hkv, w.d,
                           inp.q.dtype, device=device, kernel=kernel, **runner_kw)
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


def grad_errors(got, ref):
    """(normwise relative error, max error relative to max|ref|) of a gradient tensor."""
    got = got.double()
    ref = ref.double()
    err = got - ref
    rn = ref.norm().item()
    rm = ref.abs().max().item() if ref.numel() else 0.0
    en = err.norm().item()
    em = err.abs().max().item() if err.numel() else 0.0
    return (en / rn if rn > 0 else en), (em / rm if rm > 0 else em)


def grad_close(dtype, got, ref):
    """True when ``got`` meets the backward criterion against ``ref`` (see GRAD_REL)."""
    got = got.double()
    ref = ref.double()
    if not torch.isfinite(got).all():
        return False
    err = got - ref
    ok_norm = err.norm().item() <= GRAD_REL[dtype] * ref.norm().item() + GRAD_FLOOR
    ok_max = err.abs().max().item() <= GRAD_MAX[dtype] * ref.abs().max().item() + GRAD_FLOOR
    return ok_norm and ok_max


def assert_grad_close(dtype, got, ref, what=""):
    rel, relmax = grad_errors(got, ref)
    assert grad_close(dtype, got, ref), (
        f"{what}: normwise rel err {rel:.3e} (limit {GRAD_REL[dtype]}), max err / max|ref| {relmax:.3e} "
        f"(limit {GRAD_MAX[dtype]})")
    return rel, relmax
