"""Seeded synthetic workloads for split-KV attention: shapes, lengths and tensors.

This module only draws inputs.  It holds none of the method's arithmetic (no
costs, plans, scores or merges), so both the CUDA path and the CPU oracle can
be fed from it without sharing any computation.

The five main workloads are the short-query / long-context shapes the Split-KV
card targets ("very short queries and very long contexts", card intro): a tiny
fp32 exactness case, batched decode, a 512-token query over a 128K context, a
variable-length batch, and a 256-token query over a 1M context.  A sixth,
``specdec``, sits between decode and the tile-filling shapes: four query tokens
per sequence (16 query rows per K/V head), as in speculative decoding.

Recipe (seed = workload index unless overridden):
* lengths: ``numpy.random.default_rng(seed)``; variable-length contexts are
  log-uniform in [4096, 131072] and query lengths uniform in [64, 1024].
* a causal workload appends its queries after the context: kv_len = context +
  q_len, and the queries' own keys are the last q_len keys of the sequence.
* physical block ids: a permutation of the pool drawn from
  ``default_rng(seed + 1000)``, so logical and physical order differ.
* Q, K, V: standard normal from ``torch.Generator(device).manual_seed(seed)``
  drawn in fp32 (Q, then K and V pool in chunks of whole blocks), times
  ``q_scale`` for Q, then cast to the workload dtype.
* optional poison: key slots past kv_len in each sequence's last block are set
  to NaN, so any kernel that reads them shows it.
"""

import math
from dataclasses import dataclass, field, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    block_len: int
    n_shards: int
    causal: bool
    dtype: str  # "f32" or "bf16"
    q_len: int = 0  # fixed query length (0 with varlen)
    context: int = 0  # fixed context length (0 with varlen)
    varlen: bool = False
    ctx_range: tuple = (4096, 131072)
    q_range: tuple = (64, 1024)
    q_scale: float = 1.0
    seed: int = 0
    description: str = ""

    @property
    def G(self):
        return self.Hq // self.Hkv

    @property
    def scale(self):
        return 1.0 / math.sqrt(self.d)

    @property
    def torch_dtype(self):
        return torch.float32 if self.dtype == "f32" else torch.bfloat16

    @property
    def elem_bytes(self):
        return 4 if self.dtype == "f32" else 2


WORKLOADS = {
    "tiny": Workload(
        "tiny", B=1, Hq=4, Hkv=4, d=64, block_len=128, n_shards=4, causal=False, dtype="f32",
        q_len=16, context=2048, seed=1,
        description="B=1 Hq=Hkv=4 d=64 Lq=16 Lkv=2048 fp32, no mask, blocks of 128, S=4"),
    "decode": Workload(
        "decode", B=8, Hq=32, Hkv=8, d=128, block_len=256, n_shards=16, causal=False, dtype="bf16",
        q_len=1, context=32768, seed=2,
        description="B=8 Hq=32 Hkv=8 d=128 Lq=1 Lkv=32768 bf16, paged block_len=256, S=16"),
    "shortq": Workload(
        "shortq", B=1, Hq=32, Hkv=8, d=128, block_len=1024, n_shards=64, causal=True, dtype="bf16",
        q_len=512, context=131072, seed=3,
        description="B=1 Hq=32 Hkv=8 d=128 Lq=512 causal tail after Lkv=131072 bf16, block_len=1024, S=64"),
    "varlen": Workload(
        "varlen", B=16, Hq=32, Hkv=8, d=128, block_len=1024, n_shards=64, causal=True, dtype="bf16",
        varlen=True, seed=4,
        description="16 seqs, context log-U[4096,131072], Lq U[64,1024] causal tail, Hq=32 Hkv=8 d=128 "
                    "bf16, block_len=1024, S=64"),
    "specdec": Workload(
        "specdec", B=8, Hq=32, Hkv=8, d=128, block_len=256, n_shards=16, causal=True, dtype="bf16",
        q_len=4, context=32768, seed=6,
        description="B=8 Hq=32 Hkv=8 d=128 Lq=4 causal tail after Lkv=32768 bf16 (16 query rows per "
                    "K/V head), paged block_len=256, S=16"),
    "largest": Workload(
        "largest", B=1, Hq=32, Hkv=8, d=128, block_len=2048, n_shards=64, causal=True, dtype="bf16",
        q_len=256, context=1048576, q_scale=2.0, seed=5,
        description="B=1 Hq=32 Hkv=8 d=128 Lq=256 causal tail after Lkv=1048576 bf16, Q x2, "
                    "block_len=2048, S=64"),
}


def custom(base, **kw):
    """A workload like ``base`` (a name or a Workload) with some fields replaced."""
    w = WORKLOADS[base] if isinstance(base, str) else base
    return replace(w, **kw)


def lengths(w):
    """(q_len, kv_len) lists of the workload's sequences."""
    if w.varlen:
        rng = np.random.default_rng(w.seed)
        lo, hi = w.ctx_range
        ctx = [int(round(math.exp(rng.uniform(math.log(lo), math.log(hi))))) for _ in range(w.B)]
        ql = [int(rng.integers(w.q_range[0], w.q_range[1] + 1)) for _ in range(w.B)]
    else:
        ctx = [w.context] * w.B
        ql = [w.q_len] * w.B
    kv = [c + q if w.causal else c for c, q in zip(ctx, ql)]
    return ql, kv


def blocks_per_seq(kv_len, block_len):
    return [-(-int(n) // block_len) for n in kv_len]


@dataclass
class Inputs:
    w: Workload
    q_len: list
    kv_len: list
    q: torch.Tensor  # [total_q, Hq, d]
    k_pool: torch.Tensor  # [n_pool_blocks, block_len, Hkv, d]
    v_pool: torch.Tensor
    block_table: torch.Tensor  # int32 [B, max_blocks]
    extra: dict = field(default_factory=dict)

    @property
    def total_q(self):
        return int(sum(self.q_len))

    @property
    def n_pool_blocks(self):
        return int(self.k_pool.shape[0])


def _randn_blocks(shape, gen, device, dtype, chunk_elems=1 << 26):
    """Standard normal of ``shape`` drawn in fp32, chunked along dim 0, cast to dtype."""
    out = torch.empty(shape, dtype=dtype, device=device)
    per = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    step = max(1, chunk_elems // max(per, 1))
    for i in range(0, shape[0], step):
        n = min(step, shape[0] - i)
        out[i : i + n] = torch.randn((n,) + tuple(shape[1:]), generator=gen, device=device,
                                     dtype=torch.float32).to(dtype)
    return out


def make_inputs(w, device="cpu", poison_tail=False, spare_blocks=0, lens=None):
    """Draw the workload's tensors on ``device`` (see the module docstring)."""
    q_len, kv_len = lens if lens is not None else lengths(w)
    nblk = blocks_per_seq(kv_len, w.block_len)
    n_used = sum(nblk)
    n_pool = n_used + spare_blocks
    perm = np.random.default_rng(w.seed + 1000).permutation(n_pool)[:n_used]
    max_blocks = max(nblk) if nblk else 0
    table = np.zeros((w.B, max(max_blocks, 1)), dtype=np.int32)
    g = 0
    for b in range(w.B):
        for j in range(nblk[b]):
            table[b, j] = perm[g]
            g += 1
    gen = torch.Generator(device=device)
    gen.manual_seed(w.seed)
    dt = w.torch_dtype
    total_q = int(sum(q_len))
    q = (torch.randn((total_q, w.Hq, w.d), generator=gen, device=device, dtype=torch.float32)
         * w.q_scale).to(dt)
    shape = (n_pool, w.block_len, w.Hkv, w.d)
    k_pool = _randn_blocks(shape, gen, device, dt)
    v_pool = _randn_blocks(shape, gen, device, dt)
    if poison_tail:
        for b in range(w.B):
            rem = kv_len[b] - (nblk[b] - 1) * w.block_len
            if nblk[b] and rem < w.block_len:
                pb = int(table[b, nblk[b] - 1])
                k_pool[pb, rem:] = float("nan")
                v_pool[pb, rem:] = float("nan")
    return Inputs(w, list(q_len), list(kv_len), q, k_pool, v_pool,
                  torch.from_numpy(table).to(device))
