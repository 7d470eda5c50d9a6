"""fp64 softmax attention over paged K/V: unsharded, per-shard partial, and merge.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Conventions (the pages give no notation beyond Q, K/V blocks and shards; these
follow the problem statement of short queries appended to a long context):

* ``q``            [total_q, Hq, d]   - queries of all sequences, concatenated
                                         sequence after sequence.
* ``k_pool``/``v_pool`` [n_pool_blocks, block_len, Hkv, d] - paged K/V.
* ``block_table``  [B, max_blocks]    - physical block id of logical block j of
                                         sequence b.
* ``q_len``/``kv_len`` [B]            - queries and keys of each sequence.
* query head h reads K/V head h // G, G = Hq // Hkv (contiguous grouping).
* query token t of sequence b sits at key position kv_len - q_len + t: the
  short query is appended after the long context, so its own keys are the last
  q_len keys of the paged sequence.  Causal: key j is visible iff j <= that
  position.  Non-causal: all kv_len keys are visible.
* ``scale`` multiplies q . k before the softmax; L is the natural-log
  log-sum-exp of the scaled scores.
"""

import math

import numpy as np
import torch


def visible_keys(q_len, kv_len, t, causal):
    """Number of keys (a prefix 0..n-1 of the sequence) that query token t sees."""
    if not causal:
        return int(kv_len)
    return int(kv_len) - int(q_len) + int(t) + 1


def gather_sequence(pool, table_row, kv_len, block_len):
    """The first ``kv_len`` keys of a paged sequence as one [kv_len, Hkv, d] fp64 tensor."""
    n_blocks = -(-int(kv_len) // int(block_len))
    if n_blocks == 0:
        return torch.zeros((0,) + tuple(pool.shape[2:]), dtype=torch.float64)
    blocks = [pool[int(table_row[j])].to(torch.float64) for j in range(n_blocks)]
    return torch.cat(blocks, dim=0)[: int(kv_len)]


def _attend(qh, kh, vh, mask, scale):
    """Softmax attention of query rows ``qh`` [n, d] over keys ``kh`` [m, d].

    ``mask`` [n, m] marks the keys each row may see.  Returns O [n, dv] (the
    softmax-weighted mean of the visible values) and L [n] (log-sum-exp of the
    visible scaled scores).  A row that sees no key gets O = 0 and L = -inf:
    an empty sum has weight zero in any later merge.
    """
    s = scale * (qh @ kh.T)
    s = torch.where(mask, s, torch.full_like(s, -math.inf))
    m = s.max(dim=1).values
    any_visible = mask.any(dim=1)
    m_safe = torch.where(any_visible, m, torch.zeros_like(m))
    e = torch.exp(s - m_safe[:, None])  # exp(-inf) = 0 on masked keys
    l = e.sum(dim=1)
    o = (e @ vh) / torch.where(any_visible, l, torch.ones_like(l))[:, None]
    lse = torch.where(any_visible, m_safe + torch.log(l), torch.full_like(m, -math.inf))
    return o, lse


def _offsets(q_len):
    cu = [0]
    for n in q_len:
        cu.append(cu[-1] + int(n))
    return cu


def partial(q, k_pool, v_pool, block_table, q_len, kv_len, block_len, causal, scale, key_blocks):
    """One shard's partial attention: only the keys in the shard's own blocks.

    ``key_blocks[b]`` lists the logical block indices of sequence b that the
    shard holds (possibly none).  Returns (O_i [total_q, Hq, d], L_i [total_q, Hq])
    in fp64, where O_i is the attention output restricted to those keys and
    L_i their log-sum-exp; rows with no visible key in the shard get O_i = 0
    and L_i = -inf.
    """
    total_q, hq, d = q.shape
    hkv = k_pool.shape[2]
    g = hq // hkv
    cu = _offsets(q_len)
    o_out = torch.zeros((total_q, hq, v_pool.shape[3]), dtype=torch.float64)
    l_out = torch.full((total_q, hq), -math.inf, dtype=torch.float64)
    for b in range(len(q_len)):
        lq, lk = int(q_len[b]), int(kv_len[b])
        if lq == 0:
            continue
        k_seq = gather_sequence(k_pool, block_table[b], lk, block_len)
        v_seq = gather_sequence(v_pool, block_table[b], lk, block_len)
        pos = torch.arange(lk)
        in_shard = torch.zeros(lk, dtype=torch.bool)
        for j in key_blocks[b]:
            in_shard |= (pos >= int(j) * block_len) & (pos < (int(j) + 1) * block_len)
        vis = torch.tensor([visible_keys(lq, lk, t, causal) for t in range(lq)])
        mask = (pos[None, :] < vis[:, None]) & in_shard[None, :]
        qb = q[cu[b] : cu[b] + lq].to(torch.float64)
        for h in range(hq):
            o, lse = _attend(qb[:, h], k_seq[:, h // g], v_seq[:, h // g], mask, scale)
            o_out[cu[b] : cu[b] + lq, h] = o
            l_out[cu[b] : cu[b] + lq, h] = lse
    return o_out, l_out


def attention(q, k_pool, v_pool, block_table, q_len, kv_len, block_len, causal, scale):
    """Unsharded attention: every visible key of each sequence in one softmax.

    This is the result an exact sharded method must reproduce.  Returns
    (O [total_q, Hq, d], L [total_q, Hq]) in fp64.
    """
    all_blocks = [list(range(-(-int(n) // int(block_len)))) for n in kv_len]
    return partial(q, k_pool, v_pool, block_table, q_len, kv_len, block_len, causal, scale, all_blocks)


def attention_rows(q, k_pool, v_pool, block_table, q_len, kv_len, block_len, causal, scale, rows):
    """Unsharded attention for selected output rows only.

    ``rows`` is a list of (b, t, h): sequence, query token within it, query head.
    Returns (O [n, d], L [n]) in fp64.  Used where the full output would take
    too long on the CPU; every row is computed exactly as ``attention`` does.
    """
    hq = q.shape[1]
    hkv = k_pool.shape[2]
    g = hq // hkv
    cu = _offsets(q_len)
    o_out = torch.zeros((len(rows), v_pool.shape[3]), dtype=torch.float64)
    l_out = torch.zeros(len(rows), dtype=torch.float64)
    cache = {}
    for i, (b, t, h) in enumerate(rows):
        lq, lk = int(q_len[b]), int(kv_len[b])
        key = (b, h // g)
        if key not in cache:
            cache.clear()  # one (sequence, K/V head) at a time keeps host memory small
            k_seq = gather_sequence(k_pool[:, :, h // g], block_table[b], lk, block_len)
            v_seq = gather_sequence(v_pool[:, :, h // g], block_table[b], lk, block_len)
            cache[key] = (k_seq, v_seq)
        k_seq, v_seq = cache[key]
        n_vis = visible_keys(lq, lk, t, causal)
        mask = (torch.arange(lk) < n_vis)[None, :]
        qrow = q[cu[b] + t, h].to(torch.float64)[None, :]
        o, lse = _attend(qrow, k_seq, v_seq, mask, scale)
        o_out[i] = o[0]
        l_out[i] = lse[0]
    return o_out, l_out


def merge(partials):
    """Exact combination of per-shard partials (O_i, L_i).

    With L = log sum_i exp(L_i) and weights w_i = exp(L_i - L), the unsharded
    output is O = sum_i w_i O_i: each O_i is the softmax mean over shard i's
    keys, and exp(L_i) is that shard's share of the full softmax denominator.
    Shards with L_i = -inf (nothing visible) carry weight 0.  Only the
    query-sized O_i and L_i enter, never K or V.
    """
    ls = torch.stack([p[1] for p in partials])  # [S, ...]
    os_ = torch.stack([p[0] for p in partials])  # [S, ..., d]
    m = ls.max(dim=0).values
    finite = torch.isfinite(m)
    m_safe = torch.where(finite, m, torch.zeros_like(m))
    w = torch.exp(ls - m_safe[None])  # 0 for -inf partials
    denom = w.sum(dim=0)
    lse = torch.where(finite, m_safe + torch.log(denom), torch.full_like(m, -math.inf))
    wn = w / torch.where(finite, denom, torch.ones_like(denom))[None]
    o = (wn[..., None] * os_).sum(dim=0)
    return o, lse


def as_numpy(x):
    return np.asarray(x.detach().cpu().numpy())
