"""fp64 gradients of softmax attention over paged K/V, unsharded and per shard.

TEST INFRASTRUCTURE ONLY (see the package docstring).

The Split-KV card places the method in training ("asymmetric training scenarios
with very short queries and very long contexts", card intro) and states it is
exact ("All Facts").  For the backward pass the same split holds: with the
merged output O and log-sum-exp L saved by the forward pass, a shard needs only
query-sized tensors (Q, dO, L and D = rowsum(dO * O)) to compute
* dK_j, dV_j of its own keys exactly, and
* a partial dQ_i over its own keys; the shards' partials sum to dQ.
The formulas are the chain rule through s = scale * q.k, P = exp(s - L),
O = P V:
    dV_j = sum_r P_rj dO_r
    dP_rj = dO_r . V_j
    dS_rj = P_rj (dP_rj - D_r)
    dQ_r = scale * sum_j dS_rj K_j
    dK_j = scale * sum_r dS_rj Q_r
with r over the query rows (every query head of the K/V head's group) that see
key j.  Conventions (layouts, positions, GQA) are those of ``attn``.
"""

import math

import torch

from .attn import _offsets, gather_sequence, visible_keys


def _shard_mask(lq, lk, block_len, causal, key_blocks):
    pos = torch.arange(lk)
    in_shard = torch.zeros(lk, dtype=torch.bool)
    for j in key_blocks:
        in_shard |= (pos >= int(j) * block_len) & (pos < (int(j) + 1) * block_len)
    vis = torch.tensor([visible_keys(lq, lk, t, causal) for t in range(lq)])
    return (pos[None, :] < vis[:, None]) & in_shard[None, :]


def delta(o, do):
    """D = rowsum(dO * O) per (query row, head), fp64."""
    return (do.to(torch.float64) * o.to(torch.float64)).sum(dim=-1)


def partial_backward(q, k_pool, v_pool, block_table, q_len, kv_len, block_len, causal, scale, do, lse, dlt,
                     key_blocks):
    """One shard's backward over its own keys.

    ``lse`` and ``dlt`` are the merged forward's L and D ([total_q, Hq]).
    ``key_blocks[b]`` lists the logical blocks of sequence b the shard holds.
    Returns (dQ_i [total_q, Hq, d], dK [n_pool, block_len, Hkv, d],
    dV [n_pool, block_len, Hkv, d]) in fp64; dK / dV are zero outside the
    shard's keys.
    """
    total_q, hq, d = q.shape
    hkv = k_pool.shape[2]
    g = hq // hkv
    cu = _offsets(q_len)
    dq = torch.zeros((total_q, hq, d), dtype=torch.float64)
    dk = torch.zeros(tuple(k_pool.shape), dtype=torch.float64)
    dv = torch.zeros(tuple(v_pool.shape), dtype=torch.float64)
    for b in range(len(q_len)):
        lq, lk = int(q_len[b]), int(kv_len[b])
        if lq == 0 or lk == 0:
            continue
        ks = gather_sequence(k_pool, block_table[b], lk, block_len)
        vs = gather_sequence(v_pool, block_table[b], lk, block_len)
        mask = _shard_mask(lq, lk, block_len, causal, key_blocks[b])
        dk_seq = torch.zeros((lk, hkv, d), dtype=torch.float64)
        dv_seq = torch.zeros((lk, hkv, d), dtype=torch.float64)
        sl = slice(cu[b], cu[b] + lq)
        for h in range(hq):
            kh, vh = ks[:, h // g], vs[:, h // g]
            qh = q[sl, h].to(torch.float64)
            doh = do[sl, h].to(torch.float64)
            s = scale * (qh @ kh.T)
            p = torch.where(mask, torch.exp(s - lse[sl, h].to(torch.float64)[:, None]), torch.zeros_like(s))
            dv_seq[:, h // g] += p.T @ doh
            dp = doh @ vh.T
            ds = p * (dp - dlt[sl, h].to(torch.float64)[:, None])
            dq[sl, h] = scale * (ds @ kh)
            dk_seq[:, h // g] += scale * (ds.T @ qh)
        for j in range(-(-lk // block_len)):
            lo, hi = j * block_len, min(lk, (j + 1) * block_len)
            pb = int(block_table[b][j])
            dk[pb, : hi - lo] = dk_seq[lo:hi]
            dv[pb, : hi - lo] = dv_seq[lo:hi]
    return dq, dk, dv


def attention_backward(q, k_pool, v_pool, block_table, q_len, kv_len, block_len, causal, scale, do, lse, dlt):
    """Unsharded backward: every visible key of each sequence."""
    all_blocks = [list(range(-(-int(n) // int(block_len)))) for n in kv_len]
    return partial_backward(q, k_pool, v_pool, block_table, q_len, kv_len, block_len, causal, scale, do, lse, dlt,
                            all_blocks)


def _seq_head(pool, table_row, lk, block_len, kvh):
    return gather_sequence(pool[:, :, kvh], table_row, lk, block_len)


def backward_rows(q, k_pool, v_pool, block_table, q_len, kv_len, block_len, causal, scale, do, rows):
    """dQ of selected rows (b, t, h), each from its own full forward over the visible keys.

    Returns dQ [n, d] in fp64.  Every step follows ``partial_backward`` for one row.
    """
    hq = q.shape[1]
    g = hq // k_pool.shape[2]
    cu = _offsets(q_len)
    out = torch.zeros((len(rows), q.shape[2]), dtype=torch.float64)
    cache = {}
    for i, (b, t, h) in enumerate(rows):
        lq, lk = int(q_len[b]), int(kv_len[b])
        key = (b, h // g)
        if key not in cache:
            cache.clear()
            cache[key] = (_seq_head(k_pool, block_table[b], lk, block_len, h // g),
                          _seq_head(v_pool, block_table[b], lk, block_len, h // g))
        kh, vh = cache[key]
        n_vis = visible_keys(lq, lk, t, causal)
        qr = q[cu[b] + t, h].to(torch.float64)
        dor = do[cu[b] + t, h].to(torch.float64)
        s = scale * (kh[:n_vis] @ qr)
        p = torch.softmax(s, dim=0)
        o = p @ vh[:n_vis]
        dp = vh[:n_vis] @ dor
        ds = p * (dp - torch.dot(dor, o))
        out[i] = scale * (ds @ kh[:n_vis])
    return out


def backward_keys(q, k_pool, v_pool, block_table, q_len, kv_len, block_len, causal, scale, do, keys, row_chunk=64):
    """dK, dV of selected keys (b, kvh, position): every query row of the K/V head's
    group contributes, with L and D from the oracle's own forward over all keys.

    Returns (dK [n, d], dV [n, d]) in fp64.
    """
    hq = q.shape[1]
    g = hq // k_pool.shape[2]
    cu = _offsets(q_len)
    dk = torch.zeros((len(keys), q.shape[2]), dtype=torch.float64)
    dv = torch.zeros((len(keys), q.shape[2]), dtype=torch.float64)
    groups = {}
    for i, (b, kvh, pos) in enumerate(keys):
        groups.setdefault((b, kvh), []).append((i, pos))
    for (b, kvh), members in groups.items():
        lq, lk = int(q_len[b]), int(kv_len[b])
        kh = _seq_head(k_pool, block_table[b], lk, block_len, kvh)
        vh = _seq_head(v_pool, block_table[b], lk, block_len, kvh)
        idx = torch.tensor([pos for _, pos in members])
        pos_all = torch.arange(lk)
        for h in range(kvh * g, (kvh + 1) * g):
            for t0 in range(0, lq, row_chunk):
                t1 = min(lq, t0 + row_chunk)
                qr = q[cu[b] + t0: cu[b] + t1, h].to(torch.float64)
                dor = do[cu[b] + t0: cu[b] + t1, h].to(torch.float64)
                vis = torch.tensor([visible_keys(lq, lk, t, causal) for t in range(t0, t1)])
                mask = pos_all[None, :] < vis[:, None]
                s = scale * (qr @ kh.T)
                s = torch.where(mask, s, torch.full_like(s, -math.inf))
                lse = torch.logsumexp(s, dim=1)
                p_all = torch.exp(s - lse[:, None])
                o = p_all @ vh
                dlt = (dor * o).sum(dim=1)
                p = p_all[:, idx]                              # [rows, n_sel]
                dp = dor @ vh[idx].T
                ds = p * (dp - dlt[:, None])
                dvs = p.T @ dor
                dks = scale * (ds.T @ qr)
                for m, (i, _) in enumerate(members):
                    dv[i] += dvs[m]
                    dk[i] += dks[m]
    return dk, dv
