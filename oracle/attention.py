"""Oracle causal attention in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring).

For a query row at position P of request b and query head h (KV head
h // g with g = Hq / Hkv, reading R5), over the visible key positions
k in [lo, min(hi, P + 1)) (reading R3; lo = 0, hi = inf for full-KV
attention):

    S_k = scale * sum_c q[h, c] * K[b, k, h // g, c]
    L   = log(sum_k exp(S_k))                      (natural log, reading R4)
    O   = sum_k exp(S_k - L) * V[b, k, h // g, :]

This is the partial output O_j with its log-sum-exp L_j of the blog
"什么是 Context Parallelism", §3.3 ("each rank computes a partial output and
its LSE over its KV shard"), and with the full window it is plain dense causal
attention.  An empty window gives O = 0, L = -inf (reading R6).

The arithmetic uses NumPy matrix products as a library primitive; the max is
subtracted before exponentiating only to keep exp() in range, which does not
change the value of L or O.
"""

import numpy as np


def attention_rows(q, k, v, positions, kv_row0, scale, kv_lo=0, kv_hi=None):
    """Attention for selected query rows.

    q:         [R, Hq, d]     float64 query rows
    k:         [KV, Hkv, d]   float64 key buffer (all requests, prefix first)
    v:         [KV, Hkv, dv]  float64 value buffer
    positions: [R]            position of each row within its request
    kv_row0:   [R]            KV-buffer row of key position 0 of the row's request
    kv_lo/hi:  key-position window [kv_lo, kv_hi) intersected with [0, P]
    returns (O [R, Hq, dv], L [R, Hq])
    """
    q = np.asarray(q, dtype=np.float64)
    R, Hq, d = q.shape
    Hkv = k.shape[1]
    dv = v.shape[2]
    g = Hq // Hkv
    O = np.zeros((R, Hq, dv), dtype=np.float64)
    L = np.full((R, Hq), -np.inf, dtype=np.float64)
    for i in range(R):
        P = int(positions[i])
        lo = max(0, int(kv_lo))
        hi = P + 1 if kv_hi is None else min(int(kv_hi), P + 1)
        if hi <= lo:
            continue
        base = int(kv_row0[i])
        Kr = np.asarray(k[base + lo: base + hi], dtype=np.float64)   # [n, Hkv, d]
        Vr = np.asarray(v[base + lo: base + hi], dtype=np.float64)   # [n, Hkv, dv]
        qg = q[i].reshape(Hkv, g, d)
        S = scale * np.einsum("nkc,kgc->kgn", Kr, qg)                 # [Hkv, g, n]
        m = S.max(axis=2, keepdims=True)
        lse = m[..., 0] + np.log(np.exp(S - m).sum(axis=2))          # [Hkv, g]
        Pm = np.exp(S - lse[..., None])
        Oi = np.einsum("kgn,nkv->kgv", Pm, Vr)                        # [Hkv, g, dv]
        O[i] = Oi.reshape(Hq, dv)
        L[i] = lse.reshape(Hq)
    return O, L


def token_tables(new_lens, prefix_lens):
    """Per flat new token: position within its request and the request's KV start."""
    pos, kv0 = [], []
    kv = 0
    for n, p in zip(new_lens, prefix_lens):
        for t in range(int(n)):
            pos.append(int(p) + t)
            kv0.append(kv)
        kv += int(p) + int(n)
    return np.asarray(pos, dtype=np.int64), np.asarray(kv0, dtype=np.int64)


def dense_causal_attention(q_flat, k, v, new_lens, prefix_lens, scale, rows=None,
                           kv_lo=0, kv_hi=None):
    """Unsharded causal attention of the batch's new tokens (original order).

    q_flat: [sum(new_lens), Hq, d]; ``rows`` selects flat token indices
    (default: all).  Returns (O, L) for the selected rows.
    """
    pos, kv0 = token_tables(new_lens, prefix_lens)
    if rows is None:
        rows = np.arange(len(pos))
    rows = np.asarray(rows, dtype=np.int64)
    return attention_rows(np.asarray(q_flat[rows], dtype=np.float64), k, v,
                          pos[rows], kv0[rows], scale, kv_lo, kv_hi)


def decode_attention(q, k, v, scale, key_rows):
    """No causal mask: every query row sees exactly the key rows ``key_rows``.

    Used for the decode-style merge sweep (blog "什么是 Context Parallelism",
    §2.2 / §3.3.1: a few query tokens against a KV cache sharded by token,
    token i on rank i mod C, each rank producing (O_j, L_j)).
    q: [R, Hq, d]; returns (O [R, Hq, dv], L [R, Hq]).
    """
    key_rows = np.asarray(key_rows, dtype=np.int64)
    R, Hq, d = q.shape
    Hkv = k.shape[1]
    dv = v.shape[2]
    g = Hq // Hkv
    if len(key_rows) == 0:
        return np.zeros((R, Hq, dv)), np.full((R, Hq), -np.inf)
    Kr = np.asarray(k[key_rows], dtype=np.float64)
    Vr = np.asarray(v[key_rows], dtype=np.float64)
    qg = np.asarray(q, dtype=np.float64).reshape(R, Hkv, g, d)
    S = scale * np.einsum("nkc,rkgc->rkgn", Kr, qg)
    m = S.max(axis=3, keepdims=True)
    lse = m[..., 0] + np.log(np.exp(S - m).sum(axis=3))
    Pm = np.exp(S - lse[..., None])
    O = np.einsum("rkgn,nkv->rkgv", Pm, Vr).reshape(R, Hq, dv)
    return O, lse.reshape(R, Hq)
