"""Oracle end-to-end sharded pipelines.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Full-KV mode (SGLang docs, "Prefill Context Parallelism", introduction and
§Attention backend integration: each rank computes attention for its local
queries against the all-gathered KV, with per-block query and KV lengths):

    plan -> for each rank, for each of its segments: attention of the segment's
    rows against key positions 0..P -> O_cat (rank order) -> restore.

Partial-KV mode (blog "什么是 Context Parallelism", §2.1 item 2 and §3.1:
a rank's queries meet the KV one block at a time, each block gives
(O_j, L_j), and the LSE merge makes the result equal to single-GPU dense
attention):

    for each KV block j: partial of the rank's rows against key positions in
    block j -> merge over j -> restore.
"""

import numpy as np

from .attention import attention_rows
from .merge import lse_merge
from .plan import make_plan


def segment_rows(seg):
    """O_cat rows and positions of one segment."""
    rows = np.arange(seg.q_row0, seg.q_row0 + seg.q_len)
    pos = seg.q_pos0 + seg.q_pos_step * np.arange(seg.q_len)
    return rows, pos


def shard_partials(plan, q_cat, k, v, scale, kv_lo=0, kv_hi=None):
    """Every rank's partial (O, L) over one key window, written at O_cat rows."""
    n = q_cat.shape[0]
    Hq = q_cat.shape[1]
    dv = v.shape[2]
    O = np.zeros((n, Hq, dv))
    L = np.full((n, Hq), -np.inf)
    for r in range(plan.cp_size):
        for seg in plan.segments[r]:
            rows, pos = segment_rows(seg)
            o, l = attention_rows(q_cat[rows], k, v, pos,
                                  np.full(seg.q_len, seg.kv_row0), scale, kv_lo, kv_hi)
            O[rows] = o
            L[rows] = l
    return O, L


def sharded_attention(q_flat, k, v, new_lens, prefix_lens, cp_size, strategy, scale):
    """Full-KV CP: plan, per-shard attention, restore to original order."""
    plan = make_plan(new_lens, prefix_lens, cp_size, strategy)
    q_cat = np.asarray(q_flat, dtype=np.float64)[np.asarray(plan.gather_idx, dtype=np.int64)]
    O_cat, L_cat = shard_partials(plan, q_cat, k, v, scale)
    ri = np.asarray(plan.restore_idx, dtype=np.int64)
    return O_cat[ri], L_cat[ri], plan


def partial_kv_attention(q_flat, k, v, new_lens, prefix_lens, cp_size, strategy, scale,
                         kv_block):
    """Partial-KV CP: per-KV-block partials of each shard, LSE merge, restore."""
    plan = make_plan(new_lens, prefix_lens, cp_size, strategy)
    q_cat = np.asarray(q_flat, dtype=np.float64)[np.asarray(plan.gather_idx, dtype=np.int64)]
    longest = max(int(p) + int(n) for n, p in zip(new_lens, prefix_lens))
    nblk = (longest + kv_block - 1) // kv_block
    parts_o, parts_l = [], []
    for j in range(nblk):
        o, l = shard_partials(plan, q_cat, k, v, scale, j * kv_block, (j + 1) * kv_block)
        parts_o.append(o)
        parts_l.append(l)
    O_cat, L_cat = lse_merge(np.stack(parts_o), np.stack(parts_l))
    ri = np.asarray(plan.restore_idx, dtype=np.int64)
    return O_cat[ri], L_cat[ri], plan
