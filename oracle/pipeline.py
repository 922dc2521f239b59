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

Pass-Q ring (blog "什么是 Context Parallelism", §3.3.2 "Pass Q", and the
persistent-KV bullet of §3.5): KV stays resident, split per request into 2C
blocks with rank r keeping blocks r and 2C-1-r; each rank's query shard
travels round the ring with an accumulator (O_acc, L_acc) that starts empty,
and at every hop the host rank merges the shard's partial against its
resident KV into the accumulator with the LSE rule.  After C hops the
accumulator is the exact result.

    acc = (0, -inf); for hop s, rank r: acc[shard (r-s) mod C] <-
    merge(acc, partial(shard, KV blocks of r)) -> restore.
"""

import numpy as np

from .attention import attention_rows
from .merge import lse_merge
from .plan import make_plan, zigzag_block_sizes, zigzag_ranks_of_blocks


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


def resident_kv_windows(kv_total, cp_size):
    """Key-position windows of the KV blocks rank r keeps in the pass-Q ring.

    The request's KV positions 0..kv_total-1 are cut into 2C blocks like the
    zigzag query split (the remainder to the first blocks) and rank r keeps
    blocks r and 2C-1-r (blog §3.5, persistent KV: 2N blocks, rank i takes
    the first/last pair).  Returns, per rank, a list of (lo, hi).
    """
    sizes = zigzag_block_sizes(kv_total, cp_size)
    owner = zigzag_ranks_of_blocks(cp_size)
    start = np.concatenate([[0], np.cumsum(sizes)]).astype(int)
    wins = [[] for _ in range(cp_size)]
    for b, r in enumerate(owner):
        wins[r].append((int(start[b]), int(start[b + 1])))
    return wins


def pass_q_attention(q_flat, k, v, new_lens, prefix_lens, cp_size, strategy, scale):
    """Pass-Q ring CP: carried accumulators merged hop by hop, then restore."""
    plan = make_plan(new_lens, prefix_lens, cp_size, strategy)
    q_cat = np.asarray(q_flat, dtype=np.float64)[np.asarray(plan.gather_idx, dtype=np.int64)]
    n, Hq, dv = q_cat.shape[0], q_cat.shape[1], v.shape[2]
    O_acc = np.zeros((n, Hq, dv))
    L_acc = np.full((n, Hq), -np.inf)
    wins = [resident_kv_windows(int(p) + int(nn), cp_size)
            for nn, p in zip(new_lens, prefix_lens)]
    for hop in range(cp_size):
        for r in range(cp_size):
            shard = (r - hop) % cp_size
            for seg in plan.segments[shard]:
                rows, pos = segment_rows(seg)
                for lo, hi in wins[seg.req][r]:
                    o, l = attention_rows(q_cat[rows], k, v, pos,
                                          np.full(seg.q_len, seg.kv_row0), scale, lo, hi)
                    O_acc[rows], L_acc[rows] = lse_merge(np.stack([O_acc[rows], o]),
                                                         np.stack([L_acc[rows], l]))
    ri = np.asarray(plan.restore_idx, dtype=np.int64)
    return O_acc[ri], L_acc[ri], plan
