"""Oracle shard plans: zigzag and interleave query sharding, restore index.

TEST INFRASTRUCTURE ONLY (see the package docstring).

A plan says, for every new (uncached) token of a batch, which CP rank owns
its query row and where that row sits in the rank-concatenated buffer
``O_cat`` (rank 0's rows, then rank 1's, ...), which is what an all-gather of
the ranks' outputs produces.

Batch model (both pages): request b has ``prefix_lens[b]`` cached tokens and
``new_lens[b]`` new tokens.  Its new tokens have positions
``prefix_lens[b] + t`` for t = 0..new_lens[b]-1.  The flattened new-token
index runs over the batch in request order.  The KV buffer holds, per
request in batch order, positions 0..prefix+new-1 (prefix first).

A *segment* is a maximal run of one rank's rows that belong to one request
and whose positions advance by a constant step.  It carries the causal
metadata an attention call needs ("separate query and KV lengths for the
early and late blocks, including any cached prefix" -- SGLang docs,
"Prefill Context Parallelism", §Zigzag strategy; "per-request sharding
metadata preserves those boundaries and each query's causal extent" --
same page, §Interleave strategy).

Plain loops over tokens are used on purpose: the plan is written the way the
pages describe it, one token at a time.
"""

from dataclasses import dataclass
from typing import List

ZIGZAG = "zigzag"
INTERLEAVE = "interleave"


@dataclass(frozen=True)
class Segment:
    q_row0: int      # first row of the segment in O_cat / Q_cat
    q_len: int       # number of rows
    q_pos0: int      # position of row 0 within its request (prefix included)
    q_pos_step: int  # position increment from one row to the next
    kv_row0: int     # row of key position 0 of the request in the KV buffer
    kv_len: int      # key positions visible to the last row (= its position + 1)
    req: int         # request index
    rank: int        # owning CP rank


@dataclass
class Plan:
    cp_size: int
    strategy: str
    rank_rows: List[List[int]]   # per rank: flat new-token indices, in row order
    segments: List[List[Segment]]  # per rank
    row_offsets: List[int]       # [C+1]: first O_cat row of each rank
    gather_idx: List[int]        # O_cat row -> flat new-token index
    positions: List[int]         # O_cat row -> position within its request
    restore_idx: List[int]       # flat new-token index -> O_cat row


def request_tables(new_lens, prefix_lens):
    """Flat start of each request's new tokens and KV start of each request."""
    flat_start, kv_start = [], []
    f = kv = 0
    for n, p in zip(new_lens, prefix_lens):
        flat_start.append(f)
        kv_start.append(kv)
        f += n
        kv += p + n
    return flat_start, kv_start


def zigzag_block_sizes(n, cp_size):
    """Sizes of the 2C contiguous blocks of one request's n new tokens.

    SGLang docs, "Prefill Context Parallelism", §Zigzag strategy: split into
    2C contiguous blocks; "early blocks receive the remainder".  Reading R1:
    each of the first n mod 2C blocks gets one extra token.
    """
    nb = 2 * cp_size
    return [n // nb + (1 if k < n % nb else 0) for k in range(nb)]


def zigzag_ranks_of_blocks(cp_size):
    """Rank owning each of the 2C blocks: rank r takes blocks r and 2C-1-r."""
    owner = [None] * (2 * cp_size)
    for r in range(cp_size):
        owner[r] = r
        owner[2 * cp_size - 1 - r] = r
    return owner


def zigzag_plan(new_lens, prefix_lens, cp_size):
    """Zigzag plan (SGLang docs, "Prefill Context Parallelism", §Zigzag strategy).

    Per request (the split restarts for every request) the new tokens are cut
    into 2C contiguous blocks; rank r receives block r and block 2C-1-r.
    Reading R2: a rank's rows are its blocks request by request in batch
    order, the early block (r) before the late block (2C-1-r).
    """
    C = cp_size
    flat_start, kv_start = request_tables(new_lens, prefix_lens)
    rank_rows = [[] for _ in range(C)]
    rank_blocks = [[] for _ in range(C)]  # (req, first local token, length)
    for b, n in enumerate(new_lens):
        sizes = zigzag_block_sizes(n, C)
        starts = [sum(sizes[:k]) for k in range(2 * C)]
        for r in range(C):
            for k in (r, 2 * C - 1 - r):
                rank_blocks[r].append((b, starts[k], sizes[k]))
                for t in range(starts[k], starts[k] + sizes[k]):
                    rank_rows[r].append(flat_start[b] + t)
    row_offsets = [0]
    for r in range(C):
        row_offsets.append(row_offsets[-1] + len(rank_rows[r]))
    segments = [[] for _ in range(C)]
    for r in range(C):
        row = row_offsets[r]
        for (b, t0, ln) in rank_blocks[r]:
            if ln == 0:
                continue
            p = prefix_lens[b]
            segments[r].append(Segment(q_row0=row, q_len=ln, q_pos0=p + t0,
                                       q_pos_step=1, kv_row0=kv_start[b],
                                       kv_len=p + t0 + ln, req=b, rank=r))
            row += ln
    return _finish(C, ZIGZAG, new_lens, prefix_lens, rank_rows, segments, row_offsets)


def interleave_plan(new_lens, prefix_lens, cp_size):
    """Interleave plan (SGLang docs, "Prefill Context Parallelism", §Interleave strategy).

    Rank r receives flattened new-token indices r, r+C, r+2C, ...; the index
    runs across the whole batch and does not reset at request boundaries;
    positions keep their original values.  A segment is a maximal run of a
    rank's rows inside one request (positions advance by C within it).
    """
    C = cp_size
    flat_start, kv_start = request_tables(new_lens, prefix_lens)
    total = sum(new_lens)
    req_of, local_of = [], []
    for b, n in enumerate(new_lens):
        for t in range(n):
            req_of.append(b)
            local_of.append(t)
    rank_rows = [[] for _ in range(C)]
    for i in range(total):
        rank_rows[i % C].append(i)
    row_offsets = [0]
    for r in range(C):
        row_offsets.append(row_offsets[-1] + len(rank_rows[r]))
    segments = [[] for _ in range(C)]
    for r in range(C):
        j = 0
        rows = rank_rows[r]
        while j < len(rows):
            b = req_of[rows[j]]
            k = j
            while k + 1 < len(rows) and req_of[rows[k + 1]] == b:
                k += 1
            p = prefix_lens[b]
            first, last = local_of[rows[j]], local_of[rows[k]]
            segments[r].append(Segment(q_row0=row_offsets[r] + j, q_len=k - j + 1,
                                       q_pos0=p + first, q_pos_step=C,
                                       kv_row0=kv_start[b], kv_len=p + last + 1,
                                       req=b, rank=r))
            j = k + 1
    return _finish(C, INTERLEAVE, new_lens, prefix_lens, rank_rows, segments, row_offsets)


def _finish(C, strategy, new_lens, prefix_lens, rank_rows, segments, row_offsets):
    flat_start, _ = request_tables(new_lens, prefix_lens)
    req_of, local_of = [], []
    for b, n in enumerate(new_lens):
        for t in range(n):
            req_of.append(b)
            local_of.append(t)
    gather_idx = [i for r in range(C) for i in rank_rows[r]]
    positions = [prefix_lens[req_of[i]] + local_of[i] for i in gather_idx]
    # Restore index (blog "什么是 Context Parallelism", §2.1: a restore index
    # puts the all-gathered, interleaved token order back into causal order).
    restore_idx = [None] * len(gather_idx)
    for row, i in enumerate(gather_idx):
        restore_idx[i] = row
    return Plan(cp_size=C, strategy=strategy, rank_rows=rank_rows, segments=segments,
                row_offsets=row_offsets, gather_idx=gather_idx, positions=positions,
                restore_idx=restore_idx)


def make_plan(new_lens, prefix_lens, cp_size, strategy):
    new_lens = [int(x) for x in new_lens]
    prefix_lens = [int(x) for x in prefix_lens]
    if strategy == ZIGZAG:
        return zigzag_plan(new_lens, prefix_lens, cp_size)
    if strategy == INTERLEAVE:
        return interleave_plan(new_lens, prefix_lens, cp_size)
    raise ValueError(strategy)


def restore(o_cat, restore_idx):
    """O_orig[i] = O_cat[restore_idx[i]] (row gather into causal order)."""
    return [o_cat[restore_idx[i]] for i in range(len(restore_idx))]


def block_tile_loads(block_owner, cp_size):
    """Causal (query block, key block) tile loads per rank at block granularity.

    Blog "什么是 Context Parallelism", §2, the load-balance figure: with the
    sequence in 2C blocks and a causal mask, query block i computes against
    key blocks 0..i, so it costs i + 1 tiles.  ``block_owner[i]`` is the rank
    of query block i.
    """
    loads = [0] * cp_size
    for i, r in enumerate(block_owner):
        for j in range(len(block_owner)):
            if j <= i:
                loads[r] += 1
    return loads


def sequential_block_owner(cp_size):
    """Contiguous split: rank r owns blocks 2r and 2r+1 of 2C."""
    return [k // 2 for k in range(2 * cp_size)]


def visible_pairs(plan, new_lens, prefix_lens):
    """Visible (query, key) pairs per rank, counted one query at a time."""
    out = [0] * plan.cp_size
    for r in range(plan.cp_size):
        for seg in plan.segments[r]:
            for i in range(seg.q_len):
                out[r] += seg.q_pos0 + i * seg.q_pos_step + 1
    return out
