"""GPU parity of the shard-plan kernels against the oracle: bit-exact."""

import pytest
import torch

import context_causal_attention_cp_gb300 as cpa
from context_causal_attention_cp_gb300 import workloads as W
from oracle import plan as oplan

pytestmark = pytest.mark.gpu


def _oracle_segments(op):
    out = []
    for r in range(op.cp_size):
        for s in op.segments[r]:
            out.append([s.q_row0, s.q_len, s.q_pos0, s.q_pos_step, s.kv_row0, s.kv_len,
                        op.gather_idx[s.q_row0], s.req])
    return out


def _tile_key(seg, t):
    last = min(seg[1], (t + 1) * 128) - 1
    keys = seg[2] + last * seg[3] + 1
    return min((keys + 127) // 128, 4095)


def check_plan(new, pre, C, strategy):
    status = cpa.new_status()
    plan = cpa.make_plan(new, pre, C, strategy, status=status)
    cpa.check_status(status, "cp_shard_plan")
    op = oplan.make_plan(new, pre, C, strategy)
    N, S, T = plan.total_rows, plan.total_segs, plan.total_tiles
    segs = plan.segs[:S].cpu().tolist()
    assert segs == _oracle_segments(op)
    seg_off = [0]
    for r in range(C):
        seg_off.append(seg_off[-1] + len(op.segments[r]))
    assert plan.seg_offsets.cpu().tolist() == seg_off
    assert plan.row_offsets.cpu().tolist() == op.row_offsets
    assert plan.gather_idx[:N].cpu().tolist() == op.gather_idx
    assert plan.positions[:N].cpu().tolist() == op.positions
    assert plan.restore_idx[:N].cpu().tolist() == op.restore_idx
    # tile list: every (segment, tile) exactly once, heaviest first
    tiles = [tuple(x) for x in plan.tiles[:T].cpu().tolist()]
    expect = sorted((s, t) for s, seg in enumerate(segs)
                    for t in range((seg[1] + 127) // 128))
    assert sorted(tiles) == expect
    keys = [_tile_key(segs[s], t) for s, t in tiles]
    assert keys == sorted(keys, reverse=True)


def test_page_examples():
    check_plan([16], [0], 4, "zigzag")
    check_plan([16], [0], 4, "interleave")
    check_plan([5, 3], [0, 0], 4, "interleave")


@pytest.mark.parametrize("seed", range(24))
@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_random_batches(seed, strategy):
    new, pre = W.random_batch(seed, max_reqs=9, max_new=900, max_prefix=300)
    C = [1, 2, 3, 4, 8, 7][seed % 6]
    check_plan(new, pre, C, strategy)


def test_short_and_empty_requests():
    check_plan([3, 0, 1, 7], [17, 0, 2, 0], 4, "zigzag")
    check_plan([3, 0, 1, 7], [17, 0, 2, 0], 4, "interleave")
    check_plan([0, 0], [5, 0], 2, "zigzag")


def test_many_requests():
    new = [(i * 37) % 23 for i in range(3000)]
    pre = [(i * 11) % 5 for i in range(3000)]
    check_plan(new, pre, 8, "zigzag")
    check_plan(new, pre, 8, "interleave")


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_workload_plans(name):
    w = W.WORKLOADS[name]
    for strategy in w.strategies:
        check_plan(w.new_lens, w.prefix_lens, w.cp_size, strategy)


def test_size_mismatch_sets_status():
    plan = cpa.alloc_plan([100, 50], [0, 0], 4, "zigzag")
    plan.rows_per_rank = [x + 1 for x in plan.rows_per_rank]   # lie about the totals
    status = cpa.new_status()
    cpa.cp_shard_plan(plan, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -1


def test_maximum_cp_size():
    """C = CPATTN_MAX_CP (1024): 2048 zigzag blocks per request, most of them
    empty or single-token."""
    check_plan([2100, 5, 4096], [0, 3, 100], 1024, "zigzag")
    check_plan([2100, 5, 4096], [0, 3, 100], 1024, "interleave")


def test_maximum_request_count():
    """num_reqs = CPATTN_MAX_REQS (65536) tiny requests, including empty ones."""
    n = 65536
    new = [(i * 7) % 5 for i in range(n)]
    pre = [(i * 3) % 4 for i in range(n)]
    check_plan(new, pre, 2, "zigzag")
    check_plan(new, pre, 3, "interleave")

