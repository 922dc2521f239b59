"""GPU parity of the benchmark-size workloads against the oracle on at least
512 query rows x all heads, through the exact calls the bench times.

Rows: every segment's first and last row, both edge rows of the plan's
128-row query tiles (every tile, or every few tiles on the 128K workload),
and seeded random rows up to at least 512.  The oracle evaluates exactly those
rows in fp64 (spread over host processes by ``oracle_rows``).  Tolerances as
everywhere: max-abs 2e-2 on O, 1e-5 relative (floor 1) on the natural-log LSE.
"""

import numpy as np
import pytest
import torch

import context_causal_attention_cp_gb300 as cpa
from context_causal_attention_cp_gb300 import workloads as W
from oracle import attention as oatt
from oracle import plan as oplan

import oracle_rows
from gpu_common import assert_attn_close, np64

pytestmark = pytest.mark.gpu

MIN_ROWS = 512


def scale_rows(w, strategy, seed, tile_stride=1, target=MIN_ROWS):
    """Flat token indices: segment edges, query-tile edges and random rows."""
    plan = oplan.make_plan(w.new_lens, w.prefix_lens, w.cp_size, strategy)
    rows = set()
    for r in range(w.cp_size):
        for s in plan.segments[r]:
            rows.add(plan.gather_idx[s.q_row0])
            rows.add(plan.gather_idx[s.q_row0 + s.q_len - 1])
            for t in range(0, (s.q_len + 127) // 128, tile_stride):
                rows.add(plan.gather_idx[s.q_row0 + 128 * t])
                rows.add(plan.gather_idx[s.q_row0 + min(s.q_len, 128 * t + 128) - 1])
    while len(rows) < target + 32:
        rows |= set(W.sample_rows(seed, w.total_new, target + 32 - len(rows)))
        seed += 1000
    rows = sorted(rows)
    assert len(rows) >= target
    return rows


def oracle_for(w, inputs, rows):
    q = np64(inputs["q"][torch.as_tensor(rows, dtype=torch.long)])
    k64 = np64(inputs["k"])
    v64 = k64[:, :, : w.dv] if w.v_is_k_prefix else np64(inputs["v"])
    pos, kv0 = oatt.token_tables(w.new_lens, w.prefix_lens)
    r = np.asarray(rows, dtype=np.int64)
    return oracle_rows.attention_rows_parallel(q, k64, v64, pos[r], kv0[r], w.scale,
                                               v_is_k_prefix=w.v_is_k_prefix)


def check_rows(o, lse, rows, O_ref, L_ref, what):
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    assert o.shape[1] == O_ref.shape[1]          # all heads
    assert_attn_close(o[idx], lse[idx], O_ref, L_ref, f"{what} ({len(rows)} rows x all heads)")


def test_llama8b_32k_bench_call_at_scale():
    """cp_attn_prefill (queries read and O / LSE written by token index), the
    call the 32K bench step times, after the device plan."""
    w = W.WORKLOADS["llama8b_32k"]
    inputs = W.make_inputs(w)
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", status=status)
    q, k, v = inputs["q"].cuda(), inputs["k"].cuda(), inputs["v"].cuda()
    o, lse = cpa.cp_attn_prefill(plan.segs, q, k, v, w.scale, num_segs=plan.total_segs,
                                 tiles=plan.tiles, num_tiles=plan.total_tiles, status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    rows = scale_rows(w, "zigzag", 31)
    O_ref, L_ref = oracle_for(w, inputs, rows)
    check_rows(o, lse, rows, O_ref, L_ref, "32k cp_attn_prefill")


def test_mla_16k_bench_call_at_scale():
    """The MLA bench step: query gather into shard order, then
    cp_attn_partial_restore (V = the latent view of K, the restore in the
    store)."""
    w = W.WORKLOADS["mla_16k"]
    inputs = W.make_inputs(w)
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "interleave", status=status)
    k = inputs["k"].cuda()
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
    o, lse = cpa.cp_attn_partial_restore(plan.segs, q_cat, k, k[:, :, : w.dv], w.scale,
                                         plan.gather_idx, num_out_rows=w.total_new,
                                         num_segs=plan.total_segs, tiles=plan.tiles,
                                         num_tiles=plan.total_tiles, status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    rows = scale_rows(w, "interleave", 32)
    O_ref, L_ref = oracle_for(w, inputs, rows)
    check_rows(o, lse, rows, O_ref, L_ref, "mla 16k cp_attn_partial_restore")


@pytest.fixture(scope="module")
def case_128k():
    w = W.WORKLOADS["partialkv_128k"]
    inputs = W.make_inputs(w)
    rows = scale_rows(w, "zigzag", 33, tile_stride=8)
    O_ref, L_ref = oracle_for(w, inputs, rows)
    return w, inputs, rows, O_ref, L_ref


def test_partialkv_128k_one_call_at_scale(case_128k):
    """cp_attn_partial_kv (layout, split-KV attention over 16 KV blocks of
    8192, fused LSE merge and restore), the call the 128K bench step times."""
    w, inputs, rows, O_ref, L_ref = case_128k
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", status=status)
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
    o, lse, ws = cpa.cp_attn_partial_kv(plan, q_cat, inputs["k"].cuda(), inputs["v"].cuda(),
                                        w.scale, w.kv_block, status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    del ws
    check_rows(o, lse, rows, O_ref, L_ref, "128k cp_attn_partial_kv")


def test_partialkv_128k_pass_q_ring_at_scale(case_128k):
    """The pass-Q ring (cp_attn_pass_q over the library's schedule) and the
    restore of O and LSE, as the bench's pass-Q step runs them."""
    w, inputs, rows, O_ref, L_ref = case_128k
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", status=status)
    N = w.total_new
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[:N], status=status)
    o_cat, l_cat = cpa.cp_pass_q_attention(q_cat, inputs["k"].cuda(), inputs["v"].cuda(), plan,
                                           w.scale, status=status)
    o = cpa.cp_restore(o_cat, plan.restore_idx[:N], status=status)
    lse = cpa.cp_restore(l_cat, plan.restore_idx[:N], status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    check_rows(o, lse, rows, O_ref, L_ref, "128k pass-Q ring")
