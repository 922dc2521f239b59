"""GPU parity of the fused store variants.

* Restore fused into the attention store (cp_attn_partial_restore, blog
  "什么是 Context Parallelism" §2.1: the restore index after the all-gather):
  bit-identical to attention followed by a separate restore pass, and equal
  to the oracle.
* One pass-Q hop (cp_attn_partial_accumulate, blog §3.3.2 "Pass Q"): the new
  partial merged into a carried accumulator equals the oracle's LSE merge of
  the two, including empty sides.
* The pass-Q ring built from those hops equals dense causal attention.
"""

import math

import numpy as np
import pytest
import torch

import context_causal_attention_cp_gb300 as cpa
from context_causal_attention_cp_gb300 import workloads as W
from oracle import attention as oatt
from oracle import merge as omerge

from gpu_common import assert_attn_close, boundary_rows, np64, oracle_dense_rows

pytestmark = pytest.mark.gpu

SMALL = [("single1k_d64", "zigzag"), ("varlen6_gqa", "zigzag"), ("varlen6_gqa", "interleave")]


def setup(w, strategy, inputs=None):
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, strategy, status=status)
    inputs = inputs or W.make_inputs(w)
    q = inputs["q"].cuda()
    k = inputs["k"].cuda()
    v = k[:, :, : w.dv] if w.v_is_k_prefix else inputs["v"].cuda()
    return status, plan, inputs, q, k, v


def mla_case(new, pre, Hq, C, seed):
    return W.Workload(name=f"mla{seed}", new_lens=new, prefix_lens=pre, Hq=Hq, Hkv=1, d=576,
                      dv=512, scale=1 / math.sqrt(192), std=0.1, cp_size=C,
                      strategies=["zigzag", "interleave"], seed=seed, v_is_k_prefix=True)


def dense_ref(w, inputs):
    k64 = np64(inputs["k"])
    v64 = k64[:, :, : w.dv] if w.v_is_k_prefix else np64(inputs["v"])
    return oatt.dense_causal_attention(np64(inputs["q"]), k64, v64, w.new_lens, w.prefix_lens,
                                       w.scale)


# ---------------------------------------------------------- fused restore ----

@pytest.mark.parametrize("name,strategy",
                         SMALL + [("llama8b_32k", "zigzag"), ("mla_16k", "interleave")])
def test_fused_restore_is_bit_identical_to_separate_restore(name, strategy):
    w = W.WORKLOADS[name]
    status, plan, inputs, q, k, v = setup(w, strategy)
    o1, l1 = cpa.cp_prefill_attention(q, k, v, plan, w.scale, status=status)
    o2, l2 = cpa.cp_prefill_attention(q, k, v, plan, w.scale, status=status, fuse_restore=True)
    torch.cuda.synchronize()
    cpa.check_status(status, name)
    assert torch.equal(o1, o2)
    assert torch.equal(l1, l2)


@pytest.mark.parametrize("name,strategy", SMALL)
def test_fused_restore_all_rows(name, strategy):
    w = W.WORKLOADS[name]
    status, plan, inputs, q, k, v = setup(w, strategy)
    o, lse = cpa.cp_prefill_attention(q, k, v, plan, w.scale, status=status, fuse_restore=True)
    torch.cuda.synchronize()
    cpa.check_status(status, name)
    O_ref, L_ref = dense_ref(w, inputs)
    assert_attn_close(o, lse, O_ref, L_ref, f"{name}/{strategy}/fused")


@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_fused_restore_mla_small(strategy):
    w = mla_case([300, 77], [0, 40], 4, 3, 931)
    status, plan, inputs, q, k, v = setup(w, strategy)
    o, lse = cpa.cp_prefill_attention(q, k, v, plan, w.scale, status=status, fuse_restore=True)
    torch.cuda.synchronize()
    cpa.check_status(status, "mla")
    O_ref, L_ref = dense_ref(w, inputs)
    assert_attn_close(o, lse, O_ref, L_ref, f"mla/{strategy}/fused")


def test_fused_restore_bad_destination_sets_range():
    """A destination outside the output sets CPATTN_ERR_RANGE; that row alone
    is skipped, every other row is written as usual."""
    w = W.WORKLOADS["single1k_d64"]
    status, plan, inputs, q, k, v = setup(w, "zigzag")
    N = w.total_new
    q_cat = cpa.cp_restore(q, plan.gather_idx[:N])
    ref_o, ref_l = cpa.cp_attn_partial_restore(plan.segs, q_cat, k, v, w.scale, plan.gather_idx,
                                               num_out_rows=N, num_segs=plan.total_segs)
    dst = plan.gather_idx[:N].clone()
    lost = int(dst[5].item())
    dst[5] = N + 3
    o = torch.full((N, w.Hq, w.dv), float("nan"), dtype=torch.bfloat16, device="cuda")
    lse = torch.full((N, w.Hq), float("nan"), dtype=torch.float32, device="cuda")
    status.zero_()
    cpa.cp_attn_partial_restore(plan.segs, q_cat, k, v, w.scale, dst, num_out_rows=N,
                                num_segs=plan.total_segs, out=o, lse=lse, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    assert torch.isnan(o[lost]).all() and torch.isnan(lse[lost]).all()
    keep = torch.ones(N, dtype=torch.bool, device="cuda")
    keep[lost] = False
    assert torch.equal(o[keep], ref_o[keep])
    assert torch.equal(lse[keep], ref_l[keep])


# ------------------------------------------------------ pass-Q accumulate ----

@pytest.mark.parametrize("shape", [(8, 8, 64), (32, 8, 128), (4, 1, 576)])
def test_accumulate_merges_into_carried_partial(shape):
    """One hop: (O_acc, L_acc) random, some rows empty; the key window
    [100, 250) leaves the rows at positions < 100 with an empty new partial."""
    Hq, Hkv, d = shape
    mla = d == 576
    dv = 512 if mla else d
    w = W.Workload(name=f"acc{d}", new_lens=[300], prefix_lens=[40], Hq=Hq, Hkv=Hkv, d=d, dv=dv,
                   scale=1 / math.sqrt(192 if mla else d), std=0.1 if mla else 1.0, cp_size=2,
                   strategies=["zigzag"], seed=1201 + d, v_is_k_prefix=mla)
    status, plan, inputs, q, k, v = setup(w, "zigzag")
    N = w.total_new
    q_cat = cpa.cp_restore(q, plan.gather_idx[:N])
    gen = torch.Generator().manual_seed(55 + d)
    o0 = torch.randn((N, Hq, dv), generator=gen, dtype=torch.float32)
    l0 = torch.randn((N, Hq), generator=gen, dtype=torch.float32) * 3.0 + 2.0
    o0[:10] = 0.0          # cat rows 0..9 (positions 40..49): both sides empty
    l0[:10] = float("-inf")
    o0[200:220] = 0.0      # empty accumulator, non-empty new partial
    l0[200:220] = float("-inf")
    o_acc = o0.cuda()
    la = l0.cuda()
    lb = torch.full_like(la, float("nan"))
    cpa.cp_attn_partial_accumulate(plan.segs, q_cat, k, v, w.scale, o_acc, la, lb,
                                   num_segs=plan.total_segs, kv_lo=100, kv_hi=250, status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    flat = plan.gather_idx[:N].cpu().numpy()
    k64 = np64(inputs["k"])
    v64 = k64[:, :, :dv] if mla else np64(inputs["v"])
    O_p, L_p = oracle_dense_rows(inputs, w.new_lens, w.prefix_lens, w.scale, flat, kv_lo=100,
                                 kv_hi=250, k64=k64, v64=v64)
    assert np.isneginf(L_p[:10]).all()
    O_ref, L_ref = omerge.lse_merge(np.stack([o0.double().numpy(), O_p]),
                                    np.stack([l0.double().numpy(), L_p]))
    assert_attn_close(o_acc, lb, O_ref, L_ref, f"{w.name}/accumulate")
    assert torch.equal(la.cpu(), l0)  # the input LSE is only read


@pytest.mark.parametrize("shape", [(32, 8, 128), (4, 1, 576)])
def test_accumulate_per_segment_windows_match_single_calls(shape):
    """Per-segment key windows (one launch) give bit for bit what one call per
    segment with that window gives, including empty and unbounded windows."""
    Hq, Hkv, d = shape
    mla = d == 576
    dv = 512 if mla else d
    w = W.Workload(name=f"win{d}", new_lens=[517, 33, 1000, 3], prefix_lens=[0, 17, 256, 5],
                   Hq=Hq, Hkv=Hkv, d=d, dv=dv, scale=1 / math.sqrt(192 if mla else d),
                   std=0.1 if mla else 1.0, cp_size=3, strategies=["zigzag"], seed=1301 + d,
                   v_is_k_prefix=mla)
    status, plan, inputs, q, k, v = setup(w, "zigzag")
    N = w.total_new
    q_cat = cpa.cp_restore(q, plan.gather_idx[:N])
    S = plan.total_segs
    gen = torch.Generator().manual_seed(77 + d)
    lo = torch.randint(0, 600, (S,), generator=gen, dtype=torch.int32)
    hi = lo + torch.randint(0, 700, (S,), generator=gen, dtype=torch.int32)
    hi[::5] = -1                       # unbounded
    lo[1::7] = 2000                    # past every row: empty window
    wins = torch.stack([lo, hi], 1).contiguous()
    o0 = torch.randn((N, Hq, dv), generator=gen, dtype=torch.float32)
    l0 = torch.randn((N, Hq), generator=gen, dtype=torch.float32)
    o_a, la, lb = o0.cuda(), l0.cuda(), torch.full((N, Hq), float("nan"), device="cuda")
    cpa.cp_attn_partial_accumulate(plan.segs, q_cat, k, v, w.scale, o_a, la, lb, num_segs=S,
                                   seg_windows=wins.cuda(), status=status)
    o_b, lc, ld = o0.cuda(), l0.cuda(), torch.full((N, Hq), float("nan"), device="cuda")
    for i in range(S):
        cpa.cp_attn_partial_accumulate(plan.segs[i:i + 1], q_cat, k, v, w.scale, o_b, lc, ld,
                                       kv_lo=int(lo[i]), kv_hi=int(hi[i]), status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    assert torch.equal(o_a, o_b)
    assert torch.equal(lb, ld)


def test_accumulate_refuses_overlapping_lse():
    w = W.WORKLOADS["single1k_d64"]
    status, plan, inputs, q, k, v = setup(w, "zigzag")
    N = w.total_new
    o_acc = torch.zeros((N, w.Hq, w.dv), dtype=torch.float32, device="cuda")
    la = torch.full((N, w.Hq), float("-inf"), device="cuda")
    with pytest.raises(cpa.api.L.CpAttnError):
        cpa.cp_attn_partial_accumulate(plan.segs, q, k, v, w.scale, o_acc, la, la,
                                       num_segs=plan.total_segs)


# ----------------------------------------------------------- pass-Q ring ----

def run_pass_q(w, strategy, inputs=None):
    status, plan, inputs, q, k, v = setup(w, strategy, inputs)
    N = w.total_new
    q_cat = cpa.cp_restore(q, plan.gather_idx[:N])
    o_cat, l_cat = cpa.cp_pass_q_attention(q_cat, k, v, plan, w.scale, status=status)
    o = cpa.cp_restore(o_cat, plan.restore_idx[:N])
    lse = cpa.cp_restore(l_cat, plan.restore_idx[:N])
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    return o, lse, inputs


@pytest.mark.parametrize("name,strategy", SMALL)
def test_pass_q_ring_all_rows(name, strategy):
    w = W.WORKLOADS[name]
    o, lse, inputs = run_pass_q(w, strategy)
    O_ref, L_ref = dense_ref(w, inputs)
    assert_attn_close(o, lse, O_ref, L_ref, f"{name}/{strategy}/pass-q")


@pytest.mark.parametrize("seed", range(4))
def test_pass_q_ring_random_batches(seed):
    new, pre = W.random_batch(300 + seed, max_reqs=4, max_new=300, max_prefix=150)
    if sum(new) == 0:
        new[0] = 7
    w = W.Workload(name=f"pq{seed}", new_lens=new, prefix_lens=pre, Hq=4, Hkv=2, d=128, dv=128,
                   scale=1 / math.sqrt(128), std=1.0, cp_size=[2, 3, 4, 8][seed],
                   strategies=["zigzag", "interleave"], seed=6100 + seed)
    inputs = W.make_inputs(w)
    O_ref, L_ref = dense_ref(w, inputs)
    for strategy in w.strategies:
        o, lse, _ = run_pass_q(w, strategy, inputs)
        assert_attn_close(o, lse, O_ref, L_ref, f"{w.name}/{strategy}/pass-q")


def test_pass_q_ring_mla_small():
    w = mla_case([260, 33], [20, 0], 4, 2, 941)
    o, lse, inputs = run_pass_q(w, "zigzag")
    O_ref, L_ref = dense_ref(w, inputs)
    assert_attn_close(o, lse, O_ref, L_ref, "mla/pass-q")


def test_pass_q_ring_128k_sampled():
    w = W.WORKLOADS["partialkv_128k"]
    o, lse, inputs = run_pass_q(w, "zigzag")
    rows = boundary_rows(w.new_lens, w.prefix_lens, w.cp_size, "zigzag",
                         W.sample_rows(21, w.total_new, 4))[::2]
    O_ref, L_ref = oracle_dense_rows(inputs, w.new_lens, w.prefix_lens, w.scale, rows)
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    assert_attn_close(o[idx], lse[idx], O_ref, L_ref, "128k/pass-q")


# ------------------------------------------------------ host pipeline ----

def _host_batch(w, b, v_is_k_prefix=False):
    ho = torch.empty((w.total_new, w.Hq, w.dv), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((w.total_new, w.Hq), dtype=torch.float32).pin_memory()
    return (b["q"].pin_memory(), b["k"].pin_memory(),
            None if v_is_k_prefix else b["v"].pin_memory(), ho, hl)


@pytest.mark.parametrize("name,strategy", [("varlen6_gqa", "zigzag"), ("varlen6_gqa", "interleave"),
                                           ("single1k_d64", "zigzag")])
def test_prefill_host_matches_single_calls(name, strategy):
    """Batches run host to host by cp_prefill_host (two device buffer sets,
    three streams) give exactly what one cp_prefill_attention call gives on
    each batch, and match the oracle."""
    w = W.WORKLOADS[name]
    batches = [W.make_inputs(w, seed_offset=i) for i in range(5)]
    host = [_host_batch(w, b) for b in batches]
    status = cpa.new_status()
    _, streams = cpa.cp_prefill_host(w.new_lens, w.prefix_lens, w.cp_size, strategy, w.Hq, w.Hkv,
                                     w.d, w.dv, w.scale, host, status=status)
    streams[2].synchronize()
    cpa.check_status(status, "host prefill")
    for b, (_, _, _, ho, hl) in zip(batches, host):
        st, plan, _, q, k, v = setup(w, strategy, b)
        o, lse = cpa.cp_prefill_attention(q, k, v, plan, w.scale, status=st, fuse_restore=True)
        torch.cuda.synchronize()
        assert torch.equal(ho, o.cpu())
        assert torch.equal(hl, lse.cpu())
    O_ref, L_ref = dense_ref(w, batches[-1])
    assert_attn_close(host[-1][3], host[-1][4], O_ref, L_ref, f"{name}/{strategy}/host prefill")


def test_prefill_host_mla_latent_view():
    w = mla_case([300, 77], [0, 40], 4, 3, 951)
    b = W.make_inputs(w)
    host = [_host_batch(w, b, v_is_k_prefix=True)]
    status = cpa.new_status()
    _, streams = cpa.cp_prefill_host(w.new_lens, w.prefix_lens, w.cp_size, "interleave", w.Hq,
                                     w.Hkv, w.d, w.dv, w.scale, host, v_is_k_prefix=True,
                                     status=status)
    streams[2].synchronize()
    cpa.check_status(status, "host prefill mla")
    O_ref, L_ref = dense_ref(w, b)
    assert_attn_close(host[0][3], host[0][4], O_ref, L_ref, "mla/host prefill")


def test_prefill_host_one_stream():
    """The same call with one stream for all three roles (nothing overlaps)."""
    w = W.WORKLOADS["varlen6_gqa"]
    b = W.make_inputs(w, seed_offset=3)
    host = [_host_batch(w, b) for _ in range(3)]
    s = torch.cuda.Stream()
    status = cpa.new_status()
    cpa.cp_prefill_host(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", w.Hq, w.Hkv, w.d, w.dv,
                        w.scale, host, status=status, streams=(s, s, s))
    s.synchronize()
    cpa.check_status(status, "host prefill, one stream")
    O_ref, L_ref = dense_ref(w, b)
    for i in range(3):
        assert_attn_close(host[i][3], host[i][4], O_ref, L_ref, f"one stream, batch {i}")


# -------------------------------------------------- token-order prefill ----

@pytest.mark.parametrize("name", ["single1k_d64", "varlen6_gqa", "llama8b_32k"])
def test_token_rows_prefill_matches_gather_path(name):
    """cp_attn_prefill (queries read and outputs written by token index, zigzag
    plan) equals, bit for bit, the gather + attention with the restore store."""
    w = W.WORKLOADS[name]
    status, plan, inputs, q, k, v = setup(w, "zigzag")
    N = w.total_new
    o1, l1 = cpa.cp_attn_prefill(plan.segs, q, k, v, w.scale, num_segs=plan.total_segs,
                                 tiles=plan.tiles, num_tiles=plan.total_tiles, status=status)
    q_cat = cpa.cp_restore(q, plan.gather_idx[:N], status=status)
    o2, l2 = cpa.cp_attn_partial_restore(plan.segs, q_cat, k, v, w.scale, plan.gather_idx,
                                         num_out_rows=N, num_segs=plan.total_segs,
                                         tiles=plan.tiles, num_tiles=plan.total_tiles,
                                         status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, name)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_token_rows_prefill_mla_small():
    w = mla_case([300, 77], [0, 40], 4, 3, 961)
    status, plan, inputs, q, k, v = setup(w, "zigzag")
    o, lse = cpa.cp_attn_prefill(plan.segs, q, k, v, w.scale, num_segs=plan.total_segs,
                                 status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, "mla token rows")
    O_ref, L_ref = dense_ref(w, inputs)
    assert_attn_close(o, lse, O_ref, L_ref, "mla token rows")


def test_token_rows_prefill_refuses_strided_segments():
    """Interleave segments (position step C > 1) are not token runs: their
    tiles set CPATTN_ERR_RANGE and are skipped."""
    w = W.WORKLOADS["varlen6_gqa"]
    status, plan, inputs, q, k, v = setup(w, "interleave")
    status.zero_()
    out = torch.full((w.total_new, w.Hq, w.dv), float("nan"), dtype=torch.bfloat16,
                     device="cuda")
    cpa.cp_attn_prefill(plan.segs, q, k, v, w.scale, num_segs=plan.total_segs, out=out,
                        status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    assert torch.isnan(out).all()


# ------------------------------------------------------------ empty batch ----

@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_batch_without_new_tokens_is_a_no_op(strategy):
    """Requests with a cached prefix but no new tokens: every path returns
    empty outputs and a clean status, and launches nothing that could read
    the empty query buffer."""
    w = W.Workload(name="empty", new_lens=[0, 0], prefix_lens=[5, 0], Hq=4, Hkv=2, d=128,
                   dv=128, scale=1 / math.sqrt(128), std=1.0, cp_size=2,
                   strategies=[strategy], seed=17, kv_block=64)
    status, plan, _, q, k, v = setup(w, strategy)
    assert q.shape[0] == 0 and plan.total_segs == 0
    outs = [cpa.cp_prefill_attention(q, k, v, plan, w.scale, status=status, fuse_restore=f)
            for f in (False, True)]
    o, lse, _ = cpa.cp_attn_partial_kv(plan, q, k, v, w.scale, w.kv_block, status=status)
    outs.append((o, lse))
    outs.append(cpa.cp_pass_q_attention(q, k, v, plan, w.scale, status=status))
    torch.cuda.synchronize()
    cpa.check_status(status, "empty batch")
    for o, lse in outs:
        assert tuple(o.shape) == (0, w.Hq, w.dv) and tuple(lse.shape) == (0, w.Hq)
