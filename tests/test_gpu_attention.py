"""GPU parity of shard attention, merge and restore against the oracle.

Small workloads are compared on every row; the large ones (32K, MLA 16K,
128K partial-KV) on seeded row samples that always include each segment's
first and last rows and tile boundaries.  Tolerances: max-abs 2e-2 on O,
1e-5 relative (floor 1) on the natural-log LSE, exact for permutations.
"""

import math

import numpy as np
import pytest
import torch

import context_causal_attention_cp_gb300 as cpa
from context_causal_attention_cp_gb300 import workloads as W
from oracle import attention as oatt
from oracle import merge as omerge
from oracle import plan as oplan

from gpu_common import (assert_attn_close, boundary_rows, np64, oracle_dense_rows,
                        stepwise_partial_kv)

pytestmark = pytest.mark.gpu


def run_full_kv(w, strategy, inputs):
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, strategy, status=status)
    q = inputs["q"].cuda()
    k = inputs["k"].cuda()
    v = k[:, :, : w.dv] if w.v_is_k_prefix else inputs["v"].cuda()
    o, lse = cpa.cp_prefill_attention(q, k, v, plan, w.scale, status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    return o, lse


def random_case(seed, Hq, Hkv, d, max_reqs=4, max_new=400, max_prefix=200):
    new, pre = W.random_batch(seed, max_reqs=max_reqs, max_new=max_new, max_prefix=max_prefix)
    if sum(new) == 0:
        new[0] = 5
    w = W.Workload(name=f"rand{seed}", new_lens=new, prefix_lens=pre, Hq=Hq, Hkv=Hkv, d=d,
                   dv=d, scale=1.0 / math.sqrt(d), std=1.0, cp_size=[1, 2, 3, 4, 8][seed % 5],
                   strategies=["zigzag", "interleave"], seed=5000 + seed)
    return w


# ------------------------------------------------------------- full rows ----

@pytest.mark.parametrize("strategy", ["zigzag"])
def test_single1k_d64_all_rows(strategy):
    w = W.WORKLOADS["single1k_d64"]
    inputs = W.make_inputs(w)
    o, lse = run_full_kv(w, strategy, inputs)
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]),
                                               np64(inputs["v"]), w.new_lens, w.prefix_lens,
                                               w.scale)
    assert_attn_close(o, lse, O_ref, L_ref, w.name)


@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_varlen6_gqa_all_rows(strategy):
    w = W.WORKLOADS["varlen6_gqa"]
    inputs = W.make_inputs(w)
    o, lse = run_full_kv(w, strategy, inputs)
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]),
                                               np64(inputs["v"]), w.new_lens, w.prefix_lens,
                                               w.scale)
    assert_attn_close(o, lse, O_ref, L_ref, f"{w.name}/{strategy}")


@pytest.mark.parametrize("seed", range(10))
@pytest.mark.parametrize("heads", [(4, 2, 64), (2, 2, 128), (6, 2, 128), (3, 1, 64)])
def test_random_batches_all_rows(seed, heads):
    Hq, Hkv, d = heads
    w = random_case(seed, Hq, Hkv, d)
    inputs = W.make_inputs(w)
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]),
                                               np64(inputs["v"]), w.new_lens, w.prefix_lens,
                                               w.scale)
    for strategy in w.strategies:
        o, lse = run_full_kv(w, strategy, inputs)
        assert_attn_close(o, lse, O_ref, L_ref, f"{w.name}/{strategy}/{heads}")


# ---------------------------------------------------------- large, sampled ----

def test_llama8b_32k_sampled():
    w = W.WORKLOADS["llama8b_32k"]
    inputs = W.make_inputs(w)
    o, lse = run_full_kv(w, "zigzag", inputs)
    rows = boundary_rows(w.new_lens, w.prefix_lens, w.cp_size, "zigzag",
                         W.sample_rows(7, w.total_new, 24))
    O_ref, L_ref = oracle_dense_rows(inputs, w.new_lens, w.prefix_lens, w.scale, rows)
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    assert_attn_close(o[idx], lse[idx], O_ref, L_ref, w.name)


def test_partial_kv_small_all_rows():
    # ring-style decomposition on a small batch: windows of 192 keys (not a
    # multiple of the 128-key tile), merged and scattered to original order
    w = W.Workload(name="pkv_small", new_lens=[700, 300, 5], prefix_lens=[0, 130, 9], Hq=8,
                   Hkv=2, d=128, dv=128, scale=1 / math.sqrt(128), std=1.0, cp_size=3,
                   strategies=["zigzag", "interleave"], seed=777, kv_block=192)
    inputs = W.make_inputs(w)
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]),
                                               np64(inputs["v"]), w.new_lens, w.prefix_lens,
                                               w.scale)
    for strategy in w.strategies:
        status = cpa.new_status()
        plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, strategy, status=status)
        q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
        o, lse = stepwise_partial_kv(q_cat, inputs["k"].cuda(), inputs["v"].cuda(), plan,
                                             w.scale, w.kv_block, status=status)
        torch.cuda.synchronize()
        cpa.check_status(status, "partial kv")
        assert_attn_close(o, lse, O_ref, L_ref, f"pkv/{strategy}")


def test_partialkv_128k_sampled():
    w = W.WORKLOADS["partialkv_128k"]
    inputs = W.make_inputs(w)
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", status=status)
    k = inputs["k"].cuda()
    v = inputs["v"].cuda()
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
    o, lse = stepwise_partial_kv(q_cat, k, v, plan, w.scale, w.kv_block, status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    rows = sorted(set(W.sample_rows(11, w.total_new, 16) +
                      [0, 8191, 8192, 65535, 65536, 131071]))
    O_ref, L_ref = oracle_dense_rows(inputs, w.new_lens, w.prefix_lens, w.scale, rows)
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    assert_attn_close(o[idx], lse[idx], O_ref, L_ref, w.name)


# --------------------------------------------------------------- partials ----

@pytest.mark.parametrize("Hq,Hkv,d", [(4, 2, 128), (8, 8, 64), (2, 1, 576), (1, 1, 576)])
def test_windowed_partials_and_empty_windows(Hq, Hkv, d):
    """cp_attn_partial in partial mode: fp32 O, windows, empty rows -> (0, -inf);
    every kernel family (MLA: the pair kernel for two heads, the single-SM
    kernel for one)."""
    mla = d == 576
    if mla:
        new, pre = W.random_batch(3, max_reqs=4, max_new=500, max_prefix=50)
        w = W.Workload(name="win_mla", new_lens=new, prefix_lens=pre, Hq=Hq, Hkv=Hkv, d=576,
                       dv=512, scale=1 / math.sqrt(192), std=0.5, cp_size=2,
                       strategies=["zigzag"], seed=5103, v_is_k_prefix=True)
    else:
        w = random_case(3, Hq, Hkv, d, max_new=500, max_prefix=50)
    inputs = W.make_inputs(w)
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, 2, "zigzag", status=status)
    N = w.total_new
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[:N], status=status)
    k = inputs["k"].cuda()
    v = k[:, :, :512] if mla else inputs["v"].cuda()
    op = oplan.make_plan(w.new_lens, w.prefix_lens, 2, "zigzag")
    pos = np.asarray(op.positions)
    kv0 = np.asarray([oatt.token_tables(w.new_lens, w.prefix_lens)[1][i] for i in op.gather_idx])
    q64 = np64(inputs["q"])[np.asarray(op.gather_idx)]
    k64 = np64(inputs["k"])
    v64 = k64[:, :, :512] if mla else np64(inputs["v"])
    for lo, hi in [(0, 100), (37, 300), (256, 384), (400, 10 ** 6), (10 ** 6, -1)]:
        o, lse = cpa.cp_attn_partial(plan.segs, q_cat, k, v, w.scale,
                                     num_segs=plan.total_segs, kv_lo=lo, kv_hi=hi,
                                     out_fp32=True, status=status)
        torch.cuda.synchronize()
        cpa.check_status(status, "window")
        O_ref, L_ref = oatt.attention_rows(q64, k64, v64, pos, kv0, w.scale, lo,
                                           None if hi < 0 else hi)
        assert o.dtype == torch.float32
        assert_attn_close(o, lse, O_ref, L_ref, f"window {lo}:{hi}")


def test_merge_matches_oracle():
    g = torch.Generator().manual_seed(42)
    for n, rows, Hq, dv in [(1, 5, 3, 128), (3, 77, 4, 64), (8, 64, 32, 128), (16, 33, 2, 512),
                            (5, 10, 8, 4)]:
        o = torch.randn(n, rows, Hq, dv, generator=g)
        l = torch.randn(n, rows, Hq, generator=g) * 4
        l[0, 0, 0] = -math.inf
        if n > 1:
            l[:, 1, :] = -math.inf                            # all parts empty
            l[1:, 2, 1] = -math.inf
        out, lse = cpa.cp_lse_merge(o.cuda(), l.cuda(), lse_out=torch.empty(rows, Hq).cuda())
        O_ref, L_ref = omerge.lse_merge(o.double().numpy(), l.double().numpy())
        err = np.abs(np64(out) - O_ref).max()
        assert err < 1e-5, err
        assert_attn_close(out, lse, O_ref, L_ref, f"merge n={n}")


def test_merge_scatter_and_bf16_output():
    g = torch.Generator().manual_seed(43)
    o = torch.randn(4, 50, 8, 128, generator=g)
    l = torch.randn(4, 50, 8, generator=g)
    perm = torch.randperm(50, generator=g).to(torch.int32)
    out = torch.zeros(50, 8, 128, dtype=torch.bfloat16).cuda()
    lse = torch.zeros(50, 8).cuda()
    cpa.cp_lse_merge(o.cuda(), l.cuda(), dst_rows=perm.cuda(), out=out, lse_out=lse)
    O_ref, L_ref = omerge.lse_merge(o.double().numpy(), l.double().numpy())
    inv = np.empty(50, dtype=np.int64)
    inv[perm.numpy()] = np.arange(50)
    assert_attn_close(out, lse, O_ref[inv], L_ref[inv], "merge scatter")


def test_gpu_partials_merge_to_dense():
    """Merging the kernel's per-block partials equals one full-window call."""
    w = random_case(8, 4, 2, 64, max_new=600, max_prefix=100)
    inputs = W.make_inputs(w)
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, 1, "zigzag")
    N = w.total_new
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[:N])
    k, v = inputs["k"].cuda(), inputs["v"].cuda()
    full_o, full_l = cpa.cp_attn_partial(plan.segs, q_cat, k, v, w.scale, out_fp32=True,
                                         num_segs=plan.total_segs)
    cuts = [0, 128, 200, 512, 700, 10 ** 6]
    po = torch.empty(len(cuts) - 1, N, w.Hq, w.dv, device="cuda")
    pl = torch.empty(len(cuts) - 1, N, w.Hq, device="cuda")
    for j, (a, b) in enumerate(zip(cuts, cuts[1:])):
        cpa.cp_attn_partial(plan.segs, q_cat, k, v, w.scale, kv_lo=a, kv_hi=b, out=po[j],
                            lse=pl[j], num_segs=plan.total_segs)
    mo, ml = cpa.cp_lse_merge(po, pl, lse_out=torch.empty(N, w.Hq, device="cuda"))
    # both sides round P to bf16 (relative 2^-9 per element) against different
    # row maxima, so O may differ by about 2 * 2^-9 * max|v|
    vmax = v.float().abs().max().item()
    assert (mo - full_o).abs().max().item() < 2 * 2 ** -9 * vmax
    fin = torch.isfinite(full_l)
    assert ((ml - full_l).abs()[fin] <= 1e-5 * full_l.abs()[fin].clamp(min=1)).all()


def test_restore_is_exact():
    g = torch.Generator().manual_seed(3)
    src = torch.randn(1000, 8, 64, generator=g).to(torch.bfloat16).cuda()
    idx = torch.randperm(1000, generator=g).to(torch.int32).cuda()
    out = cpa.cp_restore(src, idx)
    assert torch.equal(out, src[idx.long()])
    lse = torch.randn(1000, 4, generator=g).cuda()
    assert torch.equal(cpa.cp_restore(lse, idx), lse[idx.long()])
    # row sizes around the warp-per-row path (>= 32 16-byte chunks): ragged
    # chunk counts, more chunks than one pass of a warp, 4-byte rows
    for rows, cols, dt in [(37, 264, torch.bfloat16), (1003, 300, torch.float32),
                           (9, 4800, torch.bfloat16), (77, 31, torch.float32),
                           (130, 3, torch.float32)]:
        src = torch.randn(rows, cols, generator=g).to(dt).cuda()
        idx = torch.randint(0, rows, (rows,), generator=g, dtype=torch.int32).cuda()
        assert torch.equal(cpa.cp_restore(src, idx), src[idx.long()]), (rows, cols, dt)


def test_restore_bad_index_sets_range():
    src = torch.zeros(64, 256, dtype=torch.float32, device="cuda")
    idx = torch.arange(64, dtype=torch.int32, device="cuda")
    idx[5] = 64
    status = cpa.new_status()
    out = torch.full_like(src, 7.0)
    cpa.cp_restore(src, idx, out=out, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    assert torch.all(out[5] == 7.0) and torch.all(out[:5] == 0) and torch.all(out[6:] == 0)


def test_bad_segment_sets_range_status():
    q = torch.zeros(256, 2, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(256, 1, 64, dtype=torch.bfloat16, device="cuda")
    seg = torch.tensor([[200, 100, 0, 1, 0, 100, 0, 0]], dtype=torch.int32, device="cuda")
    status = cpa.new_status()
    cpa.cp_attn_partial(seg, q, k, k, 0.125, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6
    bad_idx = torch.tensor([0, 5000], dtype=torch.int32, device="cuda")
    status.zero_()
    cpa.cp_restore(q, bad_idx, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6


# --------------------------------------------------------- absorbed MLA ----

def mla_case(new, pre, Hq, C, seed):
    return W.Workload(name=f"mla{seed}", new_lens=new, prefix_lens=pre, Hq=Hq, Hkv=1, d=576,
                      dv=512, scale=1 / math.sqrt(192), std=0.1, cp_size=C,
                      strategies=["interleave", "zigzag"], seed=seed, v_is_k_prefix=True)


@pytest.mark.parametrize("seed", range(3))
def test_mla_small_all_rows(seed):
    w = mla_case([300, 77, 5][: 1 + seed], [0, 40, 3][: 1 + seed], 4, [4, 2, 3][seed], 900 + seed)
    inputs = W.make_inputs(w)
    k64 = np64(inputs["k"])
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), k64, k64[:, :, :512],
                                               w.new_lens, w.prefix_lens, w.scale)
    for strategy in w.strategies:
        o, lse = run_full_kv(w, strategy, inputs)
        assert_attn_close(o, lse, O_ref, L_ref, f"mla/{strategy}")


def test_mla_small_odd_head_count_all_rows():
    """An odd number of query heads runs on the single-SM MLA kernel (the pair
    kernel needs head pairs)."""
    w = mla_case([190, 61], [0, 17], 3, 4, 905)
    inputs = W.make_inputs(w)
    k64 = np64(inputs["k"])
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), k64, k64[:, :, :512],
                                               w.new_lens, w.prefix_lens, w.scale)
    for strategy in w.strategies:
        o, lse = run_full_kv(w, strategy, inputs)
        assert_attn_close(o, lse, O_ref, L_ref, f"mla-odd/{strategy}")


# ------------------------------------------------- running max that moves ----

def _growing_keys(w, inputs, grow_from=0):
    """Scale every KV row of a request by 1 + pos/48 (pos = its position in
    the request), columns [grow_from:] only, re-rounded to bf16: later keys
    score higher, so the running row max keeps rising by more than the
    lazy-max slack and every kernel's O-rescale path runs."""
    k = inputs["k"].float()
    kv0 = 0
    for n, p in zip(w.new_lens, w.prefix_lens):
        f = 1.0 + torch.arange(n + p, dtype=torch.float32) / 48.0
        k[kv0: kv0 + n + p, :, grow_from:] *= f[:, None, None]
        kv0 += n + p
    out = dict(inputs)
    out["k"] = k.to(torch.bfloat16)
    return out


@pytest.mark.parametrize("Hq,Hkv,d", [(8, 2, 128), (3, 3, 128), (4, 2, 64), (2, 1, 576),
                                      (1, 1, 576)])
def test_running_max_moves_all_rows(Hq, Hkv, d):
    """Keys whose scores grow along the sequence make the row max move by more
    than the lazy-max slack many times; O is rescaled in tensor memory each
    time (in the MLA pair kernel by both halves of every row).  All rows
    against the oracle, both strategies: the two-head and one-head d = 128
    kernels, d = 64, the MLA pair kernel (even head count) and the single-SM
    MLA kernel (odd)."""
    mla = d == 576
    w = W.Workload(name=f"grow{Hq}x{d}", new_lens=[700, 130], prefix_lens=[100, 0], Hq=Hq,
                   Hkv=Hkv, d=d, dv=512 if mla else d,
                   scale=1 / math.sqrt(192 if mla else d), std=1.0, cp_size=2,
                   strategies=["zigzag", "interleave"], seed=7300 + d + Hq,
                   v_is_k_prefix=mla)
    # MLA: grow only the rope columns, so that V (the latent) keeps its scale
    inputs = _growing_keys(w, W.make_inputs(w), grow_from=512 if mla else 0)
    k64 = np64(inputs["k"])
    v64 = k64[:, :, :512] if mla else np64(inputs["v"])
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), k64, v64, w.new_lens,
                                               w.prefix_lens, w.scale)
    for strategy in w.strategies:
        o, lse = run_full_kv(w, strategy, inputs)
        assert_attn_close(o, lse, O_ref, L_ref, f"{w.name}/{strategy}")


def test_running_max_moves_split_kv_and_packed_heads():
    """The same growing keys through the split-KV call (blocks of 256 keys:
    per-block partials, the fused merge) with and without two query heads
    packed per tile (segments of at most 64 rows)."""
    w = W.Workload(name="grow_split", new_lens=[500, 60], prefix_lens=[300, 0], Hq=8, Hkv=2,
                   d=128, dv=128, scale=1 / math.sqrt(128), std=1.0, cp_size=8,
                   strategies=["zigzag"], seed=7400)
    inputs = _growing_keys(w, W.make_inputs(w))
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]),
                                               np64(inputs["v"]), w.new_lens, w.prefix_lens,
                                               w.scale)
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", status=status)
    q, k, v = inputs["q"].cuda(), inputs["k"].cuda(), inputs["v"].cuda()
    q_cat = cpa.cp_restore(q, plan.gather_idx[: w.total_new], status=status)
    for packed in (False, True):
        # zigzag blocks here have at most 32 rows: packing is allowed, 0 turns it off
        o, lse, _ = cpa.cp_attn_partial_kv(plan, q_cat, k, v, w.scale, 256, status=status,
                                           max_seg_rows=None if packed else 0)
        torch.cuda.synchronize()
        cpa.check_status(status, w.name)
        assert_attn_close(o, lse, O_ref, L_ref, f"{w.name}/packed={packed}")


def test_mla_16k_sampled():
    w = W.WORKLOADS["mla_16k"]
    inputs = W.make_inputs(w)
    o, lse = run_full_kv(w, "interleave", inputs)
    rows = boundary_rows(w.new_lens, w.prefix_lens, w.cp_size, "interleave",
                         W.sample_rows(13, w.total_new, 10) + [0, 1, 2, 3, 16383])
    k64 = np64(inputs["k"])
    O_ref, L_ref = oracle_dense_rows(inputs, w.new_lens, w.prefix_lens, w.scale, rows, k64=k64,
                                     v64=k64[:, :, :512])
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    assert_attn_close(o[idx], lse[idx], O_ref, L_ref, w.name)


def test_mla_requires_v_as_latent_view():
    q = torch.zeros(128, 2, 576, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(128, 1, 576, dtype=torch.bfloat16, device="cuda")
    v = torch.zeros(128, 1, 512, dtype=torch.bfloat16, device="cuda")
    seg = torch.tensor([[0, 128, 0, 1, 0, 128, 0, 0]], dtype=torch.int32, device="cuda")
    with pytest.raises(cpa.api.L.CpAttnError):
        cpa.cp_attn_partial(seg, q, k, v, 0.1)


# ------------------------------------------------ decode-style merge sweep ----

def test_merge_sweep_interleaved_kv_shards():
    """64 single-token queries x 32 heads over 65536 keys, key i on shard i mod 8:
    per-shard partials (no causal mask) merged by the LSE rule equal attention
    over all keys."""
    m = W.MERGE_SWEEP
    inputs = W.make_merge_sweep_inputs()
    q = inputs["q"].cuda()
    k = inputs["k"].cuda()
    v = inputs["v"].cuda()
    S, n_kv = m["shards"], m["kv_tokens"] // m["shards"]
    seg = torch.tensor([[0, m["queries"], n_kv - 1, 0, 0, n_kv, 0, 0]], dtype=torch.int32,
                       device="cuda")
    po = torch.empty(S, m["queries"], m["Hq"], m["dv"], device="cuda")
    pl = torch.empty(S, m["queries"], m["Hq"], device="cuda")
    status = cpa.new_status()
    for j in range(S):
        idx = torch.arange(j, m["kv_tokens"], S, dtype=torch.int32, device="cuda")
        kj = cpa.cp_restore(k, idx, status=status)
        vj = cpa.cp_restore(v, idx, status=status)
        cpa.cp_attn_partial(seg, q, kj, vj, m["scale"], out=po[j], lse=pl[j], status=status)
    out, lse = cpa.cp_lse_merge(po, pl, lse_out=torch.empty(m["queries"], m["Hq"], device="cuda"),
                                status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, "merge sweep")
    O_ref, L_ref = oatt.decode_attention(np64(inputs["q"]), np64(inputs["k"]), np64(inputs["v"]),
                                         m["scale"], np.arange(m["kv_tokens"]))
    assert_attn_close(out, lse, O_ref, L_ref, "merge sweep")


# ------------------------------------------------- bounded pipeline waits ----

@pytest.mark.parametrize("shape", [(2, 1, 128, 128), (4, 1, 128, 128), (1, 1, 64, 64),
                                   (1, 1, 576, 512), (2, 1, 576, 512)])
def test_wait_limit_reports_timeout_and_context_survives(shape):
    """With the query load withheld, the MMA thread's wait runs out: the kernel
    reports CPATTN_ERR_TIMEOUT, drains its own copies, frees TMEM and returns.
    The CUDA context stays usable: the same call without the hook is correct."""
    Hq, Hkv, d, dv = shape
    lib = cpa.api.L.load()
    g = torch.Generator().manual_seed(17)
    n = 300
    q = (torch.randn(n, Hq, d, generator=g) * 0.3).to(torch.bfloat16).cuda()
    k = (torch.randn(n, Hkv, d, generator=g) * 0.3).to(torch.bfloat16).cuda()
    v = k[:, :, :dv] if d == 576 else (torch.randn(n, Hkv, dv, generator=g)).to(torch.bfloat16).cuda()
    seg = torch.tensor([[0, n, 0, 1, 0, n, 0, 0]], dtype=torch.int32, device="cuda")
    status = cpa.new_status()
    assert lib.cp_attn_debug(cpa.api.L.DEBUG_WAIT_LIMIT_NS, 20_000_000) == 0
    assert lib.cp_attn_debug(cpa.api.L.DEBUG_WITHHOLD_Q, 1) == 0
    try:
        cpa.cp_attn_partial(seg, q, k, v, 0.1, status=status)
        torch.cuda.synchronize()
        assert int(status.item()) == cpa.api.L.ERR_TIMEOUT
    finally:
        lib.cp_attn_debug(cpa.api.L.DEBUG_WITHHOLD_Q, 0)
        lib.cp_attn_debug(cpa.api.L.DEBUG_WAIT_LIMIT_NS, 4_000_000_000)
    status.zero_()
    o, lse = cpa.cp_attn_partial(seg, q, k, v, 0.1, status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, "after timeout")
    pos = np.arange(n)
    O_ref, L_ref = oatt.attention_rows(np64(q), np64(k), np64(v), pos, np.zeros(n, np.int64), 0.1)
    assert_attn_close(o, lse, O_ref, L_ref, "after timeout")
    assert lib.cp_attn_debug(99, 1) == cpa.api.L.ERR_INVALID_ARG


# ------------------------------------------- partial-KV in one library call ----

@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_partial_kv_fused_small_all_rows(strategy):
    w = W.Workload(name="pkv_fused", new_lens=[700, 300, 5], prefix_lens=[0, 130, 9], Hq=8,
                   Hkv=2, d=128, dv=128, scale=1 / math.sqrt(128), std=1.0, cp_size=3,
                   strategies=[strategy], seed=778, kv_block=192)
    inputs = W.make_inputs(w)
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]),
                                               np64(inputs["v"]), w.new_lens, w.prefix_lens,
                                               w.scale)
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, strategy, status=status)
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
    k, v = inputs["k"].cuda(), inputs["v"].cuda()
    o, lse, ws = cpa.cp_attn_partial_kv(plan, q_cat, k, v, w.scale, w.kv_block,
                                        status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, "fused partial kv")
    assert_attn_close(o, lse, O_ref, L_ref, f"pkv fused/{strategy}")
    # cat order, fp32 output, workspace reused
    o2, lse2, _ = cpa.cp_attn_partial_kv(plan, q_cat, k, v, w.scale, w.kv_block,
                                         workspace=ws, dst_rows=None, out_fp32=True,
                                         status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, "fused partial kv, cat order")
    gi = plan.gather_idx[: w.total_new].long().cpu().numpy()
    assert_attn_close(o2, lse2, O_ref[gi], L_ref[gi], "pkv fused cat order")


def test_partial_kv_fused_mla_small():
    w = mla_case([260, 70], [0, 33], 4, 2, 990)
    inputs = W.make_inputs(w)
    k64 = np64(inputs["k"])
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), k64, k64[:, :, :512],
                                               w.new_lens, w.prefix_lens, w.scale)
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", status=status)
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
    k = inputs["k"].cuda()
    o, lse, _ = cpa.cp_attn_partial_kv(plan, q_cat, k, k[:, :, :512], w.scale, 100,
                                       status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, "fused partial kv mla")
    assert_attn_close(o, lse, O_ref, L_ref, "pkv fused mla")


def test_partialkv_128k_fused_sampled():
    w = W.WORKLOADS["partialkv_128k"]
    inputs = W.make_inputs(w)
    status = cpa.new_status()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", status=status)
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
    o, lse, ws = cpa.cp_attn_partial_kv(plan, q_cat, inputs["k"].cuda(), inputs["v"].cuda(),
                                        w.scale, w.kv_block, status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, w.name)
    del ws
    rows = sorted(set(W.sample_rows(12, w.total_new, 16) +
                      [0, 8191, 8192, 65535, 65536, 131071]))
    O_ref, L_ref = oracle_dense_rows(inputs, w.new_lens, w.prefix_lens, w.scale, rows)
    idx = torch.as_tensor(rows, dtype=torch.long, device=o.device)
    assert_attn_close(o[idx], lse[idx], O_ref, L_ref, w.name + " fused")


def test_partial_kv_workspace_too_small_is_reported():
    plan = cpa.make_plan([500], [0], 2, "zigzag")
    q = torch.zeros(500, 2, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(500, 1, 64, dtype=torch.bfloat16, device="cuda")
    need = cpa.cp_partial_kv_workspace_size([500], [0], 2, "zigzag", 64, 2, 64)[0]
    small = torch.empty(need // 3, dtype=torch.uint8, device="cuda")
    status = cpa.new_status()
    cpa.cp_attn_partial_kv(plan, q, k, k, 0.125, 64,
                           workspace=small, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) in (cpa.api.L.ERR_INVALID_ARG, cpa.api.L.ERR_RANGE)


@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
@pytest.mark.parametrize("C", [4, 8])
def test_many_tiny_requests_all_rows(strategy, C):
    """400 requests of 0..20 new tokens after 0..10 cached ones: hundreds of
    one-tile segments, many with a single row, and empty requests."""
    new = [(i * 13) % 21 for i in range(400)]
    pre = [(i * 7) % 11 for i in range(400)]
    w = W.Workload(name=f"tiny{C}", new_lens=new, prefix_lens=pre, Hq=4, Hkv=2, d=64, dv=64,
                   scale=0.125, std=1.0, cp_size=C, strategies=[strategy], seed=7100 + C)
    inputs = W.make_inputs(w)
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]),
                                               np64(inputs["v"]), w.new_lens, w.prefix_lens,
                                               w.scale)
    o, lse = run_full_kv(w, strategy, inputs)
    assert_attn_close(o, lse, O_ref, L_ref, f"tiny/{strategy}/C{C}")


def test_merge_sweep_strided_kv_views_match_copies():
    """A shard's interleaved keys passed as a strided view of the KV buffer
    (row stride 8 rows) give exactly the partial of a gathered copy."""
    m = W.MERGE_SWEEP
    inputs = W.make_merge_sweep_inputs()
    q, k, v = inputs["q"].cuda(), inputs["k"].cuda(), inputs["v"].cuda()
    S, n_kv = m["shards"], m["kv_tokens"] // m["shards"]
    seg = torch.tensor([[0, m["queries"], n_kv - 1, 0, 0, n_kv, 0, 0]], dtype=torch.int32,
                       device="cuda")
    status = cpa.new_status()
    for j in (0, 3, 7):
        idx = torch.arange(j, m["kv_tokens"], S, dtype=torch.int32, device="cuda")
        o1, l1 = cpa.cp_attn_partial(seg, q, cpa.cp_restore(k, idx), cpa.cp_restore(v, idx),
                                     m["scale"], out_fp32=True, status=status)
        o2, l2 = cpa.cp_attn_partial(seg, q, k[j::S], v[j::S], m["scale"], out_fp32=True,
                                     status=status)
        torch.cuda.synchronize()
        cpa.check_status(status, "strided views")
        assert torch.equal(o1, o2) and torch.equal(l1, l2)


@pytest.mark.parametrize("kv_block", [512, 1024, 8192])
def test_decode_sweep_split_kv(kv_block):
    """The decode path: each shard's partial through cp_attn_split_kv (keys in
    blocks of kv_block over separate CTAs, merged in the library), then the
    8 shard partials merged; equals attention over all 65536 keys."""
    m = W.MERGE_SWEEP
    inputs = W.make_merge_sweep_inputs()
    q, k, v = inputs["q"].cuda(), inputs["k"].cuda(), inputs["v"].cuda()
    S, n_kv = m["shards"], m["kv_tokens"] // m["shards"]
    seg = torch.tensor([[0, m["queries"], n_kv - 1, 0, 0, n_kv, 0, 0]], dtype=torch.int32,
                       device="cuda")
    po = torch.empty(S, m["queries"], m["Hq"], m["dv"], device="cuda")
    pl = torch.empty(S, m["queries"], m["Hq"], device="cuda")
    status = cpa.new_status()
    ws = None
    for j in range(S):
        _, _, ws = cpa.cp_attn_split_kv(seg, q, k[j::S], v[j::S], m["scale"], kv_block,
                                        out=po[j], lse_out=pl[j], workspace=ws, status=status)
    out, lse = cpa.cp_lse_merge(po, pl, lse_out=torch.empty(m["queries"], m["Hq"], device="cuda"),
                                status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, "decode split")
    O_ref, L_ref = oatt.decode_attention(np64(inputs["q"]), np64(inputs["k"]), np64(inputs["v"]),
                                         m["scale"], np.arange(m["kv_tokens"]))
    assert_attn_close(out, lse, O_ref, L_ref, f"decode split {kv_block}")


@pytest.mark.parametrize("kv_block", [2048, 4096, 8192])
def test_decode_step_as_one_merge_over_all_ranks(kv_block):
    """The decode step in one call with no second merge: the 8 ranks' KV
    caches (each rank's interleaved tokens contiguous, rank after rank) form
    one segment, its keys split in blocks of kv_block that never straddle two
    ranks' caches, so every block partial is part of one rank's partial and
    the library's LSE merge of all of them is the merge of the 8 rank
    partials.  Equals attention over all 65536 keys."""
    m = W.MERGE_SWEEP
    inputs = W.make_merge_sweep_inputs()
    q, k, v = inputs["q"].cuda(), inputs["k"].cuda(), inputs["v"].cuda()
    S, nq = m["shards"], m["queries"]
    n_kv = m["kv_tokens"] // S
    assert n_kv % kv_block == 0
    Hkv, d, dv = k.shape[1], k.shape[2], v.shape[2]
    k_rank = k.view(n_kv, S, Hkv, d).transpose(0, 1).contiguous().view(S * n_kv, Hkv, d)
    v_rank = v.view(n_kv, S, Hkv, dv).transpose(0, 1).contiguous().view(S * n_kv, Hkv, dv)
    seg = torch.tensor([[0, nq, S * n_kv - 1, 0, 0, S * n_kv, 0, 0]], dtype=torch.int32)
    status = cpa.new_status()
    out, lse, _ = cpa.cp_attn_split_kv(seg.cuda(), q, k_rank, v_rank, m["scale"], kv_block,
                                       segs_host=seg, status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, "decode one merge")
    O_ref, L_ref = oatt.decode_attention(np64(inputs["q"]), np64(inputs["k"]), np64(inputs["v"]),
                                         m["scale"], np.arange(m["kv_tokens"]))
    assert_attn_close(out, lse, O_ref, L_ref, f"decode one merge {kv_block}")


@pytest.mark.parametrize("kv_block", [512, 4096])
def test_decode_one_call_over_all_ranks(kv_block):
    """The decode step as the bench times it: each rank's KV cache holds its
    interleaved tokens contiguously, every rank holds all queries, and one
    cp_attn_split_kv call over the 8 ranks' segments gives the 8 shard
    partials, bit-identical to one call per rank on strided views; their
    merge equals attention over all 65536 keys."""
    m = W.MERGE_SWEEP
    inputs = W.make_merge_sweep_inputs()
    q, k, v = inputs["q"].cuda(), inputs["k"].cuda(), inputs["v"].cuda()
    S, nq, Hq, dv = m["shards"], m["queries"], m["Hq"], m["dv"]
    n_kv = m["kv_tokens"] // S
    Hkv, d = k.shape[1], k.shape[2]
    k_rank = k.view(n_kv, S, Hkv, d).transpose(0, 1).contiguous().view(S * n_kv, Hkv, d)
    v_rank = v.view(n_kv, S, Hkv, dv).transpose(0, 1).contiguous().view(S * n_kv, Hkv, dv)
    q_rank = q.repeat(S, 1, 1).contiguous()
    segs = torch.tensor([[j * nq, nq, n_kv - 1, 0, j * n_kv, n_kv, j * nq, j] for j in range(S)],
                        dtype=torch.int32)
    status = cpa.new_status()
    po, pl, _ = cpa.cp_attn_split_kv(segs.cuda(), q_rank, k_rank, v_rank, m["scale"], kv_block,
                                     segs_host=segs, status=status)
    seg1 = torch.tensor([[0, nq, n_kv - 1, 0, 0, n_kv, 0, 0]], dtype=torch.int32)
    po1 = torch.empty(S, nq, Hq, dv, device="cuda")
    pl1 = torch.empty(S, nq, Hq, device="cuda")
    for j in range(S):
        cpa.cp_attn_split_kv(seg1.cuda(), q, k[j::S], v[j::S], m["scale"], kv_block,
                             segs_host=seg1, out=po1[j], lse_out=pl1[j], status=status)
    out, lse = cpa.cp_lse_merge(po.view(S, nq, Hq, dv), pl.view(S, nq, Hq),
                                lse_out=torch.empty(nq, Hq, device="cuda"), status=status)
    torch.cuda.synchronize()
    cpa.check_status(status, "decode one call")
    assert torch.equal(po.view(S, nq, Hq, dv), po1) and torch.equal(pl.view(S, nq, Hq), pl1)
    O_ref, L_ref = oatt.decode_attention(np64(inputs["q"]), np64(inputs["k"]), np64(inputs["v"]),
                                         m["scale"], np.arange(m["kv_tokens"]))
    assert_attn_close(out, lse, O_ref, L_ref, f"decode one call {kv_block}")


@pytest.mark.parametrize("d,Hq,Hkv", [(128, 32, 8), (64, 16, 2), (128, 8, 8)])
def test_split_kv_packed_heads_short_segments(d, Hq, Hkv):
    """Segments of at most 64 rows (decode queries and short causal chunks at
    several positions, some ragged) through cp_attn_split_kv: with two query
    heads packed per tile (Hq / Hkv a multiple of 4) the result is
    bit-identical to unpacked tiles and equals the oracle; with a head ratio
    that cannot pack, the hint changes nothing."""
    gen = torch.Generator().manual_seed(4100 + d + Hq)
    n_kv = 3000
    k = (torch.randn(n_kv, Hkv, d, generator=gen)).to(torch.bfloat16)
    v = (torch.randn(n_kv, Hkv, d, generator=gen)).to(torch.bfloat16)
    # (q_len, q_pos0, q_pos_step, kv_row0, kv_len)
    spec = [(64, 2999, 0, 0, 3000), (37, 1200, 1, 0, 1237), (1, 5, 0, 0, 6),
            (50, 700, 1, 1000, 750), (64, 0, 1, 2000, 64), (13, 90, 7, 0, 175)]
    rows, seg_rows = 0, []
    for ql, p0, st, kv0, kvl in spec:
        seg_rows.append([rows, ql, p0, st, kv0, kvl, rows, 0])
        rows += ql
    segs = torch.tensor(seg_rows, dtype=torch.int32)
    q = (torch.randn(rows, Hq, d, generator=gen)).to(torch.bfloat16)
    scale = 1 / math.sqrt(d)
    status = cpa.new_status()
    outs = []
    for hint in (None, 0):
        o, l, _ = cpa.cp_attn_split_kv(segs.cuda(), q.cuda(), k.cuda(), v.cuda(), scale, 256,
                                       segs_host=segs, max_seg_rows=hint, status=status)
        outs.append((o, l))
    torch.cuda.synchronize()
    cpa.check_status(status, "packed heads")
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
    pos = np.concatenate([p0 + st * np.arange(ql) for ql, p0, st, _, _ in spec])
    kv0 = np.concatenate([np.full(ql, kv) for ql, _, _, kv, _ in spec])
    O_ref, L_ref = oatt.attention_rows(np64(q), np64(k), np64(v), pos, kv0, scale)
    assert_attn_close(outs[0][0], outs[0][1], O_ref, L_ref, f"packed d={d} Hq={Hq}")


def test_packed_heads_reject_a_longer_segment():
    """A max_seg_rows hint that a segment exceeds: RANGE, the segment skipped."""
    segs = torch.tensor([[0, 100, 0, 1, 0, 100, 0, 0]], dtype=torch.int32)
    q = torch.zeros(100, 8, 128, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(100, 2, 128, dtype=torch.bfloat16, device="cuda")
    status = cpa.new_status()
    cpa.cp_attn_split_kv(segs.cuda(), q, k, k, 0.1, 64, segs_host=segs, max_seg_rows=64,
                         status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == -6


def test_partial_kv_short_requests_pack_heads():
    """Plan-based partial-KV over short requests (every segment <= 64 rows):
    the call packs two query heads per tile, bit-identical to unpacked tiles
    and equal to the oracle, for both strategies."""
    w = W.Workload(name="pkv_short", new_lens=[100, 37, 90, 5, 128], prefix_lens=[0, 20, 300, 3, 0],
                   Hq=8, Hkv=2, d=128, dv=128, scale=1 / math.sqrt(128), std=1.0, cp_size=2,
                   strategies=["zigzag", "interleave"], seed=4321, kv_block=64)
    inputs = W.make_inputs(w)
    O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]),
                                               np64(inputs["v"]), w.new_lens, w.prefix_lens,
                                               w.scale)
    k, v = inputs["k"].cuda(), inputs["v"].cuda()
    for strategy in w.strategies:
        assert cpa.cp_partial_kv_workspace_size(w.new_lens, w.prefix_lens, w.cp_size, strategy,
                                            w.kv_block, w.Hq, w.dv)[2] <= 64
        status = cpa.new_status()
        plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, strategy, status=status)
        q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
        outs = [cpa.cp_attn_partial_kv(plan, q_cat, k, v, w.scale, w.kv_block,
                                       max_seg_rows=hint, status=status)[:2]
                for hint in (None, 0)]
        torch.cuda.synchronize()
        cpa.check_status(status, f"pkv short {strategy}")
        assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
        assert_attn_close(outs[0][0], outs[0][1], O_ref, L_ref, f"pkv short/{strategy}")
