"""Guard bands around every output buffer of every device entry point.

Each output (and each caller workspace) is carved out of a larger device
buffer whose bytes before and after it hold a canary pattern; after the call
the bands must still hold it, so no kernel wrote outside the buffer it was
given.  The cases are small and ragged (odd lengths, cached prefixes, a few
heads) and every result is also compared with the oracle.
"""

import math

import numpy as np
import pytest
import torch

import context_causal_attention_cp_gb300 as cpa
from context_causal_attention_cp_gb300 import _lib as L
from context_causal_attention_cp_gb300 import workloads as W
from oracle import attention as oatt
from oracle import merge as omerge

from gpu_common import assert_attn_close, np64

pytestmark = pytest.mark.gpu

GUARD = 4096          # canary bytes on each side (keeps the payload 256-byte aligned)
CANARY = 0xA5


class Guarded:
    """A tensor of ``shape`` / ``dtype`` inside a byte buffer with canary bands."""

    def __init__(self, shape, dtype, fill=None, device="cuda"):
        elem = torch.empty((), dtype=dtype).element_size()
        self.n = max(1, math.prod(shape)) * elem
        pad = (self.n + 255) // 256 * 256
        self.raw = torch.full((GUARD + pad + GUARD,), CANARY, dtype=torch.uint8, device=device)
        self.t = self.raw[GUARD: GUARD + self.n].view(dtype)[: math.prod(shape)].view(shape)
        if fill is not None:
            self.t.fill_(fill)

    def check(self, what):
        torch.cuda.synchronize()
        head = self.raw[:GUARD]
        tail = self.raw[GUARD + self.n:]
        assert bool((head == CANARY).all()), f"{what}: bytes written before the buffer"
        assert bool((tail == CANARY).all()), f"{what}: bytes written after the buffer"


def case(d=128, Hq=4, Hkv=2, C=3, seed=71):
    return W.Workload(name=f"guard{d}", new_lens=[37, 130, 5], prefix_lens=[3, 0, 250], Hq=Hq,
                      Hkv=Hkv, d=d, dv=d, scale=1 / math.sqrt(d), std=1.0, cp_size=C,
                      strategies=["zigzag", "interleave"], seed=seed, kv_block=64)


def guarded_plan(w, strategy):
    rows, segs, tiles = cpa.cp_shard_plan_sizes(w.new_lens, w.prefix_lens, w.cp_size, strategy)
    N, S, T = sum(rows), sum(segs), sum(tiles)
    i32 = torch.int32
    g = {name: Guarded(shape, i32) for name, shape in
         (("segs", (S, 8)), ("seg_offsets", (w.cp_size + 1,)), ("row_offsets", (w.cp_size + 1,)),
          ("gather_idx", (N,)), ("positions", (N,)), ("restore_idx", (N,)), ("tiles", (T, 2)))}
    plan = cpa.ShardPlan(
        cp_size=w.cp_size, strategy=cpa.api._strategy(strategy), rows_per_rank=rows,
        segs_per_rank=segs, tiles_per_rank=tiles, segs=g["segs"].t,
        seg_offsets=g["seg_offsets"].t, row_offsets=g["row_offsets"].t,
        gather_idx=g["gather_idx"].t, positions=g["positions"].t, restore_idx=g["restore_idx"].t,
        tiles=g["tiles"].t, new_lens_dev=torch.tensor(w.new_lens, dtype=i32, device="cuda"),
        prefix_lens_dev=torch.tensor(w.prefix_lens, dtype=i32, device="cuda"),
        num_reqs=len(w.new_lens), new_lens=list(w.new_lens), prefix_lens=list(w.prefix_lens))
    status = cpa.new_status()
    cpa.cp_shard_plan(plan, status=status)
    for name, gb in g.items():
        gb.check(f"plan.{name}")
    cpa.check_status(status, "plan")
    return plan


def dense_ref(w, inputs):
    return oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]), np64(inputs["v"]),
                                       w.new_lens, w.prefix_lens, w.scale)


@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
@pytest.mark.parametrize("d", [64, 128])
def test_attention_entry_points_write_only_their_outputs(strategy, d):
    w = case(d=d)
    inputs = W.make_inputs(w)
    O_ref, L_ref = dense_ref(w, inputs)
    plan = guarded_plan(w, strategy)
    N, Hq = w.total_new, w.Hq
    q, k, v = inputs["q"].cuda(), inputs["k"].cuda(), inputs["v"].cuda()
    status = cpa.new_status()
    q_cat_g = Guarded((N, Hq, d), torch.bfloat16)
    cpa.cp_restore(q, plan.gather_idx[:N], out=q_cat_g.t, status=status)
    q_cat_g.check("cp_restore (query gather)")
    gi = plan.gather_idx[:N].long().cpu().numpy()
    for o_dtype in (torch.bfloat16, torch.float32):
        og, lg = Guarded((N, Hq, d), o_dtype), Guarded((N, Hq), torch.float32)
        cpa.cp_attn_partial(plan.segs, q_cat_g.t, k, v, w.scale, num_segs=plan.total_segs,
                            tiles=plan.tiles, num_tiles=plan.total_tiles, out=og.t, lse=lg.t,
                            status=status)
        og.check("cp_attn_partial O")
        lg.check("cp_attn_partial LSE")
        assert_attn_close(og.t, lg.t, O_ref[gi], L_ref[gi], f"cp_attn_partial {o_dtype}")
    og, lg = Guarded((N, Hq, d), torch.bfloat16), Guarded((N, Hq), torch.float32)
    cpa.cp_attn_partial_restore(plan.segs, q_cat_g.t, k, v, w.scale, plan.gather_idx,
                                num_out_rows=N, num_segs=plan.total_segs, tiles=plan.tiles,
                                num_tiles=plan.total_tiles, out=og.t, lse=lg.t, status=status)
    og.check("cp_attn_partial_restore O")
    lg.check("cp_attn_partial_restore LSE")
    assert_attn_close(og.t, lg.t, O_ref, L_ref, "cp_attn_partial_restore")
    if strategy == "zigzag":
        og, lg = Guarded((N, Hq, d), torch.bfloat16), Guarded((N, Hq), torch.float32)
        cpa.cp_attn_prefill(plan.segs, q, k, v, w.scale, num_segs=plan.total_segs,
                            tiles=plan.tiles, num_tiles=plan.total_tiles, out=og.t, lse=lg.t,
                            status=status)
        og.check("cp_attn_prefill O")
        lg.check("cp_attn_prefill LSE")
        assert_attn_close(og.t, lg.t, O_ref, L_ref, "cp_attn_prefill")
    # restore of the outputs from cat order
    o_cat = torch.as_tensor(O_ref[gi], dtype=torch.float32).cuda()
    rg = Guarded((N, Hq, d), torch.float32)
    cpa.cp_restore(o_cat, plan.restore_idx[:N], out=rg.t, status=status)
    rg.check("cp_restore (outputs)")
    assert torch.equal(rg.t.cpu(), torch.as_tensor(O_ref, dtype=torch.float32))
    torch.cuda.synchronize()
    cpa.check_status(status, "guards")


@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_partial_kv_and_pass_q_write_only_their_outputs(strategy):
    w = case(d=128, Hq=8, Hkv=2, C=2)
    inputs = W.make_inputs(w)
    O_ref, L_ref = dense_ref(w, inputs)
    plan = guarded_plan(w, strategy)
    N, Hq, d = w.total_new, w.Hq, w.d
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[:N])
    k, v = inputs["k"].cuda(), inputs["v"].cuda()
    status = cpa.new_status()
    need = cpa.cp_partial_kv_workspace_size(w.new_lens, w.prefix_lens, w.cp_size, strategy,
                                            w.kv_block, Hq, d)[0]
    wsg = Guarded((need,), torch.uint8)
    og, lg = Guarded((N, Hq, d), torch.bfloat16), Guarded((N, Hq), torch.float32)
    cpa.cp_attn_partial_kv(plan, q_cat, k, v, w.scale, w.kv_block, workspace=wsg.t, out=og.t,
                           lse_out=lg.t, status=status)
    wsg.check("cp_attn_partial_kv workspace")
    og.check("cp_attn_partial_kv O")
    lg.check("cp_attn_partial_kv LSE")
    assert_attn_close(og.t, lg.t, O_ref, L_ref, f"cp_attn_partial_kv {strategy}")
    sched = cpa.pass_q_schedule(plan)
    acc = [Guarded((N, Hq, d), torch.float32), Guarded((N, Hq), torch.float32),
           Guarded((N, Hq), torch.float32)]
    o_cat, l_cat = cpa.cp_pass_q_attention(q_cat, k, v, plan, w.scale, schedule=sched,
                                           status=status, out=tuple(a.t for a in acc))
    for a, name in zip(acc, ("O_acc", "LSE", "LSE scratch")):
        a.check(f"cp_attn_pass_q {name}")
    gi = plan.gather_idx[:N].long().cpu().numpy()
    assert_attn_close(o_cat, l_cat, O_ref[gi], L_ref[gi], f"pass-Q {strategy}")
    torch.cuda.synchronize()
    cpa.check_status(status, "guards")


def test_accumulate_and_merge_write_only_their_outputs():
    w = case(d=128, Hq=4, Hkv=2, C=3)
    inputs = W.make_inputs(w)
    plan = guarded_plan(w, "zigzag")
    N, Hq, d = w.total_new, w.Hq, w.d
    q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[:N])
    k, v = inputs["k"].cuda(), inputs["v"].cuda()
    status = cpa.new_status()
    og = Guarded((N, Hq, d), torch.float32, fill=0.0)
    la = Guarded((N, Hq), torch.float32, fill=float("-inf"))
    lb = Guarded((N, Hq), torch.float32, fill=float("-inf"))
    cpa.cp_attn_partial_accumulate(plan.segs, q_cat, k, v, w.scale, og.t, la.t, lb.t,
                                   num_segs=plan.total_segs, kv_lo=0, kv_hi=100, status=status)
    cpa.cp_attn_partial_accumulate(plan.segs, q_cat, k, v, w.scale, og.t, lb.t, la.t,
                                   num_segs=plan.total_segs, kv_lo=100, kv_hi=-1, status=status)
    for g, name in ((og, "O_acc"), (la, "LSE a"), (lb, "LSE b")):
        g.check(f"cp_attn_partial_accumulate {name}")
    O_ref, L_ref = dense_ref(w, inputs)
    gi = plan.gather_idx[:N].long().cpu().numpy()
    assert_attn_close(og.t, la.t, O_ref[gi], L_ref[gi], "two accumulate hops")
    # merge of 3 random partials with a scatter, fp32 and bf16 outputs
    rng = np.random.default_rng(3)
    rows, parts, dv = 77, 3, 64
    po = rng.standard_normal((parts, rows, Hq, dv)).astype(np.float32)
    pl = (rng.standard_normal((parts, rows, Hq)) * 3).astype(np.float32)
    pl[1, :5] = -np.inf
    dst = torch.as_tensor(rng.permutation(rows).astype(np.int32)).cuda()
    O_m, L_m = omerge.lse_merge(po.astype(np.float64), pl.astype(np.float64))
    for o_dtype in (torch.float32, torch.bfloat16):
        mo, ml = Guarded((rows, Hq, dv), o_dtype), Guarded((rows, Hq), torch.float32)
        cpa.cp_lse_merge(torch.as_tensor(po).cuda(), torch.as_tensor(pl).cuda(), dst_rows=dst,
                         out=mo.t, lse_out=ml.t, num_out_rows=rows, status=status)
        mo.check(f"cp_lse_merge O {o_dtype}")
        ml.check("cp_lse_merge LSE")
        back = dst.cpu().long()          # merged row i went to output row dst[i]
        assert_attn_close(mo.t.cpu()[back], ml.t.cpu()[back], O_m, L_m, f"cp_lse_merge {o_dtype}")
    torch.cuda.synchronize()
    cpa.check_status(status, "guards")


@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_host_prefill_writes_only_its_outputs(strategy):
    """cp_prefill_host: guard bands around its device workspace, and canary
    bytes around every host output (pinned host buffers)."""
    w = case(d=128, Hq=4, Hkv=2, C=3)
    batches = [W.make_inputs(w, seed_offset=i) for i in range(3)]
    N, Hq, d = w.total_new, w.Hq, w.d
    need = cpa.cp_prefill_host_workspace_size(w.new_lens, w.prefix_lens, w.cp_size, strategy, Hq,
                                              w.Hkv, d, d)
    wsg = Guarded((need,), torch.uint8)
    host = []
    for b in batches:
        ob = torch.full((GUARD + N * Hq * d * 2 + GUARD,), CANARY, dtype=torch.uint8).pin_memory()
        lb = torch.full((GUARD + N * Hq * 4 + GUARD,), CANARY, dtype=torch.uint8).pin_memory()
        ho = ob[GUARD: GUARD + N * Hq * d * 2].view(torch.bfloat16).view(N, Hq, d)
        hl = lb[GUARD: GUARD + N * Hq * 4].view(torch.float32).view(N, Hq)
        host.append(((b["q"].pin_memory(), b["k"].pin_memory(), b["v"].pin_memory(), ho, hl),
                     ob, lb))
    status = cpa.new_status()
    _, streams = cpa.cp_prefill_host(w.new_lens, w.prefix_lens, w.cp_size, strategy, Hq, w.Hkv,
                                     d, d, w.scale, [h[0] for h in host], workspace=wsg.t,
                                     status=status)
    streams[2].synchronize()
    wsg.check("cp_prefill_host workspace")
    cpa.check_status(status, "host prefill")
    for i, (args, ob, lb) in enumerate(host):
        for buf, n, name in ((ob, N * Hq * d * 2, "O"), (lb, N * Hq * 4, "LSE")):
            assert bool((buf[:GUARD] == CANARY).all()) and bool((buf[GUARD + n:] == CANARY).all()), \
                f"host {name} of batch {i}: bytes written outside the buffer"
        O_ref, L_ref = dense_ref(w, batches[i])
        assert_attn_close(args[3], args[4], O_ref, L_ref, f"host prefill batch {i}")


def test_nvtx_ranges_change_nothing():
    """With the NVTX ranges turned on, a call gives bit-identical results."""
    w = case(d=128)
    inputs = W.make_inputs(w)
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag")
    q, k, v = inputs["q"].cuda(), inputs["k"].cuda(), inputs["v"].cuda()
    lib = L.load()
    outs = []
    try:
        for on in (0, 1):
            assert lib.cp_attn_debug(L.DEBUG_NVTX, on) == L.OK
            outs.append(cpa.cp_prefill_attention(q, k, v, plan, w.scale, fuse_restore=True))
    finally:
        lib.cp_attn_debug(L.DEBUG_NVTX, 0)
    torch.cuda.synchronize()
    assert torch.equal(outs[0][0], outs[1][0]) and torch.equal(outs[0][1], outs[1][1])
