"""cp_attn_partial_kv_noalloc through the C ABI, against the oracle and against
cp_attn_partial_kv.

The no-allocation entry point serves callers that cannot call cudaMalloc:
engines whose allocator owns all device memory, deployments with a fixed
memory budget, and hot paths that cannot take the implicit synchronisation of
cudaMalloc / cudaFree.  It runs the same computation on a scratch array that
lives inside the library, so its results must equal the oracle's (fp64 dense
causal attention) within the parity tolerance and the caller-workspace entry
point's bit for bit.  Two calls in a row with different inputs check that
nothing stale from the previous call leaks into the next one.  This file is
collected last, so a run that stops at the first failure has already run
every other test; it also passes when run alone in a fresh process.
"""

import ctypes
import math

import pytest
import torch

import context_causal_attention_cp_gb300 as cpa
from context_causal_attention_cp_gb300 import _lib as L
from context_causal_attention_cp_gb300 import workloads as W
from oracle import attention as oatt

from gpu_common import assert_attn_close, np64

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(plan, q_cat, k, v, scale, kv_block, max_blocks, max_rows, need, out, lse, status):
    lib = L.load()
    N, Hq, d = q_cat.shape
    Hkv, dv = v.shape[1], v.shape[2]
    return lib.cp_attn_partial_kv_noalloc(
        _p(plan.segs), plan.total_segs, _p(plan.tiles), plan.total_tiles, _p(q_cat), N, _p(k),
        k.stride(0), k.stride(1), _p(v), v.stride(0), v.stride(1), k.shape[0], Hq, Hkv, d, dv,
        float(scale), kv_block, max_blocks, max_rows, _p(plan.gather_idx), _p(out), 0, _p(lse),
        out.shape[0], need, _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_noalloc_matches_oracle_and_workspace_entry_point_twice(strategy):
    new, pre, C, kv_block = [700, 300, 5], [0, 130, 9], 3, 192
    Hq, Hkv, d = 8, 2, 128
    need, max_blocks, max_rows = cpa.cp_partial_kv_workspace_size(new, pre, C, strategy, kv_block,
                                                                  Hq, d)
    assert need <= L.NOALLOC_SCRATCH_BYTES
    for call, seed in enumerate((31, 32)):
        w = W.Workload(name="noalloc", new_lens=new, prefix_lens=pre, Hq=Hq, Hkv=Hkv, d=d, dv=d,
                       scale=1 / math.sqrt(d), std=1.0, cp_size=C, strategies=[strategy],
                       seed=seed)
        inputs = W.make_inputs(w)
        status = cpa.new_status()
        plan = cpa.make_plan(new, pre, C, strategy, status=status)
        q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
        k, v = inputs["k"].cuda(), inputs["v"].cuda()
        out = torch.full((w.total_new, Hq, d), float("nan"), dtype=torch.bfloat16, device="cuda")
        lse = torch.full((w.total_new, Hq), float("nan"), device="cuda")
        rc = _noalloc(plan, q_cat, k, v, w.scale, kv_block, max_blocks, max_rows, need, out, lse,
                      status)
        assert rc == L.OK, L.status_string(rc)
        ref_o, ref_l, _ = cpa.cp_attn_partial_kv(plan, q_cat, k, v, w.scale, kv_block,
                                                 status=status)
        torch.cuda.synchronize()
        cpa.check_status(status, f"no-alloc call {call}")
        O_ref, L_ref = oatt.dense_causal_attention(np64(inputs["q"]), np64(inputs["k"]),
                                                   np64(inputs["v"]), new, pre, w.scale)
        assert_attn_close(out, lse, O_ref, L_ref, f"no-alloc call {call} vs oracle")
        assert torch.equal(out, ref_o) and torch.equal(lse, ref_l), \
            f"no-alloc call {call} differs from cp_attn_partial_kv"


def test_noalloc_rejects_problems_beyond_its_scratch():
    plan = cpa.make_plan([64], [0], 1, "zigzag")
    q = torch.zeros(64, 2, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(64, 1, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(64, 2, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(64, 2, device="cuda")
    status = cpa.new_status()
    rc = _noalloc(plan, q, k, k, 0.125, 64, 1, 0, L.NOALLOC_SCRATCH_BYTES + 1, out, lse, status)
    assert rc == L.ERR_TOO_LARGE
    assert "scratch" in L.status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0


def test_noalloc_with_an_understated_need_reports_on_the_device():
    """The size check trusts the caller's figure: a problem that needs more
    than the scratch array but is declared small launches, and the device
    reports the shortfall in the status word instead of writing past the
    array."""
    new, pre, C, kv_block, Hq, d = [12000], [0], 1, 512, 16, 128
    need, max_blocks, max_rows = cpa.cp_partial_kv_workspace_size(new, pre, C, "zigzag",
                                                                  kv_block, Hq, d)
    assert need > L.NOALLOC_SCRATCH_BYTES
    plan = cpa.make_plan(new, pre, C, "zigzag")
    q = torch.zeros(new[0], Hq, d, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(new[0], 1, d, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(new[0], Hq, d, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(new[0], Hq, device="cuda")
    status = cpa.new_status()
    rc = _noalloc(plan, q, k, k, 0.1, kv_block, max_blocks, max_rows, 1024, out, lse, status)
    assert rc == L.OK
    torch.cuda.synchronize()
    assert int(status.item()) in (L.ERR_INVALID_ARG, L.ERR_RANGE)
