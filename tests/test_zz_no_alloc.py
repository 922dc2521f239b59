"""cp_attn_partial_kv_noalloc against cp_attn_partial_kv, through the C ABI.

The no-allocation entry point serves callers that cannot call cudaMalloc:
engines whose allocator owns all device memory, deployments with a fixed
memory budget, and hot paths that cannot take the implicit synchronisation of
cudaMalloc / cudaFree.  It runs the same computation on a scratch array that
lives inside the library, so its results must match the caller-workspace entry
point; two calls in a row (different inputs) check that nothing stale from
the previous call leaks into the next one.  This file is collected last.
"""

import ctypes
import math

import pytest
import torch

import context_causal_attention_cp_gb300 as cpa
from context_causal_attention_cp_gb300 import _lib as L
from context_causal_attention_cp_gb300 import workloads as W

from gpu_common import assert_attn_close, np64

pytestmark = pytest.mark.gpu


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _noalloc(plan, q_cat, k, v, scale, kv_block, max_blocks, need, out, lse, status):
    lib = L.load()
    N, Hq, d = q_cat.shape
    Hkv, dv = v.shape[1], v.shape[2]
    return lib.cp_attn_partial_kv_noalloc(
        _p(plan.segs), plan.total_segs, _p(plan.tiles), plan.total_tiles, _p(q_cat), N, _p(k),
        k.stride(0), k.stride(1), _p(v), v.stride(0), v.stride(1), k.shape[0], Hq, Hkv, d, dv,
        float(scale), kv_block, max_blocks, 0, _p(plan.gather_idx), _p(out), 0, _p(lse),
        out.shape[0], need, _p(status), ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))


def test_noalloc_matches_workspace_entry_point_twice():
    new, pre, C, kv_block = [700, 300, 5], [0, 130, 9], 3, 192
    Hq, Hkv, d = 8, 2, 128
    need, max_blocks = cpa.cp_partial_kv_workspace_size(new, pre, C, "zigzag", kv_block, Hq, d)
    assert need <= L.NOALLOC_SCRATCH_BYTES
    for call, seed in enumerate((31, 32)):
        w = W.Workload(name="noalloc", new_lens=new, prefix_lens=pre, Hq=Hq, Hkv=Hkv, d=d, dv=d,
                       scale=1 / math.sqrt(d), std=1.0, cp_size=C, strategies=["zigzag"],
                       seed=seed)
        inputs = W.make_inputs(w)
        status = cpa.new_status()
        plan = cpa.make_plan(new, pre, C, "zigzag", status=status)
        q_cat = cpa.cp_restore(inputs["q"].cuda(), plan.gather_idx[: w.total_new], status=status)
        k, v = inputs["k"].cuda(), inputs["v"].cuda()
        ref_o, ref_l, _ = cpa.cp_attn_partial_kv(plan, q_cat, k, v, w.scale, kv_block,
                                                 new_lens=new, prefix_lens=pre, status=status)
        out = torch.full_like(ref_o, float("nan"))
        lse = torch.full_like(ref_l, float("nan"))
        rc = _noalloc(plan, q_cat, k, v, w.scale, kv_block, max_blocks, need, out, lse, status)
        assert rc == L.OK, L.status_string(rc)
        torch.cuda.synchronize()
        cpa.check_status(status, f"no-alloc call {call}")
        assert_attn_close(out, lse, np64(ref_o), np64(ref_l), f"no-alloc call {call}")


def test_noalloc_rejects_problems_beyond_its_scratch():
    plan = cpa.make_plan([64], [0], 1, "zigzag")
    q = torch.zeros(64, 2, 64, dtype=torch.bfloat16, device="cuda")
    k = torch.zeros(64, 1, 64, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros(64, 2, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.zeros(64, 2, device="cuda")
    status = cpa.new_status()
    rc = _noalloc(plan, q, k, k, 0.125, 64, 1, L.NOALLOC_SCRATCH_BYTES + 1, out, lse, status)
    assert rc == L.ERR_TOO_LARGE
    assert "scratch" in L.status_string(rc)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
