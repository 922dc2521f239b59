"""Shared helpers for the GPU parity tests (oracle side + comparisons)."""

import numpy as np
import torch

from oracle import attention as oatt
from oracle import plan as oplan

O_ATOL = 2e-2        # max-abs error of attention outputs (bf16 inputs, fp32 accumulation)
LSE_RTOL = 1e-5      # |dL| <= LSE_RTOL * max(1, |L|)


def np64(t):
    return t.detach().to("cpu", torch.float32).numpy().astype(np.float64)


def assert_attn_close(o_gpu, l_gpu, o_ref, l_ref, what=""):
    o = np64(o_gpu)
    l = np64(l_gpu)
    o_ref = np.asarray(o_ref)
    l_ref = np.asarray(l_ref)
    assert o.shape == o_ref.shape, (o.shape, o_ref.shape)
    assert np.isfinite(o).all(), f"{what}: non-finite outputs"
    err = np.abs(o - o_ref).max() if o.size else 0.0
    assert err <= O_ATOL, f"{what}: max |dO| = {err:.3e}"
    inf_ref = np.isneginf(l_ref)
    assert (np.isneginf(l) == inf_ref).all(), f"{what}: -inf pattern of LSE differs"
    fin = ~inf_ref
    if fin.any():
        dl = np.abs(l[fin] - l_ref[fin]) / np.maximum(1.0, np.abs(l_ref[fin]))
        assert dl.max() <= LSE_RTOL, f"{what}: max rel |dL| = {dl.max():.3e}"
    return err


def oracle_dense_rows(inputs, w_new, w_pre, scale, flat_rows, kv_lo=0, kv_hi=None, k64=None,
                      v64=None):
    """Oracle (O, L) for selected flat tokens of a batch."""
    q = np64(inputs["q"][torch.as_tensor(flat_rows, dtype=torch.long)])
    if k64 is None:
        k64 = np64(inputs["k"])
    if v64 is None:
        v64 = np64(inputs["v"])
    pos, kv0 = oatt.token_tables(w_new, w_pre)
    fr = np.asarray(flat_rows, dtype=np.int64)
    return oatt.attention_rows(q, k64, v64, pos[fr], kv0[fr], scale, kv_lo, kv_hi)


def boundary_rows(new_lens, prefix_lens, cp_size, strategy, extra):
    """Flat tokens at every segment's first and last row plus ``extra``."""
    plan = oplan.make_plan(new_lens, prefix_lens, cp_size, strategy)
    rows = set(int(x) for x in extra)
    for r in range(cp_size):
        for s in plan.segments[r]:
            rows.add(plan.gather_idx[s.q_row0])
            rows.add(plan.gather_idx[s.q_row0 + s.q_len - 1])
            if s.q_len > 128:
                rows.add(plan.gather_idx[s.q_row0 + 127])
                rows.add(plan.gather_idx[s.q_row0 + 128])
    return sorted(rows)


def stepwise_partial_kv(q_cat, k, v, plan, scale, kv_block, status=None):
    """The ring's pass-KV schedule emulated call by call through the C ABI
    (a test cross-check of the one-call cp_attn_partial_kv): for every segment
    and every visible block of ``kv_block`` keys one cp_attn_partial with that
    key window gives the fp32 partial (O_j, L_j), then one cp_lse_merge per
    segment merges them, scattered to original token order.
    Returns (O bf16 [N, Hq, dv], LSE [N, Hq]) in original order."""
    import context_causal_attention_cp_gb300 as cpa

    N, Hq, _ = q_cat.shape
    dv = v.shape[2]
    dev = q_cat.device
    out = torch.empty((N, Hq, dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((N, Hq), dtype=torch.float32, device=dev)
    for si, s in enumerate(cpa.segments_host(plan)):
        ql = s["q_len"]
        nb = (s["q_pos0"] + (ql - 1) * s["q_pos_step"]) // kv_block + 1
        po = torch.empty((nb, ql, Hq, dv), dtype=torch.float32, device=dev)
        pl = torch.empty((nb, ql, Hq), dtype=torch.float32, device=dev)
        for j in range(nb):
            cpa.cp_attn_partial(plan.segs[si: si + 1], q_cat, k, v, scale, kv_lo=j * kv_block,
                                kv_hi=(j + 1) * kv_block, out=po[j], lse=pl[j],
                                out_row_base=s["q_row0"], num_out_rows=ql, status=status)
        cpa.cp_lse_merge(po, pl, dst_rows=plan.gather_idx[s["q_row0"]: s["q_row0"] + ql],
                         out=out, lse_out=lse, num_out_rows=N, status=status)
    return out, lse
