"""CPU-only checks of the C-ABI library: it loads, exports every entry point
declared in include/cpattn.h, and its host-side logic (plan sizes, argument
validation that returns before any device work) matches the oracle."""

import ctypes
import os
import re

import pytest

from context_causal_attention_cp_gb300 import _lib as L
from context_causal_attention_cp_gb300 import api, workloads as W
from oracle import plan as oplan

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def header_functions():
    src = open(os.path.join(ROOT, "include", "cpattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\s*\*?\s*(cp_\w+)\s*\(", src, flags=re.M)))


def test_library_exports_every_declared_symbol():
    lib = L.load()
    names = header_functions()
    assert {"cp_shard_plan_sizes", "cp_shard_plan", "cp_attn_partial", "cp_lse_merge",
            "cp_attn_partial_restore", "cp_attn_partial_accumulate",
            "cp_restore"} <= set(names)
    for n in names:
        assert hasattr(lib, n), n
        assert n in L.SIGNATURES, f"binding lacks {n}"


def _oracle_sizes(new, pre, C, strategy):
    plan = oplan.make_plan(new, pre, C, strategy)
    rows = [len(plan.rank_rows[r]) for r in range(C)]
    segs = [len(plan.segments[r]) for r in range(C)]
    tiles = [sum((s.q_len + 127) // 128 for s in plan.segments[r]) for r in range(C)]
    return rows, segs, tiles


@pytest.mark.parametrize("seed", range(30))
@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_plan_sizes_match_oracle(seed, strategy):
    new, pre = W.random_batch(seed, max_new=700)
    C = [1, 2, 3, 4, 8, 5][seed % 6]
    assert api.cp_shard_plan_sizes(new, pre, C, strategy) == _oracle_sizes(new, pre, C, strategy)


@pytest.mark.parametrize("name", sorted(W.WORKLOADS))
def test_plan_sizes_workloads(name):
    w = W.WORKLOADS[name]
    for strategy in w.strategies:
        got = api.cp_shard_plan_sizes(w.new_lens, w.prefix_lens, w.cp_size, strategy)
        assert got == _oracle_sizes(w.new_lens, w.prefix_lens, w.cp_size, strategy)


def test_invalid_arguments_are_rejected_on_host():
    lib = L.load()
    a = (ctypes.c_int32 * 2)(4, 5)
    out = (ctypes.c_int32 * 4)()
    assert lib.cp_shard_plan_sizes(a, a, 2, 0, 0, out, out, out) == L.ERR_INVALID_ARG
    assert lib.cp_shard_plan_sizes(a, a, 2, 4, 7, out, out, out) == L.ERR_INVALID_ARG
    neg = (ctypes.c_int32 * 2)(4, -1)
    assert lib.cp_shard_plan_sizes(neg, a, 2, 4, 0, out, out, out) == L.ERR_INVALID_ARG
    assert lib.cp_shard_plan_sizes(a, a, -1, 4, 0, out, out, out) == L.ERR_INVALID_ARG
    # attention: Hq not a multiple of Hkv, unsupported head dims, bad scale
    # (never dereferenced: every call below fails validation before any launch)
    nul = None
    fake = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(5)]
    args = [fake[0], 1, nul, 0, fake[1], 128, fake[2], 1024, 128, fake[3], 1024, 128, 256]
    o, lse = fake[4], ctypes.c_void_p(0x90000)
    assert lib.cp_attn_partial(*args, 6, 4, 128, 128, 0.1, 0, -1, o, 0, lse, 0, 128, nul,
                               nul) == L.ERR_INVALID_ARG
    assert lib.cp_attn_partial(*args, 8, 4, 96, 96, 0.1, 0, -1, o, 0, lse, 0, 128, nul,
                               nul) == L.ERR_UNSUPPORTED
    assert lib.cp_attn_partial(*args, 8, 4, 128, 128, 0.0, 0, -1, o, 0, lse, 0, 128, nul,
                               nul) == L.ERR_INVALID_ARG
    assert lib.cp_attn_partial(*args, 8, 4, 128, 128, 0.1, 0, -1, nul, 0, lse, 0, 128, nul,
                               nul) == L.ERR_INVALID_ARG
    # partial-KV: block count limits and workspace sizing on the host
    assert lib.cp_attn_partial_kv(*args, 8, 4, 128, 128, 0.1, 64, 33, 0, nul, o, 0, lse, 128,
                                  fake[1], 1 << 20, nul, nul) == L.ERR_INVALID_ARG
    assert lib.cp_attn_partial_kv(*args, 8, 4, 128, 128, 0.1, 64, 4, -1, nul, o, 0, lse, 128,
                                  fake[1], 1 << 20, nul, nul) == L.ERR_INVALID_ARG
    nbytes, mb = ctypes.c_int64(), ctypes.c_int32()
    one = (ctypes.c_int32 * 1)(1000)
    zero = (ctypes.c_int32 * 1)(0)
    msr = ctypes.c_int32()
    assert lib.cp_partial_kv_workspace_size(one, zero, 1, 2, 0, 0, 8, 128, ctypes.byref(nbytes),
                                            ctypes.byref(mb), None) == L.ERR_INVALID_ARG
    assert lib.cp_partial_kv_workspace_size(one, zero, 1, 2, 0, 256, 8, 128, ctypes.byref(nbytes),
                                            ctypes.byref(mb), ctypes.byref(msr)) == L.OK
    assert (mb.value, msr.value) == (4, 250)
    # a batch without new tokens: max_blocks 0, and the call is a no-op
    assert lib.cp_partial_kv_workspace_size(zero, one, 1, 2, 0, 256, 8, 128, ctypes.byref(nbytes),
                                            ctypes.byref(mb), ctypes.byref(msr)) == L.OK
    assert (mb.value, msr.value) == (0, 0)
    empty = [fake[0], 0] + args[2:]
    assert lib.cp_attn_partial_kv(*empty, 8, 4, 128, 128, 0.1, 64, 0, 0, nul, nul, 0, nul, 0,
                                  nul, 0, nul, nul) == L.OK
    assert lib.cp_attn_partial_kv(*args, 8, 4, 128, 128, 0.1, 64, 0, 0, nul, o, 0, lse, 128,
                                  fake[1], 1 << 20, nul, nul) == L.ERR_INVALID_ARG
    # merge: part count and dv limits
    assert lib.cp_lse_merge(nul, nul, 0, 0, 0, 4, 2, 128, nul, nul, 1, nul, 4, nul,
                            nul) == L.ERR_INVALID_ARG
    assert lib.cp_lse_merge(nul, nul, 33, 0, 0, 4, 2, 128, nul, nul, 1, nul, 4, nul,
                            nul) == L.ERR_INVALID_ARG
    assert lib.cp_lse_merge(nul, nul, 2, 0, 0, 4, 2, 126, nul, nul, 1, nul, 4, nul,
                            nul) == L.ERR_INVALID_ARG
    # restore: row bytes must be a multiple of 4
    assert lib.cp_restore(nul, 4, nul, 4, 22, nul, nul, nul) == L.ERR_INVALID_ARG
    # misaligned pointers are refused before any launch
    assert lib.cp_restore(ctypes.c_void_p(0x1002), 4, ctypes.c_void_p(0x2000), 4, 32,
                          ctypes.c_void_p(0x3000), nul, nul) == L.ERR_ALIGNMENT


def test_restore_and_accumulate_calls_validate_on_host():
    """Argument checks of the fused-restore and pass-Q accumulate entry points
    (every call fails validation before any launch; pointers are never used)."""
    lib = L.load()
    nul = None
    fake = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
    args = [fake[0], 1, nul, 0, fake[1], 128, fake[2], 1024, 128, fake[3], 1024, 128, 256]
    o, lse, dst = fake[4], fake[5], fake[6]
    # restore: the destination index is required, shapes checked as for cp_attn_partial
    assert lib.cp_attn_partial_restore(*args, 8, 4, 128, 128, 0.1, 0, -1, nul, o, 0, lse, 128,
                                       nul, nul) == L.ERR_INVALID_ARG
    assert lib.cp_attn_partial_restore(*args, 6, 4, 128, 128, 0.1, 0, -1, dst, o, 0, lse, 128,
                                       nul, nul) == L.ERR_INVALID_ARG
    assert lib.cp_attn_partial_restore(*args, 8, 4, 96, 96, 0.1, 0, -1, dst, o, 0, lse, 128,
                                       nul, nul) == L.ERR_UNSUPPORTED
    assert lib.cp_attn_partial_restore(*args, 8, 4, 128, 128, 0.1, 0, -1, dst,
                                       ctypes.c_void_p(0x40008), 0, lse, 128, nul,
                                       nul) == L.ERR_ALIGNMENT
    # accumulate: the two LSE buffers (128 rows x 8 heads x 4 B = 4096 B) must not overlap
    la = 0x80000
    for lb in (la, la + 16, la + 4092, la - 4092):
        assert lib.cp_attn_partial_accumulate(*args, 8, 4, 128, 128, 0.1, 0, -1, nul, o,
                                              ctypes.c_void_p(la), ctypes.c_void_p(lb), 0, 128,
                                              nul, nul) == L.ERR_INVALID_ARG, hex(lb)
    # adjacent buffers are fine (the call then fails on the unsupported shape)
    for lb in (la + 4096, la - 4096):
        assert lib.cp_attn_partial_accumulate(*args, 8, 4, 96, 96, 0.1, 0, -1, nul, o,
                                              ctypes.c_void_p(la), ctypes.c_void_p(lb), 0, 128,
                                              nul, nul) == L.ERR_UNSUPPORTED, hex(lb)
    assert lib.cp_attn_partial_accumulate(*args, 8, 4, 128, 128, 0.1, 0, -1, nul, nul,
                                          ctypes.c_void_p(la), ctypes.c_void_p(la + 8192), 0,
                                          128, nul, nul) == L.ERR_INVALID_ARG
    assert lib.cp_attn_partial_accumulate(*args, 8, 4, 128, 128, 0.1, 0, -1, nul,
                                          ctypes.c_void_p(0x40004), ctypes.c_void_p(la),
                                          ctypes.c_void_p(la + 8192), 0, 128, nul,
                                          nul) == L.ERR_ALIGNMENT
    # per-segment windows must be int32-aligned
    assert lib.cp_attn_partial_accumulate(*args, 8, 4, 128, 128, 0.1, 0, -1,
                                          ctypes.c_void_p(0x50002), o, ctypes.c_void_p(la),
                                          ctypes.c_void_p(la + 8192), 0, 128, nul,
                                          nul) == L.ERR_ALIGNMENT


def test_ring_and_host_prefill_calls_validate_on_host():
    """Argument checks of cp_attn_pass_q and cp_prefill_host (every call fails
    validation before anything is queued; pointers are never used)."""
    lib = L.load()
    nul = None
    fake = [ctypes.c_void_p(0x10000 * (i + 1)) for i in range(8)]
    first = (ctypes.c_int32 * 3)(0, 4, 2)        # decreasing: invalid
    qkv = [fake[2], 128, fake[3], 1024, 128, fake[3], 1024, 128, 256, 8, 8, 128, 128, 0.1]
    assert lib.cp_attn_pass_q(fake[0], fake[1], first, 2, *qkv, fake[4], fake[5], fake[6], nul,
                              nul) == L.ERR_INVALID_ARG
    assert lib.cp_attn_pass_q(fake[0], fake[1], first, 1, *qkv, nul, fake[5], fake[6], nul,
                              nul) == L.ERR_INVALID_ARG
    assert lib.cp_attn_pass_q(fake[0], fake[1], first, 1, *qkv, ctypes.c_void_p(0x40008),
                              fake[5], fake[6], nul, nul) == L.ERR_ALIGNMENT
    lens = (ctypes.c_int32 * 1)(1000)
    pre = (ctypes.c_int32 * 1)(0)
    nbytes = ctypes.c_int64()
    assert lib.cp_prefill_host_workspace_size(lens, pre, 1, 4, 0, 8, 8, 128, 128, 0,
                                              ctypes.byref(nbytes)) == L.OK
    set_bytes = 2 * (1000 * 8 * 128 * 2) + 1000 * 8 * 128 * 2 + 1000 * 8 * 4
    assert nbytes.value >= 2 * set_bytes
    ptrs = (ctypes.c_void_p * 1)(0x1000)
    args = [lens, pre, 1, 4, 0, 8, 8, 128, 128, 0.1, 0, 1, ptrs, ptrs, ptrs, ptrs, ptrs]
    # too small a workspace, a misaligned one, a missing host pointer, a bad strategy
    assert lib.cp_prefill_host(*args, fake[0], nbytes.value - 1, nul, nul, nul,
                               nul) == L.ERR_INVALID_ARG
    assert lib.cp_prefill_host(*args, ctypes.c_void_p(0x10010), nbytes.value, nul, nul, nul,
                               nul) == L.ERR_ALIGNMENT
    none = (ctypes.c_void_p * 1)(None)
    bad = args[:12] + [none] + args[13:]
    assert lib.cp_prefill_host(*bad, fake[0], nbytes.value, nul, nul, nul,
                               nul) == L.ERR_INVALID_ARG
    bad = args[:4] + [7] + args[5:]
    assert lib.cp_prefill_host(*bad, fake[0], nbytes.value, nul, nul, nul,
                               nul) == L.ERR_INVALID_ARG
    # no batches: nothing to do
    zero = args[:11] + [0] + args[12:]
    assert lib.cp_prefill_host(*zero, nul, 0, nul, nul, nul, nul) == L.OK


def test_select_pass_cost_matches_oracle():
    """Host logic of cp_select_pass_cost against the oracle on a grid: the
    same exposed times (to rounding) and the same choice."""
    from oracle import select as osel
    for Hq, Hkv in ((128, 8), (32, 8), (64, 64)):
        for T in (1, 7, 1000, 16384, 131072):
            for P in (0, 3, 4096, 124518):
                for C in (1, 2, 4, 8):
                    for tf, link, merge in ((620.0, 50.0, 3000.0), (1500.0, 450.0, 6000.0)):
                        got, ekv, eq = api.cp_select_pass_cost(T, P, Hq, Hkv, 128, C, tf, link,
                                                               merge)
                        r_kv, r_q = osel.exposed_times(T, P, Hq, Hkv, 128, C, tf, link, merge)
                        assert ekv == pytest.approx(r_kv, rel=1e-12, abs=1e-18)
                        assert eq == pytest.approx(r_q, rel=1e-12, abs=1e-18)
                        if abs(r_kv - r_q) > 1e-9 * max(r_kv, r_q):
                            assert got == osel.select_by_cost(T, P, Hq, Hkv, 128, C, tf, link,
                                                              merge)
    lib = L.load()
    for bad in ((0, 0, 8, 8, 128, 4, 1.0, 1.0, 1.0), (1, 0, 8, 8, 128, 4, 0.0, 1.0, 1.0),
                (1, 0, 8, 8, 128, 4, 1.0, float("inf"), 1.0), (1, 0, 8, 3, 128, 4, 1.0, 1.0, 1.0),
                (1, 0, 8, 8, 0, 4, 1.0, 1.0, 1.0), (1, 0, 8, 8, 128, 0, 1.0, 1.0, 1.0)):
        assert lib.cp_select_pass_cost(*bad, None, None) == L.ERR_INVALID_ARG, bad


def test_status_strings():
    for code in (L.OK, L.ERR_INVALID_ARG, L.ERR_UNSUPPORTED, L.ERR_CUDA, L.ERR_TIMEOUT,
                 L.ERR_ALIGNMENT, L.ERR_RANGE, L.ERR_TOO_LARGE):
        assert L.status_string(code) not in ("", "unknown status")


@pytest.mark.parametrize("seed", range(20))
@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_partial_kv_workspace_matches_oracle_segments(seed, strategy):
    """Workspace rows = sum over the oracle plan's segments of (visible KV blocks x rows)."""
    new, pre = W.random_batch(seed, max_new=700, max_prefix=300)
    C = [1, 2, 3, 4, 8][seed % 5]
    kv_block = [64, 100, 128, 1000][seed % 4]
    Hq, dv = 4, 64
    op = oplan.make_plan(new, pre, C, strategy)
    segs = [s for r in range(C) for s in op.segments[r]]
    rows = sum(((s.q_pos0 + (s.q_len - 1) * s.q_pos_step) // kv_block + 1) * s.q_len for s in segs)
    mb = max([(s.q_pos0 + (s.q_len - 1) * s.q_pos_step) // kv_block + 1 for s in segs] or [0])
    longest = max([s.q_len for s in segs] or [0])
    r256 = lambda x: (x + 255) // 256 * 256  # noqa: E731
    expect = r256((2 * len(segs) + 2) * 8) + r256(rows * Hq * dv * 4) + r256(rows * Hq * 4) + 256
    assert api.cp_partial_kv_workspace_size(new, pre, C, strategy, kv_block, Hq, dv) == \
        (expect, mb, longest)


def test_select_pass_matches_oracle():
    """Host logic of cp_select_pass against the oracle on a grid, both rules."""
    from oracle import select as osel
    for Hq, Hkv in ((32, 8), (128, 8), (64, 64), (12, 1)):
        for T in (1, 2, 3, 100, 1500, 16384, 131072):
            for P in (0, 1, 5, 999, 16384, 114688, 10 ** 7):
                got, score = api.cp_select_pass(T, P, Hq, Hkv, "message")
                assert got == osel.select_by_messages(T, P, Hq, Hkv), (T, P, Hq, Hkv)
                got, score = api.cp_select_pass(T, P, Hq, Hkv, "fitted")
                assert got == osel.select_fitted(T, P)
                assert score == pytest.approx(osel.fitted_score(T, P), rel=1e-12, abs=1e-12)


def test_select_pass_rejects_bad_arguments():
    lib = L.load()
    for args in ((0, 5, 8, 8, 0), (5, -1, 8, 8, 0), (5, 5, 6, 4, 0), (5, 5, 8, 8, 2),
                 (1 << 41, 0, 8, 8, 0)):
        assert lib.cp_select_pass(*args, None) == L.ERR_INVALID_ARG


def test_plan_limits_refused_on_host():
    """cp_size above CPATTN_MAX_CP and more than CPATTN_MAX_REQS requests."""
    with pytest.raises(L.CpAttnError):
        api.cp_shard_plan_sizes([5], [0], 1025, "zigzag")
    with pytest.raises(L.CpAttnError):
        api.cp_shard_plan_sizes([1] * 65537, [0] * 65537, 2, "zigzag")
    rows, _, _ = api.cp_shard_plan_sizes([2100, 5, 4096], [0, 3, 100], 1024, "zigzag")
    assert sum(rows) == 2100 + 5 + 4096 and len(rows) == 1024


def test_binding_refuses_host_tensors_before_any_launch():
    """A host tensor (or wrong dtype / shape) never reaches a kernel as a
    device pointer: the binding raises first."""
    import torch
    q = torch.zeros(8, 2, 64, dtype=torch.bfloat16)
    segs = torch.zeros(1, 8, dtype=torch.int32)
    idx = torch.zeros(8, dtype=torch.int32)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.cp_attn_partial(segs, q, q, q, 0.1)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.cp_attn_partial_restore(segs, q, q, q, 0.1, idx)
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.cp_attn_partial_accumulate(segs, q, q, q, 0.1, torch.zeros(8, 2, 64),
                                       torch.zeros(8, 2), torch.zeros(8, 2))
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.cp_lse_merge(torch.zeros(2, 8, 2, 64), torch.zeros(2, 8, 2))
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.cp_restore(q, idx)
    plan = api.alloc_plan([16], [0], 4, "zigzag", device="cpu")
    with pytest.raises(ValueError, match="CUDA tensor"):
        api.cp_shard_plan(plan)


@pytest.mark.parametrize("seed", range(6))
@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_workspace_size_from_segments_matches_plan_sizing(seed, strategy):
    """cp_partial_kv_workspace_size_segs over a plan's own segments gives the
    plan-based sizing, and decode-style segments (step 0) size by hand."""
    import torch
    new, pre = W.random_batch(400 + seed, max_reqs=5, max_new=700, max_prefix=300)
    C, kv_block, Hq, dv = [2, 3, 4, 8, 1, 5][seed], [64, 100, 256, 512, 7, 1000][seed], 8, 64
    op = oplan.make_plan(new, pre, C, strategy)
    rows = [[s.q_row0, s.q_len, s.q_pos0, s.q_pos_step, s.kv_row0, s.kv_len,
             op.gather_idx[s.q_row0], s.req] for r in range(C) for s in op.segments[r]]
    lib = L.load()
    seg = torch.tensor(rows or [[0] * 8], dtype=torch.int32)
    b1, m1, r1 = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
    assert lib.cp_partial_kv_workspace_size_segs(ctypes.c_void_p(seg.data_ptr()), len(rows),
                                                 kv_block, Hq, dv, ctypes.byref(b1),
                                                 ctypes.byref(m1), ctypes.byref(r1)) == L.OK
    assert (b1.value, m1.value, r1.value) == api.cp_partial_kv_workspace_size(
        new, pre, C, strategy, kv_block, Hq, dv)


def test_workspace_size_for_decode_segment():
    import torch
    lib = L.load()
    seg = torch.tensor([[0, 64, 8191, 0, 0, 8192, 0, 0]], dtype=torch.int32)
    b, m, r = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
    assert lib.cp_partial_kv_workspace_size_segs(ctypes.c_void_p(seg.data_ptr()), 1, 512, 32, 128,
                                                 ctypes.byref(b), ctypes.byref(m), None) == L.OK
    rows = 16 * 64                       # 16 blocks of 512 keys, 64 rows each
    expect = 256 + ((rows * 32 * 128 * 4 + 255) // 256) * 256 + ((rows * 32 * 4 + 255) // 256) * 256 + 256
    assert (b.value, m.value) == (expect, 16)
    assert api.cp_partial_kv_workspace_size_segs(seg, 512, 32, 128) == (expect, 16, 64)


def _oracle_segments(new, pre, C, strategy):
    """The oracle plan's segments in table order, as cp_segment_t rows."""
    op = oplan.make_plan(new, pre, C, strategy)
    rows, shard = [], []
    for r in range(C):
        for s in op.segments[r]:
            rows.append([s.q_row0, s.q_len, s.q_pos0, s.q_pos_step, s.kv_row0, s.kv_len,
                         op.gather_idx[s.q_row0], s.req])
            shard.append(r)
    return rows, shard


@pytest.mark.parametrize("seed", range(12))
def test_pass_q_schedule_covers_every_visible_key_once(seed):
    """The library's ring schedule (host call) against the oracle: every entry
    is a copy of an oracle plan segment, its window is the oracle's resident
    KV block of rank (shard + hop) mod C, no launch holds a segment twice, and
    over all launches each segment meets every key its rows can see exactly
    once."""
    from oracle import pipeline as opipe
    new, pre = W.random_batch(900 + seed, max_reqs=5, max_new=400, max_prefix=200)
    C = [1, 2, 3, 4, 8, 5][seed % 6]
    strategy = "zigzag" if seed % 2 == 0 else "interleave"
    segs, shard = _oracle_segments(new, pre, C, strategy)
    sched = api.pass_q_schedule_host(new, pre, C, strategy)
    assert sched.num_launches <= 2 * C
    assert sched.launch_first[-1] == len(sched.seg_ids)
    seen = {i: [] for i in range(len(segs))}
    rows, wins = sched.segs.tolist(), sched.windows.tolist()
    for li in range(sched.num_launches):
        hop, block = sched.hops[li], sched.blocks[li]
        ids = sched.seg_ids[sched.launch_first[li]: sched.launch_first[li + 1]]
        assert ids and len(set(ids)) == len(ids)
        for e in range(sched.launch_first[li], sched.launch_first[li + 1]):
            i = sched.seg_ids[e]
            assert rows[e] == segs[i]
            req = segs[i][7]
            host = (shard[i] + hop) % C
            expect = opipe.resident_kv_windows(new[req] + pre[req], C)[host][block]
            assert tuple(wins[e]) == tuple(expect)
            seen[i].append(tuple(wins[e]))
    for i, sg in enumerate(segs):
        last = sg[2] + (sg[1] - 1) * sg[3]
        keys = [k for lo, hi in sorted(seen[i]) for k in range(lo, min(hi, last + 1))]
        assert keys == list(range(last + 1)), (i, sorted(seen[i]))


@pytest.mark.parametrize("seed", range(8))
@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_host_segment_table_matches_oracle_plan(seed, strategy):
    """The library's host mirror of the plan, read back through the ring
    schedule's segment copies, holds exactly the oracle plan's segments, field
    by field."""
    new, pre = W.random_batch(1700 + seed, max_reqs=6, max_new=600, max_prefix=300)
    C = [1, 2, 3, 4, 8, 6, 16, 5][seed]
    segs, _ = _oracle_segments(new, pre, C, strategy)
    sched = api.pass_q_schedule_host(new, pre, C, strategy)
    got = {}
    for e, i in enumerate(sched.seg_ids):
        got[i] = sched.segs[e].tolist()
    # every segment appears: at some hop it visits the rank holding key 0
    assert sorted(got) == list(range(len(segs)))
    assert [got[i] for i in range(len(segs))] == segs


def _c_param_kind(decl):
    """ctypes kind of one C parameter declaration of the header."""
    d = " ".join(decl.split())
    if "*" in d or d.startswith("cudaStream_t"):
        return "ptr"
    base = d.rsplit(" ", 1)[0].replace("const ", "")
    return {"int": "i32", "int32_t": "i32", "cp_strategy_t": "i32", "int64_t": "i64",
            "long long": "i64", "float": "f32", "double": "f64"}[base]


def _ctypes_kind(t):
    import ctypes
    if t in (ctypes.c_void_p, ctypes.c_char_p) or hasattr(t, "_type_") and \
            isinstance(getattr(t, "_type_"), type):
        return "ptr"
    return {ctypes.c_int32: "i32", ctypes.c_int64: "i64", ctypes.c_longlong: "i64",
            ctypes.c_float: "f32", ctypes.c_double: "f64"}.get(t, repr(t))


def test_binding_signatures_match_the_header():
    """Every prototype in include/cpattn.h has a binding entry with the same
    number of arguments and the same kind (pointer, 32 / 64-bit integer,
    float) at each position, so no ctypes call can shift its arguments."""
    src = open(os.path.join(ROOT, "include", "cpattn.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    protos = re.findall(r"\b(?:int|const\s+char\s*\*)\s*(cp_\w+)\s*\(([^;{]*?)\)\s*;", src,
                        flags=re.S)
    assert len(protos) == len(header_functions())
    for name, params in protos:
        decls = [p.strip() for p in params.split(",")] if params.strip() not in ("", "void") else []
        want = [_c_param_kind(p) for p in decls]
        got = [_ctypes_kind(t) for t in L.SIGNATURES[name][1]]
        assert got == want, (name, got, want)


@pytest.mark.parametrize("seed", range(10))
def test_sizing_reports_the_longest_segment(seed):
    """The longest-segment figure of the library's sizing call (it decides head
    packing in the partial-KV call) equals the longest segment of the
    oracle's plan."""
    new, pre = W.random_batch(1300 + seed, max_reqs=6, max_new=500, max_prefix=100)
    C = [1, 2, 3, 4, 8][seed % 5]
    for strategy in ("zigzag", "interleave"):
        op = oplan.make_plan(new, pre, C, strategy)
        longest = max([s.q_len for r in range(C) for s in op.segments[r]] or [0])
        assert api.cp_partial_kv_workspace_size(new, pre, C, strategy, 512, 8, 64)[2] == longest


def test_nvtx_knob():
    """The NVTX switch of cp_attn_debug toggles, and host validation is the
    same with the ranges on (no tool attached: the ranges are no-ops)."""
    lib = L.load()
    try:
        assert lib.cp_attn_debug(L.DEBUG_NVTX, 1) == L.OK
        assert lib.cp_restore(None, 4, None, 4, 22, None, None, None) == L.ERR_INVALID_ARG
        assert lib.cp_attn_debug(L.DEBUG_NVTX, 0) == L.OK
    finally:
        lib.cp_attn_debug(L.DEBUG_NVTX, 0)
    assert lib.cp_attn_debug(99, 1) == L.ERR_INVALID_ARG
