"""Python binding of the C ABI (argument marshalling only).

Every function here converts torch tensors to raw pointers and sizes and calls
the same-named entry point of ``libcpattn.so``; all device work runs in the
library's CUDA kernels.  PyTorch supplies device memory and streams.

Layouts (see include/cpattn.h):
    q      bf16 [rows, Hq, d]          (cat rows: shard rows in rank order)
    k, v   bf16 [kv_rows, Hkv, d|dv]   (last dim contiguous; v may view k)
    o      bf16 or fp32 [rows, Hq, dv]; lse fp32 [rows, Hq] (natural log)
"""

from dataclasses import dataclass
from typing import List, Sequence

import ctypes
import math
import torch

from . import _lib as L

SEGMENT_FIELDS = ("q_row0", "q_len", "q_pos0", "q_pos_step", "kv_row0", "kv_len", "tok0", "req")
STRATEGIES = {"zigzag": L.ZIGZAG, "interleave": L.INTERLEAVE}


def _strategy(s):
    if isinstance(s, str):
        return STRATEGIES[s]
    return int(s)


def _stream(stream):
    return ctypes.c_void_p((stream or torch.cuda.current_stream()).cuda_stream)


def _p(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else None


def _dev(t, name, dtype=None, ref=None, contiguous=True):
    """Check a device argument before its pointer reaches a kernel: a CUDA
    tensor (on ref's device), of dtype, contiguous.  None passes through."""
    if t is None:
        return
    if not isinstance(t, torch.Tensor) or not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if ref is not None and t.device != ref.device:
        raise ValueError(f"{name} is on {t.device}, the call runs on {ref.device}")
    if dtype is not None and t.dtype not in (dtype if isinstance(dtype, tuple) else (dtype,)):
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if contiguous and not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _shape(t, name, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def _segments(segs, num_segs, tiles, num_tiles, ref):
    _dev(segs, "segs", torch.int32, ref)
    if segs.dim() != 2 or segs.shape[1] != 8:
        raise ValueError("segs must be int32 [S, 8] (cp_segment_t rows)")
    ns = segs.shape[0] if num_segs is None else int(num_segs)
    if ns < 0 or ns > segs.shape[0]:
        raise ValueError("num_segs exceeds the segment table")
    nt = 0
    if tiles is not None:
        _dev(tiles, "tiles", torch.int32, ref)
        if tiles.dim() != 2 or tiles.shape[1] != 2:
            raise ValueError("tiles must be int32 [T, 2]")
        nt = tiles.shape[0] if num_tiles is None else int(num_tiles)
        if nt < 0 or nt > tiles.shape[0]:
            raise ValueError("num_tiles exceeds the tile list")
    return ns, nt


def _status(status, ref):
    if status is not None:
        _dev(status, "status", torch.int32, ref)
        if status.numel() < 1:
            raise ValueError("status needs one int32")


def _i32_array(xs):
    xs = [int(x) for x in xs]
    return (ctypes.c_int32 * max(1, len(xs)))(*xs), len(xs)


def new_status(device="cuda"):
    """A zeroed device status word (int32[1])."""
    return torch.zeros(1, dtype=torch.int32, device=device)


def check_status(status, where="device"):
    """Synchronise on the status word and raise if a kernel reported an error."""
    code = int(status.item())
    if code != L.OK:
        raise L.CpAttnError(code, where)


# --------------------------------------------------------------------- plan --
def cp_shard_plan_sizes(new_lens: Sequence[int], prefix_lens: Sequence[int], cp_size: int,
                        strategy):
    lib = L.load()
    nl, n = _i32_array(new_lens)
    pl, n2 = _i32_array(prefix_lens)
    if n != n2:
        raise ValueError("new_lens and prefix_lens differ in length")
    rows = (ctypes.c_int32 * cp_size)()
    segs = (ctypes.c_int32 * cp_size)()
    tiles = (ctypes.c_int32 * cp_size)()
    L.check(lib.cp_shard_plan_sizes(nl, pl, n, cp_size, _strategy(strategy), rows, segs, tiles),
            "cp_shard_plan_sizes")
    return list(rows), list(segs), list(tiles)


@dataclass
class ShardPlan:
    cp_size: int
    strategy: int
    rows_per_rank: List[int]
    segs_per_rank: List[int]
    tiles_per_rank: List[int]
    segs: torch.Tensor          # int32 [S, 8] (cp_segment_t)
    seg_offsets: torch.Tensor   # int32 [C+1]
    row_offsets: torch.Tensor   # int32 [C+1]
    gather_idx: torch.Tensor    # int32 [N]
    positions: torch.Tensor     # int32 [N]
    restore_idx: torch.Tensor   # int32 [N]
    tiles: torch.Tensor         # int32 [T, 2]
    new_lens_dev: torch.Tensor
    prefix_lens_dev: torch.Tensor
    num_reqs: int
    new_lens: List[int]          # host copies of the lengths the plan was made from
    prefix_lens: List[int]

    @property
    def total_rows(self):
        return sum(self.rows_per_rank)

    @property
    def total_segs(self):
        return sum(self.segs_per_rank)

    @property
    def total_tiles(self):
        return sum(self.tiles_per_rank)


def alloc_plan(new_lens, prefix_lens, cp_size, strategy, device="cuda") -> ShardPlan:
    """Host size pass plus device buffers for a plan (nothing launched)."""
    rows, segs, tiles = cp_shard_plan_sizes(new_lens, prefix_lens, cp_size, strategy)
    N, S, T = sum(rows), sum(segs), sum(tiles)
    i32 = dict(dtype=torch.int32, device=device)
    return ShardPlan(
        cp_size=cp_size, strategy=_strategy(strategy), rows_per_rank=rows, segs_per_rank=segs,
        tiles_per_rank=tiles, segs=torch.empty((max(S, 1), 8), **i32),
        seg_offsets=torch.empty(cp_size + 1, **i32), row_offsets=torch.empty(cp_size + 1, **i32),
        gather_idx=torch.empty(max(N, 1), **i32), positions=torch.empty(max(N, 1), **i32),
        restore_idx=torch.empty(max(N, 1), **i32), tiles=torch.empty((max(T, 1), 2), **i32),
        new_lens_dev=torch.tensor([int(x) for x in new_lens] or [0], **i32),
        prefix_lens_dev=torch.tensor([int(x) for x in prefix_lens] or [0], **i32),
        num_reqs=len(new_lens), new_lens=[int(x) for x in new_lens],
        prefix_lens=[int(x) for x in prefix_lens])


def cp_shard_plan(plan: ShardPlan, status=None, stream=None) -> ShardPlan:
    """Fill ``plan``'s device buffers (kernel launches on ``stream``)."""
    lib = L.load()
    for name in ("new_lens_dev", "prefix_lens_dev", "segs", "seg_offsets", "row_offsets",
                 "gather_idx", "positions", "restore_idx", "tiles"):
        _dev(getattr(plan, name), "plan." + name, torch.int32, plan.segs)
    _status(status, plan.segs)
    L.check(lib.cp_shard_plan(
        _p(plan.new_lens_dev), _p(plan.prefix_lens_dev), plan.num_reqs, plan.cp_size, plan.strategy,
        plan.total_rows, plan.total_segs, plan.total_tiles, _p(plan.segs), _p(plan.seg_offsets),
        _p(plan.row_offsets), _p(plan.gather_idx), _p(plan.positions), _p(plan.restore_idx),
        _p(plan.tiles), _p(status), _stream(stream)), "cp_shard_plan")
    return plan


def make_plan(new_lens, prefix_lens, cp_size, strategy, device="cuda", status=None,
              stream=None) -> ShardPlan:
    return cp_shard_plan(alloc_plan(new_lens, prefix_lens, cp_size, strategy, device), status,
                         stream)


# ---------------------------------------------------------------- attention --
def _check_qkv(q, k, v):
    _dev(q, "q", torch.bfloat16)
    _dev(k, "k", torch.bfloat16, q, contiguous=False)
    _dev(v, "v", torch.bfloat16, q, contiguous=False)
    if q.dim() != 3 or k.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k and v are [rows, heads, dim]")
    if k.shape[1] != v.shape[1] or k.shape[0] != v.shape[0]:
        raise ValueError("k and v disagree on rows or heads")
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise TypeError("q, k and v must be bfloat16")
    if not q.is_contiguous() or k.stride(2) != 1 or v.stride(2) != 1:
        raise ValueError("q must be contiguous; k and v need a contiguous last dim")


def _attn_outputs(out, lse, n_out, Hq, dv, out_fp32, ref):
    """Allocate or check the O [n, Hq, dv] (bf16 / fp32) and LSE [n, Hq] outputs."""
    if out is None:
        out = torch.empty((n_out, Hq, dv), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=ref.device)
    _dev(out, "out", (torch.bfloat16, torch.float32), ref)
    if out.dim() != 3 or tuple(out.shape[1:]) != (Hq, dv):
        raise ValueError(f"out must be [rows, {Hq}, {dv}], got {tuple(out.shape)}")
    if lse is None:
        lse = torch.empty((out.shape[0], Hq), dtype=torch.float32, device=ref.device)
    _dev(lse, "lse", torch.float32, ref)
    _shape(lse, "lse", (out.shape[0], Hq))
    return out, lse


def cp_attn_partial(segs, q, k, v, scale, *, num_segs=None, tiles=None, num_tiles=None,
                    kv_lo=0, kv_hi=-1, out=None, lse=None, out_fp32=False, out_row_base=0,
                    num_out_rows=None, status=None, stream=None):
    """Partial causal attention of every segment row (see cp_attn_partial in cpattn.h)."""
    lib = L.load()
    _check_qkv(q, k, v)
    rows, Hq, d = q.shape
    Hkv, dv = v.shape[1], v.shape[2]
    n_out = rows if num_out_rows is None else num_out_rows
    out, lse = _attn_outputs(out, lse, n_out, Hq, dv, out_fp32, q)
    ns, nt = _segments(segs, num_segs, tiles, num_tiles, q)
    _status(status, q)
    L.check(lib.cp_attn_partial(
        _p(segs), ns, _p(tiles), nt, _p(q), rows, _p(k), k.stride(0), k.stride(1), _p(v),
        v.stride(0), v.stride(1), k.shape[0], Hq, Hkv, d, dv, float(scale), int(kv_lo),
        int(kv_hi), _p(out), 1 if out.dtype == torch.float32 else 0, _p(lse), int(out_row_base),
        out.shape[0], _p(status), _stream(stream)), "cp_attn_partial")
    return out, lse


def cp_attn_prefill(segs, q, k, v, scale, *, num_segs=None, tiles=None, num_tiles=None,
                    out=None, lse=None, out_fp32=False, status=None, stream=None):
    """Full-KV attention with q, O and LSE in original token order (segment
    rows addressed by token index; every segment a consecutive token run,
    e.g. a zigzag plan): the shard gather and the restore happen in the
    kernel.  See cp_attn_prefill in cpattn.h."""
    lib = L.load()
    _check_qkv(q, k, v)
    n, Hq, d = q.shape
    Hkv, dv = v.shape[1], v.shape[2]
    out, lse = _attn_outputs(out, lse, n, Hq, dv, out_fp32, q)
    if out.shape[0] != n:
        raise ValueError("out needs one row per token")
    ns, nt = _segments(segs, num_segs, tiles, num_tiles, q)
    _status(status, q)
    L.check(lib.cp_attn_prefill(
        _p(segs), ns, _p(tiles), nt, _p(q), n, _p(k), k.stride(0), k.stride(1), _p(v),
        v.stride(0), v.stride(1), k.shape[0], Hq, Hkv, d, dv, float(scale), _p(out),
        1 if out.dtype == torch.float32 else 0, _p(lse), _p(status), _stream(stream)),
        "cp_attn_prefill")
    return out, lse


def cp_attn_partial_restore(segs, q, k, v, scale, dst_rows, *, num_out_rows=None,
                            num_segs=None, tiles=None, num_tiles=None, kv_lo=0, kv_hi=-1,
                            out=None, lse=None, out_fp32=False, status=None, stream=None):
    """cp_attn_partial storing query row i at output row dst_rows[i] (restore fused)."""
    lib = L.load()
    _check_qkv(q, k, v)
    rows, Hq, d = q.shape
    Hkv, dv = v.shape[1], v.shape[2]
    _dev(dst_rows, "dst_rows", torch.int32, q)
    if dst_rows.dim() != 1 or dst_rows.shape[0] < rows:
        raise ValueError("dst_rows must be int32 with one entry per query row")
    n_out = rows if num_out_rows is None else num_out_rows
    out, lse = _attn_outputs(out, lse, n_out, Hq, dv, out_fp32, q)
    ns, nt = _segments(segs, num_segs, tiles, num_tiles, q)
    _status(status, q)
    L.check(lib.cp_attn_partial_restore(
        _p(segs), ns, _p(tiles), nt, _p(q), rows, _p(k), k.stride(0), k.stride(1), _p(v),
        v.stride(0), v.stride(1), k.shape[0], Hq, Hkv, d, dv, float(scale), int(kv_lo),
        int(kv_hi), _p(dst_rows), _p(out), 1 if out.dtype == torch.float32 else 0, _p(lse),
        out.shape[0], _p(status), _stream(stream)), "cp_attn_partial_restore")
    return out, lse


def cp_attn_partial_accumulate(segs, q, k, v, scale, o_acc, lse_acc, lse_out, *, num_segs=None,
                               tiles=None, num_tiles=None, kv_lo=0, kv_hi=-1, seg_windows=None,
                               out_row_base=0, status=None, stream=None):
    """One pass-Q hop: merge this window's partial into (o_acc, lse_acc) -> (o_acc, lse_out).

    ``seg_windows``: optional int32 [num_segs, 2] on the device; segment s
    then uses key window [lo, hi) = seg_windows[s] in place of (kv_lo, kv_hi).
    """
    lib = L.load()
    _check_qkv(q, k, v)
    rows, Hq, d = q.shape
    Hkv, dv = v.shape[1], v.shape[2]
    _dev(o_acc, "o_acc", torch.float32, q)
    _dev(lse_acc, "lse_acc", torch.float32, q)
    _dev(lse_out, "lse_out", torch.float32, q)
    if o_acc.dim() != 3 or tuple(o_acc.shape[1:]) != (Hq, dv):
        raise ValueError("o_acc must be [rows, Hq, dv]")
    _shape(lse_acc, "lse_acc", (o_acc.shape[0], Hq))
    _shape(lse_out, "lse_out", (o_acc.shape[0], Hq))
    ns, nt = _segments(segs, num_segs, tiles, num_tiles, q)
    if seg_windows is not None:
        _dev(seg_windows, "seg_windows", torch.int32, q)
        if seg_windows.dim() != 2 or seg_windows.shape[1] != 2 or seg_windows.shape[0] < ns:
            raise ValueError("seg_windows must be int32 [num_segs, 2]")
    _status(status, q)
    L.check(lib.cp_attn_partial_accumulate(
        _p(segs), ns, _p(tiles), nt, _p(q), rows, _p(k), k.stride(0), k.stride(1), _p(v),
        v.stride(0), v.stride(1), k.shape[0], Hq, Hkv, d, dv, float(scale), int(kv_lo),
        int(kv_hi), _p(seg_windows), _p(o_acc), _p(lse_acc), _p(lse_out), int(out_row_base),
        o_acc.shape[0], _p(status), _stream(stream)), "cp_attn_partial_accumulate")
    return o_acc, lse_out


# -------------------------------------------------------------------- merge --
def cp_lse_merge(o_parts, lse_parts, *, dst_rows=None, out=None, lse_out=None, out_fp32=True,
                 num_out_rows=None, status=None, stream=None):
    """LSE merge over axis 0 of o_parts [n, rows, Hq, dv] / lse_parts [n, rows, Hq]."""
    lib = L.load()
    _dev(o_parts, "o_parts", torch.float32, contiguous=False)
    _dev(lse_parts, "lse_parts", torch.float32, o_parts, contiguous=False)
    if o_parts.dim() != 4 or lse_parts.dim() != 3:
        raise ValueError("o_parts is [n, rows, Hq, dv] and lse_parts [n, rows, Hq]")
    n, rows, Hq, dv = o_parts.shape
    if tuple(lse_parts.shape) != (n, rows, Hq):
        raise ValueError("lse_parts disagrees with o_parts")
    if o_parts[0].stride() != (Hq * dv, dv, 1) or lse_parts[0].stride() != (Hq, 1):
        raise ValueError("each partial must be contiguous")
    if dst_rows is not None:
        _dev(dst_rows, "dst_rows", torch.int32, o_parts)
        if dst_rows.dim() != 1 or dst_rows.shape[0] < rows:
            raise ValueError("dst_rows needs one int32 per row")
    n_out = rows if num_out_rows is None else num_out_rows
    if out is None:
        out = torch.empty((n_out, Hq, dv), dtype=torch.float32 if out_fp32 else torch.bfloat16,
                          device=o_parts.device)
    _dev(out, "out", (torch.bfloat16, torch.float32), o_parts)
    if out.dim() != 3 or tuple(out.shape[1:]) != (Hq, dv):
        raise ValueError("out must be [rows, Hq, dv]")
    if lse_out is not None:
        _dev(lse_out, "lse_out", torch.float32, o_parts)
        _shape(lse_out, "lse_out", (out.shape[0], Hq))
    _status(status, o_parts)
    L.check(lib.cp_lse_merge(
        _p(o_parts), _p(lse_parts), n, o_parts.stride(0), lse_parts.stride(0), rows, Hq, dv,
        _p(dst_rows), _p(out), 1 if out.dtype == torch.float32 else 0, _p(lse_out), out.shape[0],
        _p(status), _stream(stream)), "cp_lse_merge")
    return out, lse_out


# ------------------------------------------------------------------ restore --
def cp_restore(src, idx, *, out=None, status=None, stream=None):
    """out[i] = src[idx[i]] (rows along dim 0)."""
    lib = L.load()
    _dev(src, "src")
    _dev(idx, "idx", torch.int32, src)
    if idx.dim() != 1:
        raise ValueError("idx must be a 1-D int32 index")
    rows = idx.shape[0]
    row_bytes = math.prod(src.shape[1:]) * src.element_size()
    if out is None:
        out = torch.empty((rows,) + tuple(src.shape[1:]), dtype=src.dtype, device=src.device)
    _dev(out, "out", src.dtype, src)
    _shape(out, "out", (rows,) + tuple(src.shape[1:]))
    _status(status, src)
    L.check(lib.cp_restore(_p(src), src.shape[0], _p(idx), rows, row_bytes, _p(out), _p(status),
                           _stream(stream)), "cp_restore")
    return out


# --------------------------------------------------------------- pipelines --
def cp_prefill_attention(q, k, v, plan: ShardPlan, scale, *, status=None, stream=None,
                         q_is_cat=False, workspace=None, fuse_restore=False):
    """Full-KV prefill CP on one GPU: shard rows -> attention -> restore.

    ``fuse_restore``: the attention store writes original order directly
    (cp_attn_partial_restore with the plan's gather index) instead of a
    separate cp_restore pass over O and LSE; with a zigzag plan and q in
    original order the kernel also reads the queries by token index
    (cp_attn_prefill), so no gather runs either.

    q: bf16 [N, Hq, d] in original (flat) order, or already in cat order when
    ``q_is_cat``.  Returns (O [N, Hq, dv] bf16, LSE [N, Hq] fp32) in original order.
    """
    N, Hq, _ = q.shape
    dv = v.shape[2]
    ws = workspace or {}
    if fuse_restore and not q_is_cat and plan.strategy == L.ZIGZAG:
        # zigzag segments are consecutive token runs: no gather, no restore pass
        return cp_attn_prefill(plan.segs, q, k, v, scale, num_segs=plan.total_segs,
                               tiles=plan.tiles, num_tiles=plan.total_tiles, out=ws.get("o"),
                               lse=ws.get("lse"), status=status, stream=stream)
    q_cat = q if q_is_cat else cp_restore(q, plan.gather_idx[:N], out=ws.get("q_cat"),
                                          status=status, stream=stream)
    if fuse_restore:
        return cp_attn_partial_restore(plan.segs, q_cat, k, v, scale, plan.gather_idx,
                                       num_out_rows=N, num_segs=plan.total_segs,
                                       tiles=plan.tiles, num_tiles=plan.total_tiles,
                                       out=ws.get("o"), lse=ws.get("lse"), status=status,
                                       stream=stream)
    o_cat, lse_cat = cp_attn_partial(plan.segs, q_cat, k, v, scale, num_segs=plan.total_segs,
                                     tiles=plan.tiles, num_tiles=plan.total_tiles,
                                     out=ws.get("o_cat"), lse=ws.get("lse_cat"),
                                     status=status, stream=stream)
    o = cp_restore(o_cat, plan.restore_idx[:N], out=ws.get("o"), status=status, stream=stream)
    lse = cp_restore(lse_cat, plan.restore_idx[:N], out=ws.get("lse"), status=status,
                     stream=stream)
    return o, lse


def cp_prefill_host_workspace_size(new_lens, prefix_lens, cp_size, strategy, Hq, Hkv, d, dv,
                                   v_is_k_prefix=False) -> int:
    """Device bytes cp_prefill_host needs (plan buffers and two buffer sets)."""
    lib = L.load()
    nl, n = _i32_array(new_lens)
    pl, _ = _i32_array(prefix_lens)
    nbytes = ctypes.c_int64()
    L.check(lib.cp_prefill_host_workspace_size(nl, pl, n, cp_size, _strategy(strategy), Hq, Hkv,
                                                d, dv, 1 if v_is_k_prefix else 0,
                                                ctypes.byref(nbytes)),
            "cp_prefill_host_workspace_size")
    return nbytes.value


def _host(t, name, dtype, shape):
    if not isinstance(t, torch.Tensor) or t.is_cuda:
        raise ValueError(f"{name} must be a host tensor")
    if t.dtype != dtype or tuple(t.shape) != tuple(shape) or not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous {dtype} {tuple(shape)}")


def cp_prefill_host(new_lens, prefix_lens, cp_size, strategy, Hq, Hkv, d, dv, scale, batches, *,
                    v_is_k_prefix=False, workspace=None, status=None, streams=None,
                    device="cuda"):
    """Host-to-host full-KV CP prefill of same-shaped batches (cp_prefill_host in cpattn.h).

    ``batches``: list of (q, k, v, o, lse) host tensors (pinned for the copies
    to overlap; v may be None with ``v_is_k_prefix``); o and lse are written.
    ``streams``: (compute, upload, download) CUDA streams (default: three new
    ones).  Returns (workspace, streams); the outputs are valid once the
    download stream has completed (``streams[2].synchronize()``).
    """
    lib = L.load()
    dev = torch.device(device)
    nl, n = _i32_array(new_lens)
    pl, _ = _i32_array(prefix_lens)
    N, KV = int(sum(new_lens)), int(sum(new_lens) + sum(prefix_lens))
    for i, (q, k, v, o, lse) in enumerate(batches):
        _host(q, f"q[{i}]", torch.bfloat16, (N, Hq, d))
        _host(k, f"k[{i}]", torch.bfloat16, (KV, Hkv, d))
        if not v_is_k_prefix:
            _host(v, f"v[{i}]", torch.bfloat16, (KV, Hkv, dv))
        _host(o, f"o[{i}]", torch.bfloat16, (N, Hq, dv))
        _host(lse, f"lse[{i}]", torch.float32, (N, Hq))
    nbytes = cp_prefill_host_workspace_size(new_lens, prefix_lens, cp_size, strategy, Hq, Hkv,
                                            d, dv, v_is_k_prefix)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    _dev(workspace, "workspace", torch.uint8)
    if workspace.numel() < nbytes:
        raise ValueError(f"workspace needs {nbytes} bytes")
    _status(status, workspace)
    if streams is None:
        streams = tuple(torch.cuda.Stream(dev) for _ in range(3))
    nb = len(batches)
    ptrs = lambda xs: (ctypes.c_void_p * max(1, nb))(  # noqa: E731
        *[x.data_ptr() if x is not None else None for x in xs])
    q_p, k_p = ptrs([b[0] for b in batches]), ptrs([b[1] for b in batches])
    v_p = ptrs([b[2] if not v_is_k_prefix else None for b in batches])
    o_p, l_p = ptrs([b[3] for b in batches]), ptrs([b[4] for b in batches])
    L.check(lib.cp_prefill_host(
        nl, pl, n, cp_size, _strategy(strategy), Hq, Hkv, d, dv, float(scale),
        1 if v_is_k_prefix else 0, nb, q_p, k_p, v_p, o_p, l_p, _p(workspace), workspace.numel(),
        _p(status), ctypes.c_void_p(streams[0].cuda_stream),
        ctypes.c_void_p(streams[1].cuda_stream), ctypes.c_void_p(streams[2].cuda_stream)),
        "cp_prefill_host")
    return workspace, streams


def segments_host(plan: ShardPlan):
    """Copy the plan's segment table to the host (list of dicts)."""
    s = plan.segs[: plan.total_segs].cpu().tolist()
    return [dict(zip(SEGMENT_FIELDS, row)) for row in s]


def cp_partial_kv_workspace_size(new_lens, prefix_lens, cp_size, strategy, kv_block, Hq, dv):
    """(workspace bytes, max blocks per segment, longest segment) for
    cp_attn_partial_kv over the plan these lengths make."""
    lib = L.load()
    nl, n = _i32_array(new_lens)
    pl, _ = _i32_array(prefix_lens)
    nbytes = ctypes.c_int64()
    mb = ctypes.c_int32()
    msr = ctypes.c_int32()
    L.check(lib.cp_partial_kv_workspace_size(nl, pl, n, cp_size, _strategy(strategy), kv_block,
                                             Hq, dv, ctypes.byref(nbytes), ctypes.byref(mb),
                                             ctypes.byref(msr)),
            "cp_partial_kv_workspace_size")
    return nbytes.value, mb.value, msr.value


def cp_partial_kv_workspace_size_segs(segs_host, kv_block, Hq, dv):
    """The same sizing for an explicit host segment table (int32 [S, 8])."""
    lib = L.load()
    sh = torch.as_tensor(segs_host, dtype=torch.int32).contiguous()
    if sh.dim() != 2 or sh.shape[1] != 8:
        raise ValueError("segs_host must be int32 [S, 8] (cp_segment_t rows)")
    nbytes, mb, msr = ctypes.c_int64(), ctypes.c_int32(), ctypes.c_int32()
    L.check(lib.cp_partial_kv_workspace_size_segs(
        ctypes.c_void_p(sh.data_ptr()), sh.shape[0], int(kv_block), Hq, dv, ctypes.byref(nbytes),
        ctypes.byref(mb), ctypes.byref(msr)), "cp_partial_kv_workspace_size_segs")
    return nbytes.value, mb.value, msr.value


def cp_attn_partial_kv(plan: ShardPlan, q_cat, k, v, scale, kv_block, *, workspace=None,
                       dst_rows="restore", out=None, lse_out=None, out_fp32=False,
                       max_seg_rows=None, status=None, stream=None):
    """Partial-KV decomposition in one library call (layout, split attention, merge).

    ``dst_rows="restore"`` scatters the merged rows to original token order
    (the plan's gather index); ``None`` keeps cat order.  ``max_seg_rows``
    (default: the longest segment of the plan, from the library's sizing
    call) lets the library pack two query heads per tile when every segment
    has at most 64 rows; 0 turns packing off.  Returns (O, LSE, workspace).
    """
    lib = L.load()
    N, Hq, d = q_cat.shape
    Hkv, dv = v.shape[1], v.shape[2]
    nbytes, max_blocks, longest = cp_partial_kv_workspace_size(
        plan.new_lens, plan.prefix_lens, plan.cp_size, plan.strategy, kv_block, Hq, dv)
    _check_qkv(q_cat, k, v)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q_cat.device)
    _dev(workspace, "workspace", torch.uint8, q_cat)
    idx = plan.gather_idx[:N] if isinstance(dst_rows, str) else dst_rows
    if idx is not None:
        _dev(idx, "dst_rows", torch.int32, q_cat)
        if idx.dim() != 1 or idx.shape[0] < N:
            raise ValueError("dst_rows needs one int32 per query row")
    out, lse_out = _attn_outputs(out, lse_out, N, Hq, dv, out_fp32, q_cat)
    _segments(plan.segs, plan.total_segs, plan.tiles, plan.total_tiles, q_cat)
    _status(status, q_cat)
    L.check(lib.cp_attn_partial_kv(
        _p(plan.segs), plan.total_segs, _p(plan.tiles), plan.total_tiles, _p(q_cat), N, _p(k),
        k.stride(0), k.stride(1), _p(v), v.stride(0), v.stride(1), k.shape[0], Hq, Hkv, d, dv,
        float(scale), int(kv_block), int(max_blocks),
        longest if max_seg_rows is None else int(max_seg_rows), _p(idx), _p(out),
        1 if out.dtype == torch.float32 else 0, _p(lse_out), out.shape[0], _p(workspace),
        workspace.numel(), _p(status), _stream(stream)), "cp_attn_partial_kv")
    return out, lse_out, workspace


def cp_attn_split_kv(segs, q, k, v, scale, kv_block, *, segs_host=None, num_out_rows=None,
                     dst_rows=None, out=None, lse_out=None, out_fp32=True, workspace=None,
                     max_seg_rows=None, status=None, stream=None):
    """cp_attn_partial over any segment table with every segment's keys split
    into blocks of ``kv_block`` attended by separate CTAs, then merged by the
    LSE rule inside the library (cp_attn_partial_kv without a plan).  Meant for
    few query rows over many keys, e.g. a decode step against one KV shard.
    ``max_seg_rows`` (default: the longest segment of ``segs_host``) is passed
    to the library; at most 64 lets it pack two query heads per tile, 0
    turns packing off.
    ``dst_rows`` (int32, one per query row) scatters the output; otherwise row
    i of the output is query row i.  Returns (O, LSE, workspace).
    """
    lib = L.load()
    _check_qkv(q, k, v)
    rows, Hq, d = q.shape
    Hkv, dv = v.shape[1], v.shape[2]
    ns, _ = _segments(segs, None, None, None, q)
    if segs_host is None:
        segs_host = segs.cpu()
    nbytes, max_blocks, longest = cp_partial_kv_workspace_size_segs(segs_host[:ns], kv_block, Hq,
                                                                    dv)
    max_rows = longest if max_seg_rows is None else int(max_seg_rows)
    if workspace is None:
        workspace = torch.empty(nbytes, dtype=torch.uint8, device=q.device)
    _dev(workspace, "workspace", torch.uint8, q)
    if dst_rows is not None:
        _dev(dst_rows, "dst_rows", torch.int32, q)
        if dst_rows.dim() != 1 or dst_rows.shape[0] < rows:
            raise ValueError("dst_rows needs one int32 per query row")
    n_out = rows if num_out_rows is None else num_out_rows
    out, lse_out = _attn_outputs(out, lse_out, n_out, Hq, dv, out_fp32, q)
    _status(status, q)
    L.check(lib.cp_attn_partial_kv(
        _p(segs), ns, None, 0, _p(q), rows, _p(k), k.stride(0), k.stride(1), _p(v), v.stride(0),
        v.stride(1), k.shape[0], Hq, Hkv, d, dv, float(scale), int(kv_block),
        max(1, int(max_blocks)), max_rows, _p(dst_rows), _p(out),
        1 if out.dtype == torch.float32 else 0, _p(lse_out), out.shape[0], _p(workspace),
        workspace.numel(), _p(status), _stream(stream)), "cp_attn_partial_kv")
    return out, lse_out, workspace


@dataclass
class PassQSchedule:
    """The pass-Q ring schedule from cp_pass_q_schedule: launch i covers
    entries launch_first[i] .. launch_first[i+1]-1 at ring hop hops[i] and
    resident block blocks[i] (0: block r of the request's 2C KV blocks, 1:
    block 2C-1-r).  ``segs`` (int32 [E, 8], device) are copies of the plan's
    segment rows, ``windows`` (int32 [E, 2], device) their key windows and
    ``seg_ids`` (host) their indices in the plan's segment table."""
    launch_first: List[int]
    hops: List[int]
    blocks: List[int]
    segs: torch.Tensor
    windows: torch.Tensor
    seg_ids: List[int]

    @property
    def num_launches(self):
        return len(self.hops)


def pass_q_schedule(plan: ShardPlan, device=None) -> PassQSchedule:
    """The library's pass-Q ring schedule for the plan's lengths (host call),
    with its entry arrays copied to the plan's device."""
    return pass_q_schedule_host(plan.new_lens, plan.prefix_lens, plan.cp_size, plan.strategy,
                                plan.segs.device if device is None else device)


def pass_q_schedule_host(new_lens, prefix_lens, cp_size, strategy, device="cpu") -> PassQSchedule:
    """cp_pass_q_schedule for these lengths; entry arrays on ``device``."""
    lib = L.load()
    nl, n = _i32_array(new_lens)
    pl, _ = _i32_array(prefix_lens)
    strategy = _strategy(strategy)
    nlaunch, nent = ctypes.c_int32(), ctypes.c_int32()
    L.check(lib.cp_pass_q_schedule_size(nl, pl, n, cp_size, strategy,
                                        ctypes.byref(nlaunch), ctypes.byref(nent)),
            "cp_pass_q_schedule_size")
    nL, nE = nlaunch.value, nent.value
    first = (ctypes.c_int32 * (nL + 1))()
    hops = (ctypes.c_int32 * max(1, nL))()
    blocks = (ctypes.c_int32 * max(1, nL))()
    segs = torch.zeros((max(1, nE), 8), dtype=torch.int32)
    wins = torch.zeros((max(1, nE), 2), dtype=torch.int32)
    ids = (ctypes.c_int32 * max(1, nE))()
    L.check(lib.cp_pass_q_schedule(nl, pl, n, cp_size, strategy, first, hops, blocks,
                                   ctypes.c_void_p(segs.data_ptr()),
                                   ctypes.cast(ctypes.c_void_p(wins.data_ptr()), L.c_i32p), ids),
            "cp_pass_q_schedule")
    return PassQSchedule(launch_first=list(first), hops=list(hops)[:nL],
                         blocks=list(blocks)[:nL], segs=segs.to(device), windows=wins.to(device),
                         seg_ids=list(ids)[:nE])


def cp_pass_q_attention(q_cat, k, v, plan: ShardPlan, scale, *, schedule=None, status=None,
                        stream=None, out=None):
    """Pass-Q ring CP on one GPU (cp_attn_pass_q in cpattn.h): every query
    shard travels round the ring with an fp32 accumulator that each hop's
    partial against the host rank's resident KV is merged into.
    ``schedule``: from pass_q_schedule(plan) (built when omitted).
    ``out``: optional (O_acc fp32 [N, Hq, dv], LSE [N, Hq], LSE scratch [N, Hq]).
    Returns (O fp32 [N, Hq, dv], LSE [N, Hq]) in cat order.
    """
    lib = L.load()
    _check_qkv(q_cat, k, v)
    N, Hq, d = q_cat.shape
    Hkv, dv = v.shape[1], v.shape[2]
    dev = q_cat.device
    sched = pass_q_schedule(plan, dev) if schedule is None else schedule
    if out is None:
        out = (torch.empty((max(N, 1), Hq, dv), dtype=torch.float32, device=dev),
               torch.empty((max(N, 1), Hq), dtype=torch.float32, device=dev),
               torch.empty((max(N, 1), Hq), dtype=torch.float32, device=dev))
    o_acc, lse, lse_b = out
    for t, name in ((o_acc, "o_acc"), (lse, "lse"), (lse_b, "lse_scratch")):
        _dev(t, name, torch.float32, q_cat)
    if o_acc.shape[0] < N or tuple(o_acc.shape[1:]) != (Hq, dv):
        raise ValueError("o_acc must be [N, Hq, dv]")
    if lse.shape[0] < N or lse_b.shape[0] < N or lse.shape[1:] != (Hq,) or \
            lse_b.shape[1:] != (Hq,):
        raise ValueError("lse buffers must be [N, Hq]")
    _dev(sched.segs, "schedule.segs", torch.int32, q_cat)
    _dev(sched.windows, "schedule.windows", torch.int32, q_cat)
    _status(status, q_cat)
    first = (ctypes.c_int32 * len(sched.launch_first))(*sched.launch_first)
    L.check(lib.cp_attn_pass_q(
        _p(sched.segs), _p(sched.windows), first, sched.num_launches, _p(q_cat), N, _p(k),
        k.stride(0), k.stride(1), _p(v), v.stride(0), v.stride(1), k.shape[0], Hq, Hkv, d, dv,
        float(scale), _p(o_acc), _p(lse), _p(lse_b), _p(status), _stream(stream)),
        "cp_attn_pass_q")
    return o_acc[:N], lse[:N]


def cp_select_pass(new_tokens: int, cached_tokens: int, Hq: int, Hkv: int, rule="message"):
    """Pass-KV or pass-Q for a step (see cp_select_pass in cpattn.h).

    rule: "message" (miss rate against 2*Hkv/Hq) or "fitted" (the fitted
    heuristic h(T, P)).  Returns ("pass_kv" | "pass_q", score).
    """
    lib = L.load()
    rules = {"message": L.SELECT_MESSAGE, "fitted": L.SELECT_FITTED}
    score = ctypes.c_double()
    r = lib.cp_select_pass(int(new_tokens), int(cached_tokens), int(Hq), int(Hkv), rules[rule],
                           ctypes.byref(score))
    if r < 0:
        L.check(r, "cp_select_pass")
    return ("pass_q" if r == L.PASS_Q else "pass_kv"), score.value


def cp_select_pass_cost(new_tokens: int, cached_tokens: int, Hq: int, Hkv: int, head_dim: int,
                        cp_size: int, attn_tflops: float, link_gbs: float, merge_gbs: float):
    """Pass-KV or pass-Q by exposed communication (see cp_select_pass_cost in
    cpattn.h).  Returns ("pass_kv" | "pass_q", E_kv seconds, E_q seconds)."""
    lib = L.load()
    ekv, eq = ctypes.c_double(), ctypes.c_double()
    r = lib.cp_select_pass_cost(int(new_tokens), int(cached_tokens), int(Hq), int(Hkv),
                                int(head_dim), int(cp_size), float(attn_tflops), float(link_gbs),
                                float(merge_gbs), ctypes.byref(ekv), ctypes.byref(eq))
    if r < 0:
        L.check(r, "cp_select_pass_cost")
    return ("pass_q" if r == L.PASS_Q else "pass_kv"), ekv.value, eq.value
