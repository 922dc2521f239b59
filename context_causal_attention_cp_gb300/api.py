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
from typing import List, Optional, Sequence

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
        num_reqs=len(new_lens))


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


class PrefillPipeline:
    """Full-KV CP prefill over a stream of same-shaped batches held in host memory.

    Every ``submit`` copies one batch's q, k (and v) from pinned host memory,
    runs plan -> query gather -> attention with the restore fused into its
    store, and copies O and LSE back to pinned host memory.  Two device
    buffer sets and three CUDA streams (upload, compute, download) let batch
    n's attention overlap batch n+1's upload and batch n-1's download; events
    order every reuse of a buffer set.  ``synchronize`` waits for all
    submitted batches; host outputs of a batch are valid after it.
    """

    def __init__(self, new_lens, prefix_lens, cp_size, strategy, Hq, Hkv, d, dv, scale, *,
                 v_is_k_prefix=False, device="cuda"):
        dev = torch.device(device)
        self.N = int(sum(new_lens))
        kv_rows = int(sum(new_lens) + sum(prefix_lens))
        self.scale = scale
        self.dv = dv
        self.v_is_k_prefix = v_is_k_prefix
        self.plan = alloc_plan(new_lens, prefix_lens, cp_size, strategy, device=dev)
        self.status = new_status(dev)
        bf = dict(dtype=torch.bfloat16, device=dev)
        self.bufs = []
        for _ in range(2):
            b = {"q": torch.empty((self.N, Hq, d), **bf), "k": torch.empty((kv_rows, Hkv, d), **bf),
                 "q_cat": torch.empty((self.N, Hq, d), **bf),
                 "o": torch.empty((self.N, Hq, dv), **bf),
                 "lse": torch.empty((self.N, Hq), dtype=torch.float32, device=dev)}
            b["v"] = None if v_is_k_prefix else torch.empty((kv_rows, Hkv, dv), **bf)
            self.bufs.append(b)
        self.s_up = torch.cuda.Stream(dev)
        self.s_comp = torch.cuda.Stream(dev)
        self.s_down = torch.cuda.Stream(dev)
        self.ev_up = [torch.cuda.Event() for _ in range(2)]
        self.ev_comp = [torch.cuda.Event() for _ in range(2)]
        self.ev_down = [torch.cuda.Event() for _ in range(2)]
        self.n = 0

    def submit(self, hq, hk, hv, ho, hlse):
        """Queue one batch: host q, k, v (v ignored when it is a view of k) in,
        host O [N, Hq, dv] bf16 and LSE [N, Hq] fp32 out (all pinned)."""
        i = self.n % 2
        b = self.bufs[i]
        reuse = self.n >= 2
        if reuse:
            self.s_up.wait_event(self.ev_comp[i])     # batch n-2 is done reading set i
        with torch.cuda.stream(self.s_up):
            b["q"].copy_(hq, non_blocking=True)
            b["k"].copy_(hk, non_blocking=True)
            if b["v"] is not None:
                b["v"].copy_(hv, non_blocking=True)
            self.ev_up[i].record(self.s_up)
        self.s_comp.wait_event(self.ev_up[i])
        if reuse:
            self.s_comp.wait_event(self.ev_down[i])   # batch n-2's outputs are downloaded
        with torch.cuda.stream(self.s_comp):
            v = b["k"][:, :, : self.dv] if b["v"] is None else b["v"]
            cp_shard_plan(self.plan, status=self.status, stream=self.s_comp)
            cp_prefill_attention(b["q"], b["k"], v, self.plan, self.scale, status=self.status,
                                 stream=self.s_comp, fuse_restore=True,
                                 workspace={"q_cat": b["q_cat"], "o": b["o"], "lse": b["lse"]})
            self.ev_comp[i].record(self.s_comp)
        self.s_down.wait_event(self.ev_comp[i])
        with torch.cuda.stream(self.s_down):
            ho.copy_(b["o"], non_blocking=True)
            hlse.copy_(b["lse"], non_blocking=True)
            self.ev_down[i].record(self.s_down)
        self.n += 1

    def synchronize(self):
        for s in (self.s_up, self.s_comp, self.s_down):
            s.synchronize()
        check_status(self.status, "prefill pipeline")


def segments_host(plan: ShardPlan):
    """Copy the plan's segment table to the host (list of dicts)."""
    s = plan.segs[: plan.total_segs].cpu().tolist()
    return [dict(zip(SEGMENT_FIELDS, row)) for row in s]


def partial_kv_layout(segs_host, kv_block):
    """Visible KV blocks per segment and the offset of its partial slots."""
    out, slot = [], 0
    for s in segs_host:
        last_pos = s["q_pos0"] + (s["q_len"] - 1) * s["q_pos_step"]
        nb = last_pos // kv_block + 1
        out.append((slot, nb))
        slot += nb * s["q_len"]
    return out, slot


def cp_partial_kv_workspace_size(new_lens, prefix_lens, cp_size, strategy, kv_block, Hq, dv):
    """(workspace bytes, max blocks per segment) for cp_attn_partial_kv."""
    lib = L.load()
    nl, n = _i32_array(new_lens)
    pl, _ = _i32_array(prefix_lens)
    nbytes = ctypes.c_int64()
    mb = ctypes.c_int32()
    L.check(lib.cp_partial_kv_workspace_size(nl, pl, n, cp_size, _strategy(strategy), kv_block,
                                             Hq, dv, ctypes.byref(nbytes), ctypes.byref(mb)),
            "cp_partial_kv_workspace_size")
    return nbytes.value, mb.value


def plan_max_segment_rows(new_lens, cp_size, strategy) -> int:
    """Upper bound on the rows of any segment a plan makes: a zigzag block
    holds at most ceil(n / 2C) tokens of its request, an interleave run at
    most ceil(n / C)."""
    per = 2 * cp_size if _strategy(strategy) == L.ZIGZAG else cp_size
    return max([(int(n) + per - 1) // per for n in new_lens] or [0])


def cp_attn_partial_kv(plan: ShardPlan, q_cat, k, v, scale, kv_block, *, new_lens, prefix_lens,
                       workspace=None, dst_rows="restore", out=None, lse_out=None,
                       out_fp32=False, max_seg_rows=None, status=None, stream=None):
    """Partial-KV decomposition in one library call (layout, split attention, merge).

    ``dst_rows="restore"`` scatters the merged rows to original token order
    (the plan's gather index); ``None`` keeps cat order.  ``max_seg_rows``
    (default: the plan's bound from the request lengths) lets the library
    pack two query heads per tile when every segment has at most 64 rows; 0
    turns packing off.  Returns (O, LSE, workspace).
    """
    lib = L.load()
    N, Hq, d = q_cat.shape
    Hkv, dv = v.shape[1], v.shape[2]
    nbytes, max_blocks = cp_partial_kv_workspace_size(new_lens, prefix_lens, plan.cp_size,
                                                      plan.strategy, kv_block, Hq, dv)
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
        plan_max_segment_rows(new_lens, plan.cp_size, plan.strategy) if max_seg_rows is None
        else int(max_seg_rows), _p(idx), _p(out),
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
    sh = segs_host.to(torch.int32).contiguous()
    # the longest segment: decode-sized segments (<= 64 rows) let the kernel
    # pack two query heads into each 128-row tile
    max_rows = (int(sh[:ns, 1].max()) if ns > 0 else 0) if max_seg_rows is None \
        else int(max_seg_rows)
    nbytes, max_blocks = ctypes.c_int64(), ctypes.c_int32()
    L.check(lib.cp_partial_kv_workspace_size_segs(
        ctypes.c_void_p(sh.data_ptr()), ns, int(kv_block), Hq, dv, ctypes.byref(nbytes),
        ctypes.byref(max_blocks)), "cp_partial_kv_workspace_size_segs")
    if workspace is None:
        workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=q.device)
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
        max(1, int(max_blocks.value)), max_rows, _p(dst_rows), _p(out),
        1 if out.dtype == torch.float32 else 0, _p(lse_out), out.shape[0], _p(workspace),
        workspace.numel(), _p(status), _stream(stream)), "cp_attn_partial_kv")
    return out, lse_out, workspace


def cp_partial_kv_attention(q_cat, k, v, plan: ShardPlan, scale, kv_block, *, segs_host=None,
                            parts_o=None, parts_lse=None, out=None, lse_out=None, status=None,
                            stream=None):
    """Partial-KV (ring-style) CP on one GPU, one KV block at a time.

    Emulates the ring schedule step by step: for every segment and every
    visible block of ``kv_block`` keys, one cp_attn_partial call gives the fp32
    partial (O_j, L_j); then one cp_lse_merge per segment merges them and
    scatters straight to original token order.  cp_attn_partial_kv computes
    the same in three launches.
    Returns (O [N, Hq, dv] bf16, LSE [N, Hq]).
    """
    N, Hq, _ = q_cat.shape
    dv = v.shape[2]
    segs_host = segs_host or segments_host(plan)
    layout, total_slot_rows = partial_kv_layout(segs_host, kv_block)
    dev = q_cat.device
    if parts_o is None:
        parts_o = torch.empty((total_slot_rows, Hq, dv), dtype=torch.float32, device=dev)
    if parts_lse is None:
        parts_lse = torch.empty((total_slot_rows, Hq), dtype=torch.float32, device=dev)
    if out is None:
        out = torch.empty((N, Hq, dv), dtype=torch.bfloat16, device=dev)
    if lse_out is None:
        lse_out = torch.empty((N, Hq), dtype=torch.float32, device=dev)
    for si, s in enumerate(segs_host):
        base, nb = layout[si]
        ql = s["q_len"]
        for j in range(nb):
            o_j = parts_o[base + j * ql: base + (j + 1) * ql]
            l_j = parts_lse[base + j * ql: base + (j + 1) * ql]
            cp_attn_partial(plan.segs[si: si + 1], q_cat, k, v, scale, kv_lo=j * kv_block,
                            kv_hi=(j + 1) * kv_block, out=o_j, lse=l_j,
                            out_row_base=s["q_row0"], num_out_rows=ql, status=status,
                            stream=stream)
    for si, s in enumerate(segs_host):
        base, nb = layout[si]
        ql = s["q_len"]
        o_parts = parts_o[base: base + nb * ql].view(nb, ql, Hq, dv)
        l_parts = parts_lse[base: base + nb * ql].view(nb, ql, Hq)
        cp_lse_merge(o_parts, l_parts, dst_rows=plan.gather_idx[s["q_row0"]: s["q_row0"] + ql],
                     out=out, lse_out=lse_out, num_out_rows=N, status=status, stream=stream)
    return out, lse_out


def pass_q_kv_blocks(kv_total: int, cp_size: int):
    """Resident KV shards of the pass-Q ring for one request.

    The request's KV positions 0..kv_total-1 are cut into 2C near-equal blocks
    (the remainder to the first blocks, as for the zigzag query split) and
    rank r keeps blocks r and 2C-1-r.  Returns, per rank, its two (lo, hi)
    position ranges.
    """
    nb = 2 * cp_size
    base, rem = divmod(int(kv_total), nb)
    starts = [0]
    for i in range(nb):
        starts.append(starts[-1] + base + (1 if i < rem else 0))
    return [[(starts[r], starts[r + 1]), (starts[nb - 1 - r], starts[nb - r])]
            for r in range(cp_size)]


@dataclass
class PassQLaunch:
    """One accumulate launch of the pass-Q ring: at ring hop ``hop`` every
    rank merges the query shard visiting it against resident block ``block``
    of its KV (0: block r of the request's 2C, 1: block 2C-1-r; see
    pass_q_kv_blocks).  ``segs`` holds copies of the plan's segment rows that
    see that block (int32 [n, 8]), ``windows`` their key windows (int32
    [n, 2]), ``seg_ids`` their indices in the plan."""
    hop: int
    block: int
    segs: torch.Tensor
    windows: torch.Tensor
    seg_ids: List[int]


def pass_q_schedule(plan: ShardPlan, segs_host=None) -> List[PassQLaunch]:
    """Host schedule of the pass-Q ring: one launch per (hop, resident block).

    At hop s the shard of rank q visits rank (q + s) mod C.  Each launch
    takes every segment of every shard, with the key window of its host
    rank's block for the segment's request; a segment that cannot see the
    block (the block is empty or starts after the segment's last position)
    is left out.  All windows of one launch belong to different rows, so one
    launch merges every rank's hop at once: at most 2C launches for any
    batch.  The segment copies are taken from the plan as it is now: build
    the schedule again after re-planning a different batch.
    """
    C = plan.cp_size
    segs_host = segs_host or segments_host(plan)
    new_lens = plan.new_lens_dev.cpu().tolist()[: plan.num_reqs]
    prefix_lens = plan.prefix_lens_dev.cpu().tolist()[: plan.num_reqs]
    blocks = [pass_q_kv_blocks(p + n, C) for n, p in zip(new_lens, prefix_lens)]
    shard_of = []
    for r, c in enumerate(plan.segs_per_rank):
        shard_of += [r] * c
    raw = plan.segs[: plan.total_segs].cpu()
    dev = plan.segs.device
    launches = []
    for hop in range(C):
        for b in (0, 1):
            ids, wins = [], []
            for i, sg in enumerate(segs_host):
                lo, hi = blocks[sg["req"]][(shard_of[i] + hop) % C][b]
                last = sg["q_pos0"] + (sg["q_len"] - 1) * sg["q_pos_step"]
                if hi > lo and lo <= last:
                    ids.append(i)
                    wins.append((lo, hi))
            if ids:
                launches.append(PassQLaunch(
                    hop=hop, block=b, segs=raw[ids].contiguous().to(dev),
                    windows=torch.tensor(wins, dtype=torch.int32).to(dev), seg_ids=ids))
    return launches


def cp_pass_q_attention(q_cat, k, v, plan: ShardPlan, scale, *, schedule=None, status=None,
                        stream=None, out=None):
    """Pass-Q ring CP on one GPU, hop by hop.

    KV stays resident: rank r holds the KV blocks of pass_q_kv_blocks.  Each
    rank's query shard travels round the ring with an fp32 accumulator
    (O_acc, L_acc) that starts empty (0, -inf); at hop s rank r merges the
    partial of the visiting shard (of rank (r - s) mod C) against its own KV
    blocks into that accumulator.  One cp_attn_partial_accumulate per launch
    of pass_q_schedule covers every rank of a hop for one of its two blocks,
    each segment with its own key window.  After C hops every accumulator is
    the exact result.
    ``out``: optional (O_acc fp32 [N, Hq, dv], LSE [N, Hq], LSE scratch [N, Hq]).
    Returns (O fp32 [N, Hq, dv], LSE [N, Hq]) in cat order.
    """
    N, Hq, _ = q_cat.shape
    dv = v.shape[2]
    dev = q_cat.device
    sched = pass_q_schedule(plan) if schedule is None else schedule
    with torch.cuda.stream(stream):  # the fills and LSE copies run on the launches' stream
        if out is None:
            o_acc = torch.empty((max(N, 1), Hq, dv), dtype=torch.float32, device=dev)
            lse_a = torch.empty((max(N, 1), Hq), dtype=torch.float32, device=dev)
            lse_b = torch.empty_like(lse_a)
        else:
            o_acc, lse_a, lse_b = out
        o_acc.zero_()
        lse_a.fill_(float("-inf"))
        lse_b.fill_(float("-inf"))
        for launch in sched:
            cp_attn_partial_accumulate(launch.segs, q_cat, k, v, scale, o_acc, lse_a, lse_b,
                                       seg_windows=launch.windows, status=status, stream=stream)
            # rows outside the launch hold equal values in both buffers
            lse_a.copy_(lse_b)
    return o_acc[:N], lse_a[:N]


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
