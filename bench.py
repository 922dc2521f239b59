#!/usr/bin/env python
"""Benchmark: causal prefill context-parallel attention on one GB300.

Default workload: one 32768-token prompt, Llama-3-8B-shaped attention (32
query / 8 KV heads, head dim 128), CP = 8 zigzag (16 blocks of 2048), bf16
N(0,1) synthetic inputs.  One step is the whole hot path on the device:
shard plan -> causal attention of all 8 shards against the gathered KV in
one launch that reads each shard's query rows and writes O and LSE by token
index (zigzag shards are runs of consecutive tokens: the query gather and the
restore happen in the kernel's own loads and stores).  ``value`` is causal attention TFLOP/s over the step (2*Hq*(d+dv)
flops per visible (query, key) pair), L2 flushed between steps.

The line also carries the LSE-merge GB/s of the 131072-token partial-KV
decomposition (16 KV blocks of 8192, 136 visible fp32 partials merged and
scattered to causal order), that decomposition end to end as one call
(pass-KV) and through the pass-Q ring, the GB/s of the standalone restore kernel (the
two-pass path's cp_restore of O and LSE), the attention kernel's
roofline, clocks under load, an end-to-end figure through the public API with
host buffers, and the CPU oracle timed on a bounded sample of the same
workload.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""

import argparse
import json
import math
import os
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal CP-prefill attention TFLOPS & % of GB300 bf16 peak; LSE-merge GB/s"
UNIT = "TFLOP/s"
WORKLOAD = "llama8b_32k"
MERGE_WORKLOAD = "partialkv_128k"
DECODE_KV_BLOCK = 4096  # keys per CTA in the decode step (2 blocks per rank)
# ncu summary under profiles/ holding the attention kernel's DRAM bytes per launch
PROFILE_MD = {"llama8b_32k": "attn_fwd_llama8b_32k.md", "mla_16k": "attn_mla_mla_16k.md"}


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            p = json.load(f)
        return dict(hbm_gbs=float(p["hbm_gbs"]), bf16_tflops=float(p["bf16_tflops"]),
                    bf16_tflops_sustained=float(p.get("bf16_tflops_sustained", p["bf16_tflops"])),
                    source="measured")
    except Exception:  # noqa: BLE001 - the recipe's fallback
        return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0,
                    source="fallback")


def profiled_traffic(kernel_md="attn_fwd_llama8b_32k.md"):
    """DRAM bytes per launch recorded by the ncu summary under profiles/, or
    None when the kernel's sources changed since the counters were taken
    (the summary records a SHA-256 prefix of each source file)."""
    import hashlib
    import re

    if not kernel_md:
        return None
    path = os.path.join(ROOT, "profiles", kernel_md)
    try:
        text = open(path).read()
    except OSError:
        return None
    m = re.search(r"traffic_bytes_per_launch:\s*(\d+)", text)
    h = re.search(r"source_sha256_prefix:\s*(.+)", text)
    if not m or not h:
        return None
    csrc = os.path.join(ROOT, "context_causal_attention_cp_gb300", "csrc")
    for name, prefix in re.findall(r"([\w.]+) ([0-9a-f]{16})", h.group(1)):
        try:
            digest = hashlib.sha256(open(os.path.join(csrc, name), "rb").read()).hexdigest()
        except OSError:
            return None
        if not digest.startswith(prefix):
            return None
    return int(m.group(1))


def visible_pairs(new_lens, prefix_lens):
    # every new token at position P sees P + 1 keys
    return sum(n * p + n * (n + 1) // 2 for n, p in zip(new_lens, prefix_lens))


def algorithmic_bytes(w):
    """Bytes an attention launch must move: Q, K, V once, O (bf16) and LSE once."""
    kv = w.total_kv * w.Hkv * (w.d + (0 if w.v_is_k_prefix else w.dv)) * 2
    return w.total_new * w.Hq * (w.d * 2 + w.dv * 2 + 4) + kv


def attention_flops(w):
    return 2.0 * w.Hq * (w.d + w.dv) * visible_pairs(w.new_lens, w.prefix_lens)


def reduce_max_over_ranks(value, world, device="cpu"):
    """Max of a per-rank float over the process group (identity at world 1)."""
    if world <= 1:
        return float(value)
    import torch
    import torch.distributed as dist

    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(flops_per_rank, world, steps, max_total_ms):
    """Whole-job TFLOP/s: the work of every rank over the slowest rank's time."""
    return flops_per_rank * world * steps / (max_total_ms * 1e-3) / 1e12


def kernel_label(w):
    if w.d == 576:
        return "attn_mla_kernel (tcgen05; 128 rows x 1 head x one 256-column output half per CTA)"
    nq = 2 if (w.Hq // w.Hkv) % 2 == 0 else 1
    return f"attn_fwd_kernel (tcgen05; {nq} head(s) x 128 rows per CTA)"


def config_of(w, extra=None):
    cfg = {"workload": f"{w.name}: {w.description}", "new_lens": w.new_lens,
           "prefix_lens": w.prefix_lens, "heads_q": w.Hq, "heads_kv": w.Hkv, "d": w.d,
           "dv": w.dv, "cp_size": w.cp_size, "strategy": w.strategies[0],
           "l2": "flushed between steps (256 MiB write outside the step's events)"}
    if extra:
        cfg.update(extra)
    return cfg


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 50 ms; entering
    waits (up to 3 s) for the first sample so that the samples kept, those
    read between entering and leaving, fall inside the timed region."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []
        self.keep = False

    def _reader(self):
        for line in self.proc.stdout:
            if self.keep:
                self.lines.append(line)
            self.first.set()

    def __enter__(self):
        import threading
        self.first = threading.Event()
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except Exception:  # noqa: BLE001
            self.proc = None
            return self
        self.thread = threading.Thread(target=self._reader, daemon=True)
        self.thread.start()
        self.first.wait(timeout=3.0)
        self.keep = True
        return self

    def __exit__(self, *a):
        self.keep = False
        self.out = "".join(self.lines)
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()

    def summary(self):
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in (self.out or "").strip().splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sms.append(float(parts[1]))
                mx = float(parts[2])
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        if not sms:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"]}
        sms.sort()
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# ------------------------------------------------------------- oracle leg --
def oracle_sample_rate(w, inputs, budget_s, seed=0):
    """Time the CPU oracle on seeded query rows of the workload for ~budget_s.

    Returns (flops per second, rows, seconds, threads)."""
    import numpy as np
    import torch
    from oracle import attention as oatt

    threads = len(os.sched_getaffinity(0))
    torch.set_num_threads(threads)
    k64 = inputs["k"].float().numpy().astype(np.float64)
    v64 = (k64[:, :, : w.dv] if w.v_is_k_prefix else
           inputs["v"].float().numpy().astype(np.float64))
    pos, kv0 = oatt.token_tables(w.new_lens, w.prefix_lens)
    g = torch.Generator().manual_seed(seed)
    order = torch.randperm(w.total_new, generator=g).tolist()
    done, flops, t0 = 0, 0.0, time.perf_counter()
    while done < len(order):
        i = order[done]
        q = inputs["q"][i: i + 1].float().numpy().astype(np.float64)
        oatt.attention_rows(q, k64, v64, pos[i: i + 1], kv0[i: i + 1], w.scale)
        flops += 2.0 * w.Hq * (w.d + w.dv) * (int(pos[i]) + 1)
        done += 1
        if time.perf_counter() - t0 > budget_s:
            break
    dt = time.perf_counter() - t0
    return flops / dt, done, dt, threads


def run_reference(args):
    """The oracle as the reference arm, on the host cores (rank 0 only)."""
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return 0
    from context_causal_attention_cp_gb300 import workloads as W

    w = W.WORKLOADS[args.workload]
    inputs = W.make_inputs(w)
    rates, rows_total, secs = [], 0, 0.0
    threads = len(os.sched_getaffinity(0))
    for s in range(args.warmup + args.steps):
        rate, rows, dt, threads = oracle_sample_rate(w, inputs, args.ref_step_seconds, seed=s)
        if s >= args.warmup:
            rates.append(rate)
            rows_total += rows
            secs += dt
    value = sum(rates) / len(rates) / 1e12
    ms = attention_flops(w) / (value * 1e12) * 1e3
    sample = (f"{rows_total} random query rows x all {w.Hq} heads of the workload over "
              f"{args.steps} steps of ~{args.ref_step_seconds:.0f} s; rate extrapolated to "
              f"the full workload")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference", "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": threads, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- our arm --
def run_ours(args):
    import torch
    import torch.distributed as dist

    import context_causal_attention_cp_gb300 as cpa
    from context_causal_attention_cp_gb300 import workloads as W

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    w = W.WORKLOADS[args.workload]
    strategy = w.strategies[0]
    inputs = W.make_inputs(w)
    q = inputs["q"].to(dev)
    k = inputs["k"].to(dev)
    v = k[:, :, : w.dv] if w.v_is_k_prefix else inputs["v"].to(dev)
    N, Hq, dv = w.total_new, w.Hq, w.dv
    status = cpa.new_status(dev)
    stream = torch.cuda.current_stream(dev)
    plan = cpa.alloc_plan(w.new_lens, w.prefix_lens, w.cp_size, strategy, device=dev)
    ws = {"q_cat": torch.empty_like(q),
          "o": torch.empty((N, Hq, dv), dtype=torch.bfloat16, device=dev),
          "lse": torch.empty((N, Hq), dtype=torch.float32, device=dev)}
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    token_rows = strategy == "zigzag"   # zigzag shards are runs of consecutive tokens

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        cpa.cp_shard_plan(plan, status=status, stream=stream)
        if not token_rows:
            qc = cpa.cp_restore(q, plan.gather_idx[:N], out=ws["q_cat"], status=status,
                                stream=stream)
        if ev:
            ev[1].record(stream)
        if token_rows:
            # zigzag: each shard's rows are token runs; the kernel reads its
            # queries and writes O and LSE by token index (no gather, no restore)
            cpa.cp_attn_prefill(plan.segs, q, k, v, w.scale, num_segs=plan.total_segs,
                                tiles=plan.tiles, num_tiles=plan.total_tiles, out=ws["o"],
                                lse=ws["lse"], status=status, stream=stream)
        else:
            # attention of every shard; the store puts O and LSE in causal order
            cpa.cp_attn_partial_restore(plan.segs, qc, k, v, w.scale, plan.gather_idx,
                                        num_out_rows=N, num_segs=plan.total_segs,
                                        tiles=plan.tiles, num_tiles=plan.total_tiles,
                                        out=ws["o"], lse=ws["lse"], status=status,
                                        stream=stream)
        if ev:
            ev[2].record(stream)

    launches_per_step = 3 + (0 if token_rows else 1) + 1  # plan, [Q gather], attention
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    cpa.check_status(status, "warmup")

    evs = [[E() for _ in range(3)] for _ in range(args.steps)]
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize(dev)
    with ClockSampler(local) as clk:
        t_wall0 = time.perf_counter()
        for i in range(args.steps):
            flush.zero_()
            step(evs[i])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        dist.barrier()
    cpa.check_status(status, "timed steps")
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    prep_ms = [e[0].elapsed_time(e[1]) for e in evs]
    total_ms = reduce_max_over_ranks(sum(step_ms), world, dev)
    flops = attention_flops(w)
    value = job_throughput(flops, world, args.steps, total_ms)
    pk = peaks()
    attn_avg_ms = sum(attn_ms) / len(attn_ms)
    achieved = flops / (attn_avg_ms * 1e-3) / 1e12

    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_of(w, {"parallelism": f"replicas{world}"}),
            "wall_ms_per_step": t_wall * 1e3 / args.steps,
            "breakdown_ms": {("plan" if token_rows else "plan_and_q_gather"):
                             sum(prep_ms) / len(prep_ms),
                             ("attention_token_rows" if token_rows else
                              "attention_with_restore_store"): attn_avg_ms},
            "roofline": {"kernel": kernel_label(w),
                         "bound": "tensor", "achieved": achieved, "peak": pk["bf16_tflops"],
                         "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                         "traffic": profiled_traffic(PROFILE_MD.get(w.name, "")),
                         "traffic_unit": "bytes per launch (ncu dram read + write)",
                         "algorithmic_bytes": algorithmic_bytes(w),
                         "peak_source": f"{pk['source']} bf16 burst (MEASURED_PEAKS.json)"},
            "restore": bench_restore(args, w, plan, ws, flush, dev, stream, pk, status),
            "clocks": clk.summary(),
            "gpu_launches": launches_per_step * args.steps}
    line["gpu_launches"] += line["restore"].pop("launches")

    if not args.skip_merge:
        line["merge"] = bench_merge(args, dev, stream, pk)
        line["gpu_launches"] += line["merge"].pop("launches")
    if not args.skip_merge:
        line["partial_kv"] = bench_partial_kv(args, dev, stream, pk)
        line["gpu_launches"] += line["partial_kv"].pop("launches")
        line["pass_q"] = bench_pass_q(args, dev, stream, pk)
        line["gpu_launches"] += line["pass_q"].pop("launches")
        line["merge_sweep"] = bench_merge_sweep(args, dev, stream, pk)
        line["gpu_launches"] += line["merge_sweep"].pop("launches")
    if not args.skip_e2e:
        line["e2e"] = bench_e2e(args, w, inputs, dev, stream, world)
    del q, k, v, ws, flush
    torch.cuda.empty_cache()
    if rank == 0 and not args.skip_cpu:
        rate, rows, dt, threads = oracle_sample_rate(w, inputs, args.cpu_seconds)
        line["cpu_baseline"] = {"value": rate / 1e12, "unit": UNIT, "cores": threads,
                                "kind": "oracle",
                                "sample": f"{rows} random query rows x all {w.Hq} heads of the "
                                          f"workload in {dt:.1f} s, fp64 NumPy; rate "
                                          f"extrapolated to the full workload"}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def bench_restore(args, w, plan, ws, flush, dev, stream, pk, status):
    """The standalone restore kernel (cp_restore of O and LSE, the two-pass
    path), on the step's outputs taken in cat order; L2 flushed between reps."""
    import torch

    import context_causal_attention_cp_gb300 as cpa

    N, Hq, dv = w.total_new, w.Hq, w.dv
    o_cat = ws["o"]          # any [N, Hq, dv] rows will do: the kernel is a row gather
    lse_cat = ws["lse"]
    o = torch.empty_like(o_cat)
    lse = torch.empty_like(lse_cat)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def run():
        cpa.cp_restore(o_cat, plan.restore_idx[:N], out=o, status=status, stream=stream)
        cpa.cp_restore(lse_cat, plan.restore_idx[:N], out=lse, status=status, stream=stream)

    for _ in range(3):
        run()
    reps = max(3, args.steps // 2)
    evs = [(E(), E()) for _ in range(reps)]
    for a, b in evs:
        flush.zero_()
        a.record(stream)
        run()
        b.record(stream)
    torch.cuda.synchronize(dev)
    cpa.check_status(status, "restore")
    ms = sum(a.elapsed_time(b) for a, b in evs) / reps
    nbytes = 2 * (N * Hq * dv * 2) + 2 * (N * Hq * 4)
    gbs = nbytes / (ms * 1e-3) / 1e9
    return {"gbs": gbs, "frac_of_hbm": gbs / pk["hbm_gbs"], "bytes_per_call": nbytes,
            "ms": ms, "launches": 2 * (3 + reps),
            "path": "cp_restore of O then LSE (the step itself fuses the restore into the "
                    "attention store)"}


def bench_merge(args, dev, stream, pk):
    """LSE merge of the 128K partial-KV decomposition (136 fp32 partials)."""
    import torch

    import context_causal_attention_cp_gb300 as cpa
    from context_causal_attention_cp_gb300 import workloads as W

    w = W.WORKLOADS[MERGE_WORKLOAD]
    N, Hq, dv, B = w.total_new, w.Hq, w.dv, w.kv_block
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", device=dev)
    segs = cpa.segments_host(plan)
    layout, slot_rows = cpa.api.partial_kv_layout(segs, B)
    g = torch.Generator(device=dev).manual_seed(5)
    parts_o = torch.randn((slot_rows, Hq, dv), device=dev, generator=g)
    parts_l = torch.randn((slot_rows, Hq), device=dev, generator=g) * 3 + 10
    out = torch.empty((N, Hq, dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((N, Hq), dtype=torch.float32, device=dev)
    status = cpa.new_status(dev)

    def merge_all():
        for si, s in enumerate(segs):
            base, nb = layout[si]
            ql = s["q_len"]
            cpa.cp_lse_merge(parts_o[base: base + nb * ql].view(nb, ql, Hq, dv),
                             parts_l[base: base + nb * ql].view(nb, ql, Hq),
                             dst_rows=plan.gather_idx[s["q_row0"]: s["q_row0"] + ql], out=out,
                             lse_out=lse, num_out_rows=N, status=status, stream=stream)

    for _ in range(3):
        merge_all()
    reps = max(3, args.steps // 2)
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        merge_all()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    cpa.check_status(status, "merge")
    read = slot_rows * Hq * (dv + 1) * 4
    written = N * Hq * (dv * 2 + 4)
    ms = sorted(times)[len(times) // 2]
    gbs = (read + written) / (ms * 1e-3) / 1e9
    del parts_o, parts_l
    return {"workload": f"{w.name}: {w.description}", "kernel": "lse_merge_kernel",
            "ms": ms, "gbs": gbs, "frac_of_hbm": gbs / pk["hbm_gbs"],
            "bytes_read": read, "bytes_written": written, "parts": slot_rows // (N // 16),
            "launches": len(segs) * (reps + 3),
            "note": "partials exceed L2 (18 GB), so every read comes from HBM"}


def bench_partial_kv(args, dev, stream, pk):
    """The 128K partial-KV decomposition as one library call per step.

    Step = plan + query gather + cp_attn_partial_kv (layout, split-KV
    attention over the 136 visible (query block, KV block) pairs, fp32
    partials in an 18.4 GB workspace, LSE merge scattered to causal order)."""
    import torch

    import context_causal_attention_cp_gb300 as cpa
    from context_causal_attention_cp_gb300 import workloads as W

    torch.cuda.empty_cache()
    w = W.WORKLOADS[MERGE_WORKLOAD]
    inputs = W.make_inputs(w)
    q = inputs["q"].to(dev)
    k = inputs["k"].to(dev)
    v = inputs["v"].to(dev)
    del inputs
    N, Hq, dv = w.total_new, w.Hq, w.dv
    status = cpa.new_status(dev)
    plan = cpa.alloc_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", device=dev)
    nbytes, _ = cpa.cp_partial_kv_workspace_size(w.new_lens, w.prefix_lens, w.cp_size, "zigzag",
                                                 w.kv_block, Hq, dv)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    q_cat = torch.empty_like(q)
    out = torch.empty((N, Hq, dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((N, Hq), dtype=torch.float32, device=dev)

    def step():
        cpa.cp_shard_plan(plan, status=status, stream=stream)
        cpa.cp_restore(q, plan.gather_idx[:N], out=q_cat, status=status, stream=stream)
        cpa.cp_attn_partial_kv(plan, q_cat, k, v, w.scale, w.kv_block, new_lens=w.new_lens,
                               prefix_lens=w.prefix_lens, workspace=ws, out=out, lse_out=lse,
                               status=status, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    reps = 3
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    cpa.check_status(status, "partial kv")
    ms = sorted(times)[len(times) // 2]
    flops = attention_flops(w)
    tf = flops / (ms * 1e-3) / 1e12
    del ws, q, k, v, q_cat, out, lse
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}: {w.description}", "ms_per_step": ms,
            "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"],
            "workspace_bytes": nbytes, "launches": (3 + 1 + 3) * (reps + 3),
            "path": "cp_shard_plan + cp_restore + cp_attn_partial_kv (one call: layout, "
                    "split-KV attention, merge + restore)"}


def bench_pass_q(args, dev, stream, pk):
    """The same 128K workload through the pass-Q ring (KV resident in 2C
    blocks per rank, each query shard carried round the ring with an fp32
    accumulator; one accumulate launch per (hop, resident block) covers all
    ranks, each segment with its own key window); the pass-KV figure is the
    partial_kv entry.  Step = plan + query gather + the ring + restore of O
    and LSE to causal order."""
    import torch

    import context_causal_attention_cp_gb300 as cpa
    from context_causal_attention_cp_gb300 import workloads as W

    torch.cuda.empty_cache()
    w = W.WORKLOADS[MERGE_WORKLOAD]
    inputs = W.make_inputs(w)
    q = inputs["q"].to(dev)
    k = inputs["k"].to(dev)
    v = inputs["v"].to(dev)
    del inputs
    N, Hq, dv = w.total_new, w.Hq, w.dv
    status = cpa.new_status(dev)
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", device=dev,
                         status=status)
    sched = cpa.pass_q_schedule(plan)
    q_cat = torch.empty_like(q)
    acc = (torch.empty((N, Hq, dv), dtype=torch.float32, device=dev),
           torch.empty((N, Hq), dtype=torch.float32, device=dev),
           torch.empty((N, Hq), dtype=torch.float32, device=dev))
    o = torch.empty((N, Hq, dv), dtype=torch.float32, device=dev)
    lse = torch.empty((N, Hq), dtype=torch.float32, device=dev)

    def step():
        cpa.cp_shard_plan(plan, status=status, stream=stream)
        cpa.cp_restore(q, plan.gather_idx[:N], out=q_cat, status=status, stream=stream)
        o_cat, l_cat = cpa.cp_pass_q_attention(q_cat, k, v, plan, w.scale, schedule=sched,
                                               status=status, stream=stream, out=acc)
        cpa.cp_restore(o_cat, plan.restore_idx[:N], out=o, status=status, stream=stream)
        cpa.cp_restore(l_cat, plan.restore_idx[:N], out=lse, status=status, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    reps = 3
    times = []
    for _ in range(reps):
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        times.append(e0.elapsed_time(e1))
    cpa.check_status(status, "pass q")
    ms = sorted(times)[len(times) // 2]
    tf = attention_flops(w) / (ms * 1e-3) / 1e12
    choice, score = cpa.cp_select_pass(N, 0, Hq, w.Hkv, "message")
    del q, k, v, q_cat, acc, o, lse
    torch.cuda.empty_cache()
    return {"workload": f"{w.name}: {w.description}", "ms_per_step": ms, "tflops": tf,
            "frac_of_bf16_peak": tf / pk["bf16_tflops"], "accumulate_launches": len(sched),
            "launches": (3 + 1 + len(sched) + 2) * (reps + 3),
            "selector_message_rule": choice,
            "path": "cp_shard_plan + cp_restore + cp_pass_q_attention (one "
                    "cp_attn_partial_accumulate per hop and resident KV block, all ranks "
                    "in one launch with per-segment key windows) + cp_restore of O and LSE"}


def decode_ranks(q, k, v, shards):
    """Each rank's resident data for the decode step: its interleaved KV
    tokens (key i on rank i mod shards) contiguous, as its KV cache holds
    them, and a copy of every decode query; plus the segment table (one
    segment per rank, every query at the last position)."""
    import torch

    nq, n_kv = q.shape[0], k.shape[0] // shards
    Hkv, d, dv = k.shape[1], k.shape[2], v.shape[2]
    k_rank = k.view(n_kv, shards, Hkv, d).transpose(0, 1).reshape(shards * n_kv, Hkv, d)
    v_rank = v.view(n_kv, shards, Hkv, dv).transpose(0, 1).reshape(shards * n_kv, Hkv, dv)
    q_rank = q.repeat(shards, 1, 1).contiguous()
    segs_host = torch.tensor([[j * nq, nq, n_kv - 1, 0, j * n_kv, n_kv, j * nq, j]
                              for j in range(shards)], dtype=torch.int32)
    return q_rank, k_rank, v_rank, segs_host


def bench_merge_sweep(args, dev, stream, pk):
    """Decode-style merge sweep: 64 single-token queries x 32 heads over 65536
    keys, key i resident on shard i mod 8.  Each rank's KV cache holds its
    tokens contiguously (laid out once before timing, as a KV cache is) and
    every rank holds all decode queries.  The decode step is one
    cp_attn_split_kv call over the 8 ranks' segments (each rank's keys in
    blocks of DECODE_KV_BLOCK over separate CTAs, merged per rank in the
    library: 8 shard partials) and then one LSE merge of the 8 partials.  The
    same step with one call per rank on strided views of the original-order
    KV is reported beside it.  The merge alone (8 partials, 9.5 MB, L2-sized)
    is reported both warm (launches queued behind a GPU sleep, run back to
    back) and with L2 flushed before each call."""
    import torch

    import context_causal_attention_cp_gb300 as cpa
    from context_causal_attention_cp_gb300 import workloads as W

    m = W.MERGE_SWEEP
    inputs = W.make_merge_sweep_inputs()
    q = inputs["q"].to(dev)
    k = inputs["k"].to(dev)
    v = inputs["v"].to(dev)
    S, nq, Hq, dv = m["shards"], m["queries"], m["Hq"], m["dv"]
    n_kv = m["kv_tokens"] // S
    seg = torch.tensor([[0, nq, n_kv - 1, 0, 0, n_kv, 0, 0]], dtype=torch.int32, device=dev)
    po = torch.empty(S, nq, Hq, dv, device=dev)
    pl = torch.empty(S, nq, Hq, device=dev)
    out = torch.empty(nq, Hq, dv, device=dev)
    lse = torch.empty(nq, Hq, device=dev)
    status = cpa.new_status(dev)
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731

    def merge():
        cpa.cp_lse_merge(po, pl, out=out, lse_out=lse, status=status, stream=stream)

    seg_host = seg.cpu()
    ws = cpa.cp_attn_split_kv(seg, q, k[0::S], v[0::S], m["scale"], 512, segs_host=seg_host,
                              out=po[0], lse_out=pl[0], status=status, stream=stream)[2]

    def decode_step_per_rank():
        for j in range(S):
            cpa.cp_attn_split_kv(seg, q, k[j::S], v[j::S], m["scale"], 512, segs_host=seg_host,
                                 out=po[j], lse_out=pl[j], workspace=ws, status=status,
                                 stream=stream)
        merge()

    q_rank, k_rank, v_rank, segs_all_host = decode_ranks(q, k, v, S)
    segs_all = segs_all_host.to(dev)
    po_rows, pl_rows = po.view(S * nq, Hq, dv), pl.view(S * nq, Hq)
    ws_all = cpa.cp_attn_split_kv(segs_all, q_rank, k_rank, v_rank, m["scale"], DECODE_KV_BLOCK,
                                  segs_host=segs_all_host, out=po_rows, lse_out=pl_rows,
                                  status=status, stream=stream)[2]

    def decode_step():
        cpa.cp_attn_split_kv(segs_all, q_rank, k_rank, v_rank, m["scale"], DECODE_KV_BLOCK,
                             segs_host=segs_all_host, out=po_rows, lse_out=pl_rows,
                             workspace=ws_all, status=status, stream=stream)
        merge()

    def time_steps(fn, reps=50):
        for _ in range(5):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = E(), E()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(300_000_000)  # let the host queue the launches ahead of the GPU
        e0.record(stream)
        for _ in range(reps):
            fn()
        e1.record(stream)
        torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / reps

    per_rank_us = time_steps(decode_step_per_rank)
    step_us = time_steps(decode_step)
    reps = 50
    e0, e1 = E(), E()
    with torch.cuda.stream(stream):
        torch.cuda._sleep(50_000_000)
    e0.record(stream)
    for _ in range(reps):
        merge()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    warm_us = e0.elapsed_time(e1) * 1e3 / reps
    cold = []
    for _ in range(20):
        flush.zero_()
        a, b = E(), E()
        a.record(stream)
        merge()
        b.record(stream)
        cold.append((a, b))
    torch.cuda.synchronize(dev)
    cpa.check_status(status, "merge sweep")
    cold_us = sorted(x.elapsed_time(y) for x, y in cold)[len(cold) // 2] * 1e3
    nbytes = S * nq * Hq * (dv + 1) * 4 + nq * Hq * (dv + 1) * 4
    # both steps: one sizing call + 5 warm-up + 50 timed; then the merge alone
    launches = 3 + (3 * S + 1) * 55 + 3 + 4 * 55 + reps + 20
    del q, k, v, po, pl, flush
    torch.cuda.empty_cache()
    return {"queries": nq, "heads": Hq, "kv_tokens": m["kv_tokens"], "shards": S,
            "decode_step_us": step_us, "decode_kv_block": DECODE_KV_BLOCK,
            "decode_step_per_rank_calls_us": per_rank_us, "merge_bytes": nbytes,
            "merge_warm_us": warm_us, "merge_warm_gbs": nbytes / (warm_us * 1e-6) / 1e9,
            "merge_flushed_us": cold_us, "merge_flushed_gbs": nbytes / (cold_us * 1e-6) / 1e9,
            "merge_flushed_frac_of_hbm": nbytes / (cold_us * 1e-6) / 1e9 / pk["hbm_gbs"],
            "launches": launches,
            "path": "one cp_attn_split_kv over the 8 ranks' segments (each rank's KV cache "
                    "contiguous, keys in blocks of DECODE_KV_BLOCK, merged per rank) + "
                    "cp_lse_merge (8 partials); per_rank_calls: 8 cp_attn_split_kv calls "
                    "(blocks of 512) on strided views of the original-order KV"}


def bench_e2e(args, w, inputs, dev, stream, world=1):
    """Same step through the public API with pinned host inputs and outputs.

    Every step uploads its q, k, v from pinned host memory, runs plan ->
    gather -> attention (restore fused into the store) and downloads O and
    LSE to pinned host memory (api.PrefillPipeline: batch n's attention
    overlaps batch n+1's upload and batch n-1's download).  The timed region
    runs from before the first upload to after the last download.  With N
    ranks the replicas start together after a barrier; the figure is the work
    of all ranks over the slowest rank's time, and the bytes are the whole
    job's."""
    import torch

    import context_causal_attention_cp_gb300 as cpa

    hq = inputs["q"].pin_memory()
    hk = inputs["k"].pin_memory()
    hv = None if w.v_is_k_prefix else inputs["v"].pin_memory()
    N, Hq, dv = w.total_new, w.Hq, w.dv
    ho = torch.empty((N, Hq, dv), dtype=torch.bfloat16).pin_memory()
    hl = torch.empty((N, Hq), dtype=torch.float32).pin_memory()
    pipe = cpa.PrefillPipeline(w.new_lens, w.prefix_lens, w.cp_size, w.strategies[0], Hq, w.Hkv,
                               w.d, dv, w.scale, v_is_k_prefix=w.v_is_k_prefix, device=dev)
    for _ in range(3):
        pipe.submit(hq, hk, hv, ho, hl)
    pipe.synchronize()
    torch.cuda.synchronize(dev)
    reps = max(3, args.steps // 2)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(pipe.s_up)
    for _ in range(reps):
        pipe.submit(hq, hk, hv, ho, hl)
    pipe.s_down.wait_stream(pipe.s_up)
    pipe.s_down.wait_stream(pipe.s_comp)
    e1.record(pipe.s_down)
    pipe.synchronize()
    ms = reduce_max_over_ranks(e0.elapsed_time(e1) / reps, world, dev)
    h2d = world * (hq.numel() * 2 + hk.numel() * 2 + (0 if hv is None else hv.numel() * 2))
    d2h = world * (ho.numel() * 2 + hl.numel() * 4)
    del pipe
    torch.cuda.empty_cache()
    return {"value": world * attention_flops(w) / (ms * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "steps": reps,
            "path": "api.PrefillPipeline: per step, pinned host q/k/v upload, plan, gather, "
                    "attention with the restore in its store, O and LSE download; uploads and "
                    "downloads overlap neighbouring steps' attention"}


def run_profile_case(args):
    """One kernel, small case, for ncu: 3 warm-up launches then one launch.

    attention: the workload's attention launch as in the bench step (zigzag:
               queries and outputs by token index; else restore store).
    merge:     the heaviest query block of the 128K partial-KV workload
               (16 fp32 partials of 8192 rows x 32 heads x 128, 2.2 GB read).
    merge4:    query block 3 of that workload (4 partials, 0.54 GB read; the
               few-partial kernel).
    partial_kv: the whole 128K partial-KV call (layout, split-KV attention,
               fused merge + restore), as in the partial_kv entry.
    restore:   the O restore of the default workload (268 MB each way).
    decode:    the decode step of the merge sweep (one split-KV call over
               the 8 ranks' KV caches, then the merge of the 8 partials)."""
    import torch

    import context_causal_attention_cp_gb300 as cpa
    from context_causal_attention_cp_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    status = cpa.new_status(dev)
    if args.profile_case == "partial_kv":
        w = W.WORKLOADS[MERGE_WORKLOAD]
        inputs = W.make_inputs(w)
        plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", device=dev,
                             status=status)
        q = cpa.cp_restore(inputs["q"].to(dev), plan.gather_idx[: w.total_new], status=status)
        k, v = inputs["k"].to(dev), inputs["v"].to(dev)
        del inputs
        ws = cpa.cp_attn_partial_kv(plan, q, k, v, w.scale, w.kv_block, new_lens=w.new_lens,
                                    prefix_lens=w.prefix_lens, status=status)[2]
        run = lambda: cpa.cp_attn_partial_kv(  # noqa: E731
            plan, q, k, v, w.scale, w.kv_block, new_lens=w.new_lens, prefix_lens=w.prefix_lens,
            workspace=ws, status=status)
    elif args.profile_case == "decode":
        m = W.MERGE_SWEEP
        inputs = W.make_merge_sweep_inputs()
        S, nq, Hq, dv = m["shards"], m["queries"], m["Hq"], m["dv"]
        q_rank, k_rank, v_rank, segs_host = decode_ranks(inputs["q"].to(dev), inputs["k"].to(dev),
                                                         inputs["v"].to(dev), S)
        segs = segs_host.to(dev)
        po = torch.empty(S, nq, Hq, dv, device=dev)
        pl = torch.empty(S, nq, Hq, device=dev)
        ws = cpa.cp_attn_split_kv(segs, q_rank, k_rank, v_rank, m["scale"], DECODE_KV_BLOCK,
                                  segs_host=segs_host, out=po.view(S * nq, Hq, dv),
                                  lse_out=pl.view(S * nq, Hq), status=status)[2]

        def run():
            cpa.cp_attn_split_kv(segs, q_rank, k_rank, v_rank, m["scale"], DECODE_KV_BLOCK,
                                 segs_host=segs_host, out=po.view(S * nq, Hq, dv),
                                 lse_out=pl.view(S * nq, Hq), workspace=ws, status=status)
            cpa.cp_lse_merge(po, pl, status=status)
    elif args.profile_case in ("merge", "merge4"):
        w = W.WORKLOADS[MERGE_WORKLOAD]
        rows, Hq, dv = w.total_new // 16, w.Hq, w.dv
        nb = 16 if args.profile_case == "merge" else 4
        g = torch.Generator(device=dev).manual_seed(5)
        po = torch.randn((nb, rows, Hq, dv), device=dev, generator=g)
        pl = torch.randn((nb, rows, Hq), device=dev, generator=g)
        dst = torch.randperm(rows, device=dev).to(torch.int32)
        out = torch.empty((rows, Hq, dv), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((rows, Hq), device=dev)
        run = lambda: cpa.cp_lse_merge(po, pl, dst_rows=dst, out=out, lse_out=lse,  # noqa: E731
                                       num_out_rows=rows, status=status)
    else:
        w = W.WORKLOADS[args.workload]
        inputs = W.make_inputs(w)
        plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, w.strategies[0], device=dev)
        q = cpa.cp_restore(inputs["q"].to(dev), plan.gather_idx[: w.total_new])
        k = inputs["k"].to(dev)
        v = k[:, :, : w.dv] if w.v_is_k_prefix else inputs["v"].to(dev)
        o, l = cpa.cp_attn_partial(plan.segs, q, k, v, w.scale, num_segs=plan.total_segs,
                                   tiles=plan.tiles, num_tiles=plan.total_tiles)
        if args.profile_case == "attention" and w.strategies[0] == "zigzag":
            q_tok = inputs["q"].to(dev)   # original order, read by token index
            run = lambda: cpa.cp_attn_prefill(  # noqa: E731
                plan.segs, q_tok, k, v, w.scale, num_segs=plan.total_segs, tiles=plan.tiles,
                num_tiles=plan.total_tiles, out=o, lse=l, status=status)
        elif args.profile_case == "attention":
            run = lambda: cpa.cp_attn_partial_restore(  # noqa: E731
                plan.segs, q, k, v, w.scale, plan.gather_idx, num_out_rows=w.total_new,
                num_segs=plan.total_segs, tiles=plan.tiles, num_tiles=plan.total_tiles, out=o,
                lse=l, status=status)
        else:
            out = torch.empty_like(o)
            run = lambda: cpa.cp_restore(o, plan.restore_idx[: w.total_new], out=out,  # noqa: E731
                                         status=status)
    for _ in range(4):
        run()
    torch.cuda.synchronize(dev)
    cpa.check_status(status, args.profile_case)
    print(json.dumps({"profile_case": args.profile_case, "launches": 4}))
    return 0


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=60)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=WORKLOAD)
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    ap.add_argument("--ref-step-seconds", type=float, default=4.0)
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-merge", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--profile-case",
                    choices=["attention", "merge", "merge4", "partial_kv", "restore", "decode"],
                    default=None,
                    help="run one kernel on a small case (for ncu) instead of the bench")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    if args.profile_case:
        return run_profile_case(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
