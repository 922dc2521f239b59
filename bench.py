#!/usr/bin/env python
"""Benchmark: causal prefill context-parallel attention on one GB300.

Headline workload: one 32768-token prompt, Llama-3-8B-shaped attention (32
query / 8 KV heads, head dim 128), CP = 8 zigzag (16 blocks of 2048), bf16
N(0,1) synthetic inputs.  One step is the whole hot path on the device: shard
plan -> causal attention of all 8 shards against the gathered KV in one launch
that reads each shard's query rows and writes O and LSE by token index
(zigzag shards are runs of consecutive tokens, so the query gather and the
restore happen in the kernel's own loads and stores).  ``value`` is causal
attention TFLOP/s over the step (2*Hq*(d+dv) flops per visible (query, key)
pair), L2 flushed between steps.

``per_config`` carries every workload of the benchmark set, each with its own
roofline and the CPU oracle timed beside it on this machine's host cores:
  1   1024-token prompt, d = 64, 8/8 heads, CP=4 zigzag (all rows to the oracle)
  2   6-request varlen batch with cached prefixes, GQA 32/8, CP=4, zigzag and
      interleave (all rows to the oracle)
  3   the headline 32K workload (the top-level figures)
  4   absorbed MLA 16K, 128 heads over one 576-wide latent head, CP=4
      interleave
  5a  the 131072-token partial-KV decomposition (LSE merge GB/s of 136 fp32
      partials; the pass-KV step in one call; the pass-Q ring)
  5b  the decode-style merge sweep (64 queries x 32 heads over 65536 keys on 8
      interleaved shards)
The line also carries the standalone restore kernel's GB/s, clocks sampled
during every timed region, and an end-to-end figure through the C ABI's
host-to-host call.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference]
"""

import argparse
import json
import multiprocessing as mp
import os
import shutil
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "causal CP-prefill attention TFLOPS & % of GB300 bf16 peak; LSE-merge GB/s"
UNIT = "TFLOP/s"
WORKLOAD = "llama8b_32k"
MERGE_WORKLOAD = "partialkv_128k"
DECODE_KV_BLOCK = 4096  # keys per CTA in the decode step (2 blocks per rank)
ORACLE_SAMPLE_ROWS = 512  # rows x all heads when the oracle runs a sample of a workload
# ncu summary under profiles/ holding the attention kernel's DRAM bytes per launch
PROFILE_MD = {"llama8b_32k": "attn_fwd_llama8b_32k.md", "mla_16k": "attn_mla_mla_16k.md",
              "d64_32k": "attn_fwd_d64_32k.md"}
L2_NOTE = "flushed between steps (256 MiB write outside the step's events)"


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
        if w.Hq % 2 == 0:
            return ("attn_mla_pair_kernel (tcgen05 cta_group::2; a pair of SMs per 128 rows x "
                    "2 heads x one 256-column output half)")
        return "attn_mla_kernel (tcgen05; 128 rows x 1 head x one 256-column output half per CTA)"
    nq = 2 if (w.Hq // w.Hkv) % 2 == 0 else 1
    return f"attn_fwd_kernel<d={w.d}> (tcgen05; {nq} head(s) x 128 rows per CTA)"


def config_of(w, world=1, strategy=None):
    """The config dict of a workload; both arms print the same one."""
    return {"workload": f"{w.name}: {w.description}", "new_lens": w.new_lens,
            "prefix_lens": w.prefix_lens, "heads_q": w.Hq, "heads_kv": w.Hkv, "d": w.d,
            "dv": w.dv, "cp_size": w.cp_size, "strategy": strategy or w.strategies[0],
            "l2": L2_NOTE, "parallelism": f"replicas{world}"}


# ----------------------------------------------------------------- clocks --
class ClockSampler:
    """nvidia-smi clocks and throttle reasons sampled every 20 ms for the
    whole run.  Each sample carries nvidia-smi's own timestamp; samples are
    attributed to the timed regions (``region(name)``) whose wall-clock span
    contains them, so buffering of the tool's output cannot misplace them."""

    FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index, period_ms=20):
        self.gpu = gpu_index
        self.period_ms = period_ms
        self.proc = None
        self.lines = []
        self.regions = []

    def _reader(self):
        for line in self.proc.stdout:
            self.lines.append(line)

    def start(self):
        import threading
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", str(self.period_ms)],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True, bufsize=1)
        except Exception:  # noqa: BLE001
            self.proc = None
            return self
        threading.Thread(target=self._reader, daemon=True).start()
        t0 = time.time()
        while not self.lines and time.time() - t0 < 3.0:  # first sample in, tool running
            time.sleep(0.01)
        return self

    def stop(self):
        if self.proc is not None:
            time.sleep(2 * self.period_ms / 1000.0)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:  # noqa: BLE001
                self.proc.kill()

    class _Region:
        def __init__(self, owner, name):
            self.owner, self.name = owner, name

        def __enter__(self):
            self.t0 = time.time()
            return self

        def __exit__(self, *a):
            self.owner.regions.append((self.name, self.t0, time.time()))

    def region(self, name):
        return ClockSampler._Region(self, name)

    @staticmethod
    def parse(lines):
        """[(unix time, sm MHz, max MHz, set of active reasons)]"""
        import datetime
        out = []
        for line in lines:
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(parts[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                sm, mx = float(parts[2]), float(parts[3])
            except ValueError:
                continue
            reasons = {n for n, v in zip(ClockSampler.REASONS, parts[6:10])
                       if v.lower().startswith("active")}
            out.append((ts, sm, mx, reasons))
        return out

    def summary(self, names=None):
        """Median SM clock and active reasons over the samples inside the
        regions (all regions, or those in ``names``)."""
        spans = [(a, b) for n, a, b in self.regions if names is None or n in names]
        samples = [s for s in self.parse(self.lines)
                   if any(a - 0.01 <= s[0] <= b + 0.01 for a, b in spans)]
        if not samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sms = sorted(s[1] for s in samples)
        reasons = set().union(*[s[3] for s in samples])
        return {"sm_mhz": sms[len(sms) // 2], "sm_max_mhz": samples[-1][2],
                "reasons": sorted(reasons), "samples": len(samples),
                "period_ms": self.period_ms,
                "timed_s": round(sum(b - a for a, b in spans), 3)}


# ------------------------------------------------------------- oracle leg --
# The CPU oracle (oracle.attention.attention_rows, unchanged) on selected
# query rows, spread over spawned worker processes; each worker memory-maps
# the float64 K and V that the parent wrote once.  Spawn, not fork: the parent
# holds a CUDA context.
_ORACLE_K = None
_ORACLE_V = None


def _oracle_init(k_path, k_shape, v_path, v_shape, v_cols):
    import numpy as np
    global _ORACLE_K, _ORACLE_V
    _ORACLE_K = np.memmap(k_path, dtype=np.float64, mode="r", shape=k_shape)
    _ORACLE_V = (_ORACLE_K[:, :, :v_cols] if v_path is None else
                 np.memmap(v_path, dtype=np.float64, mode="r", shape=v_shape))


def _oracle_rows(args):
    from oracle import attention as oatt
    q, pos, kv0, scale = args
    oatt.attention_rows(q, _ORACLE_K, _ORACLE_V, pos, kv0, scale)
    return len(pos)


def oracle_workers():
    return max(1, min(16, len(os.sched_getaffinity(0))))


class OracleRows:
    """A pool of oracle workers over one workload's K and V."""

    def __init__(self, w, inputs, procs=None):
        import numpy as np
        self.w = w
        self.procs = procs or oracle_workers()
        k64 = inputs["k"].float().numpy().astype(np.float64)
        base = None
        need = k64.nbytes * (1 if w.v_is_k_prefix else 2)
        try:
            if shutil.disk_usage("/dev/shm").free > 2 * need:
                base = "/dev/shm"
        except OSError:
            pass
        self.tmp = tempfile.mkdtemp(prefix="bench_oracle_", dir=base)
        k_path = os.path.join(self.tmp, "k.f64")
        k64.tofile(k_path)
        v_path, v_shape = None, (w.total_kv, w.Hkv, w.dv)
        if not w.v_is_k_prefix:
            v_path = os.path.join(self.tmp, "v.f64")
            inputs["v"].float().numpy().astype(np.float64).tofile(v_path)
        del k64
        self.q = inputs["q"]
        from oracle import attention as oatt
        self.pos, self.kv0 = oatt.token_tables(w.new_lens, w.prefix_lens)
        self.pool = mp.get_context("spawn").Pool(
            self.procs, initializer=_oracle_init,
            initargs=(k_path, (w.total_kv, w.Hkv, w.d), v_path, v_shape, w.dv))
        self.pool.map(_oracle_rows, [(self._q([0]), self.pos[:1], self.kv0[:1], w.scale)]
                      * self.procs)  # workers up and mapped before any timing

    def _q(self, rows):
        import numpy as np
        import torch
        return self.q[torch.as_tensor(list(rows), dtype=torch.long)].float().numpy() \
            .astype(np.float64)

    def flops(self, rows):
        w = self.w
        return sum(2.0 * w.Hq * (w.d + w.dv) * (int(self.pos[r]) + 1) for r in rows)

    def run(self, rows):
        """Wall seconds the oracle takes on these rows (all heads)."""
        import numpy as np
        rows = np.asarray(rows, dtype=np.int64)
        order = rows[np.argsort(-self.pos[rows], kind="stable")]
        nchunks = max(1, min(len(rows), 4 * self.procs))
        chunks = [order[c::nchunks] for c in range(nchunks)]
        tasks = [(self._q(c), self.pos[c], self.kv0[c], self.w.scale) for c in chunks if len(c)]
        t0 = time.perf_counter()
        done = sum(self.pool.map(_oracle_rows, tasks, chunksize=1))
        dt = time.perf_counter() - t0
        assert done == len(rows)
        return dt

    def close(self):
        self.pool.terminate()
        self.pool.join()
        shutil.rmtree(self.tmp, ignore_errors=True)


def sample_rows(w, count, seed):
    from context_causal_attention_cp_gb300 import workloads as W
    if count >= w.total_new:
        return list(range(w.total_new))
    return W.sample_rows(seed, w.total_new, count)


def oracle_baseline(w, inputs, rows, what):
    """cpu_baseline entry: the oracle on ``rows`` (all heads) in TFLOP/s."""
    pool = OracleRows(w, inputs)
    try:
        dt = pool.run(rows)
        fl = pool.flops(rows)
    finally:
        pool.close()
    full = len(rows) == w.total_new
    return {"value": fl / dt / 1e12, "unit": UNIT, "cores": pool.procs, "kind": "oracle",
            "seconds": round(dt, 3), "rows": len(rows), "extrapolated": not full,
            "sample": (f"all {len(rows)} query rows" if full else
                       f"{len(rows)} seeded random query rows of {w.total_new}") +
                      f" x all {w.Hq} heads of {what}, fp64 NumPy oracle in {pool.procs} "
                      f"processes, {dt:.1f} s" +
                      ("" if full else "; the rate stands for the whole workload")}


def run_reference(args):
    """The oracle as the reference arm, on the host cores (rank 0 only).

    Every step is a bounded sample of the headline workload: ``rows_per_step``
    seeded random query rows x all heads through the fp64 oracle.  The line
    reports what actually ran: its steps, their wall time, and the oracle's
    rate on them (flops of the sampled rows / time); the time the full
    workload would take at that rate is given separately."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if rank != 0:
        return 0
    from context_causal_attention_cp_gb300 import workloads as W

    w = profile_workload(W, args.workload or WORKLOAD)
    inputs = W.make_inputs(w)
    pool = OracleRows(w, inputs)
    times, flops, rows_done = [], 0.0, 0
    try:
        for s in range(args.warmup + args.steps):
            rows = sample_rows(w, args.ref_rows_per_step, seed=100 + s)
            dt = pool.run(rows)
            if s >= args.warmup:
                times.append(dt)
                flops += pool.flops(rows)
                rows_done += len(rows)
    finally:
        pool.close()
    secs = sum(times)
    value = flops / secs / 1e12
    sample = (f"{args.ref_rows_per_step} seeded random query rows x all {w.Hq} heads per step "
              f"({rows_done} rows over {args.steps} timed steps), fp64 NumPy oracle in "
              f"{pool.procs} processes")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": secs * 1e3 / len(times),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
            "data": "synthetic", "impl": "reference", "config": config_of(w, world),
            "step": "one bounded sample of the workload (see sample)",
            "rows_per_step": args.ref_rows_per_step, "rows_timed": rows_done,
            "extrapolated": False,
            "full_workload_seconds_at_this_rate": attention_flops(w) / (value * 1e12),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": pool.procs, "kind": "oracle",
                             "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ----------------------------------------------------------------- our arm --
def _events(n, k):
    import torch
    return [[torch.cuda.Event(enable_timing=True) for _ in range(k)] for _ in range(n)]


def bench_full_kv(w, strategy, inputs, dev, stream, pk, flush, steps, warmup, clk, status,
                  region, world=1):
    """Full-KV CP step of one workload: plan, then (zigzag) the token-row
    attention launch, or (interleave) the query gather into shard order and
    the attention launch with the restore in its store.  L2 flushed before
    every step.  Returns the figures, the step / attention events' times and
    the launch count."""
    import torch

    import context_causal_attention_cp_gb300 as cpa

    q = inputs["q"].to(dev)
    k = inputs["k"].to(dev)
    v = k[:, :, : w.dv] if w.v_is_k_prefix else inputs["v"].to(dev)
    N, Hq, dv = w.total_new, w.Hq, w.dv
    plan = cpa.alloc_plan(w.new_lens, w.prefix_lens, w.cp_size, strategy, device=dev)
    q_cat = torch.empty_like(q)
    o = torch.empty((N, Hq, dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((N, Hq), dtype=torch.float32, device=dev)
    token_rows = strategy == "zigzag"   # zigzag shards are runs of consecutive tokens

    def step(ev=None):
        if ev:
            ev[0].record(stream)
        cpa.cp_shard_plan(plan, status=status, stream=stream)
        if not token_rows:
            cpa.cp_restore(q, plan.gather_idx[:N], out=q_cat, status=status, stream=stream)
        if ev:
            ev[1].record(stream)
        if token_rows:
            cpa.cp_attn_prefill(plan.segs, q, k, v, w.scale, num_segs=plan.total_segs,
                                tiles=plan.tiles, num_tiles=plan.total_tiles, out=o, lse=lse,
                                status=status, stream=stream)
        else:
            cpa.cp_attn_partial_restore(plan.segs, q_cat, k, v, w.scale, plan.gather_idx,
                                        num_out_rows=N, num_segs=plan.total_segs,
                                        tiles=plan.tiles, num_tiles=plan.total_tiles, out=o,
                                        lse=lse, status=status, stream=stream)
        if ev:
            ev[2].record(stream)

    launches_per_step = 3 + (0 if token_rows else 1) + 1  # plan, [Q gather], attention
    for _ in range(warmup):
        step()
    torch.cuda.synchronize(dev)
    cpa.check_status(status, f"{w.name} warmup")
    evs = _events(steps, 3)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    with clk.region(region):
        t_wall0 = time.perf_counter()
        for i in range(steps):
            flush.zero_()
            step(evs[i])
        torch.cuda.synchronize(dev)
        t_wall = time.perf_counter() - t_wall0
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    cpa.check_status(status, f"{w.name} timed steps")
    step_ms = [e[0].elapsed_time(e[2]) for e in evs]
    attn_ms = [e[1].elapsed_time(e[2]) for e in evs]
    prep_ms = [e[0].elapsed_time(e[1]) for e in evs]
    flops = attention_flops(w)
    attn_avg = sum(attn_ms) / len(attn_ms)
    achieved = flops / (attn_avg * 1e-3) / 1e12
    traffic = profiled_traffic(PROFILE_MD.get(w.name, ""))
    out = {"workload": f"{w.name}: {w.description}", "strategy": strategy,
           "config": config_of(w, world, strategy),
           "ms_per_step": sum(step_ms) / len(step_ms), "steps": steps,
           "tflops": flops / (sum(step_ms) / len(step_ms) * 1e-3) / 1e12,
           "attention_flops": flops,
           "breakdown_ms": {("plan" if token_rows else "plan_and_q_gather"):
                            sum(prep_ms) / len(prep_ms),
                            ("attention_token_rows" if token_rows else
                             "attention_with_restore_store"): attn_avg},
           "roofline": {"kernel": kernel_label(w), "bound": "tensor", "achieved": achieved,
                        "peak": pk["bf16_tflops"], "unit": "TFLOP/s",
                        "frac": achieved / pk["bf16_tflops"], "traffic": traffic,
                        "traffic_unit": "bytes per launch (ncu dram read + write)",
                        "algorithmic_bytes": algorithmic_bytes(w),
                        "peak_source": f"{pk['source']} bf16 burst (MEASURED_PEAKS.json)"},
           "wall_ms_per_step": t_wall * 1e3 / steps}
    launches = launches_per_step * (warmup + steps)
    del q, k, v, q_cat, o, lse
    return out, step_ms, launches, plan


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
    stream = torch.cuda.current_stream(dev)
    pk = peaks()
    flush = torch.empty(256 * 1024 * 1024 // 4, dtype=torch.float32, device=dev)
    status = cpa.new_status(dev)
    clk = ClockSampler(local).start()
    launches = 0

    # ---- headline: the 32K workload ----
    w = profile_workload(W, args.workload or WORKLOAD)
    strategy = w.strategies[0]
    inputs = W.make_inputs(w)
    main, step_ms, n, plan = bench_full_kv(w, strategy, inputs, dev, stream, pk, flush,
                                           args.steps, args.warmup, clk, status, "main", world)
    launches += n
    total_ms = reduce_max_over_ranks(sum(step_ms), world, dev)
    value = job_throughput(main["attention_flops"], world, args.steps, total_ms)
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": total_ms / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
            "data": "synthetic", "config": config_of(w, world, strategy),
            "wall_ms_per_step": main["wall_ms_per_step"],
            "breakdown_ms": main["breakdown_ms"], "roofline": main["roofline"]}
    line["restore"] = bench_restore(args, w, plan, dev, stream, pk, status, flush, clk)
    launches += line["restore"].pop("launches")

    per = {"3 llama8b_32k zigzag": {"see": "top-level value, roofline and cpu_baseline",
                                    "tflops": main["tflops"],
                                    "frac_of_bf16_peak": main["roofline"]["frac"]}}
    small = {}
    if not args.skip_configs:
        for name, strat in (("single1k_d64", "zigzag"), ("varlen6_gqa", "zigzag"),
                            ("varlen6_gqa", "interleave"), ("mla_16k", "interleave")):
            wc = W.WORKLOADS[name]
            inp = small.get(name) or W.make_inputs(wc)
            small[name] = inp
            tag = {"single1k_d64": "1", "varlen6_gqa": "2", "mla_16k": "4"}[name]
            # the small workloads are launch-bound: more steps for a stable mean
            steps = args.steps if wc.total_new > 8192 else max(args.steps, 100)
            r, _, n, _ = bench_full_kv(wc, strat, inp, dev, stream, pk, flush, steps,
                                       args.warmup, clk, status, f"cfg{tag}-{strat}", world)
            launches += n
            per[f"{tag} {name} {strat}"] = r
            if name == "mla_16k":
                del inp
                small.pop(name)
            torch.cuda.empty_cache()
    if not args.skip_merge:
        per["5a partialkv_128k"] = bench_128k(args, dev, stream, pk, status, clk)
        launches += per["5a partialkv_128k"].pop("launches")
        per["5b merge_sweep"] = bench_merge_sweep(args, dev, stream, pk, clk)
        launches += per["5b merge_sweep"].pop("launches")
    if not args.skip_e2e:
        line["e2e"] = bench_e2e(args, w, inputs, dev, world, clk)
        launches += line["e2e"].pop("launches")
    clk.stop()
    line["clocks"] = clk.summary()
    line["clocks"]["main_region"] = clk.summary(["main"])
    line["gpu_launches"] = launches
    del flush
    torch.cuda.empty_cache()

    # ---- CPU oracle beside every workload (rank 0, N = 1 only) ----
    if rank == 0 and world == 1 and not args.skip_cpu:
        line["cpu_baseline"] = oracle_baseline(
            w, inputs, sample_rows(w, ORACLE_SAMPLE_ROWS, 7), w.name)
        for key, r in per.items():
            if key.startswith("3 ") or key.startswith("5"):
                continue
            name = key.split()[1]
            wc = W.WORKLOADS[name]
            inp = small.get(name) or W.make_inputs(wc)
            if key.startswith("2 ") and "cpu_baseline" in per.get("2 varlen6_gqa zigzag", {}):
                r["cpu_baseline"] = dict(per["2 varlen6_gqa zigzag"]["cpu_baseline"],
                                         note="the same oracle run as the zigzag entry: the "
                                              "oracle computes the unsharded result")
                continue
            r["cpu_baseline"] = oracle_baseline(
                wc, inp, sample_rows(wc, ORACLE_SAMPLE_ROWS if wc.total_new > 8192 else
                                     wc.total_new, 7), name)
        if "5a partialkv_128k" in per:
            wc = W.WORKLOADS[MERGE_WORKLOAD]
            per["5a partialkv_128k"]["cpu_baseline"] = oracle_baseline(
                wc, W.make_inputs(wc), sample_rows(wc, ORACLE_SAMPLE_ROWS, 7), MERGE_WORKLOAD)
        if "5b merge_sweep" in per:
            per["5b merge_sweep"]["cpu_baseline"] = oracle_decode_baseline()
    line["per_config"] = per
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.destroy_process_group()
    return 0


def bench_restore(args, w, plan, dev, stream, pk, status, flush, clk):
    """The standalone restore kernel (cp_restore of O and LSE, the two-pass
    path) on rows in cat order; L2 flushed between reps."""
    import torch

    import context_causal_attention_cp_gb300 as cpa

    N, Hq, dv = w.total_new, w.Hq, w.dv
    o_cat = torch.randn((N, Hq, dv), device=dev).to(torch.bfloat16)
    lse_cat = torch.randn((N, Hq), device=dev)
    o = torch.empty_like(o_cat)
    lse = torch.empty_like(lse_cat)
    cpa.cp_shard_plan(plan, status=status, stream=stream)

    def run():
        cpa.cp_restore(o_cat, plan.restore_idx[:N], out=o, status=status, stream=stream)
        cpa.cp_restore(lse_cat, plan.restore_idx[:N], out=lse, status=status, stream=stream)

    for _ in range(3):
        run()
    reps = max(3, args.steps // 2)
    evs = _events(reps, 2)
    with clk.region("restore"):
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
            "ms": ms, "launches": 3 + 2 * (3 + reps),
            "roofline": {"kernel": "row_gather_kernel", "bound": "hbm", "achieved": gbs,
                         "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                         "traffic": None},
            "path": "cp_restore of O then LSE (the step itself fuses the restore into the "
                    "attention store)"}


def partial_slots(plan, kv_block):
    """Partial rows of a partial-KV decomposition laid out per segment of the
    plan (block j of segment s at rows base_s + j * q_len_s; a segment whose
    last row is at position P sees P // kv_block + 1 blocks).
    Returns ([(q_row0, q_len, base, blocks)], total rows)."""
    import context_causal_attention_cp_gb300 as cpa
    out, base = [], 0
    for s in cpa.segments_host(plan):
        nb = (s["q_pos0"] + (s["q_len"] - 1) * s["q_pos_step"]) // kv_block + 1
        out.append((s["q_row0"], s["q_len"], base, nb))
        base += nb * s["q_len"]
    return out, base


def bench_128k(args, dev, stream, pk, status, clk):
    """The 131072-token partial-KV workload: the LSE merge of its 136 fp32
    partials (16 cp_lse_merge calls on synthetic partials, 18.4 GB read), the
    pass-KV step in one library call, and the same workload through the
    pass-Q ring."""
    import torch

    import context_causal_attention_cp_gb300 as cpa
    from context_causal_attention_cp_gb300 import workloads as W

    w = W.WORKLOADS[MERGE_WORKLOAD]
    N, Hq, dv = w.total_new, w.Hq, w.dv
    E = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    out = {"workload": f"{w.name}: {w.description}", "config": config_of(w)}
    launches = 0

    # -- merge of the partials (synthetic values; the kernel reads them all) --
    torch.cuda.empty_cache()
    plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", device=dev,
                         status=status)
    slots, slot_rows = partial_slots(plan, w.kv_block)
    g = torch.Generator(device=dev).manual_seed(5)
    parts_o = torch.randn((slot_rows, Hq, dv), device=dev, generator=g)
    parts_l = torch.randn((slot_rows, Hq), device=dev, generator=g) * 3 + 10
    o = torch.empty((N, Hq, dv), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((N, Hq), dtype=torch.float32, device=dev)

    def merge_all():
        for q_row0, ql, base, nb in slots:
            cpa.cp_lse_merge(parts_o[base: base + nb * ql].view(nb, ql, Hq, dv),
                             parts_l[base: base + nb * ql].view(nb, ql, Hq),
                             dst_rows=plan.gather_idx[q_row0: q_row0 + ql], out=o, lse_out=lse,
                             num_out_rows=N, status=status, stream=stream)

    for _ in range(3):
        merge_all()
    reps = max(3, args.steps // 4)
    times = []
    with clk.region("merge"):
        for _ in range(reps):
            e0, e1 = E(), E()
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
    launches += len(slots) * (reps + 3) + 3
    out["merge"] = {"kernel": "lse_merge_kernel", "ms": ms, "gbs": gbs,
                    "frac_of_hbm": gbs / pk["hbm_gbs"], "bytes_read": read,
                    "bytes_written": written, "parts": slot_rows // (N // 16),
                    "roofline": {"kernel": "lse_merge_kernel / lse_merge_batched_kernel",
                                 "bound": "hbm", "achieved": gbs, "peak": pk["hbm_gbs"],
                                 "unit": "GB/s", "frac": gbs / pk["hbm_gbs"],
                                 "traffic": profiled_traffic("lse_merge_partialkv_128k.md"),
                                 "traffic_unit": "bytes per average launch (ncu dram read + "
                                                 "write, scaled by partials read)",
                                 "algorithmic_bytes": (read + written) // len(slots)},
                    "note": "partials exceed L2 (18 GB), so every read comes from HBM"}
    del parts_o, parts_l
    torch.cuda.empty_cache()

    # -- the pass-KV step in one call, then the pass-Q ring --
    inputs = W.make_inputs(w)
    q = inputs["q"].to(dev)
    k = inputs["k"].to(dev)
    v = inputs["v"].to(dev)
    del inputs
    nbytes = cpa.cp_partial_kv_workspace_size(w.new_lens, w.prefix_lens, w.cp_size, "zigzag",
                                              w.kv_block, Hq, dv)[0]
    ws = torch.empty(nbytes, dtype=torch.uint8, device=dev)
    q_cat = torch.empty_like(q)

    def step_kv():
        cpa.cp_shard_plan(plan, status=status, stream=stream)
        cpa.cp_restore(q, plan.gather_idx[:N], out=q_cat, status=status, stream=stream)
        cpa.cp_attn_partial_kv(plan, q_cat, k, v, w.scale, w.kv_block, workspace=ws, out=o,
                               lse_out=lse, status=status, stream=stream)

    def timed(fn, region, reps=3):
        for _ in range(3):
            fn()
        torch.cuda.synchronize(dev)
        ts = []
        with clk.region(region):
            for _ in range(reps):
                e0, e1 = E(), E()
                e0.record(stream)
                fn()
                e1.record(stream)
                torch.cuda.synchronize(dev)
                ts.append(e0.elapsed_time(e1))
        return sorted(ts)[len(ts) // 2], reps + 3

    ms, n = timed(step_kv, "partial_kv")
    cpa.check_status(status, "partial kv")
    launches += (3 + 1 + 3) * n
    flops = attention_flops(w)
    tf = flops / (ms * 1e-3) / 1e12
    out["partial_kv"] = {"ms_per_step": ms, "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"],
                         "workspace_bytes": nbytes,
                         "path": "cp_shard_plan + cp_restore + cp_attn_partial_kv (one call: "
                                 "layout, split-KV attention, merge + restore)"}
    del ws
    torch.cuda.empty_cache()

    sched = cpa.pass_q_schedule(plan)
    acc = (torch.empty((N, Hq, dv), dtype=torch.float32, device=dev),
           torch.empty((N, Hq), dtype=torch.float32, device=dev),
           torch.empty((N, Hq), dtype=torch.float32, device=dev))
    o32 = torch.empty((N, Hq, dv), dtype=torch.float32, device=dev)

    def step_q():
        cpa.cp_shard_plan(plan, status=status, stream=stream)
        cpa.cp_restore(q, plan.gather_idx[:N], out=q_cat, status=status, stream=stream)
        o_cat, l_cat = cpa.cp_pass_q_attention(q_cat, k, v, plan, w.scale, schedule=sched,
                                               status=status, stream=stream, out=acc)
        cpa.cp_restore(o_cat, plan.restore_idx[:N], out=o32, status=status, stream=stream)
        cpa.cp_restore(l_cat, plan.restore_idx[:N], out=lse, status=status, stream=stream)

    ms, n = timed(step_q, "pass_q")
    cpa.check_status(status, "pass q")
    launches += (3 + 1 + 1 + sched.num_launches + 2) * n
    tf = flops / (ms * 1e-3) / 1e12
    choice, _ = cpa.cp_select_pass(N, 0, Hq, w.Hkv, "message")
    out["pass_q"] = {"ms_per_step": ms, "tflops": tf, "frac_of_bf16_peak": tf / pk["bf16_tflops"],
                     "accumulate_launches": sched.num_launches,
                     "selector_message_rule": choice,
                     "path": "cp_shard_plan + cp_restore + cp_attn_pass_q (the library's ring "
                             "schedule: one accumulate launch per hop and resident KV block, all "
                             "ranks in one launch with per-segment key windows) + cp_restore of "
                             "O and LSE"}
    # the cost-driven selector fed with this run's measured attention and
    # merge rates, at two per-GPU ring bandwidths (an InfiniBand NDR port and
    # an NVLink 5 direction), over miss rates of a 131072-token context
    sel = {"attn_tflops_measured": out["partial_kv"]["tflops"],
           "merge_gbs_measured": out["merge"]["gbs"]}
    for link in (50.0, 900.0):
        row = {}
        for miss in (0.01, 0.05, 0.125, 0.5, 1.0):
            T = max(1, int(N * miss))
            choice, ekv, eq = cpa.cp_select_pass_cost(T, N - T, Hq, w.Hkv, w.d, w.cp_size,
                                                      out["partial_kv"]["tflops"], link,
                                                      out["merge"]["gbs"])
            row[f"miss_{miss}"] = {"choice": choice, "exposed_kv_ms": ekv * 1e3,
                                   "exposed_q_ms": eq * 1e3}
        sel[f"link_{int(link)}_gbs"] = row
    out["selector_cost_rule"] = sel
    out["launches"] = launches
    del q, k, v, q_cat, acc, o32, o, lse
    torch.cuda.empty_cache()
    return out


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


def bench_merge_sweep(args, dev, stream, pk, clk):
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

    def time_steps(fn, region, reps=50):
        for _ in range(5):
            fn()
        torch.cuda.synchronize(dev)
        e0, e1 = E(), E()
        with torch.cuda.stream(stream):
            torch.cuda._sleep(300_000_000)  # let the host queue the launches ahead of the GPU
        with clk.region(region):
            e0.record(stream)
            for _ in range(reps):
                fn()
            e1.record(stream)
            torch.cuda.synchronize(dev)
        return e0.elapsed_time(e1) * 1e3 / reps

    # the decode step as one call and one merge: the 8 ranks' caches form one
    # segment whose KV blocks never straddle two ranks, so the library's merge
    # of all block partials is the merge of the rank partials
    seg_one_host = torch.tensor([[0, nq, S * n_kv - 1, 0, 0, S * n_kv, 0, 0]], dtype=torch.int32)
    seg_one = seg_one_host.to(dev)
    one_merge_us, ws_one = {}, {}
    for kvb in (2048, 4096, 8192):
        ws_one[kvb] = cpa.cp_attn_split_kv(seg_one, q, k_rank, v_rank, m["scale"], kvb,
                                           segs_host=seg_one_host, out=out, lse_out=lse,
                                           status=status, stream=stream)[2]

        def one_merge(kvb=kvb):
            cpa.cp_attn_split_kv(seg_one, q, k_rank, v_rank, m["scale"], kvb,
                                 segs_host=seg_one_host, out=out, lse_out=lse,
                                 workspace=ws_one[kvb], status=status, stream=stream)
        one_merge_us[kvb] = time_steps(one_merge, f"decode_one_merge_{kvb}")
    best_kvb = min(one_merge_us, key=one_merge_us.get)
    per_rank_us = time_steps(decode_step_per_rank, "decode_per_rank")
    step_us = time_steps(decode_step, "decode")
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
    kv_bytes = 2 * m["kv_tokens"] * m["Hkv"] * m["d"] * 2
    # both steps: one sizing call + 5 warm-up + 50 timed; then the merge alone
    launches = 3 + (3 * S + 1) * 55 + 3 + 4 * 55 + reps + 20
    del q, k, v, po, pl, flush
    torch.cuda.empty_cache()
    best_us = one_merge_us[best_kvb]
    launches += 3 * 3 * 56
    return {"queries": nq, "heads": Hq, "kv_tokens": m["kv_tokens"], "shards": S,
            "decode_step_us": best_us, "decode_kv_block": best_kvb,
            "decode_step_one_merge_us_by_kv_block": one_merge_us,
            "decode_step_rank_partials_us": step_us, "rank_partials_kv_block": DECODE_KV_BLOCK,
            "decode_step_per_rank_calls_us": per_rank_us,
            "decode_kv_gbs": kv_bytes / (best_us * 1e-6) / 1e9,
            "merge_bytes": nbytes,
            "merge_warm_us": warm_us, "merge_warm_gbs": nbytes / (warm_us * 1e-6) / 1e9,
            "merge_flushed_us": cold_us, "merge_flushed_gbs": nbytes / (cold_us * 1e-6) / 1e9,
            "merge_flushed_frac_of_hbm": nbytes / (cold_us * 1e-6) / 1e9 / pk["hbm_gbs"],
            "roofline": {"kernel": "decode step (split-KV attention + merge)", "bound": "hbm",
                         "achieved": kv_bytes / (best_us * 1e-6) / 1e9, "peak": pk["hbm_gbs"],
                         "unit": "GB/s", "frac": kv_bytes / (best_us * 1e-6) / 1e9 / pk["hbm_gbs"],
                         "traffic": profiled_traffic("decode_step_one_merge_merge_sweep.md"),
                         "traffic_unit": "bytes per call (ncu dram read + write of its three "
                                         "launches, cold cache)",
                         "algorithmic_bytes": kv_bytes,
                         "note": "K and V of all 65536 keys (268 MB) over the whole step"},
            "launches": launches,
            "path": "decode step: one cp_attn_split_kv over the 8 ranks' KV caches as one "
                    "segment (each rank's cache contiguous, KV blocks of decode_kv_block that "
                    "never straddle two ranks, all block partials LSE-merged in the call); "
                    "rank_partials: one cp_attn_split_kv over the 8 ranks' segments (8 rank "
                    "partials) + cp_lse_merge of the 8; per_rank_calls: 8 cp_attn_split_kv "
                    "calls (blocks of 512) on strided views of the original-order KV, + the merge"}


def oracle_decode_baseline():
    """The oracle's decode step of the merge sweep, in full, in one process:
    every shard's partial (O_j, L_j) of the 64 queries against its keys
    (oracle.attention.decode_attention), then the LSE merge of the 8 partials
    (oracle.merge.lse_merge)."""
    import numpy as np

    from context_causal_attention_cp_gb300 import workloads as W
    from oracle import attention as oatt
    from oracle import merge as omerge

    m = W.MERGE_SWEEP
    inp = W.make_merge_sweep_inputs()
    f64 = lambda t: t.float().numpy().astype(np.float64)  # noqa: E731
    q, k, v = f64(inp["q"]), f64(inp["k"]), f64(inp["v"])
    S = m["shards"]
    t0 = time.perf_counter()
    parts = [oatt.decode_attention(q, k, v, m["scale"], np.arange(j, m["kv_tokens"], S))
             for j in range(S)]
    t1 = time.perf_counter()
    omerge.lse_merge(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    t2 = time.perf_counter()
    nbytes = S * m["queries"] * m["Hq"] * (m["dv"] + 1) * 4 + m["queries"] * m["Hq"] * \
        (m["dv"] + 1) * 4
    return {"decode_step_us": (t2 - t0) * 1e6, "merge_us": (t2 - t1) * 1e6,
            "merge_gbs": nbytes / (t2 - t1) / 1e9, "unit": "us", "cores": 1, "kind": "oracle",
            "extrapolated": False,
            "sample": "the whole decode step in fp64 NumPy in one process: 8 shard partials of "
                      "64 queries x 32 heads over 8192 keys each, then their LSE merge"}


def bench_e2e(args, w, inputs, dev, world, clk):
    """The same workload end to end through the C ABI's host-to-host call
    (cp_prefill_host): every step uploads its q, k, v from pinned host memory,
    builds the plan, runs the attention of all shards (O / LSE in causal token
    order) and downloads O and LSE to pinned host memory; the library overlaps
    step i's attention with step i+1's upload and step i-1's download on three
    streams.  The timed region runs from before the first upload to after the
    last download.  With N ranks the replicas start together after a barrier;
    the figure is the work of all ranks over the slowest rank's time, and the
    bytes are the whole job's."""
    import torch

    import context_causal_attention_cp_gb300 as cpa

    hq = inputs["q"].pin_memory()
    hk = inputs["k"].pin_memory()
    hv = None if w.v_is_k_prefix else inputs["v"].pin_memory()
    N, Hq, dv = w.total_new, w.Hq, w.dv
    outs = [(torch.empty((N, Hq, dv), dtype=torch.bfloat16).pin_memory(),
             torch.empty((N, Hq), dtype=torch.float32).pin_memory()) for _ in range(2)]
    reps = max(3, args.steps // 2)
    batches = [(hq, hk, hv) + outs[i % 2] for i in range(reps)]
    status = cpa.new_status(dev)
    strategy = w.strategies[0]
    # warm-up call (workspace and streams reused by the timed call)
    ws, streams = cpa.cp_prefill_host(w.new_lens, w.prefix_lens, w.cp_size, strategy, Hq, w.Hkv,
                                      w.d, dv, w.scale, batches[:3],
                                      v_is_k_prefix=w.v_is_k_prefix, status=status, device=dev)
    torch.cuda.synchronize(dev)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with clk.region("e2e"):
        e0.record(streams[1])
        cpa.cp_prefill_host(w.new_lens, w.prefix_lens, w.cp_size, strategy, Hq, w.Hkv, w.d, dv,
                            w.scale, batches, v_is_k_prefix=w.v_is_k_prefix, workspace=ws,
                            status=status, streams=streams, device=dev)
        e1.record(streams[2])
        streams[2].synchronize()
    torch.cuda.synchronize(dev)
    cpa.check_status(status, "e2e")
    ms = reduce_max_over_ranks(e0.elapsed_time(e1) / reps, world, dev)
    h2d = world * (hq.numel() * 2 + hk.numel() * 2 + (0 if hv is None else hv.numel() * 2))
    d2h = world * (N * Hq * dv * 2 + N * Hq * 4)
    per_step = 4 if strategy == "zigzag" else 5
    del ws
    torch.cuda.empty_cache()
    return {"value": world * attention_flops(w) / (ms * 1e-3) / 1e12, "unit": UNIT,
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": ms,
            "steps": reps, "launches": per_step * (3 + reps),
            "path": "C ABI cp_prefill_host: per step, pinned host q/k/v upload, plan, "
                    "attention with O / LSE stored in token order, O and LSE download; "
                    "uploads and downloads overlap neighbouring steps' attention"}


def profile_workload(W, name):
    """A bench workload, or d64_32k: the 32K workload at d = dv = 64 (scale 1/8),
    where a tile carries half the MMA work of d = 128 for the same number of
    exponentials, so the exp unit rather than the tensor pipe may bind."""
    if name == "d64_32k":
        import dataclasses
        return dataclasses.replace(
            W.WORKLOADS["llama8b_32k"], name="d64_32k", d=64, dv=64, scale=0.125,
            description="1 request, 32768 tokens, GQA 32/8, d=64, CP=8 zigzag (16 x 2048)")
    return W.WORKLOADS[name]


def run_profile_case(args):
    """One kernel, small case, for ncu: 3 warm-up launches then one launch.

    attention: the workload's attention launch as in the bench step (zigzag:
               queries and outputs by token index; else restore store);
               --workload d64_32k runs the 32K workload at d = 64.
    merge:     the heaviest query block of the 128K partial-KV workload
               (16 fp32 partials of 8192 rows x 32 heads x 128, 2.2 GB read).
    merge4:    query block 3 of that workload (4 partials, 0.54 GB read; the
               few-partial kernel).
    partial_kv: the partial-KV call (layout, split-KV attention, fused merge
               + restore) on the workload given by --workload (default: the
               128K workload; its counter captures use llama8b_32k, a quarter
               of the 128K work per launch).
    restore:   the O restore of the default workload (268 MB each way).
    decode:    the rank-partials decode step of the merge sweep (one split-KV
               call over the 8 ranks' KV caches, then the merge of the 8
               partials).
    decode1:   the decode step as one split-KV call over the ranks' caches as
               one segment (block partials merged in the call)."""
    import torch

    import context_causal_attention_cp_gb300 as cpa
    from context_causal_attention_cp_gb300 import workloads as W

    dev = torch.device("cuda", 0)
    status = cpa.new_status(dev)
    if args.profile_case == "partial_kv":
        w = W.WORKLOADS[args.workload or MERGE_WORKLOAD]
        kv_block = w.kv_block or 8192
        inputs = W.make_inputs(w)
        plan = cpa.make_plan(w.new_lens, w.prefix_lens, w.cp_size, "zigzag", device=dev,
                             status=status)
        q = cpa.cp_restore(inputs["q"].to(dev), plan.gather_idx[: w.total_new], status=status)
        k, v = inputs["k"].to(dev), inputs["v"].to(dev)
        del inputs
        ws = cpa.cp_attn_partial_kv(plan, q, k, v, w.scale, kv_block, status=status)[2]
        run = lambda: cpa.cp_attn_partial_kv(  # noqa: E731
            plan, q, k, v, w.scale, kv_block, workspace=ws, status=status)
    elif args.profile_case == "decode1":
        m = W.MERGE_SWEEP
        inputs = W.make_merge_sweep_inputs()
        S, nq, Hq, dv = m["shards"], m["queries"], m["Hq"], m["dv"]
        q = inputs["q"].to(dev)
        _, k_rank, v_rank, _ = decode_ranks(q, inputs["k"].to(dev), inputs["v"].to(dev), S)
        n_kv = m["kv_tokens"] // S
        seg_host = torch.tensor([[0, nq, S * n_kv - 1, 0, 0, S * n_kv, 0, 0]], dtype=torch.int32)
        seg = seg_host.to(dev)
        out = torch.empty(nq, Hq, dv, device=dev)
        lse = torch.empty(nq, Hq, device=dev)
        ws = cpa.cp_attn_split_kv(seg, q, k_rank, v_rank, m["scale"], DECODE_KV_BLOCK,
                                  segs_host=seg_host, out=out, lse_out=lse, status=status)[2]
        run = lambda: cpa.cp_attn_split_kv(  # noqa: E731
            seg, q, k_rank, v_rank, m["scale"], DECODE_KV_BLOCK, segs_host=seg_host, out=out,
            lse_out=lse, workspace=ws, status=status)
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
        w = profile_workload(W, args.workload or WORKLOAD)
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
    ap.add_argument("--workload", default=None,
                    help=f"workload of the headline line and of --profile-case attention "
                         f"(default {WORKLOAD}; --profile-case partial_kv: {MERGE_WORKLOAD}; "
                         f"also d64_32k, the 32K workload at d = 64)")
    ap.add_argument("--ref-rows-per-step", type=int, default=128,
                    help="query rows (x all heads) the reference arm's oracle runs per step")
    ap.add_argument("--skip-cpu", action="store_true")
    ap.add_argument("--skip-merge", action="store_true")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-configs", action="store_true")
    ap.add_argument("--profile-case",
                    choices=["attention", "merge", "merge4", "partial_kv", "restore", "decode",
                             "decode1"],
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
