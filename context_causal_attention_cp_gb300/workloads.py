"""Seeded synthetic workloads shared by the tests, the bench and the smoke test.

This module only describes shapes and draws random inputs: it holds none of
the method's arithmetic (no plan, attention, merge or restore logic), so both
the CUDA path and the CPU oracle can be fed from it without sharing code.

Inputs are drawn on the CPU with ``torch.Generator().manual_seed(seed)``
as float32 normals scaled by ``std`` and rounded once to bfloat16
(round-to-nearest-even); the oracle consumes exactly those bfloat16 values
widened to float64.

Each workload mirrors one of the synthetic prefill shapes of this library's
benchmark set: a single 1K prompt, a varlen batch with cached prefixes and
GQA, a 32K Llama-3-8B-shaped prompt, an absorbed-MLA 16K prompt and a 128K
partial-KV (ring-style) decomposition plus a decode-style merge sweep.
"""

import math
from dataclasses import dataclass
from typing import List, Optional

import torch


@dataclass(frozen=True)
class Workload:
    name: str
    new_lens: List[int]
    prefix_lens: List[int]
    Hq: int
    Hkv: int
    d: int
    dv: int
    scale: float
    std: float
    cp_size: int
    strategies: List[str]
    seed: int
    v_is_k_prefix: bool = False      # MLA: V is the first dv columns of K
    kv_block: Optional[int] = None   # partial-KV mode: KV window per partial
    description: str = ""

    @property
    def total_new(self):
        return sum(self.new_lens)

    @property
    def total_kv(self):
        return sum(n + p for n, p in zip(self.new_lens, self.prefix_lens))


WORKLOADS = {
    "single1k_d64": Workload(
        name="single1k_d64", new_lens=[1024], prefix_lens=[0], Hq=8, Hkv=8, d=64, dv=64,
        scale=1.0 / 8.0, std=1.0, cp_size=4, strategies=["zigzag"], seed=1001,
        description="1 request, 1024 new tokens, 8/8 heads, d=64, CP=4 zigzag"),
    "varlen6_gqa": Workload(
        name="varlen6_gqa", new_lens=[517, 1000, 33, 2048, 3, 1500],
        prefix_lens=[0, 256, 0, 1024, 17, 0], Hq=32, Hkv=8, d=128, dv=128,
        scale=1.0 / math.sqrt(128.0), std=1.0, cp_size=4,
        strategies=["zigzag", "interleave"], seed=1002,
        description="6 requests with cached prefixes, GQA 32/8, d=128, CP=4"),
    "llama8b_32k": Workload(
        name="llama8b_32k", new_lens=[32768], prefix_lens=[0], Hq=32, Hkv=8, d=128, dv=128,
        scale=1.0 / math.sqrt(128.0), std=1.0, cp_size=8, strategies=["zigzag"], seed=1003,
        description="1 request, 32768 tokens, GQA 32/8, d=128, CP=8 zigzag (16 x 2048)"),
    "mla_16k": Workload(
        name="mla_16k", new_lens=[16384], prefix_lens=[0], Hq=128, Hkv=1, d=576, dv=512,
        scale=1.0 / math.sqrt(192.0), std=0.1, cp_size=4, strategies=["interleave"],
        seed=1004, v_is_k_prefix=True,
        description="absorbed MLA, 16384 tokens, 128 heads over 1 latent head, "
                    "qk 576 / v 512, CP=4 interleave"),
    "partialkv_128k": Workload(
        name="partialkv_128k", new_lens=[131072], prefix_lens=[0], Hq=32, Hkv=8, d=128,
        dv=128, scale=1.0 / math.sqrt(128.0), std=1.0, cp_size=8, strategies=["zigzag"],
        seed=1005, kv_block=8192,
        description="1 request, 131072 tokens, GQA 32/8, d=128, CP=8 zigzag, "
                    "16 KV blocks of 8192, per-block fp32 partials merged by LSE"),
}

# Decode-style merge sweep: 64 single-token queries x 32 heads against 65536
# KV tokens spread over 8 shards, token i on shard i mod 8.
MERGE_SWEEP = dict(name="merge_sweep", queries=64, kv_tokens=65536, shards=8, Hq=32,
                   Hkv=8, d=128, dv=128, scale=1.0 / math.sqrt(128.0), std=1.0, seed=1006)


def _normal_bf16(gen, shape, std):
    x = torch.randn(*shape, generator=gen, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def make_inputs(w: Workload, seed_offset: int = 0):
    """Seeded bf16 inputs on the CPU.

    Returns dict(q=[total_new, Hq, d], k=[total_kv, Hkv, d], v=[total_kv, Hkv, dv]).
    For MLA workloads ``v`` is a view of the first dv columns of ``k``.
    """
    gen = torch.Generator().manual_seed(w.seed + seed_offset)
    q = _normal_bf16(gen, (w.total_new, w.Hq, w.d), w.std)
    k = _normal_bf16(gen, (w.total_kv, w.Hkv, w.d), w.std)
    if w.v_is_k_prefix:
        v = k[:, :, : w.dv]
    else:
        v = _normal_bf16(gen, (w.total_kv, w.Hkv, w.dv), w.std)
    return dict(q=q, k=k, v=v)


def make_merge_sweep_inputs(seed_offset: int = 0):
    m = MERGE_SWEEP
    gen = torch.Generator().manual_seed(m["seed"] + seed_offset)
    q = _normal_bf16(gen, (m["queries"], m["Hq"], m["d"]), m["std"])
    k = _normal_bf16(gen, (m["kv_tokens"], m["Hkv"], m["d"]), m["std"])
    v = _normal_bf16(gen, (m["kv_tokens"], m["Hkv"], m["dv"]), m["std"])
    return dict(q=q, k=k, v=v)


def random_batch(seed: int, max_reqs: int = 6, max_new: int = 300, max_prefix: int = 64):
    """Random (new_lens, prefix_lens) for plan fuzzing, including empty requests."""
    gen = torch.Generator().manual_seed(seed)
    B = int(torch.randint(1, max_reqs + 1, (1,), generator=gen))
    new = torch.randint(0, max_new + 1, (B,), generator=gen).tolist()
    pre = torch.randint(0, max_prefix + 1, (B,), generator=gen).tolist()
    return new, pre


def sample_rows(seed: int, total: int, count: int, must: Optional[List[int]] = None):
    """Seeded sample of row indices (sorted, unique), always containing ``must``."""
    gen = torch.Generator().manual_seed(seed)
    picked = set(int(x) for x in (must or []) if 0 <= int(x) < total)
    if count > len(picked):
        extra = torch.randint(0, total, (count * 2,), generator=gen).tolist()
        for x in extra:
            if len(picked) >= count:
                break
            picked.add(int(x))
    return sorted(picked)
