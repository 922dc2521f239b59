"""GB300-native prefill context-parallel causal attention (zigzag / interleave + LSE merge).

The compute path is the C-ABI library ``libcpattn.so`` (CUDA, sm_103a); this
package holds its thin Python binding (``api``), the in-tree build script and
the seeded synthetic workloads.  The library is loaded on first use and its
absence raises: there is no CPU fallback.
"""

from .api import (  # noqa: F401
    PassQSchedule,
    ShardPlan,
    alloc_plan,
    check_status,
    cp_attn_partial,
    cp_attn_partial_accumulate,
    cp_attn_partial_kv,
    cp_attn_partial_restore,
    cp_attn_prefill,
    cp_attn_split_kv,
    cp_lse_merge,
    cp_partial_kv_workspace_size,
    cp_partial_kv_workspace_size_segs,
    cp_pass_q_attention,
    cp_prefill_attention,
    cp_prefill_host,
    cp_prefill_host_workspace_size,
    cp_restore,
    cp_select_pass,
    cp_select_pass_cost,
    cp_shard_plan,
    cp_shard_plan_sizes,
    make_plan,
    new_status,
    pass_q_schedule,
    pass_q_schedule_host,
    segments_host,
)
