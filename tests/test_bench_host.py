"""Host-side helpers of bench.py on CPU: the profile lookup behind the
roofline's traffic figure (a summary whose source hashes no longer match
gives no traffic), the decode ranks' resident layout, and the work counts
the throughput figures divide by."""

import os
import shutil

import pytest
import torch

import bench
from context_causal_attention_cp_gb300 import workloads as W


def test_profile_with_a_stale_hash_gives_no_traffic(tmp_path, monkeypatch):
    csrc = tmp_path / "context_causal_attention_cp_gb300" / "csrc"
    csrc.mkdir(parents=True)
    (tmp_path / "profiles").mkdir()
    src = os.path.join(bench.ROOT, "context_causal_attention_cp_gb300", "csrc", "attn.cu")
    shutil.copy(src, csrc / "attn.cu")
    import hashlib
    good = hashlib.sha256(open(src, "rb").read()).hexdigest()[:16]
    (tmp_path / "profiles" / "k.md").write_text(
        f"traffic_bytes_per_launch: 1234\nsource_sha256_prefix: attn.cu {good}\n")
    monkeypatch.setattr(bench, "ROOT", str(tmp_path))
    assert bench.profiled_traffic("k.md") == 1234
    (csrc / "attn.cu").write_text("// edited\n")
    assert bench.profiled_traffic("k.md") is None
    assert bench.profiled_traffic("missing.md") is None
    assert bench.profiled_traffic("") is None


def test_decode_ranks_hold_their_interleaved_tokens():
    S, n_kv, nq = 4, 6, 3
    k = torch.arange(S * n_kv * 2 * 8, dtype=torch.float32).view(S * n_kv, 2, 8)
    v = -k[:, :, :4].clone()
    q = torch.randn(nq, 4, 8)
    q_rank, k_rank, v_rank, segs = bench.decode_ranks(q, k, v, S)
    for j in range(S):
        for i in range(n_kv):
            assert torch.equal(k_rank[j * n_kv + i], k[i * S + j])   # key i*S+j lives on rank j
            assert torch.equal(v_rank[j * n_kv + i], v[i * S + j])
        assert torch.equal(q_rank[j * nq:(j + 1) * nq], q)
        # q_row0, q_len, q_pos0, q_pos_step, kv_row0, kv_len, tok0, req
        assert segs[j].tolist() == [j * nq, nq, n_kv - 1, 0, j * n_kv, n_kv, j * nq, j]


def test_work_counts_of_the_headline_workload():
    w = W.WORKLOADS[bench.WORKLOAD]
    assert bench.attention_flops(w) == pytest.approx(2.0 * 32 * 256 * 536887296)
    assert bench.attention_flops(w) / 1e12 == pytest.approx(8.796, abs=5e-4)
    # Q, O (bf16) and LSE once per token, K and V once
    assert bench.algorithmic_bytes(w) == 32768 * 32 * (256 + 256 + 4) + 32768 * 8 * 256 * 2
