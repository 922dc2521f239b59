"""Pins for the CPU oracle: it is checked against what the pages and the
mathematics fix, never against itself.

* the pages' worked examples (fixtures under tests/golden/, each citing its page),
* the load-balance figure of the blog "什么是 Context Parallelism" (§2),
* a literal per-element brute force of softmax attention in pure Python,
* closed forms (one visible key; identical keys; zero query),
* the merge invariant (blog §3.1 / §3.3.2: merging per-KV-block partials is
  exact) on random splits, associativity and the -inf identity,
* permutation invariants of the plans.

A few tests plant a plausible mistake in a copy of an oracle function and
check that a pin catches it.
"""

import math
import random

import numpy as np
import pytest

from oracle import attention as oatt
from oracle import merge as omerge
from oracle import pipeline as opipe
from oracle import plan as oplan
from context_causal_attention_cp_gb300 import workloads as W


# ----------------------------------------------------------------- plans ----

def _owned(plan, r):
    return sorted(plan.rank_rows[r])


def test_zigzag_page_example(golden):
    g = golden("zigzag_cp4_16tokens.txt")
    plan = oplan.zigzag_plan([16], [0], 4)
    for r in range(4):
        assert _owned(plan, r) == [int(x) for x in g[f"rank {r}"]]
    blocks = [tuple(int(t) for t in b.split("-")) for b in g["blocks"]]
    sizes = oplan.zigzag_block_sizes(16, 4)
    assert sizes == [hi - lo + 1 for lo, hi in blocks]


def test_interleave_page_example(golden):
    g = golden("interleave_cp4_16tokens.txt")
    plan = oplan.interleave_plan([16], [0], 4)
    for r in range(4):
        assert plan.rank_rows[r] == [int(x) for x in g[f"rank {r}"]]


def test_interleave_across_requests(golden):
    g = golden("interleave_lens5_3.txt")
    C = int(g["cp_size"][0])
    lens = [int(x) for x in g["new_lens"]]
    plan = oplan.interleave_plan(lens, [0] * len(lens), C)
    assert set(int(x) for x in g["rank 0 owns"]) <= set(plan.rank_rows[0])
    assert set(int(x) for x in g["rank 1 owns"]) <= set(plan.rank_rows[1])
    # flat index 5 is the first new token of the second request
    row = plan.restore_idx[5]
    assert plan.positions[row] == 0
    segs = [s for s in plan.segments[1] if s.q_row0 <= row < s.q_row0 + s.q_len]
    assert len(segs) == 1 and segs[0].req == int(g["flat 5 request"][0])
    assert row - segs[0].q_row0 == 0 and segs[0].q_pos0 == int(g["flat 5 local token"][0])
    # with a cached prefix, positions keep their original values
    plan2 = oplan.interleave_plan(lens, [7, 11], C)
    assert plan2.positions[plan2.restore_idx[5]] == 11


def test_tile_loads_figure(golden):
    g = golden("tile_loads_cp4.txt")
    assert oplan.block_tile_loads(oplan.sequential_block_owner(4), 4) == \
        [int(x) for x in g["sequential"]]
    assert oplan.block_tile_loads(oplan.zigzag_ranks_of_blocks(4), 4) == \
        [int(x) for x in g["zigzag"]]
    # closed forms behind the figure: 4r + 3 sequential, 2C + 1 zigzag
    for C in (2, 3, 4, 8):
        assert oplan.block_tile_loads(oplan.sequential_block_owner(C), C) == \
            [4 * r + 3 for r in range(C)]
        assert oplan.block_tile_loads(oplan.zigzag_ranks_of_blocks(C), C) == [2 * C + 1] * C


def test_pair_counts_balanced_32k():
    w = W.WORKLOADS["llama8b_32k"]
    plan = oplan.zigzag_plan(w.new_lens, w.prefix_lens, w.cp_size)
    pairs = oplan.visible_pairs(plan, w.new_lens, w.prefix_lens)
    # closed form per rank: 2048^2 * (r + 15 - r) + 2 * 2048*2049/2
    assert pairs == [2048 * 2048 * 15 + 2048 * 2049] * 8
    assert sum(pairs) == 32768 * 32769 // 2


@pytest.mark.parametrize("seed", range(40))
@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
def test_plan_invariants(seed, strategy):
    new, pre = W.random_batch(seed)
    C = [1, 2, 3, 4, 8][seed % 5]
    plan = oplan.make_plan(new, pre, C, strategy)
    N = sum(new)
    assert sorted(plan.gather_idx) == list(range(N))
    for i in range(N):
        assert plan.gather_idx[plan.restore_idx[i]] == i
    flat_start, kv_start = oplan.request_tables(new, pre)
    req_of = [b for b, n in enumerate(new) for _ in range(n)]
    seen = 0
    for r in range(C):
        assert plan.row_offsets[r + 1] - plan.row_offsets[r] == len(plan.rank_rows[r])
        for s in plan.segments[r]:
            assert s.q_len > 0 and s.rank == r
            for i in range(s.q_len):
                row = s.q_row0 + i
                tok = plan.gather_idx[row]
                assert req_of[tok] == s.req
                pos = pre[s.req] + tok - flat_start[s.req]
                assert plan.positions[row] == pos == s.q_pos0 + i * s.q_pos_step
                assert plan.row_offsets[r] <= row < plan.row_offsets[r + 1]
            assert s.kv_len == s.q_pos0 + (s.q_len - 1) * s.q_pos_step + 1
            assert s.kv_row0 == kv_start[s.req]
            seen += s.q_len
    assert seen == N
    if strategy == "interleave":
        for r in range(C):
            assert all(i % C == r for i in plan.rank_rows[r])
            assert plan.rank_rows[r] == sorted(plan.rank_rows[r])
    else:
        for b, n in enumerate(new):
            sizes = oplan.zigzag_block_sizes(n, C)
            assert sum(sizes) == n and max(sizes) - min(sizes) <= 1
            # early blocks receive the remainder
            assert sizes == sorted(sizes, reverse=True)


def test_zigzag_rank_order_within_rank():
    # reading R2: request by request, early block then late block
    plan = oplan.zigzag_plan([8, 8], [0, 3], 2)
    assert plan.rank_rows[0] == [0, 1, 6, 7, 8, 9, 14, 15]
    assert plan.rank_rows[1] == [2, 3, 4, 5, 10, 11, 12, 13]
    segs = plan.segments[0]
    assert [(s.q_row0, s.q_len, s.q_pos0, s.kv_len, s.req) for s in segs] == \
        [(0, 2, 0, 2, 0), (2, 2, 6, 8, 0), (4, 2, 3, 5, 1), (6, 2, 9, 11, 1)]


def test_zigzag_short_request_has_empty_blocks():
    plan = oplan.zigzag_plan([3], [17], 4)
    assert oplan.zigzag_block_sizes(3, 4) == [1, 1, 1, 0, 0, 0, 0, 0]
    assert [len(plan.rank_rows[r]) for r in range(4)] == [1, 1, 1, 0]
    assert plan.segments[3] == []
    assert plan.positions == [17, 18, 19]


# ------------------------------------------------------------- attention ----

def literal_attention(q, k, v, pos, kv0, scale, g, lo=0, hi=None):
    """Per-element pure-Python softmax attention for one query row."""
    Hq, d = len(q), len(q[0])
    dv = len(v[0][0])
    hi = pos + 1 if hi is None else min(hi, pos + 1)
    O, L = [], []
    for h in range(Hq):
        kh = h // g
        keys = list(range(max(lo, 0), hi))
        if not keys:
            O.append([0.0] * dv)
            L.append(-math.inf)
            continue
        s = [scale * math.fsum(q[h][c] * k[kv0 + j][kh][c] for c in range(d)) for j in keys]
        m = max(s)
        lse = m + math.log(math.fsum(math.exp(x - m) for x in s))
        O.append([math.fsum(math.exp(s[t] - lse) * v[kv0 + j][kh][c]
                            for t, j in enumerate(keys)) for c in range(dv)])
        L.append(lse)
    return O, L


def _tiny(seed, B=3, Hq=4, Hkv=2, d=5, dv=3):
    rng = np.random.default_rng(seed)
    new = [int(x) for x in rng.integers(1, 7, B)]
    pre = [int(x) for x in rng.integers(0, 4, B)]
    kv = sum(new) + sum(pre)
    q = rng.standard_normal((sum(new), Hq, d))
    k = rng.standard_normal((kv, Hkv, d))
    v = rng.standard_normal((kv, Hkv, dv))
    return new, pre, q, k, v


@pytest.mark.parametrize("seed", range(6))
def test_attention_matches_literal_loops(seed):
    new, pre, q, k, v = _tiny(seed)
    scale = 0.37
    O, L = oatt.dense_causal_attention(q, k, v, new, pre, scale)
    pos, kv0 = oatt.token_tables(new, pre)
    for i in range(len(pos)):
        Oi, Li = literal_attention(q[i].tolist(), k.tolist(), v.tolist(), int(pos[i]),
                                   int(kv0[i]), scale, 2)
        np.testing.assert_allclose(O[i], Oi, rtol=0, atol=1e-12)
        np.testing.assert_allclose(L[i], Li, rtol=0, atol=1e-12)


def test_attention_window_matches_literal_loops():
    new, pre, q, k, v = _tiny(11, B=2)
    pos, kv0 = oatt.token_tables(new, pre)
    for lo, hi in [(0, 2), (1, 3), (2, 100), (5, 6), (7, 9)]:
        O, L = oatt.attention_rows(q, k, v, pos, kv0, 0.5, lo, hi)
        for i in range(len(pos)):
            Oi, Li = literal_attention(q[i].tolist(), k.tolist(), v.tolist(), int(pos[i]),
                                       int(kv0[i]), 0.5, 2, lo, hi)
            np.testing.assert_allclose(O[i], Oi, rtol=0, atol=1e-12)
            assert (np.isneginf(L[i]) == np.isneginf(Li)).all()
            fin = ~np.isneginf(Li)
            np.testing.assert_allclose(L[i][fin], np.asarray(Li)[fin], rtol=0, atol=1e-12)


def test_single_visible_key():
    # the first new token with no prefix sees only itself: O = v, L = s * q.k
    rng = np.random.default_rng(3)
    q = rng.standard_normal((1, 4, 8))
    k = rng.standard_normal((1, 2, 8))
    v = rng.standard_normal((1, 2, 6))
    O, L = oatt.dense_causal_attention(q, k, v, [1], [0], 0.25)
    for h in range(4):
        assert O[0, h].tolist() == v[0, h // 2].tolist()
        assert L[0, h] == pytest.approx(0.25 * float(q[0, h] @ k[0, h // 2]), abs=1e-14)


def test_identical_keys_closed_form():
    rng = np.random.default_rng(4)
    n = 9
    q = rng.standard_normal((n, 2, 8))
    k = np.tile(rng.standard_normal((1, 1, 8)), (n, 1, 1))
    v = rng.standard_normal((n, 1, 3))
    O, L = oatt.dense_causal_attention(q, k, v, [n], [0], 0.7)
    for t in range(n):
        for h in range(2):
            s = 0.7 * float(q[t, h] @ k[0, 0])
            assert L[t, h] == pytest.approx(s + math.log(t + 1), abs=1e-12)
            np.testing.assert_allclose(O[t, h], v[: t + 1, 0].mean(axis=0), atol=1e-12)


def test_zero_query_is_mean_of_visible_values():
    rng = np.random.default_rng(5)
    q = np.zeros((4, 1, 8))
    k = rng.standard_normal((6, 1, 8))
    v = rng.standard_normal((6, 1, 3))
    O, L = oatt.dense_causal_attention(q, k, v, [4], [2], 1.0)
    for t in range(4):
        assert L[t, 0] == pytest.approx(math.log(t + 3), abs=1e-14)
        np.testing.assert_allclose(O[t, 0], v[: t + 3, 0].mean(axis=0), atol=1e-12)


def test_decode_attention_matches_literal():
    rng = np.random.default_rng(6)
    q = rng.standard_normal((2, 4, 5))
    k = rng.standard_normal((7, 2, 5))
    v = rng.standard_normal((7, 2, 3))
    rows = [1, 3, 5]
    O, L = oatt.decode_attention(q, k, v, 0.9, rows)
    ksel, vsel = k[rows], v[rows]
    for i in range(2):
        # every selected key visible: a query "at position len-1" over the selection
        Oi, Li = literal_attention(q[i].tolist(), ksel.tolist(), vsel.tolist(), 2, 0, 0.9, 2)
        np.testing.assert_allclose(O[i], Oi, atol=1e-12)
        np.testing.assert_allclose(L[i], Li, atol=1e-12)


# ----------------------------------------------------------------- merge ----

@pytest.mark.parametrize("seed", range(8))
def test_merge_of_random_kv_splits_is_exact(seed):
    new, pre, q, k, v = _tiny(100 + seed, B=2, Hq=4, Hkv=4, d=4, dv=4)
    pos, kv0 = oatt.token_tables(new, pre)
    full_O, full_L = oatt.attention_rows(q, k, v, pos, kv0, 0.8)
    rnd = random.Random(seed)
    longest = max(n + p for n, p in zip(new, pre))
    cuts = sorted(set([0, longest] + [rnd.randrange(1, longest) for _ in range(3)]))
    parts = [oatt.attention_rows(q, k, v, pos, kv0, 0.8, a, b) for a, b in zip(cuts, cuts[1:])]
    O, L = omerge.lse_merge([p[0] for p in parts], [p[1] for p in parts])
    np.testing.assert_allclose(O, full_O, rtol=0, atol=1e-12)
    np.testing.assert_allclose(L, full_L, rtol=0, atol=1e-12)


def test_merge_associative_and_identity():
    rng = np.random.default_rng(9)
    o = rng.standard_normal((3, 5, 4))
    l = rng.standard_normal((3, 5)) * 3
    O3, L3 = omerge.lse_merge(o, l)
    O12, L12 = omerge.lse_merge(o[:2], l[:2])
    Oa, La = omerge.lse_merge(np.stack([O12, o[2]]), np.stack([L12, l[2]]))
    np.testing.assert_allclose(Oa, O3, atol=1e-13)
    np.testing.assert_allclose(La, L3, atol=1e-13)
    empty_o = np.zeros((5, 4))
    empty_l = np.full(5, -np.inf)
    Oe, Le = omerge.lse_merge(np.stack([o[0], empty_o]), np.stack([l[0], empty_l]))
    np.testing.assert_allclose(Oe, o[0], atol=0)
    np.testing.assert_allclose(Le, l[0], atol=0)
    Oz, Lz = omerge.lse_merge(np.stack([empty_o, empty_o]), np.stack([empty_l, empty_l]))
    assert (Oz == 0).all() and np.isneginf(Lz).all()


def test_merge_two_parts_closed_form():
    # two partials over disjoint single keys: L = log(e^a + e^b), O = softmax-weighted
    a, b = 0.3, -1.2
    o1, o2 = np.array([1.0, 2.0]), np.array([-3.0, 0.5])
    O, L = omerge.lse_merge(np.stack([o1, o2])[:, None], np.array([[a], [b]]))
    assert L[0] == pytest.approx(math.log(math.exp(a) + math.exp(b)), abs=1e-15)
    wa = math.exp(a) / (math.exp(a) + math.exp(b))
    np.testing.assert_allclose(O[0], wa * o1 + (1 - wa) * o2, atol=1e-15)


# -------------------------------------------------------------- pipeline ----

@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
@pytest.mark.parametrize("C", [1, 2, 3, 4])
def test_sharded_pipeline_equals_dense(strategy, C):
    new, pre, q, k, v = _tiny(40 + C, B=3, Hq=4, Hkv=2, d=6, dv=5)
    O_ref, L_ref = oatt.dense_causal_attention(q, k, v, new, pre, 0.45)
    O, L, _ = opipe.sharded_attention(q, k, v, new, pre, C, strategy, 0.45)
    np.testing.assert_allclose(O, O_ref, atol=1e-13)
    np.testing.assert_allclose(L, L_ref, atol=1e-13)
    Op, Lp, _ = opipe.partial_kv_attention(q, k, v, new, pre, C, strategy, 0.45, kv_block=3)
    np.testing.assert_allclose(Op, O_ref, atol=1e-12)
    np.testing.assert_allclose(Lp, L_ref, atol=1e-12)


def test_pass_q_resident_kv_matches_zigzag_example(golden):
    """With no prefix, the resident KV blocks of the pass-Q ring are the zigzag
    blocks of the page's CP=4 / 16-token example (rank r keeps blocks r and
    2C-1-r)."""
    g = golden("zigzag_cp4_16tokens.txt")
    wins = opipe.resident_kv_windows(16, 4)
    for r in range(4):
        owned = sorted(t for lo, hi in wins[r] for t in range(lo, hi))
        assert owned == [int(x) for x in g[f"rank {r}"]]


@pytest.mark.parametrize("total", [0, 1, 7, 16, 37, 1000])
@pytest.mark.parametrize("C", [1, 2, 3, 8])
def test_pass_q_resident_kv_partitions_positions(total, C):
    wins = opipe.resident_kv_windows(total, C)
    cover = sorted(t for r in range(C) for lo, hi in wins[r] for t in range(lo, hi))
    assert cover == list(range(total))
    sizes = [hi - lo for r in range(C) for lo, hi in wins[r]]
    assert max(sizes) - min(sizes) <= 1


@pytest.mark.parametrize("strategy", ["zigzag", "interleave"])
@pytest.mark.parametrize("C", [1, 2, 3, 4])
def test_pass_q_ring_equals_dense(strategy, C):
    """Blog §3.3.2: after C hops the carried accumulator is the exact output."""
    new, pre, q, k, v = _tiny(60 + C, B=3, Hq=4, Hkv=2, d=6, dv=5)
    O_ref, L_ref = oatt.dense_causal_attention(q, k, v, new, pre, 0.45)
    O, L, _ = opipe.pass_q_attention(q, k, v, new, pre, C, strategy, 0.45)
    np.testing.assert_allclose(O, O_ref, atol=1e-12)
    np.testing.assert_allclose(L, L_ref, atol=1e-12)


# ------------------------------------------------------ planted mistakes ----

def test_planted_mistakes_are_caught(monkeypatch):
    """Each plausible oracle mistake must break one of the pins above."""
    new, pre, q, k, v = _tiny(77)
    pos, kv0 = oatt.token_tables(new, pre)
    ref = [literal_attention(q[i].tolist(), k.tolist(), v.tolist(), int(pos[i]),
                             int(kv0[i]), 0.37, 2) for i in range(len(pos))]

    def off_by_one(q_, k_, v_, positions, kv_row0, scale, kv_lo=0, kv_hi=None):
        return oatt.attention_rows(q_, k_, v_, np.asarray(positions) - 1, kv_row0, scale,
                                   kv_lo, kv_hi)

    def wrong_group(q_, k_, v_, positions, kv_row0, scale, kv_lo=0, kv_hi=None):
        # h % Hkv instead of h // g
        Hq = q_.shape[1]
        perm = [(h % 2) * 2 + h // 2 for h in range(Hq)]
        return oatt.attention_rows(q_[:, perm], k_, v_, positions, kv_row0, scale,
                                   kv_lo, kv_hi)

    for bad in (off_by_one, wrong_group):
        O, L = bad(q, k, v, pos, kv0, 0.37)
        errs = [np.abs(np.nan_to_num(O[i]) - np.asarray(ref[i][0])).max() for i in range(len(pos))]
        assert max(errs) > 1e-3

    # a merge that forgets to renormalise the weights
    o = np.random.default_rng(1).standard_normal((2, 3, 2))
    l = np.array([[0.1, 0.2, 0.3], [1.0, -1.0, 0.0]])
    w = np.exp(l)
    bad_O = (w[..., None] * o).sum(0)
    good_O, _ = omerge.lse_merge(o, l)
    assert np.abs(bad_O - good_O).max() > 1e-2

    # remainder to the late blocks instead of the early ones
    def late_rem(n, C):
        return list(reversed(oplan.zigzag_block_sizes(n, C)))
    sizes = late_rem(13, 4)
    assert sizes != sorted(sizes, reverse=True)


def test_planted_pass_q_mistakes_are_caught(monkeypatch):
    """A ring that forgets a rank's second resident block, or merges with the
    wrong weight, must break the pass-Q pin."""
    new, pre, q, k, v = _tiny(63, B=3, Hq=4, Hkv=2, d=6, dv=5)
    O_ref, L_ref = oatt.dense_causal_attention(q, k, v, new, pre, 0.45)
    good = opipe.resident_kv_windows
    monkeypatch.setattr(opipe, "resident_kv_windows", lambda t, c: [w[:1] for w in good(t, c)])
    O, L, _ = opipe.pass_q_attention(q, k, v, new, pre, 3, "zigzag", 0.45)
    assert not np.allclose(L, L_ref, atol=1e-6)
    monkeypatch.setattr(opipe, "resident_kv_windows", good)

    real_merge = opipe.lse_merge

    def merge_without_max_weight(o_parts, l_parts):
        # plain mean of the non-empty partials instead of the LSE weights
        O, L = real_merge(o_parts, l_parts)
        w = np.where(np.isneginf(l_parts), 0.0, 1.0)
        n = np.maximum(w.sum(axis=0), 1.0)
        return (w[..., None] * o_parts).sum(axis=0) / n[..., None], L

    monkeypatch.setattr(opipe, "lse_merge", merge_without_max_weight)
    O, L, _ = opipe.pass_q_attention(q, k, v, new, pre, 3, "zigzag", 0.45)
    assert not np.allclose(O, O_ref, atol=1e-6)


# ---------------------------------------------------- pass-KV / pass-Q ----

def test_select_threshold_page_value(golden):
    """§3.5: with N_h/N_kv = 16 the switch is at a miss rate of 12.5 %."""
    from oracle import select as osel
    g = golden("pass_switch_threshold.txt")
    ratio = int(g["heads_ratio"][0])
    thr = float(g["threshold_percent"][0]) / 100.0
    Hkv = 8
    Hq = ratio * Hkv
    for total in (8, 1024, 131072):
        T = int(total * thr)
        assert T / total == thr
        assert osel.select_by_messages(T, total - T, Hq, Hkv) == "pass_q"
        assert osel.select_by_messages(T + 1, total - T - 1, Hq, Hkv) == "pass_kv"


@pytest.mark.parametrize("ratio", [4, 8, 16])
def test_select_page_statements(ratio):
    """Decode (T = 1) picks pass-Q; full prefill (P = 0) picks pass-KV (GQA)."""
    from oracle import select as osel
    for P in (1000, 131071, 10 ** 6):
        assert osel.select_by_messages(1, P, 8 * ratio, 8) == "pass_q"
    for T in (1, 4096, 131072):
        assert osel.select_by_messages(T, 0, 8 * ratio, 8) == "pass_kv"


def test_select_fitted_reading():
    """The fitted rule with natural logs: h is decreasing in T at fixed miss
    rate, and pass-Q at decode over a long cache (page: decode uses pass-Q)."""
    from oracle import select as osel
    assert osel.select_fitted(1, 131071) == "pass_q"
    assert osel.fitted_score(1000, 1000) > osel.fitted_score(2000, 2000)
    assert osel.fitted_score(1, 0) == pytest.approx(12.112)


def test_parallel_row_harness_equals_direct_oracle_calls():
    """The test harness that spreads oracle rows over spawned processes gives,
    row by row, exactly the oracle's own single-process values (also with V
    a view of K and with a key window)."""
    import oracle_rows
    rng = np.random.default_rng(5)
    new, pre = [40, 7, 65], [3, 0, 20]
    kv = sum(new) + sum(pre)
    q = rng.standard_normal((sum(new), 4, 16))
    k = rng.standard_normal((kv, 2, 16))
    v = rng.standard_normal((kv, 2, 8))
    pos, kv0 = oatt.token_tables(new, pre)
    rows = np.array([0, 5, 39, 40, 46, 47, 100, 111])
    for vv, pref, lo, hi in ((v, False, 0, None), (k[:, :, :8], True, 0, None), (v, False, 10, 30)):
        O1, L1 = oatt.attention_rows(q[rows], k, vv, pos[rows], kv0[rows], 0.3, lo, hi)
        O2, L2 = oracle_rows.attention_rows_parallel(q[rows], k, vv, pos[rows], kv0[rows], 0.3,
                                                     lo, hi, v_is_k_prefix=pref, procs=2)
        assert np.array_equal(O1, O2) and np.array_equal(L1, L2)


# ------------------------------------------------ cost-driven selector ----

@pytest.mark.parametrize("link_gbs", [25.0, 50.0, 450.0])
@pytest.mark.parametrize("ratio", [4, 8, 16])
def test_select_cost_page_statements(link_gbs, ratio):
    """§3.5: decode (T = 1) over a long cache picks pass-Q; full prefill under
    GQA picks pass-KV (its SendRecv hides behind the attention), for attention
    rates and links of real GPUs."""
    from oracle import select as osel
    Hkv = 8
    Hq = ratio * Hkv
    for C in (2, 4, 8):
        for tf in (300.0, 1000.0, 2000.0):
            for P in (4096, 131071, 10 ** 6):
                assert osel.select_by_cost(1, P, Hq, Hkv, 128, C, tf, link_gbs, 3000.0) == "pass_q"
            for T in (16384, 131072):
                assert osel.select_by_cost(T, 0, Hq, Hkv, 128, C, tf, link_gbs, 3000.0) == \
                    "pass_kv"


def test_select_cost_reduces_to_the_message_rule_without_overlap():
    """With no overlap to gain (a very slow link) and the All2All and merge
    terms negligible (a long ring, a free merge), the exposed times are the
    ring's messages, so the cost rule decides like the message rule (pinned
    to the page's 12.5 %) away from the tie."""
    from oracle import select as osel
    C = 1024
    for Hq, Hkv in ((128, 8), (32, 8), (64, 64)):
        for Tb in (1, 3, 17, 100):
            for Pb in (0, 1, 5, 64, 1000):
                T, P = Tb * C, Pb * C
                lhs, rhs = T * Hq, 2 * (T + P) * Hkv
                if abs(lhs - rhs) <= 0.02 * rhs:
                    continue
                assert osel.select_by_cost(T, P, Hq, Hkv, 128, C, 1000.0, 1e-6, 1e12) == \
                    osel.select_by_messages(T, P, Hq, Hkv), (T, P, Hq, Hkv)


def _check_slow_attention_hides_pass_kv():
    from oracle import select as osel
    for T in (1, 100, 4096):
        for P in (0, 10 ** 5):
            e_kv, e_q = osel.exposed_times(T, P, 128, 8, 128, 4, 1e-9, 50.0, 3000.0)
            assert e_kv == 0.0 and e_q > 0.0
            assert osel.select_by_cost(T, P, 128, 8, 128, 4, 1e-9, 50.0, 3000.0) == "pass_kv"


def test_select_cost_slow_attention_hides_pass_kv():
    """The roofline condition: when attention is slow enough that any hop's
    SendRecv hides behind it, pass-KV wins whatever the miss rate."""
    _check_slow_attention_hides_pass_kv()


def _check_all2all_refines_pass_q():
    from oracle import select as osel
    for C in (2, 4, 8):
        for total in (8192, 131072):
            T = total // 8                     # 12.5 %: the message rule's tie for 128 / 8 heads
            assert osel.select_by_messages(T, total - T, 128, 8) == "pass_q"
            assert osel.select_by_cost(T, total - T, 128, 8, 128, C, 1000.0, 1e-6, 1e12) == \
                "pass_kv"


def test_select_cost_all2all_refines_pass_q():
    """The page's refinement counts pass-Q's All2All: at the message rule's
    tie (equal ring messages) and without overlap, pass-Q still has its
    partials to move, so pass-KV wins."""
    _check_all2all_refines_pass_q()


def test_planted_cost_rule_mistakes_are_caught(monkeypatch):
    """Plausible slips in the cost rule each fail a pin: dropping the overlap
    with attention fails the roofline pin; charging the All2All to pass-KV
    instead of pass-Q fails the refinement pin."""
    from oracle import select as osel
    real = osel.exposed_times

    def no_overlap(T, P, Hq, Hkv, d, C, tf, link, merge):
        return real(T, P, Hq, Hkv, d, C, 1e30, link, merge)   # attention takes no time
    monkeypatch.setattr(osel, "exposed_times", no_overlap)
    with pytest.raises(AssertionError):
        _check_slow_attention_hides_pass_kv()

    def a2a_on_kv(T, P, Hq, Hkv, d, C, tf, link, merge):
        e_kv, e_q = real(T, P, Hq, Hkv, d, C, tf, link, merge)
        partials = math.ceil(T / C) * Hq * (d + 1) * 4 * (C - 1) / C / (link * 1e9)
        return e_kv + partials, e_q - partials
    monkeypatch.setattr(osel, "exposed_times", a2a_on_kv)
    with pytest.raises(AssertionError):
        _check_all2all_refines_pass_q()


def test_fitted_heuristic_readings_miss_the_page_switch_point():
    """Documents why the fitted heuristic stays unpinned: under every reading
    tried (log base e, 2 or 10; T and P in tokens, thousands of tokens or
    tokens per rank at CP=4) the switch of h(T, P) at a 131072-token context
    is nowhere near the page's measured ~5 % miss rate (blog §3.5): it is
    either absent or below 0.01 %."""
    N, C = 131072, 4
    for log in (math.log, math.log2, math.log10):
        for unit in (1.0, 1e-3, 1.0 / C):
            def h(m):
                T = m * N
                return -1.059 * log(T * unit) + 1.145 * log(T / N) + 12.112
            grid = [10 ** (-6 + 6 * i / 3000) for i in range(3001)]
            switches = [grid[i] for i in range(1, len(grid))
                        if (h(grid[i]) > 0) != (h(grid[i - 1]) > 0)]
            assert all(s < 1e-4 for s in switches), (log, unit, switches)
            assert not any(0.025 <= s <= 0.1 for s in switches)
