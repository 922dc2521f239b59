"""Oracle of the pass-KV / pass-Q choice.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Blog "什么是 Context Parallelism", §3.5 (the pass-KV / pass-Q switch): pass-KV
circulates the KV blocks (K and V of all T+P tokens, Hkv heads), pass-Q
circulates the query blocks (T tokens, Hq heads); pass-Q is chosen when its
message is the smaller one.  The page states the same rule as a miss-rate
threshold, T/(T+P) <= 2 Nkv/Nh, and gives 12.5 % for Llama-3 405B.  This
module decides by comparing the two message sizes directly.

The page's fitted heuristic h(T,P) = -1.059 log T + 1.145 log(T/(T+P)) +
12.112 (pass-KV when h > 0) names neither the logarithm's base nor the unit
of T and P; natural logarithms of token counts are taken here.  Parity
unpinned: the page's own 128K / CP=4 switch point (about 5 % miss rate) does
not follow from the formula under any base (e, 2, 10) with T and P counted
in tokens, thousands of tokens or tokens per rank.

The same section lays a roofline condition over the message rule (pass-KV is
preferred when its per-hop SendRecv hides behind that hop's attention) and
refines pass-Q by the All2All that brings its scattered partials home before
the LSE merge; it prints no formula for either.  ``exposed_times`` prices
them for one rank of a ring of C ranks (reading R10): every hop carries one
C-th of the KV (pass-KV, K and V) or of the queries (pass-Q) and overlaps it
with one C-th of that rank's attention; pass-Q then moves its partials in an
All2All and merges its C partials; whatever communication does not hide
behind attention is exposed, and the smaller exposure wins (pass-KV on a tie,
since a hidden SendRecv is what the roofline condition prefers).
"""

import math


def message_elements(T, P, Hq, Hkv, d=128):
    """Elements one ring hop sends: (pass-KV K+V block, pass-Q query block)."""
    kv = 2 * (T + P) * Hkv * d
    q = T * Hq * d
    return kv, q


def select_by_messages(T, P, Hq, Hkv):
    kv, q = message_elements(T, P, Hq, Hkv)
    return "pass_q" if q <= kv else "pass_kv"


def fitted_score(T, P):
    return -1.059 * math.log(T) + 1.145 * math.log(T / (T + P)) + 12.112


def select_fitted(T, P):
    return "pass_kv" if fitted_score(T, P) > 0 else "pass_q"


def exposed_times(T, P, Hq, Hkv, d, C, attn_tflops, link_gbs, merge_gbs):
    """(exposed pass-KV seconds, exposed pass-Q seconds) of one rank of a ring
    of C ranks, messages in bf16 and partials in fp32 (reading R10)."""
    pairs = T * P + T * (T + 1) / 2            # visible (query, key) pairs of the step
    flops = 2 * Hq * (d + d) * pairs
    hop_attention = flops / C / C / (attn_tflops * 1e12)
    q_rows = math.ceil(T / C)                  # one rank's query block
    kv_rows = math.ceil((T + P) / C)           # one rank's KV block
    kv_message = 2 * kv_rows * Hkv * d * 2     # K and V, bf16
    q_message = q_rows * Hq * d * 2            # Q, bf16
    partials = q_rows * Hq * (d + 1) * 4       # one rank's (O_j, L_j), fp32
    link = link_gbs * 1e9
    pass_kv = (C - 1) * max(0.0, kv_message / link - hop_attention)
    pass_q = (C - 1) * max(0.0, q_message / link - hop_attention)
    pass_q += (C - 1) / C * partials / link    # the All2All: all but the own share move
    pass_q += C * partials / (merge_gbs * 1e9)  # merging C partials reads them all
    return pass_kv, pass_q


def select_by_cost(T, P, Hq, Hkv, d, C, attn_tflops, link_gbs, merge_gbs):
    e_kv, e_q = exposed_times(T, P, Hq, Hkv, d, C, attn_tflops, link_gbs, merge_gbs)
    return "pass_kv" if e_kv <= e_q else "pass_q"
