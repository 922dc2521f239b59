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
not follow from the formula under any base with token units.
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
