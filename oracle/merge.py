"""Oracle log-sum-exp merge of partial attention results.

TEST INFRASTRUCTURE ONLY (see the package docstring).

Blog "什么是 Context Parallelism", §3.6 (the shared component of pass-KV and
pass-Q): shard j gives a normalised output O_j and its log-sum-exp L_j; the
exact result is their online-softmax combination.  The formula itself did not
survive the page's extraction; the reading used here (reading C1) is the
standard rule, which follows from L_j = log(sum over shard j of exp S):

    L = log(sum_j exp(L_j))
    O = sum_j exp(L_j - L) * O_j

evaluated with the largest L_j subtracted first (m = max_j L_j,
w_j = exp(L_j - m), L = m + log(sum_j w_j), O = sum_j w_j O_j / sum_j w_j),
which is the same value.  An empty partial (L_j = -inf) has weight 0; if every
partial is empty the result is O = 0, L = -inf (reading R6).
"""

import numpy as np


def lse_merge(o_parts, l_parts):
    """Merge partials along axis 0.

    o_parts: [n, ..., dv] float64, l_parts: [n, ...] float64
    returns (O [..., dv], L [...])
    """
    o_parts = np.asarray(o_parts, dtype=np.float64)
    l_parts = np.asarray(l_parts, dtype=np.float64)
    m = l_parts.max(axis=0)
    empty = np.isneginf(m)
    m_safe = np.where(empty, 0.0, m)
    w = np.exp(l_parts - m_safe[None])              # exp(-inf) = 0 for empty parts
    wsum = w.sum(axis=0)
    wsum_safe = np.where(empty, 1.0, wsum)
    O = (w[..., None] * o_parts).sum(axis=0) / wsum_safe[..., None]
    L = np.where(empty, -np.inf, m_safe + np.log(wsum_safe))
    O = np.where(empty[..., None], 0.0, O)
    return O, L
