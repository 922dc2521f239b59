"""CPU oracle for prefill context-parallel causal attention.

TEST INFRASTRUCTURE ONLY.  Nothing in the product path imports this package:
only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code, table or
helper with the CUDA library in ``context_causal_attention_cp_gb300/``.

Everything here is plain Python + NumPy in float64, written to be checked by
eye against the source pages:

* "Prefill Context Parallelism" (SGLang documentation), sections
  "Zigzag strategy", "Interleave strategy" and "Attention backend
  integration" -- the shard layouts and the per-block causal metadata.
* "什么是 Context Parallelism" (zhifeiding blog), section 2 (the zigzag
  load-balance figure), section 2.1 (restore index after the all-gather),
  section 3.1 / 3.3 (partial outputs O_j with their log-sum-exp L_j),
  section 3.3.2 (the pass-Q ring with a carried accumulator), section 3.5
  (persistent KV split into 2C first/last-paired blocks; the pass-KV /
  pass-Q switch) and section 3.6 (the LSE merge, a generalisation of
  FlashAttention's online softmax).

Modules:
    plan       -- zigzag / interleave shard plans, restore index, tile-load counts
    attention  -- dense causal attention (per query row) and per-KV-window partials
    merge      -- the log-sum-exp merge of partial results
    pipeline   -- plan -> per-shard partial -> [merge] -> restore, end to end;
                  the pass-Q ring (hop-by-hop merge into a carried accumulator)
    select     -- the pass-KV / pass-Q choice (message sizes; fitted heuristic;
                  the roofline cost rule)

Readings where the pages are silent:
    R1 remainder tokens of a zigzag split go one each to blocks 0..rem-1;
    R2 a rank's rows are ordered request by request, early block first;
    R3 the query at position P sees key positions 0..P of its own request
       (bottom-right aligned when a cached prefix exists);
    R4 LSE is the natural log of sum(exp(scale * q.k));
    R5 query head h reads KV head h // (Hq // Hkv);
    R6 an empty partial has O = 0 and L = -inf, the identity of the merge;
    R7 pass-Q keeps each request's KV resident in 2C blocks split like the
       zigzag query blocks, rank r holding blocks r and 2C-1-r;
    R8 the fitted switch heuristic uses natural logarithms of token counts;
    R9 the miss-rate threshold 2 Nkv / Nh compares one ring hop's messages
       (T Hq query rows against K and V of T+P tokens), ties to pass-Q;
    R10 the roofline rule prices, for one rank of a ring of C, the part of
       each hop's message (and of pass-Q's All2All of partials) that does
       not hide behind one C-th of the attention, pass-KV on a tie;
    R11 pass-Q carries an accumulator round the ring (section 3.3.2); the
       cost rule prices the All2All variant of section 3.5.
The remainder placement (R1) and rank-local order (R2) are fixed by these
readings only: "parity unpinned" by the pages beyond their even-split
examples.  The fitted heuristic (R8) is "parity unpinned": the page's stated
switch point does not follow from its formula under any reading tried.
"""

from . import plan, attention, merge, pipeline, select  # noqa: F401
