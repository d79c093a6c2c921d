"""CPU oracle for HeadTail ring (context-parallel) causal attention.

TEST INFRASTRUCTURE ONLY. Nothing on the product path may import, call or run
anything in this package: only ``tests/``, ``__graft_entry__.smoke()`` and the
``cpu_baseline`` / ``--impl reference`` legs of ``bench.py`` use it.

It is a plain, slow, float64 statement of what the method computes, written
from the pages it follows and sharing no code with the CUDA path:

* ``headtail``  -- the chunk-level HeadTail permutation, shard and unshard.
* ``attention`` -- RoPE at global positions, single-pass masked softmax
  attention (forward O and LSE) and its analytic gradients, the log-sum-exp
  merge (SDPAMerger), and the ring variant that merges per-step partials.
* ``ulysses``   -- the Ulysses all-to-all between sequence and head shards,
  and the attention run rank by rank on head shards.

Every function is pinned by ``tests/test_oracle.py`` against facts that do not
come from the oracle itself: the pages' worked HeadTail example, brute-force
softmax, closed forms, the ring == single-pass invariant, merge algebra,
complex-number RoPE, and central finite differences.
"""
from . import attention, headtail, ulysses  # noqa: F401
