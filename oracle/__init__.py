"""Oracle for block-wise variable-length attention and the FCP block distributor.

TEST INFRASTRUCTURE. This package is a plain, slow, obviously correct CPU
restatement of what the hot path computes. Only the tests, the smoke check of
``__graft_entry__`` and the CPU-baseline leg of ``bench.py`` may import it. The
product path (``context_parallelism_fcp_gb300``) never imports it and shares no
code with it; the only module both sides use is ``workloads`` (seeded input
generators, no method arithmetic).

Sources (all from "Unleashing Scalable Context Parallelism for Foundation Models
Pre-Training via FCP", arXiv 2605.08524, and the review of the same paper):

* ``attention`` -- the attention equation of Section 2.2, with causal/full masks
  (Section 2.2 scope) and grouped-query heads (Section 2.3), computed per whole
  sequence in float64 with no blocks; its analytic gradient; and the associative
  reduction of partial results named in Section 2.3, written out as the
  log-sum-exp merge.
* ``plan`` -- the sharding function G and assignment function M of Section 3.3,
  the fixed-size blocks with packing of Section 4.1, the Zig-Zag pairing of
  Section 3.2 / Figure 4, and the LPT greedy under a per-worker token cap of
  Sections 3.2 and 4.1; plus the work list of (Q-block, KV-block, mask) pairs and
  the coalescing of Section 4.2.

Every function is pinned by tests under ``tests/`` against facts the pages and
the mathematics fix (brute force, closed forms, special cases, finite
differences, the pages' worked Zig-Zag example). Parity of the LPT tie rules
beyond those invariants is a specification both implementations follow; its
optimality is unpinned (the pages state the problem is NP-complete and do not
print their Appendix A.1).
"""
