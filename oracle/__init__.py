"""CPU oracle for the collective datapath — TEST INFRASTRUCTURE ONLY.

Only the tests, the smoke check in ``__graft_entry__`` and the CPU-baseline leg of
``bench.py`` may import this package. The library's product path never calls it and
shares no code with it (not even a header or a constant generator); the two meet only on
the seeded inputs of ``synth``.

What it computes, and where that comes from:

* A collective is a naming of an input layout and an output layout plus one operation,
  copy or reduce (Purlin article, "The Purlin PDF describes a three-layer design").
  ``oracle.naming`` evaluates any such naming by its plain definition.
* ``oracle.collectives`` writes the named collectives out directly from their
  definitions (all-reduce as every rank receiving the full sum — SiFAR review, Fig. 5
  oneshot; reduce-scatter then all-gather giving the same values — Fig. 6 twoshot;
  all-gather, broadcast, all-to-all, MoE dispatch by routing table).
* ``oracle.brute`` is an independent per-element evaluator with exact rational
  rounding, used only to pin the two modules above on tiny cases.

Readings taken where the pages are silent (each is listed in the design notes):
sums run in fixed rank order 0..R-1 (ties by ascending offset) in binary32 with
round-to-nearest-even, starting from the first term (not +0.0); bf16 outputs are rounded
once, to nearest even, from the binary32 sum.

Parity status: pinned (closed forms, invariants, brute force, hand-worked fixtures in
``tests/golden``); the pages print no worked example of their own.
"""

from .naming import validate, run_naming, ERR  # noqa: F401
from . import collectives  # noqa: F401
