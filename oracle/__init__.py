"""CPU oracle for the grammar-compressed right product y = Mx.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline leg may import or run anything in this package.
The product path never does, and this package imports nothing from it.

It is deliberately plain and slow: numpy and Python loops, float64 for
floating point, no blocking, fusion or reordering beyond what the definitions
state. Each function cites the passage of "Right Multiplication on
Grammar-Compressed Matrices: A Streaming, Memory-Bounded GPU Engine" (the
pages) that it follows.

Modules
  direct   O1: y = Mx straight from the uncompressed rows (fp64 / exact int /
           boolean OR / float32 min-plus), plus the error scale b = |M||x|;
           the left product x = M^T y (float64 with b = |M|^T |y|, exact
           int64, Boolean OR, float32 min-plus).
  grammar  CSRV encoding, a naive RePair, decompression, the W-array grammar
           evaluation (sum and min-plus), the top-down left product, levels
           (Eq. 3.1), pass-through
           completion and live-set widths (Def. 3.2, Lemma 3.3, Sec. 4.2).
  reach    Boolean-semiring fixpoint x <- x OR (M (x) x), textbook BFS, and the
           tropical fixpoint x <- min(x, M (x) x) (Bellman-Ford).

Parity status: every public function here is pinned by a ``-m "not gpu"``
test against the pages' worked example, a library routine or brute force
(see tests/test_oracle_pins.py). No function is "parity unpinned".
"""
from . import direct, grammar, reach  # noqa: F401
