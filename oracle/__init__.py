"""CPU oracle for the allreduce schedules.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously correct
simulation of every allreduce schedule the engine implements.  Only the tests,
``__graft_entry__.smoke()`` and the CPU-baseline / reference legs of
``bench.py`` may import it.  The product path (``collective_reduction_gb300``
and its CUDA library) never imports, links or calls anything here, and this
package never imports the product.

Layout:
  elementops  the element operation (sum / prod / max / min over int32,
              fp32 and bf16) and the bf16 round-to-nearest-even conversion
  chunking    the ceil chunk split
  schedules   literal step-by-step simulations of each schedule, with the
              step / byte / combine counters they imply
  direct      the plain definition of the result (brute-force reduction)

Every schedule simulation builds each step's messages from the pre-step state
and then applies them, exactly as the pages describe rounds of simultaneous
sends.  Values can be numeric NumPy arrays or symbolic expression trees
(``elementops.Symbolic``), so the same code yields both results and the exact
reduction order.

Parity status: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` (closed forms, brute force, page examples, special
cases).  The one reading left unpinned for floats is the relative order of
recursive-doubling distances (the pages do not fix it); integer results and
step / byte counts are pinned for it.
"""

from . import chunking, direct, elementops, schedules  # noqa: F401
from .elementops import Arith, Symbolic, bf16_to_f32, f32_to_bf16_rne  # noqa: F401
from .schedules import ALGOS, run  # noqa: F401
