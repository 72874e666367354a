"""CPU oracle for MLA. TEST INFRASTRUCTURE ONLY.

Plain float64 numpy (``mla_ref``) and pure-Python scalar loops (``brute``) restating the
per-head formulas of the MLA pages. Only the tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import it; the CUDA library and its Python binding
never do, and the two share no code (only the seeded input generator ``mla_inputs``).

Parity status: every function here is pinned by ``tests/test_oracle.py`` (closed forms,
invariants, brute force and the absorbed/explicit equivalence); none is "parity unpinned".
"""
from . import mla_ref, brute  # noqa: F401
