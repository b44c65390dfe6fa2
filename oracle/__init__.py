"""Plain fp64 CPU oracle for Quest sparse decode and SnapKV eviction.

TEST INFRASTRUCTURE ONLY. The test-suite, the package smoke check and the
bench's CPU-baseline leg are the only code allowed to import it. The CUDA
library and its Python binding never import it, and it imports nothing from
them: the two share no kernels, helpers, tables or constants. Only the
seeded input generators in ``synth`` serve both sides.

Every step is written from its definition, in numpy float64, with inputs
upcast exactly from bf16. Where the SparseEngine pages leave a step open, the
module docstring of the step says which reading it takes.

Parity pins: every function here is pinned by the ``-m "not gpu"`` tests in
``tests/test_oracle_*.py`` against brute force, closed forms, library
routines (numpy/torch/scipy) and invariants. The synthetic data recipe and
the group-sum reading of the Quest bound are pinned only by internal
consistency, because the pages print no worked example (parity unpinned for
those two readings; every computed step is pinned).
"""
from . import quest, snapkv, budgets  # noqa: F401
