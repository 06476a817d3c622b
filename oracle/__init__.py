"""Float64 CPU oracle of paged-KV attention forward and of the work planner.

TEST INFRASTRUCTURE ONLY: the test suite, ``__graft_entry__.smoke()`` and the benchmark's
CPU-baseline leg are the only callers.  The CUDA library neither imports this package nor
shares any code with it.
"""
from . import attention, planner  # noqa: F401
