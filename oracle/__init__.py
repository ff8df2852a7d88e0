"""Float64 CPU oracle for the MoE layer forward (test infrastructure only).

Only the tests, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The library's product path never does.
"""

from . import moe_oracle  # noqa: F401
