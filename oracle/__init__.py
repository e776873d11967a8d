"""Oracle package: TEST INFRASTRUCTURE ONLY.

A plain float64 CPU reference of the pruned-KV decode path, used by the test
suite, the package smoke check and the benchmark's CPU-baseline leg. The
library's GPU path never imports it.
"""
from .kvp_oracle import *  # noqa: F401,F403
from .kvp_oracle import CapacityError, PagedCache  # noqa: F401
