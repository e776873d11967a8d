"""Oracle package: TEST INFRASTRUCTURE ONLY.

A plain, slow, float64 CPU reference of the pruned-KV decode path, used by the
test suite, the package smoke check and the benchmark's CPU legs. The
library's GPU path never imports it.

Two implementations of the same functions, written independently:

* the C++ one (oracle/kvp_oracle.cpp, through oracle/cpp.py), threaded with
  std::thread over (batch, kv head) units and scorer rows on every host
  core. ``import oracle`` gives this one.
* the numpy one (oracle/kvp_oracle.py), kept as a cross-check: the CPU
  pins run against both, and a test compares them on the same inputs.
"""
from . import cpp as cpp_impl  # noqa: F401
from . import kvp_oracle as numpy_impl  # noqa: F401
from .cpp import *  # noqa: F401,F403
from .kvp_oracle import CapacityError, PagedCache, QuantPagedCache  # noqa: F401
