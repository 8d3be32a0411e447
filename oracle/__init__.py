"""CPU oracle for the routed-expert hot path.

TEST INFRASTRUCTURE ONLY.  Only the test suite, the package smoke check and the
CPU-baseline leg of the benchmark may import this package.  The product library
never loads it, and it imports nothing from the product package.

The arithmetic lives in ``moe_oracle.cpp`` (plain C++; OpenMP over independent
outer loops where available, results independent of the thread count); this
module compiles it with the host C++ compiler and wraps it with ctypes/numpy.
"""

from .oracle import (  # noqa: F401
    Oracle,
    build_oracle,
    load_oracle,
)
