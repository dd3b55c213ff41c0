"""CPU oracle of the ECHO decode hot path: TEST INFRASTRUCTURE ONLY.

The oracle is the plain C++ library in echo_oracle.cpp, loaded through cpp_oracle
(built on first use by oracle/build.py).  numpy_oracle is an independent numpy
restatement of the same definitions, kept as a cross-check that must agree with it."""
from .cpp_oracle import *  # noqa: F401,F403
from . import numpy_oracle  # noqa: F401
