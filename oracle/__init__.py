"""fp64 CPU oracle of the CSA hot path (test infrastructure only).

Imported only by the tests, the smoke check and the CPU-baseline leg of the
benchmark.  The product library never imports it.
"""
from .csa_oracle import *  # noqa: F401,F403
