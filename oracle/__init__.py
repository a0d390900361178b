"""OSCAR INT2 paged-KV decode: plain CPU oracle.

TEST INFRASTRUCTURE. This package is a slow, obviously-correct numpy
restatement of what the decode path computes, used only to check the CUDA
library. Only the test suite, the package's smoke check and the benchmark's
CPU-baseline leg may import it; the product library never calls it and shares
no code with it.

Parity pins: every function here is pinned by tests in ``tests/test_oracle_pins.py``
(closed forms, invariants, brute force). No function is "parity unpinned".
"""
from .oscar_oracle import *  # noqa: F401,F403
