"""Float64 CPU oracle for closed-form cross-model KV-cache transfer.

TEST INFRASTRUCTURE ONLY.  Nothing in the product package imports, links or runs
this code; only the tests, the smoke check and the benchmark's CPU-baseline leg
do.  It shares no code with the CUDA path: it is written from the pages'
formulas in plain NumPy float64, and it is pinned by the CPU tests to what the
pages and the mathematics fix (identities, closed forms, library special cases,
brute force on tiny inputs and the pages' printed sizes).

Parity status per function is listed in the docstring of `kvb_oracle`.
"""
from .kvb_oracle import *  # noqa: F401,F403
