"""CPU oracle for packed, question-isolated attention.

TEST INFRASTRUCTURE ONLY: imported by ``tests/``, ``__graft_entry__.smoke()``
and the CPU-baseline legs of ``bench.py`` -- never by the product package.
"""
from . import brute, kev_oracle  # noqa: F401
