"""fp64 CPU oracle for exact attention.  TEST INFRASTRUCTURE ONLY: imported by tests/,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``, never by the library."""
from .attention import (allowed, backward, forward, merge_stats, online_attention,  # noqa: F401
                        probabilities, stats)
