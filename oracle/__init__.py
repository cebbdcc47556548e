"""CPU oracle (test infrastructure only).

Plain float64 restatements of what the CUDA path computes, used by ``tests/``,
``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``. The
product package never imports this package.
"""
from . import attention, burst_gap, moe  # noqa: F401
