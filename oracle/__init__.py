"""CPU fp64 oracle of the fused LM-head + CE + KL distillation loss.

Test infrastructure only: imported by the test suite, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; never by the CUDA library.
"""
from . import kd_oracle  # noqa: F401
