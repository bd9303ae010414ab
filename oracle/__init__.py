"""CPU oracle for the quantized projection matmul (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never does.
"""
from .qmm_oracle import *  # noqa: F401,F403
