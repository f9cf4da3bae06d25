"""CPU oracle for the MXFP8 norm-quant + GEMM path (test infrastructure only).

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  See ``oracle/mx_oracle.py``.
"""
from .mx_oracle import *  # noqa: F401,F403
from .mx_oracle import __all__  # noqa: F401
