"""fp64 CPU oracle for quantized KV-cache decode attention (test infrastructure).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference
arm use this package; the CUDA library never imports it.
"""
from .kvq_oracle import *  # noqa: F401,F403
from .kvq_oracle import ZERO_CLAMPED, NONFINITE, ZERO_LIMIT  # noqa: F401
