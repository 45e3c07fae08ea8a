"""cattn: pluggable-map attention (Yat, s^tau, softmax) for GB300: forward and backward.

The compute path is the C-ABI library libcattn.so (hand-written sm_103a CUDA,
see include/cattn.h); this package holds its build script, the ctypes binding
and the seeded workload generators.
"""
from .attention import (backward, check_status, forward, forward_entropy, key_norms,  # noqa: F401
                        make_problem, row_stats,
                        tau_star, workspace_bytes)
from .native import CattnError  # noqa: F401
