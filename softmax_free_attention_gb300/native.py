"""ctypes binding of libcattn.so (the C ABI in include/cattn.h).

Argument marshalling only: every step of the forward runs in the library's
CUDA kernels.  If the library is missing this module raises instead of
falling back to anything else.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libcattn.so")

SOFTMAX, YAT, STAU = 0, 1, 2
F32, BF16 = 0, 1
FLAG_NORMS_READY = 1
FLAG_TEST_STALL = 2  # testing only: the forward kernel waits on a barrier nothing completes

OK = 0
ERR_INVALID_ARG = 1
ERR_SHAPE = 2
ERR_UNSUPPORTED = 3
ERR_CUDA = 4
ERR_TIMEOUT = 5
ERR_SCRATCH_LIMIT = 6

# every symbol include/cattn.h declares
EXPORTS = ("cattn_version", "cattn_error_string", "cattn_workspace_bytes", "cattn_validate",
           "cattn_key_norms", "cattn_forward", "cattn_forward_entropy", "cattn_forward_noalloc",
           "cattn_forward_host_workspace_bytes", "cattn_forward_host",
           "cattn_tau_star_workspace_bytes", "cattn_tau_star", "cattn_row_stats_workspace_bytes",
           "cattn_row_stats", "cattn_backward_workspace_bytes", "cattn_backward",
           "cattn_check_status")


class Problem(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int), ("h", ctypes.c_int), ("hkv", ctypes.c_int),
        ("Tq", ctypes.c_int), ("Tk", ctypes.c_int), ("dk", ctypes.c_int), ("dv", ctypes.c_int),
        ("dtype", ctypes.c_int), ("causal", ctypes.c_int), ("scale", ctypes.c_float),
        ("flags", ctypes.c_int), ("yat_m", ctypes.c_int),
    ]


class CattnError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        super().__init__(f"{what}: {error_string(status)} (status {status})" if what
                         else f"{error_string(status)} (status {status})")


_lib = None


def load():
    """Load libcattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"libcattn.so not found at {LIB_PATH}; build it with "
            "`python -m softmax_free_attention_gb300.build` (nvcc, sm_103a)")
    lib = ctypes.CDLL(LIB_PATH)
    vp, i, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    pp = ctypes.POINTER(Problem)
    lib.cattn_version.argtypes = []
    lib.cattn_version.restype = i
    lib.cattn_error_string.argtypes = [i]
    lib.cattn_error_string.restype = ctypes.c_char_p
    lib.cattn_workspace_bytes.argtypes = [i, pp]
    lib.cattn_workspace_bytes.restype = sz
    lib.cattn_validate.argtypes = [i, pp, vp, vp, vp, vp, vp, vp, vp, vp, sz]
    lib.cattn_validate.restype = i
    lib.cattn_key_norms.argtypes = [pp, vp, vp, sz, vp]
    lib.cattn_key_norms.restype = i
    lib.cattn_forward.argtypes = [i, pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.cattn_forward.restype = i
    lib.cattn_forward_entropy.argtypes = [i, pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.cattn_forward_entropy.restype = i
    lib.cattn_forward_noalloc.argtypes = [i, pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp]
    lib.cattn_forward_noalloc.restype = i
    lib.cattn_forward_host_workspace_bytes.argtypes = [i, pp, i]
    lib.cattn_forward_host_workspace_bytes.restype = sz
    lib.cattn_forward_host.argtypes = [i, pp] + [vp] * 16 + [sz, i, vp, vp, vp]
    lib.cattn_forward_host.restype = i
    lib.cattn_tau_star_workspace_bytes.argtypes = [pp]
    lib.cattn_tau_star_workspace_bytes.restype = sz
    lib.cattn_tau_star.argtypes = [pp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.cattn_tau_star.restype = i
    lib.cattn_row_stats_workspace_bytes.argtypes = [i, pp]
    lib.cattn_row_stats_workspace_bytes.restype = sz
    lib.cattn_row_stats.argtypes = [i, pp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp]
    lib.cattn_row_stats.restype = i
    lib.cattn_backward_workspace_bytes.argtypes = [i, pp]
    lib.cattn_backward_workspace_bytes.restype = sz
    lib.cattn_backward.argtypes = [i, pp] + [vp] * 16 + [sz, vp]
    lib.cattn_backward.restype = i
    lib.cattn_check_status.argtypes = [vp]
    lib.cattn_check_status.restype = i
    _lib = lib
    return lib


def error_string(status: int) -> str:
    try:
        return load().cattn_error_string(int(status)).decode()
    except ImportError:
        return f"status {status}"


def check(status: int, what: str = "") -> None:
    if status != OK:
        raise CattnError(status, what)
