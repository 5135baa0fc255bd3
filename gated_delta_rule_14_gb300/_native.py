"""ctypes handle on libkla_gb300.so (the C ABI of include/kla.h).

Argument marshalling only: no arithmetic of the recurrence happens in Python.
If the library has not been built, loading fails loudly; there is no fallback.
"""
from __future__ import annotations

import ctypes
import os
import threading

from . import build as _build

KLA_OK = 0
KLA_ERR_INVALID_ARG = 1
KLA_ERR_UNSUPPORTED = 2
KLA_ERR_CUDA = 3
KLA_ERR_TIMEOUT = 4

KLA_DTYPE_F32 = 0
KLA_DTYPE_BF16 = 1
KLA_GATE_SCALAR = 0
KLA_GATE_CHANNEL = 1
KLA_BETA_KACZMARZ = 0
KLA_BETA_RAW = 1

_lock = threading.Lock()
_lib = None


class KlaError(RuntimeError):
    """A KLA C-ABI call returned a status other than KLA_OK."""

    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {status_string(status)}")


def library_path() -> str:
    return _build.LIB


def _declare(lib):
    vp, fp, i, sz = ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int, ctypes.c_size_t
    lib.kla_chunk_fwd.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, vp, fp,
                                  i, i, i, i, i, i, i, i, vp, sz, vp]
    lib.kla_chunk_fwd.restype = ctypes.c_int
    lib.kla_chunk_fwd_ex.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, vp, fp,
                                     i, i, i, i, i, i, i, i, i, ctypes.c_float, vp, sz, vp]
    lib.kla_chunk_fwd_ex.restype = ctypes.c_int
    lib.kla_chunk_fwd_workspace_size.argtypes = [i, i, i, i, i, i, i, i]
    lib.kla_chunk_fwd_workspace_size.restype = sz
    lib.kla_decode_step.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, vp, i, i, i, i, i, i, vp]
    lib.kla_decode_step.restype = ctypes.c_int
    lib.kla_decode_step_ex.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, vp, i, i, i, i, i, i, i,
                                       ctypes.c_float, vp]
    lib.kla_decode_step_ex.restype = ctypes.c_int
    lib.kla_chunk_fwd_host.argtypes = [vp, vp, vp, fp, fp, fp, vp, fp, vp, vp, vp, fp, fp, fp, vp, fp, ctypes.c_float,
                                       i, i, i, i, i, i, i, i, i, ctypes.c_float, i, vp]
    lib.kla_chunk_fwd_host.restype = ctypes.c_int
    lib.kla_chunk_bwd.argtypes = [vp, vp, vp, fp, fp, ctypes.c_float, fp, vp, fp, fp, fp, fp, fp, fp, fp,
                                  i, i, i, i, i, i, i, i, ctypes.c_float, vp, sz, vp]
    lib.kla_chunk_bwd.restype = ctypes.c_int
    lib.kla_chunk_bwd_workspace_size.argtypes = [i, i, i, i, i]
    lib.kla_chunk_bwd_workspace_size.restype = sz
    lib.kla_chunk_bwd_workspace_size_ex.argtypes = [i, i, i, i, i, i, i]
    lib.kla_chunk_bwd_workspace_size_ex.restype = sz
    lib.kla_selftest_wait_timeout.argtypes = [ctypes.c_uint, vp]
    lib.kla_selftest_wait_timeout.restype = ctypes.c_int
    lib.kla_device_status.argtypes = [vp]
    lib.kla_device_status.restype = ctypes.c_int
    lib.kla_status_string.argtypes = [ctypes.c_int]
    lib.kla_status_string.restype = ctypes.c_char_p
    lib.kla_abi_version.argtypes = []
    lib.kla_abi_version.restype = ctypes.c_int
    return lib


def lib():
    """Load libkla_gb300.so once; raises if it has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise RuntimeError(
                    f"KLA CUDA library not found at {path}; build it with "
                    "`python -c 'import __graft_entry__ as g; g.build()'` (needs nvcc)")
            _lib = _declare(ctypes.CDLL(path))
        return _lib


def status_string(status: int) -> str:
    return lib().kla_status_string(int(status)).decode()


def check(status: int, what: str) -> None:
    if status != KLA_OK:
        raise KlaError(status, what)
