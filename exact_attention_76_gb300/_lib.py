"""ctypes binding of libfa_gb300.so: argument marshalling only.

Every function here has the name of the C entry point it calls (include/fa.h)
and passes raw device pointers taken from torch tensors plus the current
stream.  There is no fallback: if the library is missing or a call fails, a
RuntimeError says so.
"""
from __future__ import annotations

import ctypes
import os

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")

FA_OK = 0
STATUS_NAMES = {0: "FA_OK", 1: "FA_ERR_INVALID_ARG", 2: "FA_ERR_UNSUPPORTED", 3: "FA_ERR_ALIGNMENT",
                4: "FA_ERR_LAUNCH", 5: "FA_ERR_TIMEOUT", 6: "FA_ERR_WORKSPACE", 7: "FA_ERR_KERNEL_CONFIG"}

# (name, argtypes, restype) for every symbol include/fa.h declares.
_P, _I, _F, _Z, _U = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t, ctypes.c_uint
_L = ctypes.c_longlong
SIGNATURES = {
    "fa_fwd": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_bwd_workspace_size": ([_I, _I, _I, _I], _Z),
    "fa_bwd": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_bwd_preprocess": ([_P, _P, _P, _P, _I, _I, _I, _I, _P], _I),
    "fa_bwd_main": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_bwd_dq_convert": ([_P, _P, _I, _I, _I, _I, _F, _P], _I),
    "fa_fwd_fp8": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_status_string": ([_I], ctypes.c_char_p),
    "fa_device_error": ([_P], _I),
    "fa_debug_wait_timeout": ([_U, _P], _I),
    "fa_fwd_gqa": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_bwd_gqa": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _I, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_fp8_quantize": ([_P, _I, _I, _P, _P, _L, _I, _P], _I),
    "fa_bwd_noalloc": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_fwd_fp8_blocks": ([_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_fp8_quantize_blocks": ([_P, _I, _I, _I, _P, _P, _I, _I, _I, _P], _I),
    "fa_fwd_window": ([_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_bwd_window": ([_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _Z, _I, _I, _I, _I, _I, _I, _F, _P], _I),
    "fa_measure_ex2_rate_scratch_size": ([], _Z),
    "fa_measure_ex2_rate": ([_P, _P, _Z, _P], _I),
    "fa_debug_exp2_poly": ([_P, _P, _L, _I, _P], _I),
    "fa_decode_workspace_size": ([_I, _I, _I, _I, _I], _Z),
    "fa_bwd_gqa_workspace_size": ([_I, _I, _I, _I, _I], _Z),
    "fa_decode": ([_P, _P, _P, _P, _P, _P, _Z, _I, _I, _I, _I, _I, _F, _P], _I),
}

_lib = None


def load(path: str = LIB_PATH):
    """Loads the shared library (building nothing) and binds its signatures."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: build it with `python -m exact_attention_76_gb300.build` "
                           "(the CUDA path has no fallback)")
    lib = ctypes.CDLL(path)
    for name, (args, res) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


class FaError(RuntimeError):
    def __init__(self, fn: str, status: int):
        self.status = status
        name = STATUS_NAMES.get(status, str(status))
        super().__init__(f"{fn} returned {name}")


def check(fn: str, status: int) -> None:
    if status != FA_OK:
        raise FaError(fn, status)
