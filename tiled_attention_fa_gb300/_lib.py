"""ctypes loader for the C-ABI library ``libfa_gb300.so`` (built in-tree).

There is no fallback: if the library is missing or fails to load, every call
raises.  Build it with ``python -m tiled_attention_fa_gb300.build``.
"""

from __future__ import annotations

import ctypes
import os
import re

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "libfa_gb300.so")
HEADER = os.path.join(os.path.dirname(HERE), "include", "fa.h")

FA_OK, FA_ERR_INVALID_ARG, FA_ERR_UNSUPPORTED, FA_ERR_CUDA, FA_ERR_DEVICE_TIMEOUT = range(5)
FA_ERR_SCRATCH_TOO_SMALL = 5
FA_NOALLOC_SCRATCH_BYTES = 64 << 20
FA_F16, FA_BF16 = 0, 1

_lib = None

_vp = ctypes.c_void_p
_i = ctypes.c_int
_SIGS = {
    "fa_fwd": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _vp], _i),
    "fa_fwd_kv": ([_vp, _vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _i, _i, _i, _vp], _i),
    "fa_fwd_fp8": ([_vp] * 3 + [ctypes.c_float] * 3 + [_vp, _vp] + [_i] * 8 + [_vp], _i),
    "fa_bwd_preprocess": ([_vp, _vp, _vp, _vp, _i, _i, _i, _i, _i, _vp], _i),
    "fa_bwd_kv": ([_vp] * 11 + [_i] * 9 + [_vp], _i),
    "fa_bwd_workspace_size": ([_i, _i, _i, _i], ctypes.c_size_t),
    "fa_bwd": ([_vp] * 11 + [_i] * 8 + [_vp], _i),
    "fa_bwd_main": ([_vp] * 9 + [_i] * 8 + [_vp], _i),
    "fa_bwd_postprocess": ([_vp, _vp] + [_i] * 5 + [_vp], _i),
    "fa_bwd_noalloc": ([_vp] * 10 + [_i] * 7 + [_vp], _i),
    "fa_decode_workspace_size": ([_i] * 6, ctypes.c_size_t),
    "fa_decode": ([_vp] * 6 + [ctypes.c_size_t] + [_i] * 8 + [_vp], _i),
    "fa_decode_slices": ([_vp] * 4 + [ctypes.c_size_t] + [_i] * 8 + [_vp], _i),
    "fa_decode_merge": ([_vp, ctypes.c_size_t, _vp, _vp] + [_i] * 7 + [_vp], _i),
    "fa_check_device_error": ([_vp], _i),
    "fa_last_error_site": ([], ctypes.c_uint),
    "fa_selftest_bounded_wait": ([ctypes.c_ulonglong, _vp], _i),
    "fa_status_string": ([_i], ctypes.c_char_p),
    "fa_version": ([], ctypes.c_char_p),
}


class FAError(RuntimeError):
    """A non-zero fa_status returned by the library."""

    def __init__(self, fn: str, status: int):
        self.status = status
        text = load().fa_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{fn} failed: {text} (status {status})")


def header_functions() -> list:
    """Names of the functions declared in include/fa.h."""
    with open(HEADER) as fh:
        src = fh.read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return re.findall(r"\b(fa_[a-z_]+)\s*\(", src)


def load():
    """Load (once) and return the library with argument types declared."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with "
                           "`python -m tiled_attention_fa_gb300.build` (needs nvcc)")
    lib = ctypes.CDLL(LIB_PATH)
    for name, (args, res) in _SIGS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def check(fn: str, status: int) -> None:
    if status != FA_OK:
        raise FAError(fn, status)
