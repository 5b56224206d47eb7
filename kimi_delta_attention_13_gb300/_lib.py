"""ctypes loader for libkda_gb300.so: symbol signatures mirroring include/kda.h.

There is no fallback: if the library has not been built, loading raises.
"""
from __future__ import annotations

import ctypes
import os

from . import build as _build

KDA_OK = 0
KDA_BF16 = 0
KDA_F32 = 1
STATUS_NAMES = {
    0: "KDA_OK", 1: "KDA_ERR_INVALID_ARG", 2: "KDA_ERR_UNSUPPORTED_SHAPE", 3: "KDA_ERR_MISALIGNED",
    4: "KDA_ERR_CUDA", 5: "KDA_ERR_DEVICE_TIMEOUT", 6: "KDA_ERR_INDEX_RANGE", 7: "KDA_ERR_DEVICE_BOUNDS",
}

# name -> (restype, argtypes); every function declared in include/kda.h
_vp, _i32, _i64 = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64
_PREFILL_ARGS = [_vp, _vp, _vp, _vp, _vp, _vp, _i32, _i64, _i32, _i32, _i32, _i32, _i32, _vp, _vp,
                 _vp, _i32, _vp, _vp]
SIGNATURES = {
    "kda_abi_version": (ctypes.c_int, []),
    "kda_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kda_prefill": (ctypes.c_int, _PREFILL_ARGS),
    "kda_prefill_recurrent": (ctypes.c_int, _PREFILL_ARGS),
    "kda_prefill_precise": (ctypes.c_int, _PREFILL_ARGS),
    "kda_prefill_path": (ctypes.c_int, [_i32, _i32, _i32]),
    "kda_decode": (ctypes.c_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _i32, _i32, _i32, _i32, _i32, _i32,
                                   _vp]),
    "kda_state_copy": (ctypes.c_int, [_vp, _vp, _i64, _vp, _vp, _i64, _i64, _i32, _i32, _i32, _vp]),
    "kda_device_status": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int32), _vp]),
    "kda_diag_device_timeout": (ctypes.c_int, [_i64, _vp]),
    "kda_diag_bounds_check": (ctypes.c_int, [_i32, ctypes.POINTER(ctypes.c_int32), _vp]),
    "kda_diag_staged_handles": (ctypes.c_int, [ctypes.POINTER(ctypes.c_int64)]),
    "kda_premix": (ctypes.c_int, [_vp] * 7 + [_vp, _i32, _i64, _i32, _i32, ctypes.c_float, _i32]
                   + [_vp] * 5 + [_vp]),
    "kda_output_gate": (ctypes.c_int, [_vp, _i32, _vp, _i32, _vp, _i32, _i64, _vp]),
    "kda_cp_combine": (ctypes.c_int, [_vp, _vp, _vp, _i32, _i32, _i32, _vp, _vp, _vp]),
    "kda_cp_correct": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, _i32, _i64, _i32, _i32, _vp, _vp]),
    "kda_prefill_staged": (ctypes.c_int, [_vp] * 6 + [_i32, _i64, _i32, _i32, _i32, _vp] + [_vp] * 9
                           + [_i64, _i64, _vp]),
    "kda_prefill_staged_scratch": (ctypes.c_int64, [_vp, _i32, _i64, _i64]),
    "kda_prefill_staged_static": (ctypes.c_int, [_vp] * 6 + [_i32, _i64, _i32, _i32, _i32, _vp]
                                  + [_vp] * 8 + [_i64, _vp]),
}

_LIB = None


class KDAError(RuntimeError):
    def __init__(self, status: int, what: str = ""):
        self.status = status
        name = status_string(status) if _LIB is not None else STATUS_NAMES.get(status, str(status))
        super().__init__(f"{what}: {name}" if what else name)


def library_path() -> str:
    return _build.LIB_PATH


def load(path: str | None = None):
    """Load the built library (once).  Raises if it does not exist."""
    global _LIB
    if _LIB is not None:
        return _LIB
    path = path or library_path()
    if not os.path.exists(path):
        raise RuntimeError(
            f"libkda_gb300.so is not built ({path}); run `python -c \"import __graft_entry__ as g; "
            "g.build()\"` first.  There is no CPU fallback.")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _LIB = lib
    return lib


def status_string(status: int) -> str:
    return load().kda_status_string(int(status)).decode()


def check(status: int, what: str):
    if status != KDA_OK:
        raise KDAError(status, what)
