"""ctypes binding of libhc_gr.so (the C ABI in include/hc_gr.h).

Argument marshalling only: every step of the operation runs in the CUDA
library.  Importing this module raises if the library has not been built;
there is no fallback.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libhc_gr.so")

OK, ERR_INVALID_ARG, ERR_UNSUPPORTED, ERR_ALIAS, ERR_CUDA, ERR_TIMEOUT = range(6)
PATH_AUTO, PATH_DECODE, PATH_PREFILL = range(3)

EXPORTS = ("hc_gr_create", "hc_gr_forward", "hc_gr_forward_ex", "hc_gr_check",
           "hc_gr_destroy", "hc_gr_strerror", "hc_gr_last_cuda_error", "hc_gr_forward_noalloc",
           "hc_gr_combine", "hc_gr_mix", "hc_gr_noalloc_check")

MAX_TOKENS = 1 << 30   # HC_GR_MAX_TOKENS: largest M and max_M
MAX_WIDTH = 1 << 30    # HC_GR_MAX_WIDTH: largest K = HC * HS

_vp = ctypes.c_void_p
_fp = ctypes.c_void_p   # float* passed as an address


class Args(ctypes.Structure):
    """Mirror of struct hc_gr_args."""

    _fields_ = [
        ("M", ctypes.c_int64),
        ("HC", ctypes.c_int32), ("HS", ctypes.c_int32), ("r", ctypes.c_int32),
        ("eps", ctypes.c_float),
        ("R", _vp), ("y", _vp), ("inj", _fp), ("ld_inj", ctypes.c_int64),
        ("Wnorm", _vp), ("Wd", _vp), ("Wi", _vp), ("Wdi", _vp),
        ("n_pad", ctypes.c_int32), ("fold_w", ctypes.c_int32),
        ("Wu", _vp), ("R2", _vp), ("rrms", _fp), ("inj_next", _fp), ("x", _vp), ("lora", _fp),
        ("force_path", ctypes.c_int32), ("debug_fault", ctypes.c_int32),
        ("pdl", ctypes.c_int32),
        ("wnorm_hs", ctypes.c_int32),
    ]


class HcGrError(RuntimeError):
    def __init__(self, status: int, msg: str):
        super().__init__(f"hc_gr status {status}: {msg}")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build the CUDA library first "
            "(python -c 'import __graft_entry__ as g; g.build()')")
    lib = ctypes.CDLL(path)
    lib.hc_gr_create.argtypes = [ctypes.POINTER(_vp), ctypes.c_int, ctypes.c_int64,
                                 ctypes.c_int, ctypes.c_int, ctypes.c_int]
    lib.hc_gr_create.restype = ctypes.c_int
    lib.hc_gr_forward.argtypes = [_vp, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                  ctypes.c_float] + [_vp] * 12 + [_vp]
    lib.hc_gr_forward.restype = ctypes.c_int
    lib.hc_gr_forward_ex.argtypes = [_vp, ctypes.POINTER(Args), _vp]
    lib.hc_gr_forward_ex.restype = ctypes.c_int
    lib.hc_gr_check.argtypes = [_vp, _vp]
    lib.hc_gr_check.restype = ctypes.c_int
    lib.hc_gr_destroy.argtypes = [_vp]
    lib.hc_gr_destroy.restype = ctypes.c_int
    lib.hc_gr_strerror.argtypes = [ctypes.c_int]
    lib.hc_gr_strerror.restype = ctypes.c_char_p
    lib.hc_gr_last_cuda_error.argtypes = [_vp]
    lib.hc_gr_last_cuda_error.restype = ctypes.c_char_p
    lib.hc_gr_forward_noalloc.argtypes = [ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                          ctypes.c_float] + [_vp] * 12 + [_vp]
    lib.hc_gr_forward_noalloc.restype = ctypes.c_int
    lib.hc_gr_noalloc_check.argtypes = [_vp]
    lib.hc_gr_noalloc_check.restype = ctypes.c_int
    lib.hc_gr_combine.argtypes = [_vp, ctypes.c_int64, ctypes.c_int, ctypes.c_int, _vp, _vp, _vp,
                                  ctypes.c_int64, _vp, _vp]
    lib.hc_gr_combine.restype = ctypes.c_int
    lib.hc_gr_mix.argtypes = [_vp, ctypes.c_int64, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                              ctypes.c_float] + [_vp] * 9 + [_vp]
    lib.hc_gr_mix.restype = ctypes.c_int
    return lib


_LIB = None


def lib() -> ctypes.CDLL:
    global _LIB
    if _LIB is None:
        _LIB = load()
    return _LIB


def strerror(status: int) -> str:
    return lib().hc_gr_strerror(status).decode()
