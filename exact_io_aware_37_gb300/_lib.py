"""ctypes loader for libfa_gb300.so (argument types only; no arithmetic)."""

import ctypes
import os

from . import build as _build

FA_BF16, FA_F32, FA_F16 = 0, 1, 2
STATUS = {
    0: "FA_OK", -1: "FA_ERR_INVALID", -2: "FA_ERR_UNSUPPORTED", -3: "FA_ERR_ALIGN",
    -4: "FA_ERR_CUDA", -5: "FA_ERR_TIMEOUT", -6: "FA_ERR_WORKSPACE",
}

_LIB = None

_c = ctypes
_vp, _int, _f, _sz = _c.c_void_p, _c.c_int, _c.c_float, _c.c_size_t

SIGNATURES = {
    "fa_fwd": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _f, _int, _vp, _int, _int, _vp]),
    "fa_bwd_workspace_size": (_sz, [_int, _int, _int, _int, _vp, _int, _int]),
    "fa_bwd": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _f, _int,
                      _vp, _int, _int, _vp, _sz, _vp]),
    "fa_bwd_static_ws": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _f, _int,
                                _vp, _int, _int, _vp]),
    "fa_strerror": (_c.c_char_p, [_int]),
    "fa_get_last_device_error": (_int, [_vp]),
    "fa_set_wait_limit_ns": (None, [_c.c_ulonglong]),
    "fa_selftest_wait_timeout": (_int, [_vp]),
    "fa_selftest_tile": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _int, _vp]),
    "fa_path_name": (_c.c_char_p, [_int, _int]),
    "fa_launch_count": (_c.c_ulonglong, []),
    "fa_schedule_preview": (_int, [_int, _vp, _int, _int, _int, _int, _int, _int, _vp, _vp, _int, _vp]),
    "fa_last_error_detail": (_c.c_char_p, []),
    "fa_bwd_time_main_kernel": (None, [_vp, _vp]),
    "fa_fwd_dropout": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _f, _int, _vp, _int, _int, _f,
                              _c.c_uint64, _c.c_uint32, _vp]),
    "fa_bwd_dropout": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _f, _int,
                              _vp, _int, _int, _f, _c.c_uint64, _c.c_uint32, _vp, _sz, _vp]),
    "fa_bwd_deterministic": (_int, [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _f, _int,
                                    _vp, _int, _int, _f, _c.c_uint64, _c.c_uint32, _vp, _sz, _vp]),
    "fa_decode_workspace_size": (_sz, [_int, _int, _int, _int, _int, _int]),
    "fa_probe_ex2_rate": (_int, [_int, _c.POINTER(_c.c_double), _vp]),
    "fa_decode": (_int, [_vp, _vp, _vp, _vp, _vp, _int, _int, _int, _int, _int, _f, _int, _int, _vp, _sz, _vp]),
}


def library_path():
    return _build.LIB_PATH


def lib():
    """The loaded library.  Fails loudly when it has not been built: there is
    no fallback implementation."""
    global _LIB
    if _LIB is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m exact_io_aware_37_gb300.build` "
                "(there is no fallback path)")
        handle = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            fn = getattr(handle, name)
            fn.restype = res
            fn.argtypes = args
        _LIB = handle
    return _LIB


class FAError(RuntimeError):
    def __init__(self, status, where):
        self.status = status
        msg = lib().fa_strerror(status).decode()
        detail = lib().fa_last_error_detail().decode() if status == -4 else ""
        super().__init__(f"{where}: {STATUS.get(status, status)} ({msg})" + (f" [{detail}]" if detail else ""))
