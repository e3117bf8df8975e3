"""ctypes binding of libkd (include/kd.h). Argument marshalling only.

The library is the in-tree lib/libkd.so, built by build.py (it is rebuilt
when a source is newer). If it cannot be built or loaded, importing raises:
there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os

from . import build as _build

KD_OK = 0
KD_ERR_INVALID_ARG = 1
KD_ERR_UNSUPPORTED = 2
KD_ERR_WORKSPACE = 3
KD_ERR_CUDA = 4
KD_ERR_DEVICE_TIMEOUT = 5
KD_ERR_BAD_ID = 6
KD_BF16 = 0
KD_F32 = 1

# name -> (restype, argtypes); every symbol declared in include/kd.h,
# include/kd_testing.h and include/kd_profile.h.
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
SIGNATURES = {
    "kd_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "kd_version": (ctypes.c_int, []),
    "kd_topk_workspace_size": (_SZ, [_I64, _I64, _I32, _I32]),
    "kd_topk_cache": (ctypes.c_int, [_P, _I32, _I64, _I64, _I64, _I32, _P, _P, _P, _SZ, _P]),
    "kd_topk_cache_noalloc": (ctypes.c_int, [_P, _I32, _I64, _I64, _I64, _I32, _P, _P, _P]),
    "kd_fused_kl_workspace_size": (_SZ, [_I64, _I64, _I32, _I64]),
    "kd_fused_kl_workspace_size_ex": (_SZ, [_I64, _I64, _I32, _I64, _I32]),
    "kd_teacher_topk_workspace_size": (_SZ, [_I64, _I64, _I32, _I64]),
    "kd_teacher_topk_cache": (ctypes.c_int, [_P, _P, _I64, _I64, _I64, _I32, _I64, _P, _P, _P, _SZ, _P]),
    "kd_fused_kl_fwd": (
        ctypes.c_int,
        [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _I64, _P, _P, _P, _P, _SZ, _P],
    ),
    "kd_fused_kl_bwd": (
        ctypes.c_int,
        [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I64, ctypes.c_float, _P, _P, _P, _I32, _P, _SZ, _P],
    ),
    "kd_fused_kl_fwdbwd": (
        ctypes.c_int,
        [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _I64, ctypes.c_float, _P, _P, _P, _P, _P, _P, _I32, _P, _SZ, _P],
    ),
    "kd_fused_kl_fwd_ex": (
        ctypes.c_int,
        [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _I64, _P, _P, _P, _P, _P, _SZ, _P],
    ),
    "kd_fused_kl_bwd_ex": (
        ctypes.c_int,
        [_P, _P, _P, _P, _P, _I64, _I64, _I64, _I32, _I64, ctypes.c_float, _P, _P, _P, _I32, _P, _P, _SZ, _P],
    ),
    "kd_fused_kl_fwdbwd_ex": (
        ctypes.c_int,
        [_P, _P, _P, _P, _I64, _I64, _I64, _I32, _I64, ctypes.c_float, _P, _P, _P, _P, _P, _P, _I32, _P, _P, _SZ,
         _P],
    ),
    "kd_read_device_status": (ctypes.c_int, [_P, _P]),
    "kd_cache_create": (ctypes.c_int, [ctypes.c_char_p, _I64, _I32, _P]),
    "kd_cache_append": (ctypes.c_int, [_P, _P, _P, _I64]),
    "kd_cache_open": (ctypes.c_int, [ctypes.c_char_p, _P, _P, _P, _P]),
    "kd_cache_read": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
    "kd_cache_close": (ctypes.c_int, [_P]),
    "kd_test_gemm": (ctypes.c_int, [_P, _P, _P, _I64, _I64, _I64, _I32, _I32, _I32, _P, _P]),
    "kd_test_wait_timeout": (ctypes.c_int, [_I64, _P, _P]),
    "kd_test_set_gemm_tiles": (ctypes.c_int, [_I32, _I32]),
    "kd_test_get_gemm_tiles": (ctypes.c_int, [_P, _P]),
    "kd_test_set_topk_force_exact": (ctypes.c_int, [_I32]),
    "kd_profile_begin": (ctypes.c_int, []),
    "kd_profile_end": (ctypes.c_int, [_P, _I32, _P]),
}


class KLOptions(ctypes.Structure):
    """Mirror of kd_kl_options in include/kd.h."""

    _fields_ = [("temperature", ctypes.c_float), ("mask", ctypes.c_void_p), ("mean_over_mask", ctypes.c_int32),
                ("dH_bf16", ctypes.c_int32), ("group", ctypes.c_int32)]


class ProfEntry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char * 32), ("launches", ctypes.c_int32), ("total_ms", ctypes.c_double)]


class KDError(RuntimeError):
    def __init__(self, fn: str, code: int):
        super().__init__("%s failed: %s (%d)" % (fn, status_string(code), code))
        self.code = code


_lib = None


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) libkd and bind every exported symbol."""
    global _lib
    if _lib is not None and path is None:
        return _lib
    if path is None:
        path = _build.build()
    if not os.path.exists(path):
        raise RuntimeError("libkd not found at %s" % path)
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        f = getattr(lib, name)
        f.restype = res
        f.argtypes = args
    if path == _build.LIB:
        _lib = lib
    return lib


def lib() -> ctypes.CDLL:
    return load()


def status_string(code: int) -> str:
    return lib().kd_status_string(int(code)).decode()


def profile_begin() -> None:
    lib().kd_profile_begin()


def profile_end() -> dict:
    """{kernel name: (launches, total device ms)} since profile_begin()."""
    buf = (ProfEntry * 16)()
    n = ctypes.c_int32(0)
    check("kd_profile_end", lib().kd_profile_end(buf, 16, ctypes.byref(n)))
    return {buf[i].name.decode(): (int(buf[i].launches), float(buf[i].total_ms)) for i in range(n.value)}


def set_gemm_tiles(cta2: int = -1, wide: int = -1) -> None:
    """kd_test_set_gemm_tiles (include/kd_testing.h): -1 restores a default."""
    check("kd_test_set_gemm_tiles", lib().kd_test_set_gemm_tiles(int(cta2), int(wide)))


def get_gemm_tiles() -> tuple:
    """(cta2, wide) switch values of kd_test_get_gemm_tiles (-1 = default)."""
    a, b = ctypes.c_int32(0), ctypes.c_int32(0)
    check("kd_test_get_gemm_tiles", lib().kd_test_get_gemm_tiles(ctypes.byref(a), ctypes.byref(b)))
    return int(a.value), int(b.value)


def set_topk_force_exact(on: bool) -> None:
    """kd_test_set_topk_force_exact (include/kd_testing.h)."""
    check("kd_test_set_topk_force_exact", lib().kd_test_set_topk_force_exact(1 if on else 0))


def check(fn: str, code: int) -> None:
    if code != KD_OK:
        raise KDError(fn, code)
