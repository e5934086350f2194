"""ctypes declarations of the C ABI in include/bwd.h (argument marshalling only).

Loading fails loudly when ``libbwd.so`` has not been built: there is no
fallback implementation of any step.
"""

from __future__ import annotations

import ctypes
import os

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libbwd.so")

BWD_OK = 0
BWD_ERR_INVALID_ARG = 1
BWD_ERR_UNSUPPORTED_DTYPE = 2
BWD_ERR_CUDA = 3

BWD_MAP_SIGNED = 0
BWD_MAP_UNSIGNED = 1
BWD_F32 = 0
BWD_BF16 = 1
BWD_F16 = 2
BLOCK = 2048


class AdamHParams(ctypes.Structure):
    """Mirror of ``bwd_adam_hparams``."""

    _fields_ = [
        ("lr", ctypes.c_float),
        ("beta1", ctypes.c_float),
        ("beta2", ctypes.c_float),
        ("eps", ctypes.c_float),
        ("weight_decay", ctypes.c_float),
        ("step", ctypes.c_int64),
    ]


class BwdError(RuntimeError):
    def __init__(self, status: int, where: str, detail: str):
        self.status = status
        super().__init__(f"{where}: {detail}")


_vp = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int32
_int = ctypes.c_int
_pp = ctypes.POINTER(ctypes.c_void_p)

_SIGNATURES = {
    "bwd_num_blocks": (_i64, [_i64]),
    "bwd_build_map": (_int, [_int, _vp, _vp]),
    "bwd_init": (_int, []),
    "bwd_quantize_blockwise": (_int, [_vp, _i64, _int, _vp, _vp, _vp]),
    "bwd_dequantize_blockwise": (_int, [_vp, _vp, _i64, _int, _vp, _vp]),
    "bwd_state_init": (_int, [_vp, _vp, _vp, _vp, _i64, _vp]),
    "bwd_adam8bit_step": (_int, [_vp, _vp, _int, _vp, _vp, _vp, _vp, _i64, ctypes.POINTER(AdamHParams), _vp]),
    "bwd_adam8bit_step_multi": (
        _int,
        [_i32, _pp, _pp, _int, _pp, _pp, _pp, _pp, ctypes.POINTER(_i64), ctypes.POINTER(AdamHParams), _vp],
    ),
    "bwd_adam8bit_step_multi_ex": (
        _int,
        [_i32, _pp, _int, _pp, _int, _pp, _pp, _pp, _pp, ctypes.POINTER(_i64), ctypes.POINTER(AdamHParams), _vp],
    ),
    "bwd_zero_shard": (_int, [_i32, _vp, _i32, _i32, _vp, _vp, _vp, _vp, _vp]),
    "bwd_embedding_init": (_int, [_vp, _i64, _i64, _vp, _vp]),
    "bwd_embedding_xavier_bound": (ctypes.c_float, [_i64, _i64]),
    "bwd_embedding_forward": (
        _int, [_vp, _i64, _vp, _i64, _i64, _vp, _vp, ctypes.c_float, _vp, _vp, _vp, _vp]),
    "bwd_embedding_backward": (
        _int, [_vp, _i64, _vp, _i64, _i64, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp]),
    "bwd_check_device": (_int, [_vp]),
    "bwd_selftest_bounded_wait": (_int, [_vp]),
    "bwd_status_string": (ctypes.c_char_p, [_int]),
    "bwd_last_error": (ctypes.c_char_p, []),
}

_lib = None


def load() -> ctypes.CDLL:
    """Load ``libbwd.so`` once; raise ImportError if it is missing."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise ImportError(
            f"{LIB_PATH} is not built; run `python -m block_wise_dynamic_gb300.build` "
            "(needs nvcc) -- there is no fallback implementation"
        )
    lib = ctypes.CDLL(LIB_PATH)
    for name, (res, args) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def check(status: int, where: str) -> None:
    """Raise BwdError for a non-zero status, with the library's detail."""
    if status != BWD_OK:
        lib = load()
        detail = lib.bwd_last_error().decode() or lib.bwd_status_string(status).decode()
        raise BwdError(status, where, f"{lib.bwd_status_string(status).decode()}: {detail}")
