"""ctypes view of libeas.so (the C ABI declared in include/eas.h)."""
from __future__ import annotations

import ctypes
import os

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libeas.so")

EAS_OK = 0
EAS_ERR_INVALID_ARG = 1
EAS_ERR_INVALID_SPANS = 2
EAS_ERR_UNSUPPORTED = 3
EAS_ERR_WORKSPACE = 4
EAS_ERR_CUDA = 5
EAS_ERR_TIMEOUT = 6
EAS_ERR_SPAN_CAPACITY = 7
EAS_ERR_INVALID_LAYOUT = 8

EAS_BF16 = 0
EAS_FP32 = 1
EAS_E4M3 = 2

EAS_ROWS_ACTIVE = 0
EAS_ROWS_SPAN = 1
EAS_REUSE_FWD_ROWS = 2

EAS_DEFAULT_VOCAB_CHUNK = 16384
EAS_STATIC_SCRATCH_BYTES = 64 << 20

# name -> (restype, argtypes), in the order of include/eas.h
_P, _I64, _I32, _U32, _SZ = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_uint32, ctypes.c_size_t
SIGNATURES = {
    "eas_spans_workspace_size": (_SZ, [_I64]),
    "eas_build_active_spans": (ctypes.c_int, [_P, _I64, _I32, _P, _I64, _P, _P, _SZ, _P]),
    "eas_cp_local_layout": (ctypes.c_int, [_P, _P, _I32, _I64, _I32, _I32, _P, _P, _P, _SZ, _P]),
    "eas_lmhead_workspace_size": (_SZ, [_I64, _I64, _I64, ctypes.c_int, _I64]),
    "eas_lmhead_fwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                      ctypes.c_int, _U32, _P, _P, _P, _P, _SZ, _P]),
    "eas_lmhead_bwd": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _P, _P,
                                      _I64, _I64, _I64, ctypes.c_int, _U32, _I64,
                                      _P, _P, _P, _SZ, _P]),
    "eas_quantize_rows_e4m3": (ctypes.c_int, [_P, ctypes.c_int, _I64, _I64, _P, _P, _P]),
    "eas_lmhead_fwd_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                          _U32, _P, _P, _P, _P, _SZ, _P]),
    "eas_lmhead_bwd_fp8_workspace_size": (_SZ, [_I64, _I64, _I64, _I64]),
    "eas_lmhead_bwd_fp8": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _I64,
                                          _P, _P, _I64, _I64, _I64, _U32, _I64, _P, _P, _P, _SZ,
                                          _P]),
    "eas_lmhead_fwd_shard": (ctypes.c_int, [_P, _P, _I64, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                            ctypes.c_int, _U32, _P, _P, _SZ, _P]),
    "eas_lmhead_combine_shards": (ctypes.c_int, [_P, _I32, _I64, _P, _P, _P, _P, _P]),
    "eas_lmhead_bwd_shard": (ctypes.c_int, [_P, _P, _P, _P, _I64, _P, _P, _P, _P, _I64, _P, _P,
                                            _I64, _I64, _I64, ctypes.c_int, _U32, _I64,
                                            _P, _P, _P, _SZ, _P]),
    "eas_lmhead_fwd_noalloc": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _I64, _I64, _I64, _I64,
                                              ctypes.c_int, _U32, _P, _P, _P, _P]),
    "eas_selftest_wait_timeout": (ctypes.c_int, [_I64, _P, _SZ, _P]),
    "eas_read_device_status": (ctypes.c_int, [_P, _P]),
    "eas_trace_enable": (None, [_I32]),
    "eas_trace_read": (ctypes.c_int32, [_P, _P, _I32]),
    "eas_kernel_name": (ctypes.c_char_p, [_I32]),
    "eas_last_error": (ctypes.c_char_p, []),
    "eas_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "eas_version": (ctypes.c_int32, []),
}

_lib = None


class EasError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{status_string(status)}: {message}")
        self.status = status


def load(path: str = LIB_PATH) -> ctypes.CDLL:
    """Loads libeas.so; raises if it has not been built (there is no fallback)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(path):
        raise RuntimeError(
            f"{path} is missing: build it with entropy_active_span_gb300.build.build() "
            "(nvcc, sm_103a); this package has no CPU or Python fallback")
    lib = ctypes.CDLL(path)
    for name, (res, args) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(status: int) -> str:
    return load().eas_status_string(status).decode()


def check(status: int) -> None:
    if status != EAS_OK:
        raise EasError(status, load().eas_last_error().decode())
