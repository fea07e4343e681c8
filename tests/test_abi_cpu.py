"""The C-ABI library loads and exports every symbol include/eas.h declares,
and rejects bad host-side arguments before touching the GPU (CPU only)."""
import ctypes
import os
import re

import pytest

from entropy_active_span_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    src = open(os.path.join(ROOT, "include", "eas.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(eas_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for n in ("eas_build_active_spans", "eas_lmhead_fwd", "eas_lmhead_bwd",
              "eas_lmhead_workspace_size", "eas_spans_workspace_size",
              "eas_read_device_status", "eas_last_error"):
        assert n in names


def test_every_declared_symbol_is_exported(libeas):
    names = declared_functions()
    assert names
    for n in names:
        assert hasattr(libeas, n), n
        assert n in _lib.SIGNATURES, n


def test_version_and_strings(libeas):
    assert libeas.eas_version() >= 100
    assert libeas.eas_status_string(_lib.EAS_ERR_INVALID_SPANS) == b"EAS_ERR_INVALID_SPANS"


def test_workspace_sizes(libeas):
    f = libeas.eas_lmhead_workspace_size
    a = f(16384, 4096, 128256, _lib.EAS_BF16, 0)
    b = f(16384, 4096, 128256, _lib.EAS_BF16, 4096)
    assert a > 16384 * 4096 * 2           # at least the packed copy of hidden
    assert b < a                          # a narrower vocab chunk needs less staging
    assert f(0, 128, 1024, _lib.EAS_FP32, 0) > 0
    assert f(-1, 128, 1024, _lib.EAS_FP32, 0) == 0
    assert libeas.eas_spans_workspace_size(1000) >= 16


def _fwd(libeas, T=256, H=128, V=1024, dtype=_lib.EAS_FP32, flags=0, ws_bytes=1 << 30,
         hidden=256, ws=256):
    p = 256  # fake, aligned, never dereferenced: every call below fails on the host
    return libeas.eas_lmhead_fwd(hidden, p, p, p, p, p, 4, T, H, V, dtype, flags,
                                 p, p, p, ws, ws_bytes, None)


def test_host_side_argument_errors(libeas):
    assert _fwd(libeas, T=-1) == _lib.EAS_ERR_INVALID_ARG
    assert _fwd(libeas, V=0) == _lib.EAS_ERR_INVALID_ARG
    assert _fwd(libeas, H=100, dtype=_lib.EAS_BF16) == _lib.EAS_ERR_UNSUPPORTED
    assert _fwd(libeas, H=6, dtype=_lib.EAS_FP32) == _lib.EAS_ERR_UNSUPPORTED
    assert _fwd(libeas, flags=7) == _lib.EAS_ERR_INVALID_ARG
    assert _fwd(libeas, ws_bytes=100) == _lib.EAS_ERR_WORKSPACE
    assert _fwd(libeas, hidden=258) == _lib.EAS_ERR_INVALID_ARG     # misaligned
    assert b"align" in libeas.eas_last_error()
    assert _fwd(libeas, ws=0) == _lib.EAS_ERR_INVALID_ARG           # null workspace
    assert libeas.eas_build_active_spans(256, 10, -1, 256, 4, 256, 256, 1024, None) == \
        _lib.EAS_ERR_INVALID_ARG                                      # max_gap < 0
    assert libeas.eas_build_active_spans(256, 10, 0, 256, 4, 256, 256, 8, None) == \
        _lib.EAS_ERR_WORKSPACE
    bwd = libeas.eas_lmhead_bwd
    p = 256
    assert bwd(p, p, p, p, p, p, p, p, 4, p, p, 10, 64, 100, _lib.EAS_BF16, 0, -5,
               p, p, p, 1 << 30, None) == _lib.EAS_ERR_INVALID_ARG   # vocab_chunk < 0
    assert bwd(p, p, p, p, p, p, p, p, 4, p, p, 10, 64, 100, _lib.EAS_BF16, 0, 0,
               p + 8, p, p, 1 << 30, None) == _lib.EAS_ERR_INVALID_ARG   # misaligned dhidden
    assert b"align" in libeas.eas_last_error()
    assert bwd(p, p, p, p, p, p, p, p, 4, p, p, 10, 64, 100, _lib.EAS_BF16, 0, 0,
               p, p + 4, p, 1 << 30, None) == _lib.EAS_ERR_INVALID_ARG   # misaligned dW
    assert bwd(p, p, p, p, p, p, p, p, 4, p, p, 10, 128, 100, _lib.EAS_E4M3, 0, 0,
               p, p, p, 1 << 30, None) == _lib.EAS_ERR_UNSUPPORTED     # no e4m3 backward
    assert bwd(p, p, p, p, p, p, p, p, 4, p, p, 10, 64, 100, _lib.EAS_BF16, 8, 0,
               p, p, p, 1 << 30, None) == _lib.EAS_ERR_INVALID_ARG     # unknown flag bit
    assert bwd(p, p, p, p, p, p, p, p, 4, p, p, 10, 64, 100, _lib.EAS_BF16, 0, 0,
               p, p, p, 100, None) == _lib.EAS_ERR_WORKSPACE           # workspace too small


def test_missing_library_fails_loudly(tmp_path, monkeypatch):
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="no CPU or Python fallback"):
        _lib.load(str(tmp_path / "libeas.so"))
