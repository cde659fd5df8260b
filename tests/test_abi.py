"""The C-ABI library builds for sm_103a, loads, exports every entry point
declared in include/fp8q.h, and rejects bad arguments on the host before it
touches CUDA. No kernel runs here."""
import ctypes
import os
import re

import pytest

from conftest import ROOT
from fp8_fine_grained_25_b300 import build as fbuild


@pytest.fixture(scope="module")
def lib():
    path = fbuild.build()
    return ctypes.CDLL(path)


def _declared():
    src = open(os.path.join(ROOT, "include", "fp8q.h")).read()
    return re.findall(r"^FP8Q_API\s+[\w\s\*]*?\b(\w+)\s*\(", src, re.M)


def test_every_declared_symbol_is_exported(lib):
    names = _declared()
    assert set(names) >= {"fp8q_quant_act", "fp8q_quant_weight", "fp8_block_gemm",
                          "fp8_grouped_gemm", "fp8q_status_string"}
    for n in names:
        assert hasattr(lib, n), n


def test_only_declared_symbols_are_exported():
    out = os.popen(f"nm -D --defined-only {fbuild.LIB}").read()
    exported = {line.split()[-1] for line in out.splitlines() if " T " in line}
    assert exported == set(_declared())


def test_status_strings(lib):
    lib.fp8q_status_string.restype = ctypes.c_char_p
    for code in range(9):
        assert lib.fp8q_status_string(code)
    assert b"unknown" in lib.fp8q_status_string(99)


# Status codes, mirrored from include/fp8q.h.
OK, NULL, SHAPE, ALIGN = 0, 1, 2, 3
P = 1 << 20  # a 16-byte-aligned non-null fake pointer; never dereferenced on these paths


def _q(lib, *a):
    f = lib.fp8q_quant_act
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    return f(*a)


def _w(lib, *a):
    f = lib.fp8q_quant_weight
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    return f(*a)


def _g(lib, *a):
    f = lib.fp8_block_gemm
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
    return f(*a)


def _gg(lib, *a):
    f = lib.fp8_grouped_gemm
    f.argtypes = [ctypes.c_void_p] * 6 + [ctypes.c_int32] + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
    return f(*a)


def test_quant_act_argument_checks(lib):
    assert _q(lib, P, -1, 128, P, P, None) == SHAPE
    assert _q(lib, P, 4, 0, P, P, None) == SHAPE
    assert _q(lib, P, 4, 1 << 31, P, P, None) == SHAPE
    assert _q(lib, None, 0, 128, None, None, None) == OK  # M = 0 is a no-op
    assert _q(lib, None, 4, 128, P, P, None) == NULL
    assert _q(lib, P, 4, 128, None, P, None) == NULL
    assert _q(lib, P, 4, 128, P, None, None) == NULL
    assert _q(lib, P, 4, 120, P, P, None) == ALIGN   # K % 16 != 0
    assert _q(lib, P + 8, 4, 128, P, P, None) == ALIGN
    assert _q(lib, P, 4, 128, P + 4, P, None) == ALIGN
    assert _q(lib, P, 4, 128, P, P + 2, None) == ALIGN


def test_quant_weight_argument_checks(lib):
    assert _w(lib, P, -3, 128, P, P, None) == SHAPE
    assert _w(lib, None, 0, 128, None, None, None) == OK
    assert _w(lib, P, 4, 128, None, P, None) == NULL
    assert _w(lib, P, 4, 24, P, P, None) == ALIGN


def test_gemm_argument_checks(lib):
    assert _g(lib, P, P, P, P, P, -1, 256, 512, None) == SHAPE
    assert _g(lib, P, P, P, P, P, 128, 0, 512, None) == SHAPE
    assert _g(lib, P, P, P, P, P, 128, 256, 0, None) == SHAPE
    assert _g(lib, None, None, None, None, None, 0, 256, 512, None) == OK
    for i in range(5):
        args = [P] * 5
        args[i] = None
        assert _g(lib, *args, 128, 256, 512, None) == NULL
    assert _g(lib, P, P, P, P, P, 128, 256, 520, None) == ALIGN   # K % 16
    assert _g(lib, P, P, P, P, P, 128, 252, 512, None) == ALIGN   # N % 8
    assert _g(lib, P + 8, P, P, P, P, 128, 256, 512, None) == ALIGN
    assert _g(lib, P, P, P, P, P + 8, 128, 256, 512, None) == ALIGN


def test_grouped_argument_checks(lib):
    assert _gg(lib, P, P, P, P, P, P, 0, 64, 256, 512, None) == SHAPE      # E < 1
    assert _gg(lib, P, P, P, P, P, P, 1025, 64, 256, 512, None) == SHAPE   # E > 1024
    assert _gg(lib, P, P, P, P, P, P, 4, -1, 256, 512, None) == SHAPE
    assert _gg(lib, P, P, P, P, P, P, 1024, 64, 1 << 22, 512, None) == SHAPE  # E*N > 2^31-1
    assert _gg(lib, None, None, None, None, None, None, 4, 0, 256, 512, None) == OK
    assert _gg(lib, P, P, P, P, P, None, 4, 64, 256, 512, None) == NULL
    assert _gg(lib, P, P, P, P, P, P + 2, 4, 64, 256, 512, None) == ALIGN
    assert _gg(lib, P, P, P, P, P, P, 4, 64, 256, 500, None) == ALIGN


def _ga(lib, *a):
    f = lib.fp8q_gather_rows
    f.argtypes = [ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_int64, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    return f(*a)


def test_gather_argument_checks(lib):
    assert _ga(lib, P, P, -1, 128, P, 4, P, P, None) == SHAPE
    assert _ga(lib, P, P, 8, 0, P, 4, P, P, None) == SHAPE
    assert _ga(lib, None, None, 8, 128, None, 0, None, None, None) == OK   # R = 0
    assert _ga(lib, P, P, 8, 128, None, 4, P, P, None) == NULL
    assert _ga(lib, P, P, 8, 120, P, 4, P, P, None) == ALIGN
    assert _ga(lib, P + 8, P, 8, 128, P, 4, P, P, None) == ALIGN
    assert _ga(lib, P, P, 8, 128, P + 2, 4, P, P, None) == ALIGN


def _qt(lib, *a):
    f = lib.fp8q_quant_act_t
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                  ctypes.c_void_p, ctypes.c_void_p]
    return f(*a)


def _wt(lib, *a):
    f = lib.fp8q_quant_weight_t
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64] + [ctypes.c_void_p] * 5
    return f(*a)


def _wg(lib, *a):
    f = lib.fp8_wgrad_gemm
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
    return f(*a)


def test_quant_act_t_argument_checks(lib):
    assert _qt(lib, P, -1, 128, P, P, None) == SHAPE
    assert _qt(lib, P, 16, 0, P, P, None) == SHAPE
    assert _qt(lib, None, 0, 128, None, None, None) == OK
    assert _qt(lib, None, 16, 128, P, P, None) == NULL
    assert _qt(lib, P, 16, 128, None, P, None) == NULL
    assert _qt(lib, P, 16, 128, P, None, None) == NULL
    assert _qt(lib, P, 24, 128, P, P, None) == ALIGN   # M % 16: the row pitch of qt
    assert _qt(lib, P, 16, 120, P, P, None) == ALIGN   # K % 16
    assert _qt(lib, P, 16, 128, P + 8, P, None) == ALIGN


def test_quant_weight_t_argument_checks(lib):
    assert _wt(lib, P, -16, 128, P, P, P, P, None) == SHAPE
    assert _wt(lib, None, 0, 128, None, None, None, None, None) == OK
    assert _wt(lib, P, 16, 128, P, P, None, P, None) == NULL     # qt required
    assert _wt(lib, P, 16, 128, P, P, P, None, None) == NULL     # st required
    assert _wt(lib, P, 16, 128, P, None, P, P, None) == NULL     # q without s
    assert _wt(lib, P, 16, 128, None, P, P, P, None) == NULL     # s without q
    assert _wt(lib, P, 40, 128, None, None, P, P, None) == ALIGN  # N % 16
    assert _wt(lib, P, 16, 120, None, None, P, P, None) == ALIGN  # K % 16
    assert _wt(lib, P, 16, 128, P + 4, P, P, P, None) == ALIGN


def test_wgrad_gemm_argument_checks(lib):
    assert _wg(lib, P, P, P, P, P, -1, 256, 512, None) == SHAPE
    assert _wg(lib, None, None, None, None, None, 0, 256, 512, None) == OK
    for i in range(5):
        args = [P] * 5
        args[i] = None
        assert _wg(lib, *args, 128, 256, 512, None) == NULL
    assert _wg(lib, P, P, P, P, P, 128, 256, 520, None) == ALIGN
    assert _wg(lib, P, P, P, P, P, 128, 252, 512, None) == ALIGN


def test_ue8m0_quantizer_argument_checks(lib):
    for name in ("fp8q_quant_act_ue8m0", "fp8q_quant_weight_ue8m0"):
        f = getattr(lib, name)
        f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                      ctypes.c_void_p, ctypes.c_void_p]
        assert f(P, -1, 128, P, P, None) == SHAPE
        assert f(None, 0, 128, None, None, None) == OK
        assert f(P, 4, 128, P, None, None) == NULL
        assert f(P, 4, 120, P, P, None) == ALIGN
        assert f(P, 4, 128, P + 8, P, None) == ALIGN
        assert f(P, 4, 128, P, P + 1, None) != ALIGN  # byte scales need no alignment


def test_tile_width_setter(lib):
    # the setters only record a process-wide choice; no device is touched
    OK, UNSUPPORTED = 0, 7
    for bn in (0, 128, 160, 224, 256):
        assert lib.fp8q_set_gemm_tile_n(bn) == OK, bn
    for bn in (64, 192, 512, -1):
        assert lib.fp8q_set_gemm_tile_n(bn) == UNSUPPORTED, bn
    assert lib.fp8q_set_gemm_tile_n(0) == OK


def _gws(lib, *a):
    f = lib.fp8_block_gemm_ws
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_void_p, ctypes.c_size_t,
                                                                 ctypes.c_void_p]
    return f(*a)


def test_split_k_gemm_argument_checks(lib):
    # the same host checks as fp8_block_gemm, made before any device call
    assert _gws(lib, P, P, P, P, P, -1, 256, 512, P, 1 << 20, None) == SHAPE
    assert _gws(lib, None, None, None, None, None, 0, 256, 512, None, 0, None) == OK
    for i in range(5):
        args = [P] * 5
        args[i] = None
        assert _gws(lib, *args, 128, 256, 512, P, 1 << 20, None) == NULL
    assert _gws(lib, P, P, P, P, P, 128, 252, 512, P, 1 << 20, None) == ALIGN    # N % 8
    assert _gws(lib, P, P, P, P, P, 128, 256, 512, P + 16, 1 << 20, None) == ALIGN  # workspace
    f = lib.fp8_block_gemm_workspace_size
    f.argtypes = [ctypes.c_int64] * 3 + [ctypes.POINTER(ctypes.c_size_t)]
    n = ctypes.c_size_t(7)
    assert f(128, 256, 512, None) == NULL
    assert f(-1, 256, 512, ctypes.byref(n)) == SHAPE and n.value == 0
    assert f(0, 256, 512, ctypes.byref(n)) == OK and n.value == 0


def test_split_count_setter(lib):
    OK, UNSUPPORTED = 0, 7
    for s in range(0, 9):
        assert lib.fp8q_set_gemm_splits(s) == OK, s
    for s in (-1, 9, 64):
        assert lib.fp8q_set_gemm_splits(s) == UNSUPPORTED, s
    assert lib.fp8q_set_gemm_splits(0) == OK


def test_static_scratch_gemm_argument_checks(lib):
    f = lib.fp8_block_gemm_static
    f.argtypes = [ctypes.c_void_p] * 5 + [ctypes.c_int64] * 3 + [ctypes.c_void_p]
    assert f(P, P, P, P, P, -1, 256, 512, None) == SHAPE
    assert f(None, None, None, None, None, 0, 256, 512, None) == OK
    assert f(P, P, None, P, P, 128, 256, 512, None) == NULL
    assert f(P, P, P, P, P, 128, 252, 512, None) == ALIGN
