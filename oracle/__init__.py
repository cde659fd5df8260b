"""CPU oracle for fine-grained FP8 quantization and the block-scaled FP8 GEMM.

TEST INFRASTRUCTURE ONLY. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package. The product path
(``fp8_fine_grained_25_b300``) never imports it, and this package imports
nothing from the product.

The arithmetic lives in ``fp8_oracle.c`` (plain C, one element at a time, the
definitions written out; see that file's header for the passages it follows:
news.qq.com/rain/a/20241229A05OQF00 "FP8 低精度训练" Fig. 7a/7b, the aliyun
article §4.1 and the jxzklqfsx article §三(二)). This module only builds it,
marshals numpy arrays into it, splits rows across host threads (ctypes drops
the GIL during the call), and states the acceptance test.

Parity status: every function here is pinned by ``tests/test_oracle_*.py``
against facts outside the oracle (the E4M3 format table, a library codec,
closed forms and exact rational brute force).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading
from concurrent.futures import ThreadPoolExecutor

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fp8_oracle.c")
_LIB = os.path.join(_HERE, "libfp8_oracle.so")
_lock = threading.Lock()
_lib = None

TILE = 128
E4M3_MAX = 448.0


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/libfp8_oracle.so`` (gcc, no fast-math,
    no FP contraction) unless an up-to-date build exists."""
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off",
           "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
        i64, p = ctypes.c_int64, ctypes.c_void_p
        lib.fp8o_e4m3_decode.restype = ctypes.c_double
        lib.fp8o_e4m3_decode.argtypes = [ctypes.c_uint8]
        lib.fp8o_e4m3_encode.restype = ctypes.c_uint8
        lib.fp8o_e4m3_encode.argtypes = [ctypes.c_float]
        lib.fp8o_e4m3_encode_n.argtypes = [p, i64, p]
        lib.fp8o_quant_act.argtypes = [p, i64, i64, i64, i64, p, p]
        lib.fp8o_quant_weight.argtypes = [p, i64, i64, i64, i64, p, p]
        lib.fp8o_quant_act_ue8m0.argtypes = [p, i64, i64, i64, i64, p, p]
        lib.fp8o_quant_weight_ue8m0.argtypes = [p, i64, i64, i64, i64, p, p]
        lib.fp8o_block_partials.argtypes = [p, p, i64, i64, i64, p]
        lib.fp8o_gemm.argtypes = [p, p, p, p, i64, p, i64, p, i64, p, p]
        lib.fp8o_wgrad_gemm.argtypes = [p, p, p, p, i64, p, i64, p, i64, p, p]
        lib.fp8o_grouped_gemm.argtypes = [p, p, p, p, p, ctypes.c_int32, i64, i64,
                                          p, i64, p, i64, p, p]
        _lib = lib
        return lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags["C_CONTIGUOUS"], "oracle inputs must be C-contiguous"
    return a.ctypes.data


def _threads(threads: int | None) -> int:
    return max(1, threads if threads is not None else (os.cpu_count() or 1))


def _split(n: int, parts: int):
    parts = max(1, min(parts, n))
    step = -(-n // parts)
    return [(i, min(n, i + step)) for i in range(0, n, step)]


# ---------------------------------------------------------------- E4M3 codec
def e4m3_decode(codes) -> np.ndarray:
    """Decode uint8 E4M3 codes to float64 (NaN for 0x7F / 0xFF)."""
    lib = _load()
    codes = np.ascontiguousarray(codes, dtype=np.uint8)
    table = np.array([lib.fp8o_e4m3_decode(c) for c in range(256)], dtype=np.float64)
    return table[codes]


def e4m3_encode(values) -> np.ndarray:
    """Encode float32 values to E4M3 codes (RNE, saturating at +-448)."""
    lib = _load()
    v = np.ascontiguousarray(values, dtype=np.float32)
    out = np.empty(v.shape, dtype=np.uint8)
    lib.fp8o_e4m3_encode_n(_ptr(v), v.size, _ptr(out))
    return out


# ------------------------------------------------------------- quantization
def _as_bf16_bits(x) -> np.ndarray:
    a = np.asarray(x)
    if a.dtype == np.uint16:
        return np.ascontiguousarray(a)
    if a.dtype == np.int16:
        return np.ascontiguousarray(a).view(np.uint16)
    raise TypeError("pass bf16 data as its raw uint16 bits")


def quant_act(x_bits, threads: int | None = None):
    """Per-1x128-tile quantization of bf16 activations [M, K].

    Returns (codes uint8 [M, K], scales float32 [M, ceil(K/128)])."""
    lib = _load()
    x = _as_bf16_bits(x_bits)
    M, K = x.shape
    KB = -(-K // TILE)
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty((M, KB), dtype=np.float32)
    chunks = _split(M, _threads(threads))
    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(lambda c: lib.fp8o_quant_act(_ptr(x), M, K, c[0], c[1], _ptr(q), _ptr(s)),
                    chunks))
    return q, s


def quant_weight(w_bits, threads: int | None = None):
    """Per-128x128-block quantization of bf16 weights [N, K].

    Returns (codes uint8 [N, K], scales float32 [ceil(N/128), ceil(K/128)])."""
    lib = _load()
    w = _as_bf16_bits(w_bits)
    N, K = w.shape
    NB, KB = -(-N // TILE), -(-K // TILE)
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty((NB, KB), dtype=np.float32)
    chunks = _split(NB, _threads(threads))
    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(lambda c: lib.fp8o_quant_weight(_ptr(w), N, K, c[0], c[1], _ptr(q), _ptr(s)),
                    chunks))
    return q, s


def quant_act_ue8m0(x_bits, threads: int | None = None):
    """1x128 tiles with power-of-two (UE8M0) scales: (codes uint8 [M, K],
    scale bytes uint8 [M, ceil(K/128)]; the scale is 2^(byte - 127))."""
    lib = _load()
    x = _as_bf16_bits(x_bits)
    M, K = x.shape
    q = np.empty((M, K), dtype=np.uint8)
    s = np.empty((M, -(-K // TILE)), dtype=np.uint8)
    chunks = _split(M, _threads(threads))
    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(lambda c: lib.fp8o_quant_act_ue8m0(_ptr(x), M, K, c[0], c[1], _ptr(q), _ptr(s)),
                    chunks))
    return q, s


def quant_weight_ue8m0(w_bits, threads: int | None = None):
    """128x128 blocks with power-of-two (UE8M0) scales: (codes uint8 [N, K],
    scale bytes uint8 [ceil(N/128), ceil(K/128)])."""
    lib = _load()
    w = _as_bf16_bits(w_bits)
    N, K = w.shape
    q = np.empty((N, K), dtype=np.uint8)
    s = np.empty((-(-N // TILE), -(-K // TILE)), dtype=np.uint8)
    chunks = _split(-(-N // TILE), _threads(threads))
    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(lambda c: lib.fp8o_quant_weight_ue8m0(_ptr(w), N, K, c[0], c[1], _ptr(q), _ptr(s)),
                    chunks))
    return q, s


def ue8m0_to_f32(s_bytes) -> np.ndarray:
    """The scale a UE8M0 byte stands for: 2^(byte - 127), exact in float32
    (2^-127 is a float32 subnormal)."""
    b = np.asarray(s_bytes, dtype=np.int32)
    return np.ldexp(np.float32(1.0), b - 127).astype(np.float32)


def gemm_ue8m0(qa, sa_bytes, qb, sb_bytes, rows=None, cols=None, threads: int | None = None):
    """The block-scaled GEMM with UE8M0 scales: by definition the same
    computation as gemm() with the scales 2^(byte - 127)."""
    return gemm(qa, ue8m0_to_f32(sa_bytes), qb, ue8m0_to_f32(sb_bytes), rows, cols, threads)


def quant_act_t_ue8m0(x_bits, threads: int | None = None):
    """128x1 tiles (along M) with UE8M0 scales, written transposed: the 1x128
    UE8M0 tiles of x^T. Returns (codes uint8 [K, M], bytes uint8 [K, ceil(M/128)])."""
    x = _as_bf16_bits(x_bits)
    return quant_act_ue8m0(np.ascontiguousarray(x.T), threads)


def quant_weight_t_ue8m0(w_bits, threads: int | None = None):
    """128x128 UE8M0 blocks in both layouts: (q [N, K], s [NB, KB], qt [K, N],
    st [KB, NB]); a block's byte and codes do not depend on the orientation."""
    q, s = quant_weight_ue8m0(w_bits, threads)
    return q, s, np.ascontiguousarray(q.T), np.ascontiguousarray(s.T)


def wgrad_gemm_ue8m0(qa, sa_bytes, qb, sb_bytes, rows=None, cols=None, threads: int | None = None):
    """The weight-gradient GEMM with UE8M0 row scales on both operands: by
    definition wgrad_gemm() with the scales 2^(byte - 127)."""
    return wgrad_gemm(qa, ue8m0_to_f32(sa_bytes), qb, ue8m0_to_f32(sb_bytes), rows, cols, threads)


def quant_act_t(x_bits, threads: int | None = None):
    """Quantization of bf16 activations [M, K] in 128x1 tiles (128 consecutive
    rows of one column), written transposed: the 1x128 tiles of x^T.

    This is the layout the weight-gradient GEMM reads (it contracts over the
    M axis). Returns (codes uint8 [K, M], scales float32 [K, ceil(M/128)])."""
    x = _as_bf16_bits(x_bits)
    return quant_act(np.ascontiguousarray(x.T), threads)


def quant_weight_t(w_bits, threads: int | None = None):
    """128x128-block quantization of bf16 weights [N, K] with the codes also
    in the transposed layout. A block's amax, scale and codes do not depend
    on the orientation, so the transposed outputs are the transposes:
    returns (q [N, K], s [NB, KB], qt [K, N], st [KB, NB])."""
    q, s = quant_weight(w_bits, threads)
    return q, s, np.ascontiguousarray(q.T), np.ascontiguousarray(s.T)


# --------------------------------------------------------------------- GEMM
def block_partials(qa, qb, m: int, n: int) -> np.ndarray:
    """Exact per-128-K-block dot products of decoded codes, float64 [KB]."""
    lib = _load()
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    K = qa.shape[1]
    P = np.empty(-(-K // TILE), dtype=np.float64)
    lib.fp8o_block_partials(_ptr(qa), _ptr(qb), K, m, n, _ptr(P))
    return P


def _gemm_at(fn, qa, sa, qb, sb, rows, cols, threads):
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    M, K = qa.shape
    N = qb.shape[0]
    assert qb.shape[1] == K
    rows = np.arange(M, dtype=np.int64) if rows is None else np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    c32 = np.empty((len(rows), len(cols)), dtype=np.float32)
    S = np.empty((len(rows), len(cols)), dtype=np.float64)
    chunks = _split(len(rows), _threads(threads))

    def work(c):
        r = rows[c[0]:c[1]]
        o = np.empty((len(r), len(cols)), dtype=np.float32)
        b = np.empty((len(r), len(cols)), dtype=np.float64)
        fn(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), K, _ptr(r), len(r),
           _ptr(cols), len(cols), _ptr(o), _ptr(b))
        c32[c[0]:c[1]] = o
        S[c[0]:c[1]] = b

    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(work, chunks))
    return c32, S


def gemm(qa, sa, qb, sb, rows=None, cols=None, threads: int | None = None):
    """Block-scaled GEMM C = A * B^T at the outputs rows x cols.

    qa uint8 [M, K], sa float32 [M, KB], qb uint8 [N, K], sb float32 [NB, KB].
    Returns (c32 float32 [len(rows), len(cols)], S float64 [same])."""
    return _gemm_at(_load().fp8o_gemm, qa, sa, qb, sb, rows, cols, threads)


def wgrad_gemm(qa, sa, qb, sb, rows=None, cols=None, threads: int | None = None):
    """The weight-gradient GEMM: C = A * B^T where both operands carry one
    scale per row per 128-wide K block (1x128 tiles of the transposed
    activations): qa uint8 [M, K], sa float32 [M, KB], qb uint8 [N, K],
    sb float32 [N, KB]. Returns (c32, S) at rows x cols."""
    return _gemm_at(_load().fp8o_wgrad_gemm, qa, sa, qb, sb, rows, cols, threads)


def grouped_gemm(qa, sa, qb, sb, offsets, rows, cols=None, threads: int | None = None):
    """Grouped GEMM: row m of A uses expert e with off[e] <= m < off[e+1].

    qb uint8 [E, N, K], sb float32 [E, NB, KB], offsets int32 [E+1].
    Returns (c32, S) at rows x cols."""
    lib = _load()
    qa = np.ascontiguousarray(qa, dtype=np.uint8)
    qb = np.ascontiguousarray(qb, dtype=np.uint8)
    sa = np.ascontiguousarray(sa, dtype=np.float32)
    sb = np.ascontiguousarray(sb, dtype=np.float32)
    off = np.ascontiguousarray(offsets, dtype=np.int32)
    E, N, K = qb.shape
    assert qa.shape[1] == K and len(off) == E + 1
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.arange(N, dtype=np.int64) if cols is None else np.ascontiguousarray(cols, dtype=np.int64)
    c32 = np.empty((len(rows), len(cols)), dtype=np.float32)
    S = np.empty((len(rows), len(cols)), dtype=np.float64)
    chunks = _split(len(rows), _threads(threads))

    def work(c):
        r = rows[c[0]:c[1]]
        o = np.empty((len(r), len(cols)), dtype=np.float32)
        b = np.empty((len(r), len(cols)), dtype=np.float64)
        lib.fp8o_grouped_gemm(_ptr(qa), _ptr(sa), _ptr(qb), _ptr(sb), _ptr(off), E, N, K,
                              _ptr(r), len(r), _ptr(cols), len(cols), _ptr(o), _ptr(b))
        c32[c[0]:c[1]] = o
        S[c[0]:c[1]] = b

    with ThreadPoolExecutor(len(chunks)) as ex:
        list(ex.map(work, chunks))
    return c32, S


# --------------------------------------------------------------- acceptance
def bf16_ulp(v) -> np.ndarray:
    """One bf16 ulp at v: 2^(floor(log2|v|) - 7) for normal |v|; the smallest
    bf16 subnormal 2^-133 for zero and subnormal v."""
    v = np.abs(np.asarray(v, dtype=np.float64))
    out = np.full(v.shape, 2.0 ** -133)
    normal = v >= 2.0 ** -126
    e = np.floor(np.log2(np.where(normal, v, 1.0)))
    out[normal] = np.exp2(e[normal] - 7)
    return out


def gemm_tolerance(c32, S) -> np.ndarray:
    """Per-element acceptance bound: 1 bf16 ulp of the oracle's FP32 result
    plus 1e-5 times sum_k |a_k * b_k| (dequantized)."""
    return bf16_ulp(c32) + 1e-5 * np.asarray(S, dtype=np.float64)


def gemm_check(c_test, c32, S):
    """Return (ok, worst ratio |c_test - c32| / bound, index of the worst)."""
    c_test = np.asarray(c_test, dtype=np.float64)
    err = np.abs(c_test - np.asarray(c32, dtype=np.float64))
    tol = gemm_tolerance(c32, S)
    ratio = np.where(np.isfinite(err), err / tol, np.inf)
    idx = np.unravel_index(int(np.argmax(ratio)), ratio.shape) if ratio.size else ()
    worst = float(ratio[idx]) if ratio.size else 0.0
    return bool(np.all(ratio <= 1.0)), worst, idx
