"""CPU oracle for the Q8_0 x q8_1 block-quantized matmul -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of ``bench.py``
may import this package.  The product library never calls it, and this package never
imports the product library: the two share no code.

The arithmetic lives in ``q8_oracle.c`` (plain C, single-threaded, compiled with
``-ffp-contract=off`` so every f32 operation is rounded on its own).  This module builds
it with gcc and exposes numpy-facing wrappers:

    f32_to_f16, f16_to_f32            O0  IEEE binary16 conversions (round to nearest even)
    quantize_q8_0(w)                  O1  f32 [n,k] -> Q8_0 bytes [n, k/32*34]
    quantize_q8_1(x)                  O2  f32 [m,k] -> (int8 [m,k], f32 [m,k/32])
    block_dots(w, xq, k, rows=None)   O3  exact int32 D[t, r, b]
    matmul(w, xq, xd, k, rows=None)   O4  (y32, y64, S) with S = sum_b |d_w d_a D|
    dequant_f16(w, k)                 O5  Q8_0 -> fp16 bits [n, k]
    repack_q8_0(w, k, ldn)            O6  Q8_0 -> exact binary16 quant plane + f32 scale plane
    quantize_q4_0(w)                  O7a f32 [n,k] -> Q4_0 bytes [n, k/32*18] (data preparation)
    dequant_q4_0_f16(w, k)            O7b Q4_0 -> fp16 bits [n, k]
    block_dots_q4_0(w, xq, k, rows)   O7c exact int32 D[t, r, b] of Q4_0 weights
    matmul_q4_0(w, xq, xd, k, rows)   O7d (y32, y64, S) over Q4_0 weights
    f64_to_f16(x)                     O8  binary64 -> binary16 bits (round to nearest even)
    dequant_kq_f16(fmt, w, k)         O8a K-quant superblocks -> fp16 bits [n, k]
                                          (fmt: "q6_k", "q4_k", "q5_k")
    block_dots_kq(fmt, w, xq, k, rows)  O8b exact int32 per-32-block integers [t, r, b]
    matmul_kq(fmt, w, xq, xd, k, rows)  O8c (y32, y64, S) over K-quant weights

Each C function cites the page passage it follows (memra-engine docs.rs pages:
accprobe_bench.rs, decode_kernel_census.rs, f16_ffi.rs).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "q8_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libq8oracle.so")
_LOCK = threading.Lock()
_LIB = None

QK = 32
Q8_0_BYTES = 34
Q4_0_BYTES = 18
QK_K = 256
KQ_FORMATS = {"q6_k": (6, 210), "q4_k": (4, 144), "q5_k": (5, 176)}   # code, superblock bytes


def build(force: bool = False) -> str:
    """Compile q8_oracle.c into a shared library (idempotent); returns its path."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
           "-shared", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _bind(lib):
    P = ctypes.c_void_p
    I64 = ctypes.c_int64
    lib.oracle_f32_to_f16_array.argtypes = [P, P, I64]
    lib.oracle_f16_to_f32_array.argtypes = [P, P, I64]
    lib.oracle_quantize_q8_1.argtypes = [P, P, P, I64, I64]
    lib.oracle_quantize_q8_0.argtypes = [P, P, I64, I64]
    lib.oracle_block_dots.argtypes = [P, P, P, I64, I64, I64, P, I64]
    lib.oracle_matmul.argtypes = [P, P, P, I64, I64, I64, P, I64, P, P, P]
    lib.oracle_dequant_f16.argtypes = [P, P, I64, I64]
    lib.oracle_repack_q8_0.argtypes = [P, P, P, I64, I64, I64]
    lib.oracle_quantize_q4_0.argtypes = [P, P, I64, I64]
    lib.oracle_dequant_q4_0_f16.argtypes = [P, P, I64, I64]
    lib.oracle_block_dots_q4_0.argtypes = [P, P, P, I64, I64, I64, P, I64]
    lib.oracle_matmul_q4_0.argtypes = [P, P, P, I64, I64, I64, P, I64, P, P, P]
    I32 = ctypes.c_int
    lib.oracle_f64_to_f16.argtypes = [ctypes.c_double]
    lib.oracle_f64_to_f16.restype = ctypes.c_uint16
    lib.oracle_dequant_kq_f16.argtypes = [I32, P, P, I64, I64]
    lib.oracle_block_dots_kq.argtypes = [I32, P, P, P, I64, I64, I64, P, I64]
    lib.oracle_matmul_kq.argtypes = [I32, P, P, P, I64, I64, I64, P, I64, P, P, P]
    for name in ("oracle_f32_to_f16_array", "oracle_f16_to_f32_array",
                 "oracle_quantize_q8_1", "oracle_quantize_q8_0", "oracle_block_dots",
                 "oracle_matmul", "oracle_dequant_f16", "oracle_repack_q8_0",
                 "oracle_quantize_q4_0", "oracle_dequant_q4_0_f16", "oracle_block_dots_q4_0",
                 "oracle_matmul_q4_0", "oracle_dequant_kq_f16", "oracle_block_dots_kq",
                 "oracle_matmul_kq"):
        getattr(lib, name).restype = None
    return lib


def _lib():
    global _LIB
    with _LOCK:
        if _LIB is None:
            _LIB = _bind(ctypes.CDLL(build()))
    return _LIB


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data


def _check_k(k: int) -> None:
    if k <= 0 or k % QK:
        raise ValueError(f"k must be a positive multiple of {QK}, got {k}")


class Oracle:
    """The oracle's functions bound to one compiled copy of the C source.

    The module-level functions use the copy built from ``q8_oracle.c``; the test-suite
    also wraps deliberately broken copies (planted mistakes) to show that its pins catch
    them.
    """

    def __init__(self, lib_path: str | None = None):
        self._path = lib_path

    def lib(self):
        if self._path is None:
            return _lib()
        if not hasattr(self, "_l"):
            self._l = _bind(ctypes.CDLL(self._path))
        return self._l


def f32_to_f16(x, _o: Oracle | None = None) -> np.ndarray:
    """Element-wise binary32 -> binary16 bits (uint16), round to nearest even."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    out = np.empty(x.shape, dtype=np.uint16)
    (_o or _DEFAULT).lib().oracle_f32_to_f16_array(_ptr(x), _ptr(out), x.size)
    return out


def f16_to_f32(h, _o: Oracle | None = None) -> np.ndarray:
    """Element-wise binary16 bits (uint16) -> binary32."""
    h = np.ascontiguousarray(h, dtype=np.uint16)
    out = np.empty(h.shape, dtype=np.float32)
    (_o or _DEFAULT).lib().oracle_f16_to_f32_array(_ptr(h), _ptr(out), h.size)
    return out


def quantize_q8_0(w: np.ndarray, _o: Oracle | None = None) -> np.ndarray:
    """O1: f32 weights [n, k] -> Q8_0 bytes uint8 [n, k/32*34]."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    _check_k(k)
    out = np.empty((n, k // QK * Q8_0_BYTES), dtype=np.uint8)
    (_o or _DEFAULT).lib().oracle_quantize_q8_0(_ptr(w), _ptr(out), n, k)
    return out


def quantize_q8_1(x: np.ndarray, _o: Oracle | None = None):
    """O2: f32 activations [m, k] -> (xq int8 [m, k], xd f32 [m, k/32])."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    m, k = x.shape
    _check_k(k)
    xq = np.empty((m, k), dtype=np.int8)
    xd = np.empty((m, k // QK), dtype=np.float32)
    (_o or _DEFAULT).lib().oracle_quantize_q8_1(_ptr(x), _ptr(xq), _ptr(xd), m, k)
    return xq, xd


def _rows_arg(rows, n):
    if rows is None:
        return None, n
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    if rows.size and (rows.min() < 0 or rows.max() >= n):
        raise ValueError("row index out of range")
    return rows, rows.size


def block_dots(w: np.ndarray, xq: np.ndarray, k: int, rows=None, _o: Oracle | None = None) -> np.ndarray:
    """O3: exact int32 block dots D[t, j, b] for weight rows ``rows`` (default: all)."""
    _check_k(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    n = w.size // (k // QK * Q8_0_BYTES)
    m = xq.size // k
    rows, nr = _rows_arg(rows, n)
    D = np.empty((m, nr, k // QK), dtype=np.int32)
    (_o or _DEFAULT).lib().oracle_block_dots(_ptr(w), _ptr(xq), _ptr(D), m, n, k, _ptr(rows), nr)
    return D


def matmul(w: np.ndarray, xq: np.ndarray, xd: np.ndarray, k: int, rows=None, _o: Oracle | None = None):
    """O4: returns (y32 f32 [m, nr], y64 f64 [m, nr], S f64 [m, nr])."""
    _check_k(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xd = np.ascontiguousarray(xd, dtype=np.float32)
    n = w.size // (k // QK * Q8_0_BYTES)
    m = xq.size // k
    rows, nr = _rows_arg(rows, n)
    y32 = np.empty((m, nr), dtype=np.float32)
    y64 = np.empty((m, nr), dtype=np.float64)
    S = np.empty((m, nr), dtype=np.float64)
    (_o or _DEFAULT).lib().oracle_matmul(_ptr(w), _ptr(xq), _ptr(xd), m, n, k, _ptr(rows), nr,
                         _ptr(y32), _ptr(y64), _ptr(S))
    return y32, y64, S


def dequant_f16(w: np.ndarray, k: int, _o: Oracle | None = None) -> np.ndarray:
    """O5: Q8_0 bytes -> fp16 bits uint16 [n, k]."""
    _check_k(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    n = w.size // (k // QK * Q8_0_BYTES)
    out = np.empty((n, k), dtype=np.uint16)
    (_o or _DEFAULT).lib().oracle_dequant_f16(_ptr(w), _ptr(out), n, k)
    return out


def repack_q8_0(w: np.ndarray, k: int, ldn: int | None = None, _o: Oracle | None = None):
    """O6: Q8_0 bytes -> (wq16 binary16 bits uint16 [n, k], wdt f32 [k/32, ldn]); the
    columns n..ldn-1 of wdt are zero."""
    _check_k(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    n = w.size // (k // QK * Q8_0_BYTES)
    ldn = n if ldn is None else ldn
    wq16 = np.empty((n, k), dtype=np.uint16)
    wdt = np.zeros((k // QK, ldn), dtype=np.float32)
    (_o or _DEFAULT).lib().oracle_repack_q8_0(_ptr(w), _ptr(wq16), _ptr(wdt), n, k, ldn)
    return wq16, wdt


def quantize_q4_0(w: np.ndarray, _o: Oracle | None = None) -> np.ndarray:
    """O7a: f32 weights [n, k] -> Q4_0 bytes uint8 [n, k/32*18] (data preparation)."""
    w = np.ascontiguousarray(w, dtype=np.float32)
    n, k = w.shape
    _check_k(k)
    out = np.empty((n, k // QK * Q4_0_BYTES), dtype=np.uint8)
    (_o or _DEFAULT).lib().oracle_quantize_q4_0(_ptr(w), _ptr(out), n, k)
    return out


def dequant_q4_0_f16(w: np.ndarray, k: int, _o: Oracle | None = None) -> np.ndarray:
    """O7b: Q4_0 bytes -> fp16 bits uint16 [n, k]."""
    _check_k(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    n = w.size // (k // QK * Q4_0_BYTES)
    out = np.empty((n, k), dtype=np.uint16)
    (_o or _DEFAULT).lib().oracle_dequant_q4_0_f16(_ptr(w), _ptr(out), n, k)
    return out


def block_dots_q4_0(w: np.ndarray, xq: np.ndarray, k: int, rows=None, _o: Oracle | None = None) -> np.ndarray:
    """O7c: exact int32 block dots D[t, j, b] of Q4_0 weight rows ``rows`` (default: all)."""
    _check_k(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    n = w.size // (k // QK * Q4_0_BYTES)
    m = xq.size // k
    rows, nr = _rows_arg(rows, n)
    D = np.empty((m, nr, k // QK), dtype=np.int32)
    (_o or _DEFAULT).lib().oracle_block_dots_q4_0(_ptr(w), _ptr(xq), _ptr(D), m, n, k, _ptr(rows), nr)
    return D


def matmul_q4_0(w: np.ndarray, xq: np.ndarray, xd: np.ndarray, k: int, rows=None, _o: Oracle | None = None):
    """O7d: returns (y32 f32 [m, nr], y64 f64 [m, nr], S f64 [m, nr]) over Q4_0 weights."""
    _check_k(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xd = np.ascontiguousarray(xd, dtype=np.float32)
    n = w.size // (k // QK * Q4_0_BYTES)
    m = xq.size // k
    rows, nr = _rows_arg(rows, n)
    y32 = np.empty((m, nr), dtype=np.float32)
    y64 = np.empty((m, nr), dtype=np.float64)
    S = np.empty((m, nr), dtype=np.float64)
    (_o or _DEFAULT).lib().oracle_matmul_q4_0(_ptr(w), _ptr(xq), _ptr(xd), m, n, k, _ptr(rows), nr,
                              _ptr(y32), _ptr(y64), _ptr(S))
    return y32, y64, S


def _kq(fmt: str):
    if fmt not in KQ_FORMATS:
        raise ValueError(f"unknown K-quant format {fmt!r}")
    return KQ_FORMATS[fmt]


def _check_kk(k: int) -> None:
    if k <= 0 or k % QK_K:
        raise ValueError(f"k must be a positive multiple of {QK_K}, got {k}")


def f64_to_f16(x, _o: Oracle | None = None) -> np.ndarray:
    """O8: element-wise binary64 -> binary16 bits (uint16), round to nearest even."""
    x = np.asarray(x, dtype=np.float64)
    f = (_o or _DEFAULT).lib().oracle_f64_to_f16
    return np.array([f(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def dequant_kq_f16(fmt: str, w: np.ndarray, k: int, _o: Oracle | None = None) -> np.ndarray:
    """O8a: K-quant superblock bytes (fmt "q6_k", "q4_k" or "q5_k") -> fp16 bits uint16 [n, k],
    each the correctly rounded binary16 of the weight's exact value."""
    code, sbytes = _kq(fmt)
    _check_kk(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    n = w.size // (k // QK_K * sbytes)
    out = np.empty((n, k), dtype=np.uint16)
    (_o or _DEFAULT).lib().oracle_dequant_kq_f16(code, _ptr(w), _ptr(out), n, k)
    return out


def block_dots_kq(fmt: str, w: np.ndarray, xq: np.ndarray, k: int, rows=None, _o: Oracle | None = None):
    """O8b: the exact int32 integers of every 32-wide block [t, j, b] that the fold consumes
    (Q6_K: the scale-weighted sum of its two 16-wide dots; Q4_K / Q5_K: sum q * xq)."""
    code, sbytes = _kq(fmt)
    _check_kk(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    n = w.size // (k // QK_K * sbytes)
    m = xq.size // k
    rows, nr = _rows_arg(rows, n)
    D = np.empty((m, nr, k // QK), dtype=np.int32)
    (_o or _DEFAULT).lib().oracle_block_dots_kq(code, _ptr(w), _ptr(xq), _ptr(D), m, n, k, _ptr(rows), nr)
    return D


def matmul_kq(fmt: str, w: np.ndarray, xq: np.ndarray, xd: np.ndarray, k: int, rows=None,
              _o: Oracle | None = None):
    """O8c: returns (y32 f32 [m, nr], y64 f64 [m, nr], S f64 [m, nr]) over K-quant weights."""
    code, sbytes = _kq(fmt)
    _check_kk(k)
    w = np.ascontiguousarray(w, dtype=np.uint8)
    xq = np.ascontiguousarray(xq, dtype=np.int8)
    xd = np.ascontiguousarray(xd, dtype=np.float32)
    n = w.size // (k // QK_K * sbytes)
    m = xq.size // k
    rows, nr = _rows_arg(rows, n)
    y32 = np.empty((m, nr), dtype=np.float32)
    y64 = np.empty((m, nr), dtype=np.float64)
    S = np.empty((m, nr), dtype=np.float64)
    (_o or _DEFAULT).lib().oracle_matmul_kq(code, _ptr(w), _ptr(xq), _ptr(xd), m, n, k, _ptr(rows), nr,
                                            _ptr(y32), _ptr(y64), _ptr(S))
    return y32, y64, S


_DEFAULT = Oracle()

_PUBLIC = ("f32_to_f16", "f16_to_f32", "quantize_q8_0", "quantize_q8_1", "block_dots",
           "matmul", "dequant_f16", "repack_q8_0", "quantize_q4_0", "dequant_q4_0_f16",
           "block_dots_q4_0", "matmul_q4_0", "f64_to_f16", "dequant_kq_f16", "block_dots_kq",
           "matmul_kq")


def bound(o: Oracle):
    """A namespace with the public functions bound to the compiled copy ``o``."""
    import types
    import functools
    g = globals()
    return types.SimpleNamespace(**{n: functools.partial(g[n], _o=o) for n in _PUBLIC})
