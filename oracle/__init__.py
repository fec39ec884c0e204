"""MXFP4 oracle: plain single-threaded fp64 CPU implementation (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the CUDA library and
its binding in ``precision_bf16_mxfp4_gb300``) never imports it, and this
package imports nothing from the product.

The arithmetic lives in ``mxfp4_oracle.c`` (compiled with gcc, no CUDA); this
module only builds it and marshals numpy arrays.  Every function here cites
the page passage its C counterpart follows; see the header comment of
``mxfp4_oracle.c``.

Parity pins: every function is pinned by ``tests/test_oracle_pins.py`` against
values fixed independently of this code (hand-worked examples under
``tests/golden/``, closed forms, exhaustive comparison with an independent
threshold formulation, exact rational brute force, and reduction to a plain
matmul).  No function is "parity unpinned".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "mxfp4_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile mxfp4_oracle.c into a shared library with gcc (no fast-math)."""
    os.makedirs(os.path.dirname(_LIB_PATH), exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math",
             "-ffp-contract=off", "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            p = ctypes.c_void_p
            i64 = ctypes.c_int64
            lib.oracle_block_exponent.argtypes = [p, i64]
            lib.oracle_block_exponent.restype = ctypes.c_int
            lib.oracle_e2m1_code.argtypes = [ctypes.c_double]
            lib.oracle_e2m1_code.restype = ctypes.c_int
            lib.oracle_encode.argtypes = [ctypes.c_uint16, ctypes.c_int]
            lib.oracle_encode.restype = ctypes.c_int
            lib.oracle_quant.argtypes = [p, i64, i64, i64, p, p]
            lib.oracle_quant.restype = None
            lib.oracle_dequant.argtypes = [p, p, i64, i64, p]
            lib.oracle_dequant.restype = None
            lib.oracle_gemm.argtypes = [p, p, p, p, i64, i64, i64, p]
            lib.oracle_gemm.restype = None
            lib.oracle_gemm_entries.argtypes = [p, p, p, p, i64, p, p, i64, p]
            lib.oracle_gemm_entries.restype = None
            lib.oracle_encode_many.argtypes = [p, p, i64, p]
            lib.oracle_encode_many.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _bf16_bits(a) -> np.ndarray:
    """Accept a uint16 array of bf16 bit patterns or a torch bfloat16 tensor."""
    if hasattr(a, "dtype") and str(a.dtype) == "torch.bfloat16":
        a = a.contiguous().view(__import__("torch").int16).numpy().view(np.uint16)
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("expected bf16 bit patterns as uint16")
    return a


def block_exponent(block_bits) -> int:
    """ub of one block (submission 694791 "MXFP4 quantization": amax round-up, -2, clamp)."""
    b = _bf16_bits(block_bits)
    return int(_load().oracle_block_exponent(_ptr(b), b.size))


def e2m1_code(q: float) -> int:
    """Nearest e2m1 magnitude code of q >= 0, ties to even, saturating at 6.0."""
    return int(_load().oracle_e2m1_code(float(q)))


def encode(x_bits: int, ub: int) -> int:
    """4-bit nibble of one bf16 element under block exponent ub."""
    return int(_load().oracle_encode(int(x_bits) & 0xFFFF, int(ub)))


def encode_many(x_bits, ub) -> np.ndarray:
    """Vectorised :func:`encode` over equal-length arrays of bf16 bits and ub."""
    x = np.ascontiguousarray(x_bits, np.uint16)
    u = np.ascontiguousarray(ub, np.int32)
    if x.shape != u.shape:
        raise ValueError("shape mismatch")
    out = np.zeros(x.shape, np.uint8)
    _load().oracle_encode_many(_ptr(x), _ptr(u), x.size, _ptr(out))
    return out


def quant(a_bits, m: int | None = None, k: int | None = None):
    """bf16 [m,k] -> (fp4x2 [m,k/2] u8, e8m0 [m,k/32] u8) (submission 694791 quantizer and packing)."""
    a = _bf16_bits(a_bits)
    if a.ndim != 2:
        raise ValueError("A must be 2-D")
    m, k = a.shape
    if k % 32:
        raise ValueError("k must be a multiple of 32")
    q = np.zeros((m, k // 2), np.uint8)
    s = np.zeros((m, k // 32), np.uint8)
    _load().oracle_quant(_ptr(a), m, k, k, _ptr(q), _ptr(s))
    return q, s


def dequant(q: np.ndarray, s: np.ndarray) -> np.ndarray:
    """MXFP4 [r,k] -> fp64 [r,k]; e8m0 byte e means 2^(e-127), 0 included."""
    q = np.ascontiguousarray(q, np.uint8)
    s = np.ascontiguousarray(s, np.uint8)
    r, k = q.shape[0], q.shape[1] * 2
    out = np.zeros((r, k), np.float64)
    _load().oracle_dequant(_ptr(q), _ptr(s), r, k, _ptr(out))
    return out


def gemm(aq, a_s, bq, b_s) -> np.ndarray:
    """C = deq(A) . deq(B)^T in fp64 (submission 752099 `tl.dot_scaled` semantics)."""
    aq = np.ascontiguousarray(aq, np.uint8)
    a_s = np.ascontiguousarray(a_s, np.uint8)
    bq = np.ascontiguousarray(bq, np.uint8)
    b_s = np.ascontiguousarray(b_s, np.uint8)
    m, n, k = aq.shape[0], bq.shape[0], aq.shape[1] * 2
    if bq.shape[1] * 2 != k:
        raise ValueError("A and B disagree on k")
    c = np.zeros((m, n), np.float64)
    _load().oracle_gemm(_ptr(aq), _ptr(a_s), _ptr(bq), _ptr(b_s), m, n, k, _ptr(c))
    return c


def gemm_entries(aq, a_s, bq, b_s, rows, cols) -> np.ndarray:
    """The fp64 GEMM evaluated only at the listed (row, col) pairs."""
    aq = np.ascontiguousarray(aq, np.uint8)
    a_s = np.ascontiguousarray(a_s, np.uint8)
    bq = np.ascontiguousarray(bq, np.uint8)
    b_s = np.ascontiguousarray(b_s, np.uint8)
    rows = np.ascontiguousarray(rows, np.int64)
    cols = np.ascontiguousarray(cols, np.int64)
    k = aq.shape[1] * 2
    out = np.zeros(rows.size, np.float64)
    _load().oracle_gemm_entries(_ptr(aq), _ptr(a_s), _ptr(bq), _ptr(b_s), k,
                                _ptr(rows), _ptr(cols), rows.size, _ptr(out))
    return out


def gemm_via_dequant(aq, a_s, bq, b_s) -> np.ndarray:
    """Same definition as :func:`gemm`, with the fp64 sum taken by numpy's matmul.

    The products deq(A)[i,k]*deq(B)[j,k] and their fp64 sum are the definition
    of submission 752099 (`tl.dot_scaled`); a library matmul only changes the fp64
    summation order.  Used where the plain loop would take minutes.
    """
    return dequant(aq, a_s) @ dequant(bq, b_s).T
