"""CPU oracle for the generalized GEMM with a fused epilogue (test infrastructure).

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package.  The GPU library never
imports it and shares no code with it; the C source (``oracle.c``) is compiled
with the host C compiler, not nvcc.

What it computes (see the header of ``oracle.c`` for the passages it follows):

    D[i,j] = cast_out(act(alpha * sum_k a(i,k) b(k,j) + beta * C[i,j] + bias))

with fp64 accumulation for floating inputs, int64 for int8 inputs; and the same
GEMM over complex or dual numbers stored interleaved (``gemm_pairs``: the
section 5.4 variants of "Flexible Performant GEMM Kernels on GPUs").

Every function here is marshalling only: pointers, sizes and type codes go to
the C routines unchanged.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "liboracle.so")

# The oracle's own type codes (mirrors the enum at the top of oracle.c).
F32, F16, BF16, S8, S32 = 0, 1, 2, 3, 4
LAYOUT_N, LAYOUT_T = 0, 1
ACT_NONE, ACT_RELU = 0, 1
BIAS_NONE, BIAS_COL, BIAS_ROW = 0, 1, 2
UNIT_IMAGINARY, UNIT_DUAL = 0, 1     # complex numbers (i*i = -1), dual numbers (eps*eps = 0)

_lib = None
_lock = threading.Lock()


def build(force: bool = False) -> str:
    """Compile oracle.c into a shared library with gcc (OpenMP over rows)."""
    os.makedirs(_BUILD_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    with _lock:
        if _lib is not None:
            return _lib
        return _load_from(build())


def _load_from(path: str):
    """Load the oracle library at `path` and make it the active one."""
    global _lib
    lib = ctypes.CDLL(path)
    i64, dbl, vp, ci = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
    lib.oracle_gemm.restype = i64
    lib.oracle_gemm.argtypes = [ci, ci, ci, i64, i64, i64, dbl, vp, i64, vp, i64,
                                dbl, ci, vp, i64, ci, vp, ci, ci, ci, ci, vp, i64, ci, ci, dbl,
                                ci, dbl, ci, dbl]
    lib.oracle_gemm_entries.restype = i64
    lib.oracle_gemm_entries.argtypes = [ci, ci, ci, i64, i64, i64, dbl, vp, i64, vp, i64,
                                        dbl, ci, vp, i64, ci, vp, ci, ci, ci, ci, i64, vp, vp,
                                        vp, ci, dbl, ci, dbl, ci, dbl]
    lib.oracle_gemm_pairs.restype = i64
    lib.oracle_gemm_pairs.argtypes = [ci, ci, ci, ci, i64, i64, i64, dbl, vp, i64, vp, i64,
                                      dbl, ci, vp, i64, ci, vp, ci, ci, ci, ci, vp, i64, ci]
    lib.oracle_gemm_pairs_entries.restype = i64
    lib.oracle_gemm_pairs_entries.argtypes = [ci, ci, ci, ci, i64, i64, i64, dbl, vp, i64, vp, i64,
                                              dbl, ci, vp, i64, ci, vp, ci, ci, ci, ci, i64, vp,
                                              vp, vp, ci]
    lib.oracle_f16_to_double.restype = dbl
    lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_bf16_to_double.restype = dbl
    lib.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
    lib.oracle_f16_from_double.restype = ctypes.c_uint16
    lib.oracle_f16_from_double.argtypes = [dbl]
    lib.oracle_bf16_from_double.restype = ctypes.c_uint16
    lib.oracle_bf16_from_double.argtypes = [dbl]
    lib.oracle_max_threads.restype = ci
    lib.oracle_max_threads.argtypes = []
    _lib = lib
    return lib


def _ptr(buf):
    """Raw address of a host buffer (numpy array or CPU torch tensor), or None."""
    if buf is None:
        return None
    if isinstance(buf, np.ndarray):
        return buf.ctypes.data
    # torch tensor on the CPU
    if getattr(buf, "is_cuda", False):
        raise ValueError("the oracle reads host memory only")
    return buf.data_ptr()


_OUT_NP = {F32: np.float32, F16: np.uint16, BF16: np.uint16, S32: np.int32, S8: np.int8}


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def gemm(ab_dtype, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb,
         beta=0.0, c_dtype=F32, C=None, ldc=0, bias_dtype=F32, bias=None,
         bias_mode=BIAS_NONE, act=ACT_NONE, d_dtype=F32, ldd=None,
         loop_order=0, nthreads=None, c_act=ACT_NONE, out_scale=1.0,
         a_act=ACT_NONE, a_scale=1.0, b_act=ACT_NONE, b_scale=1.0):
    """Full D (row-major M x ldd, raw bits for 16-bit outputs) and the int32
    overflow count.  Buffers are raw storage: numpy arrays or CPU tensors.
    a_act/a_scale, b_act/b_scale: the transforms of A and B after load."""
    if ldd is None:
        ldd = N
    if nthreads is None:
        nthreads = max_threads()
    D = np.zeros((M, ldd), dtype=_OUT_NP[d_dtype])
    n = _load().oracle_gemm(ab_dtype, layout_a, layout_b, M, N, K, float(alpha),
                            _ptr(A), lda, _ptr(B), ldb, float(beta), c_dtype, _ptr(C), ldc,
                            bias_dtype, _ptr(bias), bias_mode, act, c_act, d_dtype,
                            D.ctypes.data, ldd, loop_order, nthreads, float(out_scale),
                            a_act, float(a_scale), b_act, float(b_scale))
    if n < 0:
        raise ValueError("oracle_gemm: invalid arguments")
    return D, int(n)


def gemm_entries(ab_dtype, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb,
                 rows, cols, beta=0.0, c_dtype=F32, C=None, ldc=0, bias_dtype=F32,
                 bias=None, bias_mode=BIAS_NONE, act=ACT_NONE, d_dtype=F32, nthreads=None,
                 c_act=ACT_NONE, out_scale=1.0, a_act=ACT_NONE, a_scale=1.0, b_act=ACT_NONE,
                 b_scale=1.0):
    """D at the listed (rows[e], cols[e]) entries, in d_dtype (raw bits for 16-bit)."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if nthreads is None:
        nthreads = max_threads()
    out = np.zeros(rows.shape[0], dtype=_OUT_NP[d_dtype])
    n = _load().oracle_gemm_entries(ab_dtype, layout_a, layout_b, M, N, K, float(alpha),
                                    _ptr(A), lda, _ptr(B), ldb, float(beta), c_dtype, _ptr(C),
                                    ldc, bias_dtype, _ptr(bias), bias_mode, act, c_act, d_dtype,
                                    rows.shape[0], rows.ctypes.data, cols.ctypes.data,
                                    out.ctypes.data, nthreads, float(out_scale),
                                    a_act, float(a_scale), b_act, float(b_scale))
    if n < 0:
        raise ValueError("oracle_gemm_entries: invalid arguments")
    return out, int(n)


def f16_to_double(bits: int) -> float:
    return _load().oracle_f16_to_double(bits)


def bf16_to_double(bits: int) -> float:
    return _load().oracle_bf16_to_double(bits)


def f16_from_double(x: float) -> int:
    return int(_load().oracle_f16_from_double(x))


def bf16_from_double(x: float) -> int:
    return int(_load().oracle_bf16_from_double(x))


def decode(bits: np.ndarray, dtype: int) -> np.ndarray:
    """Widen an output array to float64 (16-bit outputs are raw bits)."""
    lib = _load()
    if dtype == F16:
        f = np.vectorize(lambda b: lib.oracle_f16_to_double(int(b)), otypes=[np.float64])
        return f(bits)
    if dtype == BF16:
        f = np.vectorize(lambda b: lib.oracle_bf16_to_double(int(b)), otypes=[np.float64])
        return f(bits)
    return bits.astype(np.float64)


def gemm_pairs(unit, ab_dtype, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb,
               beta=0.0, c_dtype=F32, C=None, ldc=0, bias_dtype=F32, bias=None,
               bias_mode=BIAS_NONE, act=ACT_NONE, d_dtype=F32, ldd=None, nthreads=None,
               c_act=ACT_NONE):
    """Complex (unit UNIT_IMAGINARY) or dual (UNIT_DUAL) GEMM on interleaved
    storage; sizes and leading dimensions count pairs.  Returns D with shape
    (M, ldd, 2): [..., 0] the real parts, [..., 1] the unit parts (raw bits
    for 16-bit outputs)."""
    if ldd is None:
        ldd = N
    if nthreads is None:
        nthreads = max_threads()
    D = np.zeros((M, ldd, 2), dtype=_OUT_NP[d_dtype])
    n = _load().oracle_gemm_pairs(unit, ab_dtype, layout_a, layout_b, M, N, K, float(alpha),
                                  _ptr(A), lda, _ptr(B), ldb, float(beta), c_dtype, _ptr(C), ldc,
                                  bias_dtype, _ptr(bias), bias_mode, act, c_act, d_dtype,
                                  D.ctypes.data, ldd, nthreads)
    if n < 0:
        raise ValueError("oracle_gemm_pairs: invalid arguments")
    return D


def gemm_pairs_entries(unit, ab_dtype, layout_a, layout_b, M, N, K, alpha, A, lda, B, ldb,
                       rows, cols, beta=0.0, c_dtype=F32, C=None, ldc=0, bias_dtype=F32,
                       bias=None, bias_mode=BIAS_NONE, act=ACT_NONE, d_dtype=F32, nthreads=None,
                       c_act=ACT_NONE):
    """The output pairs at (rows[e], cols[e]); shape (n, 2)."""
    rows = np.ascontiguousarray(rows, dtype=np.int64)
    cols = np.ascontiguousarray(cols, dtype=np.int64)
    if nthreads is None:
        nthreads = max_threads()
    out = np.zeros((rows.shape[0], 2), dtype=_OUT_NP[d_dtype])
    n = _load().oracle_gemm_pairs_entries(unit, ab_dtype, layout_a, layout_b, M, N, K,
                                          float(alpha), _ptr(A), lda, _ptr(B), ldb, float(beta),
                                          c_dtype, _ptr(C), ldc, bias_dtype, _ptr(bias), bias_mode,
                                          act, c_act, d_dtype, rows.shape[0], rows.ctypes.data,
                                          cols.ctypes.data, out.ctypes.data, nthreads)
    if n < 0:
        raise ValueError("oracle_gemm_pairs_entries: invalid arguments")
    return out
