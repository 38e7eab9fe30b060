"""CPU oracle for dense GEMM -- TEST INFRASTRUCTURE ONLY.

Only the test suite, ``__graft_entry__.smoke()`` and ``bench.py``'s CPU-baseline
leg may import this package.  The product path (``dense_gemm_tcgen05_gb300``)
never imports, links or calls it, and this package never imports the product.

The arithmetic lives in ``oracle.c`` (plain C, binary64 accumulation in plain
k order, exact decoders written from the format definitions).  This module
only compiles that file and marshals numpy arrays to it.

Layouts (all element offsets):
  TN (fp16, bf16, e4m3):  A[m*lda + k], B[n*ldb + k], C[n*ldc + m]
      ("FP16 GEMM Optimization on AMD RDNA 3 and RDNA 4", "What We Are Computing")
  FP32 row-major:         A[m*lda + k], B[k*ldb + n], C[m*ldc + n]
      ("Optimizing GEMM in HIP", "GEMM fundamentals" and Step 1)

Every function here is pinned by ``tests/test_oracle.py``; none is unpinned.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB = os.path.join(_HERE, "liboracle.so")

F16, BF16, E4M3 = 0, 1, 2
_DTYPES = {"f16": F16, "fp16": F16, "bf16": BF16, "e4m3": E4M3, "fp8": E4M3}

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into liboracle.so (gcc, OpenMP).  Returns the path."""
    stale = (not os.path.exists(_LIB)) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC)
    if force or stale:
        tmp = _LIB + ".tmp.%d" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c99", "-fopenmp", "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB)
        i64, dbl, vp, i32 = ctypes.c_int64, ctypes.c_double, ctypes.c_void_p, ctypes.c_int
        lib.oracle_dec_array.argtypes = [i32, vp, i64, vp]
        lib.oracle_dec_array.restype = None
        lib.oracle_enc_array.argtypes = [i32, vp, i64, vp]
        lib.oracle_enc_array.restype = None
        lib.oracle_gemm_tn.argtypes = [i32, i64, i64, i64, vp, i64, vp, i64, dbl, dbl, vp, i64]
        lib.oracle_gemm_tn.restype = i32
        lib.oracle_gemm_tn_sampled.argtypes = [i32, i64, vp, i64, vp, i64, dbl, dbl, i64, vp, vp, vp]
        lib.oracle_gemm_tn_sampled.restype = i32
        lib.oracle_gemm_f32.argtypes = [i64, i64, i64, vp, i64, vp, i64, vp, i64]
        lib.oracle_gemm_f32.restype = i32
        lib.oracle_gemm_f32_sampled.argtypes = [i64, vp, i64, vp, i64, i64, vp, vp, vp]
        lib.oracle_gemm_f32_sampled.restype = i32
        lib.oracle_num_threads.argtypes = []
        lib.oracle_num_threads.restype = i32
        lib.oracle_set_num_threads.argtypes = [i32]
        lib.oracle_set_num_threads.restype = i32
        _lib = lib
        return lib


def _dtype_id(dtype) -> int:
    if isinstance(dtype, int):
        return dtype
    return _DTYPES[str(dtype)]


def _codes(arr: np.ndarray, dt: int) -> np.ndarray:
    want = np.uint8 if dt == E4M3 else np.uint16
    a = np.ascontiguousarray(arr)
    if a.dtype != want:
        if a.dtype.itemsize != np.dtype(want).itemsize:
            raise TypeError("storage codes must be %d-byte integers" % np.dtype(want).itemsize)
        a = a.view(want)
    return a


def _ptr(a: np.ndarray) -> int:
    return a.ctypes.data


def num_threads() -> int:
    return int(_load().oracle_num_threads())


def set_num_threads(n: int) -> int:
    """Threads for later oracle calls (n >= 1); returns the count in effect."""
    return int(_load().oracle_set_num_threads(int(n)))


def decode(dtype, codes: np.ndarray) -> np.ndarray:
    """Exact binary64 value of every storage code (fp16/bf16 as uint16, e4m3 as uint8)."""
    dt = _dtype_id(dtype)
    c = _codes(codes, dt)
    out = np.empty(c.shape, dtype=np.float64)
    _load().oracle_dec_array(dt, _ptr(c), c.size, _ptr(out))
    return out


def encode_rne(dtype, x: np.ndarray) -> np.ndarray:
    """Round binary64 values to fp16 or bf16 codes (uint16), nearest-even."""
    dt = _dtype_id(dtype)
    if dt not in (F16, BF16):
        raise ValueError("encoder exists for fp16 and bf16 only")
    xx = np.ascontiguousarray(x, dtype=np.float64)
    out = np.empty(xx.shape, dtype=np.uint16)
    _load().oracle_enc_array(dt, _ptr(xx), xx.size, _ptr(out))
    return out


def gemm_tn(dtype, M: int, N: int, K: int, A: np.ndarray, lda: int, B: np.ndarray, ldb: int,
            scale_a: float = 1.0, scale_b: float = 1.0) -> np.ndarray:
    """Full TN product in binary64, returned as a logical (M, N) array C[m, n].

    A holds storage codes with a(m,k) = A.flat[m*lda + k]; B holds b(k,n) = B.flat[n*ldb + k].
    """
    dt = _dtype_id(dtype)
    a, b = _codes(A, dt), _codes(B, dt)
    if M and K:
        assert a.size >= (M - 1) * lda + K, "A too small for M, K, lda"
    if N and K:
        assert b.size >= (N - 1) * ldb + K, "B too small for N, K, ldb"
    c = np.zeros((max(N, 0), max(M, 0)), dtype=np.float64)  # column-major C, ldc = M
    rc = _load().oracle_gemm_tn(dt, M, N, K, _ptr(a), lda, _ptr(b), ldb, float(scale_a),
                                float(scale_b), _ptr(c), max(M, 1))
    if rc:
        raise RuntimeError("oracle_gemm_tn failed: %d" % rc)
    return c.T


def gemm_tn_sampled(dtype, K: int, A: np.ndarray, lda: int, B: np.ndarray, ldb: int,
                    ms: np.ndarray, ns: np.ndarray, scale_a: float = 1.0,
                    scale_b: float = 1.0) -> np.ndarray:
    """C(ms[s], ns[s]) for every sample s, each one K-long binary64 dot product."""
    dt = _dtype_id(dtype)
    a, b = _codes(A, dt), _codes(B, dt)
    ms64 = np.ascontiguousarray(ms, dtype=np.int64)
    ns64 = np.ascontiguousarray(ns, dtype=np.int64)
    assert ms64.shape == ns64.shape
    out = np.empty(ms64.shape, dtype=np.float64)
    rc = _load().oracle_gemm_tn_sampled(dt, K, _ptr(a), lda, _ptr(b), ldb, float(scale_a),
                                        float(scale_b), ms64.size, _ptr(ms64), _ptr(ns64),
                                        _ptr(out))
    if rc:
        raise RuntimeError("oracle_gemm_tn_sampled failed: %d" % rc)
    return out


def gemm_f32(M: int, N: int, K: int, A: np.ndarray, lda: int, B: np.ndarray,
             ldb: int) -> np.ndarray:
    """Full row-major FP32 product in binary64, returned as an (M, N) array."""
    a = np.ascontiguousarray(A, dtype=np.float32)
    b = np.ascontiguousarray(B, dtype=np.float32)
    if M and K:
        assert a.size >= (M - 1) * lda + K
    if K and N:
        assert b.size >= (K - 1) * ldb + N
    c = np.zeros((max(M, 0), max(N, 0)), dtype=np.float64)
    rc = _load().oracle_gemm_f32(M, N, K, _ptr(a), lda, _ptr(b), ldb, _ptr(c), max(N, 1))
    if rc:
        raise RuntimeError("oracle_gemm_f32 failed: %d" % rc)
    return c


def gemm_f32_sampled(K: int, A: np.ndarray, lda: int, B: np.ndarray, ldb: int, ms: np.ndarray,
                     ns: np.ndarray) -> np.ndarray:
    a = np.ascontiguousarray(A, dtype=np.float32)
    b = np.ascontiguousarray(B, dtype=np.float32)
    ms64 = np.ascontiguousarray(ms, dtype=np.int64)
    ns64 = np.ascontiguousarray(ns, dtype=np.int64)
    out = np.empty(ms64.shape, dtype=np.float64)
    rc = _load().oracle_gemm_f32_sampled(K, _ptr(a), lda, _ptr(b), ldb, ms64.size, _ptr(ms64),
                                         _ptr(ns64), _ptr(out))
    if rc:
        raise RuntimeError("oracle_gemm_f32_sampled failed: %d" % rc)
    return out
