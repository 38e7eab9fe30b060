"""ctypes binding of libgemm.so with the C ABI's own names and arguments.

Argument marshalling only: every function forwards integers, floats and raw
device pointers (Python ints) to the library and returns its status code.  The
library must have been built (``dense_gemm_tcgen05_gb300.build``); loading
fails loudly otherwise -- there is no fallback of any kind.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import build as _build

LIB_PATH = _build.LIB
HEADER = os.path.join(_build.INCLUDE, "gemm.h")

GEMM_OK = 0
GEMM_ERR_INVALID_DIM = 1
GEMM_ERR_INVALID_LD = 2
GEMM_ERR_NULL_PTR = 3
GEMM_ERR_MISALIGNED = 4
GEMM_ERR_UNSUPPORTED_DEVICE = 5
GEMM_ERR_LAUNCH = 6
GEMM_ERR_TIMEOUT = 7
GEMM_ERR_INVALID_OPTION = 8
GEMM_ERR_SCRATCH = 9
GEMM_ERR_WORKSPACE = 10

_lock = threading.Lock()
_lib = None

_i64, _f32, _vp, _int = ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_int
_SIGNATURES = {
    "gemm_f32": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp], _int),
    "gemm_f16_tn": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp], _int),
    "gemm_bf16_tn": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp], _int),
    "gemm_f16_tn_acc16": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp], _int),
    "gemm_fp8_tn": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _f32, _f32, _vp, _i64, _vp], _int),
    "gemm_fp8_tn_f32": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _f32, _f32, _vp, _i64, _vp], _int),
    "gemm_status_string": ([_int], ctypes.c_char_p),
    "gemm_read_watchdog": ([_int], _int),
    "gemm_set_option": ([ctypes.c_char_p, _i64], _int),
    "gemm_tile_coord": ([_i64, _i64, _i64, _i64, _int, ctypes.POINTER(_i64), ctypes.POINTER(_i64)],
                        _int),
    "gemm_watchdog_selftest": ([_i64, _vp], _int),
    "gemm_set_workspace": ([_vp, _i64], _int),
    "gemm_bf16_tn_noalloc": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _i64, _vp], _int),
    "gemm_workspace_bytes": ([_i64, _i64, _i64], _i64),
    "gemm_f32_bf16x6": ([_i64, _i64, _i64, _vp, _i64, _vp, _i64, _vp, _i64, _vp], _int),
    "gemm_f32_bf16x6_workspace_bytes": ([_i64, _i64, _i64], _i64),
    "gemm_tn_plan": ([_int, _i64, _i64, _i64, _int, _i64, _int, ctypes.POINTER(_i64), _int],
                     _int),
}

PLAN_KINDS = {"f16": 0, "bf16": 1, "e4m3": 2, "f16_acc16": 3, "e4m3_f32out": 4}
PLAN_A_TMA, PLAN_B_TMA, PLAN_C_TMA, PLAN_A_128, PLAN_B_128, PLAN_NOALLOC = 1, 2, 4, 8, 16, 32
GEMM_NOALLOC_SCRATCH_BYTES = 24 << 20
PLAN_ALIGNED = PLAN_A_TMA | PLAN_B_TMA | PLAN_C_TMA | PLAN_A_128 | PLAN_B_128
PLAN_FIELDS = ("status", "pair", "producer", "tile_q", "half", "splits", "tail_f", "tail_ksplit",
               "stages", "grid", "copy_a", "copy_b", "tiles_p", "tiles_q",
               "kb_per_split", "tail_kb_per", "stage_bytes", "issuers", "atoms", "ring_epi")


class GemmError(RuntimeError):
    def __init__(self, status: int, where: str = ""):
        self.status = status
        super().__init__("%s failed: status %d (%s)" % (where or "gemm", status, status_text(status)))


def lib() -> ctypes.CDLL:
    """The loaded library.  Raises if libgemm.so has not been built."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    "libgemm.so is missing (%s); build it with "
                    "`python -m dense_gemm_tcgen05_gb300.build`" % LIB_PATH)
            handle = ctypes.CDLL(LIB_PATH)
            for name, (args, res) in _SIGNATURES.items():
                fn = getattr(handle, name)
                fn.argtypes = args
                fn.restype = res
            _lib = handle
        return _lib


def declared_symbols() -> list[str]:
    """Function names declared in include/gemm.h."""
    text = open(HEADER).read()
    return sorted(set(re.findall(r"^\s*(?:const\s+)?\w+\*?\s+\**(gemm_\w+)\s*\(", text, re.M)))


def status_text(status: int) -> str:
    try:
        return lib().gemm_status_string(int(status)).decode()
    except Exception:  # pragma: no cover - library not loadable
        return "status %d" % status


def _p(x) -> int | None:
    return None if x is None else int(x)


def gemm_f32(M, N, K, A, lda, B, ldb, C, ldc, stream=None) -> int:
    return lib().gemm_f32(M, N, K, _p(A), lda, _p(B), ldb, _p(C), ldc, _p(stream))


def gemm_f32_bf16x6(M, N, K, A, lda, B, ldb, C, ldc, stream=None) -> int:
    return lib().gemm_f32_bf16x6(M, N, K, _p(A), lda, _p(B), ldb, _p(C), ldc, _p(stream))


def gemm_f32_bf16x6_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib().gemm_f32_bf16x6_workspace_bytes(M, N, K)


def gemm_tn_plan(kind: str, M: int, N: int, K: int, flags: int = PLAN_ALIGNED,
                 workspace_bytes: int = 0, sms: int = 152):
    """(status, plan dict) of what a TN call would run (no GPU needed)."""
    out = (_i64 * len(PLAN_FIELDS))()
    st = lib().gemm_tn_plan(PLAN_KINDS[kind], M, N, K, flags, workspace_bytes, sms, out,
                            len(PLAN_FIELDS))
    return st, dict(zip(PLAN_FIELDS, (int(v) for v in out)))


def gemm_f16_tn(M, N, K, A, lda, B, ldb, C, ldc, stream=None) -> int:
    return lib().gemm_f16_tn(M, N, K, _p(A), lda, _p(B), ldb, _p(C), ldc, _p(stream))


def gemm_f16_tn_acc16(M, N, K, A, lda, B, ldb, C, ldc, stream=None) -> int:
    return lib().gemm_f16_tn_acc16(M, N, K, _p(A), lda, _p(B), ldb, _p(C), ldc, _p(stream))


def gemm_bf16_tn(M, N, K, A, lda, B, ldb, C, ldc, stream=None) -> int:
    return lib().gemm_bf16_tn(M, N, K, _p(A), lda, _p(B), ldb, _p(C), ldc, _p(stream))


def gemm_fp8_tn(M, N, K, A, lda, B, ldb, scale_a, scale_b, C, ldc, stream=None) -> int:
    return lib().gemm_fp8_tn(M, N, K, _p(A), lda, _p(B), ldb, float(scale_a), float(scale_b),
                             _p(C), ldc, _p(stream))


def gemm_fp8_tn_f32(M, N, K, A, lda, B, ldb, scale_a, scale_b, C, ldc, stream=None) -> int:
    return lib().gemm_fp8_tn_f32(M, N, K, _p(A), lda, _p(B), ldb, float(scale_a),
                                 float(scale_b), _p(C), ldc, _p(stream))


def gemm_status_string(status: int) -> str:
    return status_text(status)


def gemm_read_watchdog(reset: int = 0) -> int:
    return lib().gemm_read_watchdog(int(reset))


def gemm_set_option(name: str, value: int) -> int:
    return lib().gemm_set_option(name.encode(), int(value))


def gemm_tile_coord(t: int, tiles_m: int, tiles_n: int, group: int, snake: int = 0):
    tm, tn = _i64(), _i64()
    st = lib().gemm_tile_coord(t, tiles_m, tiles_n, group, int(snake), ctypes.byref(tm),
                               ctypes.byref(tn))
    return st, tm.value, tn.value


def gemm_set_workspace(ptr, nbytes: int) -> int:
    return lib().gemm_set_workspace(_p(ptr), int(nbytes))


def gemm_bf16_tn_noalloc(M, N, K, A, lda, B, ldb, C, ldc, splits=0, stream=None) -> int:
    return lib().gemm_bf16_tn_noalloc(M, N, K, _p(A), lda, _p(B), ldb, _p(C), ldc, int(splits),
                                      _p(stream))


def gemm_workspace_bytes(M: int, N: int, K: int) -> int:
    return lib().gemm_workspace_bytes(M, N, K)


def gemm_watchdog_selftest(limit_ns: int, stream=None) -> int:
    return lib().gemm_watchdog_selftest(int(limit_ns), _p(stream))
