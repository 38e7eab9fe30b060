"""Seeded synthetic inputs for dense GEMM.

This module is shared by the tests, the benchmark and the smoke check.  It
holds no GEMM arithmetic: it only draws random numbers, casts them to the
storage formats (the casts are the inputs both sides then see), and lays them
out with the leading dimensions a call asks for.  Neither the CUDA library nor
the oracle imports it.

Distributions (the pages use synthetic data only):
  "pm1"      entries uniform on {-1, +1}  ("FP16 GEMM Optimization on AMD RDNA 3
             and RDNA 4", "What We Are Computing": the exact check)
  "uniform"  entries uniform on [-1, 1)
  "normal"   entries N(0, 1) * sigma
  "ones"     every entry 1
  "identity" the identity matrix (B = I  =>  C = A; "Optimizing GEMM in HIP",
             introduction: the identity-matrix test)

Generator: ``torch.Generator('cpu').manual_seed(seed)``; A is drawn before B
from the same generator.  Sample positions use a second generator seeded with
``seed + 1000``.

FP8 E4M3 inputs are drawn in float32, then quantised per tensor with
scale = amax / 448 (scale = 1 when amax = 0): q = e4m3(clamp(x / scale, +-448)),
torch's round-to-nearest-even cast.  The scales are returned with the codes.

Padding columns (k >= K when ld > K) are filled with NaN codes so that a
kernel reading past K poisons its sums.
"""
from __future__ import annotations

import numpy as np
import torch

E4M3_MAX = 448.0
_EXACT = ("pm1", "ones", "identity", "zeros")

_TORCH_DTYPES = {
    "f16": torch.float16,
    "bf16": torch.bfloat16,
    "e4m3": torch.float8_e4m3fn,
    "f32": torch.float32,
}
_NAN_CODES = {"f16": 0x7E00, "bf16": 0x7FC0, "e4m3": 0x7F}


def torch_dtype(kind: str) -> torch.dtype:
    return _TORCH_DTYPES[kind]


def elem_size(kind: str) -> int:
    return {"f16": 2, "bf16": 2, "e4m3": 1, "f32": 4}[kind]


def draw(gen: torch.Generator, rows: int, cols: int, dist: str, sigma: float = 1.0) -> torch.Tensor:
    """A (rows, cols) float32 CPU tensor from the named distribution."""
    shape = (rows, cols)
    if dist == "pm1":
        return torch.randint(0, 2, shape, generator=gen, dtype=torch.int32).to(torch.float32) * 2 - 1
    if dist == "uniform":
        return torch.rand(shape, generator=gen, dtype=torch.float32) * 2 - 1
    if dist == "normal":
        return torch.randn(shape, generator=gen, dtype=torch.float32) * sigma
    if dist == "ones":
        return torch.ones(shape, dtype=torch.float32)
    if dist == "identity":
        return torch.eye(rows, cols, dtype=torch.float32)
    if dist == "zeros":
        return torch.zeros(shape, dtype=torch.float32)
    raise ValueError("unknown distribution %r" % dist)


def _quantise_e4m3(x: torch.Tensor):
    amax = float(x.abs().max()) if x.numel() else 0.0
    scale = amax / E4M3_MAX if amax > 0 else 1.0
    q = (x / scale).clamp_(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn)
    return q, float(scale)


def _pad(t: torch.Tensor, ld: int, kind: str) -> torch.Tensor:
    """Place t (rows, cols) into a (rows, ld) storage tensor with NaN padding."""
    rows, cols = t.shape
    if ld == cols:
        return t.contiguous()
    store = torch.empty((rows, ld), dtype=t.dtype)
    if kind == "f32":
        store.fill_(float("nan"))
    else:
        bits = torch.int16 if elem_size(kind) == 2 else torch.uint8
        code = _NAN_CODES[kind]
        if bits == torch.int16 and code >= 0x8000:
            code -= 0x10000
        store.view(bits).fill_(code)
    store[:, :cols] = t
    return store


def tn_operands(kind: str, M: int, N: int, K: int, dist: str = "normal", seed: int = 0,
                sigma: float = 1.0, lda: int | None = None, ldb: int | None = None,
                dist_b: str | None = None, quantise: bool = True) -> dict:
    """Operands of a TN GEMM as CPU storage tensors.

    Returns {"A": (M, lda) tensor, "B": (N, ldb) tensor, "scale_a", "scale_b",
    "lda", "ldb"}.  a(m, k) is A[m, k]; b(k, n) is B[n, k] (B column-major).
    ``dist_b`` overrides the distribution of B (e.g. "identity").  With
    ``quantise=False`` e4m3 operands are cast directly (clamped to +-448) and
    keep scale 1.
    """
    lda = K if lda is None else lda
    ldb = K if ldb is None else ldb
    gen = torch.Generator("cpu").manual_seed(seed)
    xa = draw(gen, M, K, dist, sigma)
    db = dist if dist_b is None else dist_b
    xb = draw(gen, N, K, db, sigma)  # row n of this is column n of B
    if kind == "e4m3":
        # Exact-valued operands (+-1, ones, identity) keep scale 1; drawn ones are quantised.
        def direct(x):
            return x.clamp(-E4M3_MAX, E4M3_MAX).to(torch.float8_e4m3fn), 1.0

        qa, sa = direct(xa) if (dist in _EXACT or not quantise) else _quantise_e4m3(xa)
        qb, sb = direct(xb) if (db in _EXACT or not quantise) else _quantise_e4m3(xb)
    else:
        qa, sa = xa.to(_TORCH_DTYPES[kind]), 1.0
        qb, sb = xb.to(_TORCH_DTYPES[kind]), 1.0
    return {"A": _pad(qa, lda, kind), "B": _pad(qb, ldb, kind), "scale_a": sa, "scale_b": sb,
            "lda": lda, "ldb": ldb}


def f32_operands(M: int, N: int, K: int, dist: str = "uniform", seed: int = 1,
                 lda: int | None = None, ldb: int | None = None, dist_b: str | None = None) -> dict:
    """Row-major FP32 operands: A (M, lda) with a(m,k) = A[m,k]; B (K, ldb) with b(k,n) = B[k,n]."""
    lda = K if lda is None else lda
    ldb = N if ldb is None else ldb
    gen = torch.Generator("cpu").manual_seed(seed)
    xa = draw(gen, M, K, dist)
    xb = draw(gen, K, N, dist if dist_b is None else dist_b)
    return {"A": _pad(xa, lda, "f32"), "B": _pad(xb, ldb, "f32"), "lda": lda, "ldb": ldb}


def codes(t: torch.Tensor) -> np.ndarray:
    """Storage codes of a CPU tensor as a numpy integer array (for the oracle)."""
    if t.dtype in (torch.float16, torch.bfloat16):
        return t.contiguous().view(torch.int16).numpy().view(np.uint16)
    if t.dtype == torch.float8_e4m3fn:
        return t.contiguous().view(torch.uint8).numpy()
    if t.dtype == torch.float32:
        return t.contiguous().numpy()
    raise TypeError(t.dtype)


def sample_positions(M: int, N: int, count: int = 4096, seed: int = 0, edges: bool = True):
    """``count`` seeded (m, n) positions, plus the corners and ragged edges when asked."""
    gen = torch.Generator("cpu").manual_seed(seed + 1000)
    ms = torch.randint(0, M, (count,), generator=gen, dtype=torch.int64)
    ns = torch.randint(0, N, (count,), generator=gen, dtype=torch.int64)
    if edges:
        em = [0, M - 1, 0, M - 1, M // 2, M - 1, 0]
        en = [0, 0, N - 1, N - 1, N - 1, N // 2, N // 2]
        ms = torch.cat([ms, torch.tensor(em, dtype=torch.int64)])
        ns = torch.cat([ns, torch.tensor(en, dtype=torch.int64)])
    return ms.numpy(), ns.numpy()
