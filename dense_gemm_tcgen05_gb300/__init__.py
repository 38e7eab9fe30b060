"""dense_gemm_tcgen05_gb300 -- dense GEMM for one NVIDIA GB300 GPU (sm_103a).

The compute lives in ``libgemm.so`` (hand-written CUDA: a persistent tcgen05
tensor-core kernel for fp16/bf16/e4m3 and a SIMT FFMA kernel for fp32), whose C
ABI is declared in ``include/gemm.h``.  ``capi`` binds that ABI one to one;
the helpers here only turn torch CUDA tensors into its pointer/size arguments.
PyTorch provides device memory and streams, nothing else.

Layouts, as torch tensors (every tensor's last stride must be 1):
  tn(a, b):   a = A, shape (M, K), row-major with lda = a.stride(0)
              b = B column-major K x N, given as its (N, K) row-major view
              returns the (N, M) row-major view of C (C column-major M x N);
              C as a logical M x N matrix is ``out.t()``.
  f32(a, b):  a (M, K), b (K, N), out (M, N), all row-major.
"""
from __future__ import annotations

import torch

from . import capi
from .capi import GemmError  # noqa: F401

__all__ = ["tn", "f32", "f32_bf16x6", "register_workspace", "capi", "GemmError", "stream_handle"]

_TN_DTYPES = {
    torch.float16: ("gemm_f16_tn", torch.float16),
    torch.bfloat16: ("gemm_bf16_tn", torch.bfloat16),
    torch.float8_e4m3fn: ("gemm_fp8_tn", torch.bfloat16),
}


def stream_handle(stream=None) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _check_2d(t: torch.Tensor, name: str):
    if t.dim() != 2 or (t.size(1) > 1 and t.stride(1) != 1):
        raise ValueError("%s must be 2-D with unit last stride" % name)
    if not t.is_cuda:
        raise ValueError("%s must be a CUDA tensor" % name)


def _ld(t: torch.Tensor) -> int:
    return max(int(t.stride(0)), int(t.size(1)), 1)


def _same_device(*ts: torch.Tensor):
    dev = ts[0].device
    for t in ts[1:]:
        if t.device != dev:
            raise ValueError("all tensors must be on one device (got %s and %s)" % (dev, t.device))


def _check_out(out: torch.Tensor, shape, dtype):
    """A caller-supplied output must match exactly: the library writes every
    element of the product, so a smaller tensor would be written past its end."""
    _check_2d(out, "out")
    if out.dtype != dtype or tuple(out.shape) != tuple(shape):
        raise ValueError("out must be %s of %s, got %s of %s" % (tuple(shape), dtype,
                                                                 tuple(out.shape), out.dtype))


def tn(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None, scale_a: float = 1.0,
       scale_b: float = 1.0, stream=None, out_dtype: torch.dtype | None = None) -> torch.Tensor:
    """C = A x B in the TN layout; returns ``out`` (N, M) holding C column-major.

    FP8 inputs give a bfloat16 C, or float32 with ``out_dtype=torch.float32``
    (``gemm_fp8_tn_f32``)."""
    if a.dtype != b.dtype or a.dtype not in _TN_DTYPES:
        raise TypeError("a and b must both be float16, bfloat16 or float8_e4m3fn")
    _check_2d(a, "a")
    _check_2d(b, "b")
    M, K = a.shape
    N, Kb = b.shape
    if K != Kb:
        raise ValueError("K mismatch: a has %d columns, b has %d" % (K, Kb))
    fn_name, default_out = _TN_DTYPES[a.dtype]
    if out_dtype is None and out is not None:
        out_dtype = out.dtype
    out_dtype = default_out if out_dtype is None else out_dtype
    if fn_name == "gemm_fp8_tn" and out_dtype == torch.float32:
        fn_name = "gemm_fp8_tn_f32"
    elif out_dtype != default_out:
        raise TypeError("output dtype %s is not available for %s inputs" % (out_dtype, a.dtype))
    if out is None:
        out = torch.empty((N, M), dtype=out_dtype, device=a.device)
    _check_out(out, (N, M), out_dtype)
    _same_device(a, b, out)
    with torch.cuda.device(a.device):
        h = stream_handle(stream)
        if fn_name in ("gemm_fp8_tn", "gemm_fp8_tn_f32"):
            st = getattr(capi, fn_name)(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b),
                                        scale_a, scale_b, out.data_ptr(), _ld(out), h)
        else:
            st = getattr(capi, fn_name)(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b),
                                        out.data_ptr(), _ld(out), h)
    if st != capi.GEMM_OK:
        raise GemmError(st, fn_name)
    return out


def f32(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
        stream=None) -> torch.Tensor:
    """C = A x B with every matrix FP32 row-major; returns ``out`` (M, N)."""
    if a.dtype != torch.float32 or b.dtype != torch.float32:
        raise TypeError("a and b must be float32")
    _check_2d(a, "a")
    _check_2d(b, "b")
    M, K = a.shape
    Kb, N = b.shape
    if K != Kb:
        raise ValueError("K mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=a.device)
    _check_out(out, (M, N), torch.float32)
    _same_device(a, b, out)
    with torch.cuda.device(a.device):
        st = capi.gemm_f32(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b), out.data_ptr(),
                           _ld(out), stream_handle(stream))
    if st != capi.GEMM_OK:
        raise GemmError(st, "gemm_f32")
    return out


def f32_bf16x6(a: torch.Tensor, b: torch.Tensor, out: torch.Tensor | None = None,
               stream=None) -> torch.Tensor:
    """The FP32 product of ``f32`` on the tensor cores (gemm_f32_bf16x6): exact
    three-way BF16 splits of A and B, six piece products summed in FP32.  Needs
    a registered workspace of at least gemm_f32_bf16x6_workspace_bytes(M, N, K)
    (see ``register_workspace``)."""
    if a.dtype != torch.float32 or b.dtype != torch.float32:
        raise TypeError("a and b must be float32")
    _check_2d(a, "a")
    _check_2d(b, "b")
    M, K = a.shape
    Kb, N = b.shape
    if K != Kb:
        raise ValueError("K mismatch")
    if out is None:
        out = torch.empty((M, N), dtype=torch.float32, device=a.device)
    _check_out(out, (M, N), torch.float32)
    _same_device(a, b, out)
    with torch.cuda.device(a.device):
        st = capi.gemm_f32_bf16x6(M, N, K, a.data_ptr(), _ld(a), b.data_ptr(), _ld(b),
                                  out.data_ptr(), _ld(out), stream_handle(stream))
    if st != capi.GEMM_OK:
        raise GemmError(st, "gemm_f32_bf16x6")
    return out


def register_workspace(nbytes: int, device=None) -> torch.Tensor:
    """Allocates ``nbytes`` of device memory and registers it as the library's
    workspace for that device (gemm_set_workspace).  Returns the buffer: the
    caller keeps it alive for as long as calls may use it, and registers
    ``None`` (``capi.gemm_set_workspace(None, 0)``) before freeing it."""
    buf = torch.empty(int(nbytes), dtype=torch.uint8, device=device or "cuda")
    with torch.cuda.device(buf.device):
        st = capi.gemm_set_workspace(buf.data_ptr(), buf.numel())
    if st != capi.GEMM_OK:
        raise GemmError(st, "gemm_set_workspace")
    return buf
