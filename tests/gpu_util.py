"""Helpers for the GPU parity tests: run the library through its C ABI on
seeded inputs and compare with the CPU oracle.

Comparison rules:
  exact       the GPU output code equals the oracle's round-to-nearest-even
              encoding of the exact result (+0 and -0 count as equal);
  contract    max |err| <= 1e-2 * sqrt(K) * max|a| * max|b|   (fp16/bf16/fp8)
              max |err| <= 2e-5 * K * max|a| * max|b|         (fp32)
  tight       |err| <= ulp_out(|c|) + 2 * K * 2^-24 * sum_k |a||b|, a bound
              derived from one output rounding plus FP32 accumulation error.
"""
from __future__ import annotations

import math

import numpy as np
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi

OUT_KIND = {"f16": "f16", "bf16": "bf16", "e4m3": "bf16"}
OUT_TORCH = {"f16": torch.float16, "bf16": torch.bfloat16, "e4m3": torch.bfloat16}
FN = {"f16": capi.gemm_f16_tn, "bf16": capi.gemm_bf16_tn}
OUT_MANT_BITS = {"f16": 10, "bf16": 7}


def stream():
    return torch.cuda.current_stream().cuda_stream


def run_tn(kind, ops, M, N, K, ldc=None, c_init=None, expect=capi.GEMM_OK):
    """Run the TN entry point for `kind` on CPU storage operands; returns the
    (N, ldc) output storage tensor on the CPU."""
    ldc = M if ldc is None else ldc
    A = ops["A"].cuda()
    B = ops["B"].cuda()
    if c_init is None:
        C = torch.empty((max(N, 1), ldc), dtype=OUT_TORCH[kind], device="cuda")
        C.view(torch.int16).fill_(0x7E00 if kind == "f16" else 0x7FC0)  # NaN sentinel
    else:
        C = c_init.cuda()
    if kind == "e4m3":
        st = capi.gemm_fp8_tn(M, N, K, A.data_ptr(), ops["lda"], B.data_ptr(), ops["ldb"],
                              ops["scale_a"], ops["scale_b"], C.data_ptr(), ldc, stream())
    else:
        st = FN[kind](M, N, K, A.data_ptr(), ops["lda"], B.data_ptr(), ops["ldb"],
                      C.data_ptr(), ldc, stream())
    assert st == expect, capi.status_text(st)
    torch.cuda.synchronize()
    return C.cpu()


def out_codes(C_store, M, N):
    """(M, N) uint16 codes of C from its (N, ldc) column-major storage."""
    return C_store[:N, :M].contiguous().view(torch.int16).numpy().view(np.uint16).T


def out_values(C_store, M, N):
    return C_store[:N, :M].to(torch.float64).numpy().T


def exact_codes(kind, c64):
    return oracle.encode_rne(OUT_KIND[kind], c64)


def assert_codes_equal(got, want):
    g = np.where(got == 0x8000, 0, got)
    w = np.where(want == 0x8000, 0, want)
    bad = np.argwhere(g != w)
    assert bad.size == 0, "%d mismatches, first at %s: got %#06x want %#06x" % (
        len(bad), tuple(bad[0]), got[tuple(bad[0])], want[tuple(bad[0])])


def maxabs_dequant(ops, kind):
    a = ops["A"][:, : ops.get("K", ops["A"].shape[1])]
    b = ops["B"][:, : ops.get("K", ops["B"].shape[1])]
    ma = float(a.to(torch.float32).abs().nan_to_num(0).max()) * ops.get("scale_a", 1.0)
    mb = float(b.to(torch.float32).abs().nan_to_num(0).max()) * ops.get("scale_b", 1.0)
    return ma, mb


def contract_tol(kind, K, ma, mb):
    if kind == "f32":
        return 2e-5 * K * ma * mb
    return 1e-2 * math.sqrt(K) * ma * mb


def tight_tol(kind, exact, absdot, K):
    """Per-element bound: one output ulp plus twice the worst FP32 sum error."""
    mant = OUT_MANT_BITS[OUT_KIND[kind]]
    mag = np.maximum(np.abs(exact), 2.0 ** -30)
    ulp = np.exp2(np.floor(np.log2(mag)) - mant)
    return ulp + 2.0 * K * 2.0 ** -24 * absdot


def decoded(ops, kind, K):
    """Dequantised float64 operands (torch decoding) for bound computations."""
    a = ops["A"][:, :K].to(torch.float64).numpy() * ops["scale_a"]
    b = ops["B"][:, :K].to(torch.float64).numpy() * ops["scale_b"]
    return a, b


def check_full(kind, ops, M, N, K, C_store):
    """Full comparison against the oracle: contract and tight tolerances."""
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), ops["lda"], si.codes(ops["B"]),
                           ops["ldb"], ops["scale_a"], ops["scale_b"])
    got = out_values(C_store, M, N)
    assert np.all(np.isfinite(got)), "non-finite outputs"
    err = np.abs(got - exact)
    ops = dict(ops, K=K)
    ma, mb = maxabs_dequant(ops, kind)
    tol = contract_tol(kind, K, ma, mb)
    assert err.max() <= tol, "max err %g > contract tol %g" % (err.max(), tol)
    a, b = decoded(ops, kind, K)
    absdot = np.abs(a) @ np.abs(b).T
    tt = tight_tol(kind, exact, absdot, K)
    worst = np.argmax(err - tt)
    assert np.all(err <= tt), "tight bound violated at %s: err %g > %g" % (
        np.unravel_index(worst, err.shape), err.flat[worst], tt.flat[worst])
    return err.max(), tol


def _rows(t, idx, K):
    """float64 copy of rows `idx`, columns [0, K), of a CPU storage tensor."""
    bits = torch.uint8 if t.element_size() == 1 else torch.int16
    rows = t.view(bits)[torch.from_numpy(np.asarray(idx)), :K].contiguous().view(t.dtype)
    return rows.to(torch.float64).numpy()


def check_sampled(kind, ops, M, N, K, C_store, seed, count=4096):
    ms, ns = si.sample_positions(M, N, count, seed)
    exact = oracle.gemm_tn_sampled(kind, K, si.codes(ops["A"]), ops["lda"], si.codes(ops["B"]),
                                   ops["ldb"], ms, ns, ops["scale_a"], ops["scale_b"])
    got = C_store[torch.from_numpy(ns), torch.from_numpy(ms)].to(torch.float64).numpy()
    assert np.all(np.isfinite(got)), "non-finite outputs"
    err = np.abs(got - exact)
    ops = dict(ops, K=K)
    ma, mb = maxabs_dequant(ops, kind)
    tol = contract_tol(kind, K, ma, mb)
    assert err.max() <= tol, "max err %g > contract tol %g" % (err.max(), tol)
    # tight bound on the samples (rows gathered as raw codes: CPU float8 has no gather)
    a = _rows(ops["A"], ms, K) * ops["scale_a"]
    b = _rows(ops["B"], ns, K) * ops["scale_b"]
    absdot = np.sum(np.abs(a) * np.abs(b), axis=1)
    tt = tight_tol(kind, exact, absdot, K)
    assert np.all(err <= tt), "tight bound violated: worst excess %g" % float(np.max(err - tt))
    return err.max(), tol
