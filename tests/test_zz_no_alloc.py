"""gemm_bf16_tn_noalloc -- BF16 TN GEMM whose split-K scratch is a fixed array
inside the library, for callers that may not allocate device memory (code
whose memory belongs to a pooled allocator it must not bypass, plugins whose
host forbids device allocation, loops where an allocation would synchronise
the device).

Each case calls the new entry point twice in a row through the C ABI and
checks both outputs against gemm_bf16_tn's (which, with no workspace
registered, does not split K) within the contract tolerance the other tests
use, 1e-2 * sqrt(K) * max|a| * max|b|.  This file sorts last so that a run
stopping at its first failure has run every other test first."""
import math

import pytest
import torch

import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.mark.parametrize("shape,splits", [((256, 512, 4096), 0), ((300, 200, 1000), 3),
                                          ((1024, 1024, 8192), 0), ((64, 2048, 2048), 0)])
def test_noalloc_matches_gemm_bf16_tn_on_two_calls(shape, splits):
    M, N, K = shape
    assert capi.gemm_set_workspace(None, 0) == capi.GEMM_OK  # reference call: no split
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=M + K, sigma=0.5)
    A, B = ops["A"].cuda(), ops["B"].cuda()
    ref = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
    st = capi.gemm_bf16_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, ref.data_ptr(), M,
                           _stream())
    assert st == capi.GEMM_OK, capi.status_text(st)
    ma = float(ops["A"].float().abs().max())
    mb = float(ops["B"].float().abs().max())
    tol = 1e-2 * math.sqrt(K) * ma * mb
    for _ in range(2):
        out = torch.full((N, M), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = capi.gemm_bf16_tn_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), K, out.data_ptr(),
                                       M, splits, _stream())
        assert st == capi.GEMM_OK, capi.status_text(st)
        torch.cuda.synchronize()
        diff = (out.double() - ref.double()).abs()
        assert bool(torch.isfinite(diff).all()), "non-finite output"
        assert float(diff.max()) <= tol


def test_noalloc_rejects_a_split_beyond_the_scratch():
    """16 forced pieces of a 4096^2 output need far more than the array holds:
    the call must refuse before launching and leave C untouched."""
    M = N = K = 4096
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.full((N, M), 3.0, dtype=torch.bfloat16, device="cuda")
    st = capi.gemm_bf16_tn_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C.data_ptr(), M,
                                   16, _stream())
    assert st == capi.GEMM_ERR_SCRATCH
    assert "scratch" in capi.status_text(st)
    torch.cuda.synchronize()
    assert bool((C == 3.0).all())
