"""Launch ordering under programmatic dependent launch.

Every tensor-core launch may start its prologue while the previous grid in
the stream is still running, and waits for that grid to complete before it
touches global memory.  These cases chain calls through shared buffers with
no host synchronisation in between and compare bit for bit with the oracle
run on the same chain:
  - read after write: a call consumes the previous call's output;
  - write after read: a call overwrites a buffer the previous call reads;
  - both across split-K launches (workspace counters) and unsplit ones."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import assert_codes_equal, exact_codes, out_codes

pytestmark = pytest.mark.gpu


def _stream():
    return torch.cuda.current_stream().cuda_stream


@pytest.fixture(params=["unsplit", "split"])
def mode(request):
    if request.param == "split":
        ws = torch.empty(1 << 27, dtype=torch.uint8, device="cuda")
        assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
        assert capi.gemm_set_option("splits", 3) == 0
        yield request.param
        capi.gemm_set_option("splits", 0)
        assert capi.gemm_set_workspace(None, 0) == 0
    else:
        yield request.param


def test_read_after_write_chain(mode):
    """C1 = A B, then C2 = C1' D with C1's storage as the next call's A
    operand, then C3 = C2' E: three calls, one sync at the end."""
    M, N, K = 192, 320, 256
    N2, N3 = 256, 200
    opsA = si.tn_operands("bf16", M, N, K, dist="pm1", seed=31)
    D = si.tn_operands("bf16", N, N2, M, dist="pm1", seed=32)["B"]      # N2 x M
    E = si.tn_operands("bf16", N2, N3, N, dist="pm1", seed=33)["B"]     # N3 x N
    A, B = opsA["A"].cuda(), opsA["B"].cuda()
    Dd, Ed = D.cuda(), E.cuda()
    C1 = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")       # column-major M x N
    C2 = torch.empty((N2, N), dtype=torch.bfloat16, device="cuda")
    C3 = torch.empty((N3, N2), dtype=torch.bfloat16, device="cuda")
    st = _stream()
    assert capi.gemm_bf16_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C1.data_ptr(), M, st) == 0
    # C1 storage row n holds M contiguous values: as a TN A operand it has N rows of K' = M.
    assert capi.gemm_bf16_tn(N, N2, M, C1.data_ptr(), M, Dd.data_ptr(), M, C2.data_ptr(), N,
                             st) == 0
    assert capi.gemm_bf16_tn(N2, N3, N, C2.data_ptr(), N, Ed.data_ptr(), N, C3.data_ptr(), N2,
                             st) == 0
    torch.cuda.synchronize()
    c1 = exact_codes("bf16", oracle.gemm_tn("bf16", M, N, K, si.codes(opsA["A"]), K,
                                            si.codes(opsA["B"]), K))           # (M, N)
    a2 = np.ascontiguousarray(c1.T)                                             # (N, M)
    c2 = exact_codes("bf16", oracle.gemm_tn("bf16", N, N2, M, a2, M, si.codes(D), M))
    a3 = np.ascontiguousarray(c2.T)                                             # (N2, N)
    c3 = exact_codes("bf16", oracle.gemm_tn("bf16", N2, N3, N, a3, N, si.codes(E), N))
    assert_codes_equal(out_codes(C1.cpu(), M, N), c1)
    assert_codes_equal(out_codes(C2.cpu(), N, N2), c2)
    assert_codes_equal(out_codes(C3.cpu(), N2, N3), c3)


def test_write_after_read(mode):
    """The second call writes its output over the first call's A operand: the
    first call must have read A completely before that."""
    M, N, K = 256, 384, 512
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=41)
    ops2 = si.tn_operands("bf16", 512, 256, 300, dist="pm1", seed=42)
    A, B = ops["A"].cuda(), ops["B"].cuda()                 # A: M x K = 256 x 512 values
    A2, B2 = ops2["A"].cuda(), ops2["B"].cuda()
    C1 = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
    st = _stream()
    assert capi.gemm_bf16_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C1.data_ptr(), M, st) == 0
    # 512 x 256 output (column-major, ldc = 512) written over A's 256 x 512 storage
    assert capi.gemm_bf16_tn(512, 256, 300, A2.data_ptr(), 300, B2.data_ptr(), 300, A.data_ptr(),
                             512, st) == 0
    torch.cuda.synchronize()
    c1 = exact_codes("bf16", oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K,
                                            si.codes(ops["B"]), K))
    c2 = exact_codes("bf16", oracle.gemm_tn("bf16", 512, 256, 300, si.codes(ops2["A"]), 300,
                                            si.codes(ops2["B"]), 300))
    assert_codes_equal(out_codes(C1.cpu(), M, N), c1)
    assert_codes_equal(out_codes(A.cpu().view(256, 512), 512, 256), c2)


def test_torch_kernels_in_between(mode):
    """A torch kernel (no programmatic launch) between two calls: it reads the
    first call's output and writes the second call's input."""
    M, N, K = 128, 512, 384
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=51)
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C1 = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
    C2 = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
    st = _stream()
    assert capi.gemm_bf16_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C1.data_ptr(), M, st) == 0
    Bn = B.clone()
    Bn.neg_()                                   # torch kernel on the same stream
    assert capi.gemm_bf16_tn(M, N, K, A.data_ptr(), K, Bn.data_ptr(), K, C2.data_ptr(), M, st) == 0
    S = C1.float() + C2.float()                 # reads both outputs
    torch.cuda.synchronize()
    c1 = exact_codes("bf16", oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K,
                                            si.codes(ops["B"]), K))
    assert_codes_equal(out_codes(C1.cpu(), M, N), c1)
    assert float(S.abs().max()) == 0.0          # C2 = -C1 exactly (negation is exact)
