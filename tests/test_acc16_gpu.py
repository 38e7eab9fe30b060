"""GPU parity of gemm_f16_tn_acc16 (FP16 inputs, FP16 accumulation in the
tensor core, FP16 output -- the mode the FP16 page measures) against the CPU
oracle, through the C ABI.

+-1 inputs with K <= 2048 keep every partial sum an integer FP16 holds, so
the result must be bit-exact.  Random inputs are checked against the contract
tolerance and a bound for FP16 accumulation: one output ulp plus
2 * K * 2^-11 * sum_k |a||b|."""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import assert_codes_equal, exact_codes, out_codes

pytestmark = pytest.mark.gpu


def run(ops, M, N, K, ldc=None):
    ldc = M if ldc is None else ldc
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C = torch.empty((max(N, 1), ldc), dtype=torch.float16, device="cuda")
    C.view(torch.int16).fill_(0x7E00)
    st = capi.gemm_f16_tn_acc16(M, N, K, A.data_ptr(), ops["lda"], B.data_ptr(), ops["ldb"],
                                C.data_ptr(), ldc, torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    torch.cuda.synchronize()
    return C.cpu()


@pytest.fixture(params=[0, 1], ids=["cta1", "pair"])
def pair_mode(request):
    assert capi.gemm_set_option("pair", request.param) == 0
    yield
    capi.gemm_set_option("pair", -1)


@pytest.mark.parametrize("shape", [(256, 256, 256), (600, 330, 2048), (301, 213, 129)])
def test_pm1_bitexact(shape, pair_mode):
    M, N, K = shape
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=K)
    C = run(ops, M, N, K)
    exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))


@pytest.mark.parametrize("shape", [(600, 330, 200), (257, 129, 1000), (1024, 512, 4096)])
def test_random_within_fp16_accumulation_bound(shape, pair_mode):
    M, N, K = shape
    ops = si.tn_operands("f16", M, N, K, dist="normal", seed=sum(shape), sigma=0.1)
    C = run(ops, M, N, K)
    exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    got = C[:N, :M].double().numpy().T
    a = ops["A"].double().numpy()
    b = ops["B"].double().numpy()
    err = np.abs(got - exact)
    contract = 1e-2 * math.sqrt(K) * np.abs(a).max() * np.abs(b).max()
    assert err.max() <= contract
    mag = np.maximum(np.abs(exact), 2.0 ** -24)
    bound = np.exp2(np.floor(np.log2(mag)) - 10) + 2.0 * K * 2.0 ** -11 * (np.abs(a) @ np.abs(b).T)
    assert np.all(err <= bound)


def test_unaligned_rows_and_workspace_does_not_split():
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    try:
        M, N, K = 301, 213, 1001
        ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=4, lda=K, ldb=K + 2)
        C = run(ops, M, N, K, ldc=M + 1)
        exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K + 2)
        assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))
    finally:
        capi.gemm_set_workspace(None, 0)


def test_pm1_8192_k2048_sampled():
    """The FP16 page's +-1 check at 8192 x 8192 x 2048, with FP16 accumulation."""
    M, N, K = 8192, 8192, 2048
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=2)
    C = run(ops, M, N, K)
    ms, ns = si.sample_positions(M, N, 4096, seed=2)
    exact = oracle.gemm_tn_sampled("f16", K, si.codes(ops["A"]), K, si.codes(ops["B"]), K, ms, ns)
    got = C[torch.from_numpy(ns), torch.from_numpy(ms)].contiguous().view(torch.int16).numpy()
    assert_codes_equal(got.view(np.uint16), exact_codes("f16", exact))
