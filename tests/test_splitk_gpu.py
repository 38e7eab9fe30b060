"""GPU parity of split-K (tiles cut along K when one wave of output tiles
cannot fill the GPU; partials in a caller-registered workspace, summed by the
last piece in piece order) against the CPU oracle, through the C ABI."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import (assert_codes_equal, check_full, check_sampled, exact_codes, out_codes,
                      run_tn)

pytestmark = pytest.mark.gpu
KINDS = ["f16", "bf16", "e4m3"]


@pytest.fixture
def workspace():
    ws = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")  # 256 MiB
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    yield ws
    assert capi.gemm_set_workspace(None, 0) == 0
    capi.gemm_set_option("splits", 0)
    capi.gemm_set_option("pair", -1)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(256, 512, 4096), (300, 200, 1000), (64, 2048, 2048)])
def test_auto_split_pm1_bitexact(kind, shape, workspace):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=M + N)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("splits", [2, 3, 7])
def test_forced_split_random(kind, pair, splits, workspace):
    M, N, K = 600, 330, 1000
    assert capi.gemm_set_option("pair", pair) == 0
    assert capi.gemm_set_option("splits", splits) == 0
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=splits, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


def test_split_is_deterministic(workspace):
    M, N, K = 512, 256, 8192
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=5)
    runs = [run_tn("bf16", ops, M, N, K) for _ in range(3)]
    for r in runs[1:]:
        assert torch.equal(r.view(torch.int16), runs[0].view(torch.int16))
    check_full("bf16", ops, M, N, K, runs[0])


def test_split_with_unaligned_rows_and_fp32_out(workspace):
    M, N, K = 301, 213, 1001
    assert capi.gemm_set_option("splits", 4) == 0
    ops = si.tn_operands("e4m3", M, N, K, dist="pm1", seed=9, lda=K, ldb=K + 2)
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C = torch.full((N, M + 3), float("nan"), device="cuda")
    st = capi.gemm_fp8_tn_f32(M, N, K, A.data_ptr(), K, B.data_ptr(), K + 2, 1.0, 1.0,
                              C.data_ptr(), M + 3, torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K + 2)
    got = C.cpu()
    np.testing.assert_array_equal(got[:, :M].numpy().T, exact.astype(np.float32))
    assert torch.all(torch.isnan(got[:, M:]))


def test_small_workspace_does_not_split_and_stays_correct():
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    try:
        M, N, K = 256, 512, 4096
        ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=1)
        C = run_tn("f16", ops, M, N, K)
        exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
        assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))
    finally:
        capi.gemm_set_workspace(None, 0)


@pytest.mark.parametrize("shape", [(128, 8192, 8192), (64, 14336, 4096), (1024, 1024, 8192),
                                   (16, 8192, 8192), (100, 8192, 2048)])
def test_skinny_sampled(shape, workspace):
    M, N, K = shape
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=3, sigma=0.05)
    C = run_tn("bf16", ops, M, N, K)
    check_sampled("bf16", ops, M, N, K, C, seed=3)
    assert capi.gemm_read_watchdog(0) == capi.GEMM_OK


def test_workspace_api_checks():
    assert capi.gemm_set_workspace(None, 10) == capi.GEMM_ERR_INVALID_DIM
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr() + 8, 512) == capi.GEMM_ERR_MISALIGNED
    assert capi.gemm_workspace_bytes(1024, 1024, 8192) > 0


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("pair", [0, 1])
def test_tail_k_pieces_full(kind, pair, workspace):
    """A partial last wave with a workspace: its tiles are cut into K pieces
    (few CTAs force several waves and a partial last one)."""
    M, N, K = 1100, 700, 1000
    for k, v in {"pair": pair, "max_ctas": 10, "tail_k": 3}.items():
        assert capi.gemm_set_option(k, v) == 0
    try:
        ops = si.tn_operands(kind, M, N, K, dist="normal", seed=pair + 11, sigma=0.5)
        C1 = run_tn(kind, ops, M, N, K)
        check_full(kind, ops, M, N, K, C1)
        C2 = run_tn(kind, ops, M, N, K)
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16)), "not deterministic"
    finally:
        capi.gemm_set_option("max_ctas", 0)
        capi.gemm_set_option("tail_k", 0)


@pytest.mark.parametrize("shape,tail_k", [((4096, 4096, 4096), 2), ((3072, 4096, 8192), 5)])
def test_tail_k_pieces_large_sampled(shape, tail_k, workspace):
    M, N, K = shape
    assert capi.gemm_set_option("tail_k", tail_k) == 0
    try:
        ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=3, sigma=0.05)
        C = run_tn("bf16", ops, M, N, K)
        check_sampled("bf16", ops, M, N, K, C, seed=3)
    finally:
        capi.gemm_set_option("tail_k", 0)
