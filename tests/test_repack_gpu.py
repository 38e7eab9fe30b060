"""GPU parity of the repack path: with a workspace registered, operands whose
rows are not 16-byte aligned (or, for compute-heavy shapes, not 128-byte
aligned) are copied into it with aligned rows and the TMA path runs.  Checked against the CPU oracle through the C ABI; inputs must be
left unchanged and C's padding untouched."""
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
    ws = torch.empty(1 << 29, dtype=torch.uint8, device="cuda")  # 512 MiB
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    yield ws
    capi.gemm_set_workspace(None, 0)
    capi.gemm_set_option("repack", 0)
    capi.gemm_set_option("splits", 0)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("lds", [(1023, 1023, 2047), (1025, 1030, 2050), (1040, 1027, 2048)])
def test_repacked_operands_full(kind, lds, workspace):
    M, N, K = 2047, 1001, 1023
    lda, ldb, ldc = lds
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=sum(lds), lda=lda, ldb=ldb)
    a_before, b_before = ops["A"].clone(), ops["B"].clone()
    C = run_tn(kind, ops, M, N, K, ldc=ldc)
    check_full(kind, ops, M, N, K, C)
    if ldc > M:
        pad = C[:N, M:ldc].contiguous().view(torch.int16)
        assert torch.all(pad == (0x7E00 if kind == "f16" else 0x7FC0))
    assert torch.equal(ops["A"].view(torch.uint8), a_before.view(torch.uint8))
    assert torch.equal(ops["B"].view(torch.uint8), b_before.view(torch.uint8))


@pytest.mark.parametrize("kind", KINDS)
def test_repack_then_split(kind, workspace):
    """Unaligned rows and too few tiles: repack, then split-K in the rest of the workspace."""
    M, N, K = 200, 300, 3001
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=5, lda=K, ldb=K + 1)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K + 1)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


def test_small_workspace_falls_back_to_load_producer():
    ws = torch.empty(1 << 16, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    try:
        M, N, K = 513, 257, 1001
        ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=6)
        C = run_tn("bf16", ops, M, N, K)
        exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
        assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))
    finally:
        capi.gemm_set_workspace(None, 0)


def test_repack_disabled_uses_load_producer(workspace):
    assert capi.gemm_set_option("repack", 1) == 0
    M, N, K = 513, 257, 1001
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=7)
    C = run_tn("f16", ops, M, N, K)
    exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))


@pytest.mark.parametrize("shape", [(8191, 8191, 8191), (2047, 3001, 1023)])
def test_bf16_tight_ld_configs_with_workspace(shape, workspace):
    """The BF16 sweep's ragged shapes with tight leading dimensions."""
    M, N, K = shape
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=3, sigma=0.05)
    C = run_tn("bf16", ops, M, N, K)
    check_sampled("bf16", ops, M, N, K, C, seed=3)


@pytest.mark.parametrize("kind", KINDS)
def test_128_byte_misaligned_rows_copied(kind, workspace):
    """Rows 16-byte but not 128-byte aligned (ld = 208 elements) on a shape
    heavy enough for the copy (MN / (M + N) = 2560 >= 1100 x element size): the
    copied path must match the oracle and, bit for bit, the same call without
    the copy (same arithmetic)."""
    M = N = 5120
    K = 200
    ld = 208
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=11, sigma=0.5, lda=ld, ldb=ld)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)
    assert capi.gemm_set_option("repack", 1) == 0
    C2 = run_tn(kind, ops, M, N, K)
    assert torch.equal(C.view(torch.int16), C2.view(torch.int16))
