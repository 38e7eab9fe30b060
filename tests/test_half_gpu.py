"""GPU parity of 64-row tiles (one CTA per tile of 64 rows of N, MMA M = 64)
against the CPU oracle, through the C ABI.

With M = 64 the accumulator row 16 q + i sits in TMEM lane 32 q + i, so each
epilogue warp stores 16 rows; these cases cover that mapping on every input
kind, ragged edges in M and N, leading dimensions that take the row-wise store
path, FP32 output, and a last wave of narrowed tiles."""
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
def half_tiles():
    assert capi.gemm_set_option("half", 1) == 0
    yield
    assert capi.gemm_set_option("half", 0) == 0
    capi.gemm_set_option("pair", -1)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(16, 8192, 512), (64, 4100, 300), (200, 1000, 257),
                                   (1, 70, 64), (130, 64, 1000)])
def test_forced_random(kind, shape, half_tiles):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=M + N + K, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("kind", KINDS)
def test_forced_pm1_bitexact(kind, half_tiles):
    M, N, K = 96, 1000, 2048
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=7)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("ldc_pad", [0, 3])
def test_forced_row_wise_stores(ldc_pad, half_tiles):
    """ldc = M + 3 with M odd: C rows are not 16-byte aligned, so the epilogue
    writes rows itself (16 per warp); the padding must keep its sentinel."""
    M, N, K = 37, 333, 200
    ldc = M + ldc_pad
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=11)
    C = run_tn("bf16", ops, M, N, K, ldc=ldc)
    check_full("bf16", ops, M, N, K, C)
    if ldc_pad:
        assert torch.all(torch.isnan(C[:N, M:].float())), "C padding was written"


def test_forced_fp8_f32_out(half_tiles):
    M, N, K = 48, 777, 512
    ops = si.tn_operands("e4m3", M, N, K, dist="pm1", seed=13)
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C = torch.full((N, M), float("nan"), device="cuda")
    st = capi.gemm_fp8_tn_f32(M, N, K, A.data_ptr(), K, B.data_ptr(), K, 1.0, 1.0, C.data_ptr(),
                              M, torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    np.testing.assert_array_equal(C.cpu().numpy().T, exact.astype(np.float32))


def test_forced_narrow_last_wave(half_tiles):
    """200 tiles of 64 x 256 on 152 SMs: the 48 tiles of the last wave are cut
    into 128-column halves, still 16 rows per epilogue warp."""
    M, N, K = 512, 64 * 100, 256
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=17)
    C = run_tn("bf16", ops, M, N, K)
    check_sampled("bf16", ops, M, N, K, C, seed=17)


def test_forced_ignored_for_pairs_and_fp16_accumulation(half_tiles):
    """Forcing 64-row tiles does not apply to CTA pairs or FP16 accumulation:
    those calls run as before and stay exact."""
    M, N, K = 512, 1024, 1024
    assert capi.gemm_set_option("pair", 1) == 0
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=19)
    C = run_tn("f16", ops, M, N, K)
    exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))
    A, B = ops["A"].cuda(), ops["B"].cuda()
    Ca = torch.empty((N, M), dtype=torch.float16, device="cuda")
    st = capi.gemm_f16_tn_acc16(M, N, K, A.data_ptr(), K, B.data_ptr(), K, Ca.data_ptr(), M,
                                torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    assert_codes_equal(out_codes(Ca.cpu(), M, N), exact_codes("f16", exact))


def _chosen(capfd, M, N, K):
    """Runs one BF16 call with the library's debug line on and returns it."""
    import os
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=M)
    os.environ["GEMM_DEBUG"] = "1"
    try:
        capfd.readouterr()
        C = run_tn("bf16", ops, M, N, K)
        err = capfd.readouterr().err
    finally:
        del os.environ["GEMM_DEBUG"]
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))
    return [ln for ln in err.splitlines() if ln.startswith("[gemm] tn")][-1]


def test_automatic_choice(capfd):
    """64-row tiles run only when forced (measured slower than 128-row tiles
    with K split in two on every skinny shape tried).  Skinny shapes whose M
    fits in 16 or 32 columns take that narrower tile instead, which leaves room
    for more ring stages of B.  Without a workspace (no split) 16-bit skinny
    shapes with M <= 64 run pairs of 64-row halves 32 or 64 wide."""
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    assert capi.gemm_set_option("half", 0) == 0
    try:
        line = _chosen(capfd, 16, 8192, 1024)
        assert "pair=0" in line and "half=0" in line and "tile_q=16" in line, line
        assert "tile_q=32" in _chosen(capfd, 20, 8192, 1024)
        assert "tile_q=64" in _chosen(capfd, 48, 8192, 1024)
        assert capi.gemm_set_option("half", 1) == 0
        line = _chosen(capfd, 16, 8192, 1024)
        assert "half=1" in line and "splits=1" in line and "grid=128" in line, line
        assert "half=0" in _chosen(capfd, 2048, 2048, 1024)   # CTA pairs: not applied
    finally:
        capi.gemm_set_option("half", 0)
        capi.gemm_set_workspace(None, 0)
    for M, width in ((16, 32), (48, 64)):
        line = _chosen(capfd, M, 8192, 1024)
        assert "pair=1" in line and "half=1" in line and f"tile_q={width}" in line, line
