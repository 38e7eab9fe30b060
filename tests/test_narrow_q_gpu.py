"""GPU parity of the narrow Q tiles (16 or 32 columns of C per tile, MMA N = 16
or 32) against the CPU oracle, through the C ABI.

These tiles are narrower than the epilogue's 64-column (32 for FP32 output)
chunk: the chunk's columns past the tile hold stale accumulator values and
must never reach C.  They are used only when all of M fits in one tile, so
those columns lie past M; the cases below check that on every input kind, for
TMA and row-wise stores, with split-K, and that a forced narrow width falls back
to 64 columns when M does not fit."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import (assert_codes_equal, check_full, exact_codes, out_codes, run_tn)

pytestmark = pytest.mark.gpu
KINDS = ["f16", "bf16", "e4m3"]


@pytest.fixture
def tile_q():
    def set_(v):
        assert capi.gemm_set_option("tile_q", v) == 0
    yield set_
    capi.gemm_set_option("tile_q", 0)
    capi.gemm_set_option("splits", 0)
    capi.gemm_set_workspace(None, 0)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("q,M", [(16, 1), (16, 16), (32, 17), (32, 32)])
def test_forced_width_random(kind, q, M, tile_q):
    tile_q(q)
    N, K = 3000, 700
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=q + M, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("kind", KINDS)
def test_automatic_pm1_bitexact(kind):
    """M = 9 takes a 16-column tile by itself (a decode-like shape)."""
    M, N, K = 9, 4096, 4096
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=21)
    C = run_tn(kind, ops, M, N, K, ldc=16)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


def test_row_wise_stores(tile_q):
    """ldc = M = 13: C rows are not 16-byte aligned, the epilogue writes them."""
    tile_q(16)
    M, N, K = 13, 1000, 300
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=23)
    C = run_tn("bf16", ops, M, N, K, ldc=M)
    check_full("bf16", ops, M, N, K, C)


def test_fp32_output_and_fp16_accumulation(tile_q):
    tile_q(32)
    M, N, K = 24, 2000, 1024
    ops = si.tn_operands("e4m3", M, N, K, dist="pm1", seed=25)
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C = torch.full((N, M), float("nan"), device="cuda")
    st = capi.gemm_fp8_tn_f32(M, N, K, A.data_ptr(), K, B.data_ptr(), K, 1.0, 1.0, C.data_ptr(),
                              M, torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    np.testing.assert_array_equal(C.cpu().numpy().T, exact.astype(np.float32))
    ops16 = si.tn_operands("f16", M, N, K, dist="pm1", seed=26)
    A16, B16 = ops16["A"].cuda(), ops16["B"].cuda()
    C16 = torch.empty((N, M), dtype=torch.float16, device="cuda")
    st = capi.gemm_f16_tn_acc16(M, N, K, A16.data_ptr(), K, B16.data_ptr(), K, C16.data_ptr(),
                                M, torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    exact16 = oracle.gemm_tn("f16", M, N, K, si.codes(ops16["A"]), K, si.codes(ops16["B"]), K)
    assert_codes_equal(out_codes(C16.cpu(), M, N), exact_codes("f16", exact16))


@pytest.mark.parametrize("splits", [0, 3])
def test_split_k(splits, tile_q):
    """16-column tiles with K pieces: partial sums cover 32 columns, the
    combined chunk 64; the columns past M stay out of C."""
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    tile_q(16)
    assert capi.gemm_set_option("splits", splits) == 0
    M, N, K = 5, 8192, 4096
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=27 + splits)
    C = run_tn("bf16", ops, M, N, K, ldc=8)
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))
    assert torch.all(torch.isnan(C[:N, M:].float())), "C padding was written"


def test_forced_width_falls_back_when_m_does_not_fit(tile_q):
    """tile_q = 16 with M = 40 would need three 16-column tiles whose chunks
    overlap their neighbours' columns: the call uses 64-column tiles instead."""
    tile_q(16)
    M, N, K = 40, 1500, 500
    ops = si.tn_operands("f16", M, N, K, dist="normal", seed=29)
    C = run_tn("f16", ops, M, N, K)
    check_full("f16", ops, M, N, K, C)
