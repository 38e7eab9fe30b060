"""GPU parity of pairs of 64-row halves against the CPU oracle, through the C ABI.

A CTA pair computes 128 rows of N (64 per CTA, tcgen05.mma cta_group::2 with
M = 128) by 128, 192 or 256 columns of M.  Each CTA holds its 64 rows for all
the tile's columns, row r and column n in TMEM lane r + 64 (n / (width / 2)),
column n % (width / 2), so each epilogue warp stores 32 rows of one half of
the columns (96 for width 192: one whole 64-column chunk and one cut at the
half's end, which the lanes store).  These cases cover that mapping on every
input kind and output type, all three tile widths, ragged edges in M, N and K
(a partial last pair tile, and a pair whose second CTA lies past N or past M),
leading dimensions that take the row-wise store path, +-1 inputs (exact), and
few CTA pairs that each walk many tiles (ring and accumulator phases)."""
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
def pair_halves():
    touched = []

    def set_(name, value):
        assert capi.gemm_set_option(name, value) == 0
        touched.append(name)
    set_("half", 3)
    yield set_
    for name in touched:
        capi.gemm_set_option(name, -1 if name == "pair" else 0)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(128, 8192, 512), (100, 1000, 257), (256, 700, 300),
                                   (200, 130, 1000), (1, 64, 64), (129, 333, 128)])
def test_forced_random(kind, shape, pair_halves):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=M + N + K, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("tile_q", [128, 256])
def test_forced_pm1_bitexact(kind, tile_q, pair_halves):
    pair_halves("tile_q", tile_q)
    M, N, K = 250, 1000, 2048
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=7)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("ctas", [2, 6])
def test_few_pairs_walk_many_tiles(ctas, pair_halves):
    """Two or six CTAs (one or three pairs) each run many tiles: every ring
    slot and both accumulator buffers cycle through several phases."""
    pair_halves("max_ctas", ctas)
    M, N, K = 300, 1200, 700
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=ctas)
    C = run_tn("bf16", ops, M, N, K)
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))


@pytest.mark.parametrize("ldc_pad", [0, 3])
def test_forced_row_wise_stores(ldc_pad, pair_halves):
    """ldc = M + 3 with M odd: C rows are not 16-byte aligned, so the epilogue
    writes rows itself (32 per warp, half the columns each); the padding must
    keep its sentinel."""
    M, N, K = 137, 333, 200
    ldc = M + ldc_pad
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=11)
    C = run_tn("bf16", ops, M, N, K, ldc=ldc)
    check_full("bf16", ops, M, N, K, C)
    if ldc_pad:
        assert torch.all(torch.isnan(C[:N, M:].float())), "C padding was written"


@pytest.mark.parametrize("M", [64, 128, 192])
def test_fp8_f32_output(M, pair_halves):
    """FP32 output: 32-column chunks, two or four per warp; the contract
    tolerance and the bound of one FP32 rounding plus the accumulation."""
    import numpy as np
    from test_fp8_f32out_gpu import run, tols

    N, K = 520, 384
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=M)
    C = run(ops, M, N, K)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K,
                           ops["scale_a"], ops["scale_b"])
    a = ops["A"][:, :K].to(torch.float64).numpy() * ops["scale_a"]
    b = ops["B"][:, :K].to(torch.float64).numpy() * ops["scale_b"]
    contract, tight = tols(ops, K, exact, np.abs(a) @ np.abs(b).T)
    err = np.abs(C[:N, :M].double().numpy().T - exact)
    assert err.max() <= contract and np.all(err <= tight)


@pytest.mark.parametrize("kind,shape", [("bf16", (128, 8192, 8192)), ("e4m3", (256, 8192, 8192)),
                                        ("f16", (128, 16384, 4096))])
def test_forced_skinny_sampled(kind, shape, pair_halves):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=5, sigma=1.0 if kind == "e4m3"
                         else 0.05)
    C = run_tn(kind, ops, M, N, K)
    check_sampled(kind, ops, M, N, K, C, seed=3)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(128, 4100, 700), (256, 900, 2048), (1, 64, 64), (200, 333, 129)])
def test_two_issuers_random(kind, shape, pair_halves):
    """Pairs of halves with two MMA-issuing warps in the leader CTA (option
    "issuers" = 2): alternate K stages into accumulators of tile_q / 2 columns
    each, added by the epilogue; units of one K stage add nothing."""
    pair_halves("issuers", 2)
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=M + N + K + 1, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("ctas", [2, 6, 0])
def test_two_issuers_pm1_bitexact(ctas, pair_halves):
    pair_halves("issuers", 2)
    pair_halves("max_ctas", ctas)
    M, N, K = 250, 1200, 2048
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=ctas + 3)
    C = run_tn("bf16", ops, M, N, K)
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("issuers", [1, 2])
@pytest.mark.parametrize("M", [192, 150, 97, 250])
def test_width_192_pm1_bitexact(kind, issuers, M, pair_halves):
    """Width 192: 96 columns per half.  M = 150 ends inside a 16-byte granule
    of the second half; M = 97 leaves the second CTA one row of A; M = 250
    adds a second column of tiles 58 wide.  N = 1000 ends inside a pair."""
    pair_halves("tile_q", 192)
    pair_halves("issuers", issuers)
    N, K = 1000, 2048
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = capi.gemm_tn_plan(kind, M, N, K, sms=sms)
    assert st == 0 and (p["pair"], p["half"], p["tile_q"], p["atoms"]) == (1, 1, 192, 1), p
    assert p["issuers"] == issuers, p
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=M + issuers)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(192, 8192, 512), (180, 700, 300), (129, 130, 1000)])
def test_width_192_random(kind, shape, pair_halves):
    pair_halves("tile_q", 192)
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=M + N + K + 2, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("M,ldc", [(192, 200), (137, 140), (191, 194)])
def test_width_192_padding_and_row_wise_stores(M, ldc, pair_halves):
    """ldc = 200 keeps C rows 16-byte aligned (TMA stores, lanes for the cut
    chunk); 140 and 194 with 16-bit output do not (row-wise stores).  The
    padding between M and ldc keeps its sentinel."""
    pair_halves("tile_q", 192)
    N, K = 333, 200
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=ldc)
    C = run_tn("bf16", ops, M, N, K, ldc=ldc)
    check_full("bf16", ops, M, N, K, C)
    assert torch.all(torch.isnan(C[:N, M:].float())), "C padding was written"


@pytest.mark.parametrize("ctas", [2, 6])
def test_width_192_few_pairs_walk_many_tiles(ctas, pair_halves):
    pair_halves("tile_q", 192)
    pair_halves("max_ctas", ctas)
    M, N, K = 400, 1200, 700
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=ctas + 20)
    C = run_tn("f16", ops, M, N, K)
    exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))


def test_width_192_fp8_f32_output(pair_halves):
    """FP32 output: three whole 32-column chunks per half, nothing cut."""
    import numpy as np
    from test_fp8_f32out_gpu import run, tols

    pair_halves("tile_q", 192)
    M, N, K = 170, 520, 384
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=M)
    C = run(ops, M, N, K)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K,
                           ops["scale_a"], ops["scale_b"])
    a = ops["A"][:, :K].to(torch.float64).numpy() * ops["scale_a"]
    b = ops["B"][:, :K].to(torch.float64).numpy() * ops["scale_b"]
    contract, tight = tols(ops, K, exact, np.abs(a) @ np.abs(b).T)
    err = np.abs(C[:N, :M].double().numpy().T - exact)
    assert err.max() <= contract and np.all(err <= tight)


def test_width_192_skinny_sampled(pair_halves):
    pair_halves("tile_q", 192)
    M, N, K = 192, 8192, 8192
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=9, sigma=0.05)
    C = run_tn("bf16", ops, M, N, K)
    check_sampled("bf16", ops, M, N, K, C, seed=4)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("issuers", [1, 2])
@pytest.mark.parametrize("M,width", [(1, 32), (16, 32), (20, 32), (32, 32), (33, 64), (48, 64),
                                     (64, 64), (100, 128), (140, 160), (160, 160), (210, 224),
                                     (224, 224)])
def test_width_from_m_pm1_bitexact(kind, issuers, M, width, pair_halves):
    """Without a tile_q option the width is 32 or 64 for M up to that, 128 up
    to 128, else M rounded up to a multiple of 32: halves of 16, 32, 80 and
    112 columns end inside their only or last 64-column chunk (16-bit output);
    widths 32 and 64 run one K atom per stage."""
    pair_halves("issuers", issuers)
    N, K = 1000, 1000
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = capi.gemm_tn_plan(kind, M, N, K, sms=sms)
    assert st == 0 and (p["pair"], p["half"], p["tile_q"], p["issuers"]) == (1, 1, width, issuers), p
    assert p["atoms"] == (2 if width == 128 else 1), p
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=M + issuers)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("M,ldc", [(150, 152), (150, 153), (211, 216), (211, 213), (137, 138),
                                   (20, 24), (20, 21), (40, 48), (57, 59)])
def test_width_from_m_padding_and_row_wise_stores(M, ldc, pair_halves):
    N, K = 300, 300
    ops = si.tn_operands("f16", M, N, K, dist="normal", seed=ldc + 1)
    C = run_tn("f16", ops, M, N, K, ldc=ldc)
    check_full("f16", ops, M, N, K, C)
    assert torch.all(torch.isnan(C[:N, M:].float())), "C padding was written"


@pytest.mark.parametrize("M", [20, 50, 150, 220])
def test_width_from_m_fp8_f32_output(M, pair_halves):
    """FP32 output, 32-column chunks: halves of 16, 80 and 112 columns end 16
    columns into their only or last chunk; halves of 32 fill one."""
    import numpy as np
    from test_fp8_f32out_gpu import run, tols

    N, K = 520, 384
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=M + 1)
    C = run(ops, M, N, K)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K,
                           ops["scale_a"], ops["scale_b"])
    a = ops["A"][:, :K].to(torch.float64).numpy() * ops["scale_a"]
    b = ops["B"][:, :K].to(torch.float64).numpy() * ops["scale_b"]
    contract, tight = tols(ops, K, exact, np.abs(a) @ np.abs(b).T)
    err = np.abs(C[:N, :M].double().numpy().T - exact)
    assert err.max() <= contract and np.all(err <= tight)


@pytest.mark.parametrize("kind,M", [("bf16", 16), ("f16", 64), ("e4m3", 32)])
def test_narrow_widths_skinny_sampled(kind, M, pair_halves):
    N, K = 8192, 8192
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=M, sigma=1.0 if kind == "e4m3"
                         else 0.05)
    C = run_tn(kind, ops, M, N, K)
    check_sampled(kind, ops, M, N, K, C, seed=5)
