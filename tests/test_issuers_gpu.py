"""GPU parity of two MMA-issuing warps (option "issuers" = 2) against the CPU
oracle, through the C ABI.

Issuer j takes the K stages s of each tile with s % 2 == j into an accumulator
of its own, and the epilogue adds the two.  These
cases cover every input kind and output type, the tile widths 16 to 128, units
with fewer K stages than issuers (the idle issuers add nothing), ragged edges,
row-wise stores, few CTAs walking many tiles, a narrowed last wave, and +-1
inputs (exact: every partial sum is an integer)."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import assert_codes_equal, check_full, exact_codes, out_codes, run_tn

pytestmark = pytest.mark.gpu
KINDS = ["f16", "bf16", "e4m3"]


@pytest.fixture(params=[2], ids=["two"])
def many(request):
    touched = []

    def set_(name, value):
        assert capi.gemm_set_option(name, value) == 0
        touched.append(name)
    set_("issuers", request.param)
    set_("pair", 0)
    set_.issuers = request.param
    yield set_
    for name in touched:
        capi.gemm_set_option(name, -1 if name == "pair" else 0)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(128, 8192, 512), (100, 1000, 257), (16, 700, 300),
                                   (30, 130, 1000), (1, 64, 64), (129, 333, 128), (64, 500, 65),
                                   (77, 260, 200)])
def test_forced_random(kind, shape, many):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=M + N + K, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("M", [16, 32, 64, 128, 200])
def test_forced_pm1_bitexact(kind, M, many):
    N, K = 1000, 2048
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=M)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("ctas,tail", [(1, 0), (3, 0), (5, 2)])
def test_few_ctas_many_tiles(ctas, tail, many):
    """One to five CTAs each run many tiles (both issuers cycle every ring slot
    and both accumulator buffers); with tail = 2 the last wave's tiles are cut
    into narrower units."""
    many("max_ctas", ctas)
    many("tail", tail)
    M, N, K = 256, 1100, 700
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=ctas)
    C = run_tn("bf16", ops, M, N, K)
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))


@pytest.mark.parametrize("ldc_pad", [0, 3])
def test_forced_row_wise_stores(ldc_pad, many):
    M, N, K = 37, 333, 200
    ldc = M + ldc_pad
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=11)
    C = run_tn("bf16", ops, M, N, K, ldc=ldc)
    check_full("bf16", ops, M, N, K, C)
    if ldc_pad:
        assert torch.all(torch.isnan(C[:N, M:].float())), "C padding was written"


@pytest.mark.parametrize("M", [16, 64, 128])
def test_fp8_f32_output(M, many):
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


def test_plan_takes_issuers_only_where_allowed(many):
    """Forced, the extra issuers run on one-CTA TMA tiles without K pieces
    whose accumulators fit in 256 TMEM columns, and nowhere else."""
    ni = many.issuers
    many("tile_q", 64)
    st, p = capi.gemm_tn_plan("bf16", 128, 8192, 8192, workspace_bytes=0)     # 64 columns
    assert st == 0 and p["issuers"] == ni and p["pair"] == 0
    many("tile_q", 128)
    st, p = capi.gemm_tn_plan("bf16", 256, 8192, 8192, workspace_bytes=0)     # 128 columns
    assert p["issuers"] == 2
    many("tile_q", 256)
    st, p = capi.gemm_tn_plan("bf16", 256, 8192, 8192, workspace_bytes=0)     # 256: no room
    assert p["issuers"] == 1
    capi.gemm_set_option("pair", -1)
    assert capi.gemm_tn_plan("bf16", 8192, 8192, 8192)[1]["issuers"] == 1      # CTA pairs
    assert capi.gemm_tn_plan("f16_acc16", 128, 8192, 8192)[1]["issuers"] == 1  # FP16 accumulation
