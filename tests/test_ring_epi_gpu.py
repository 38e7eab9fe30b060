"""GPU parity of rings that run on over the epilogue's staging area (plan field
ring_epi = 1) against the CPU oracle, through the C ABI.

Where every CTA pair of a plan of 64-row halves runs one unit, the ring takes
the epilogue's 32 KB of staging buffers as well; the epilogue writes them only
after the accumulator-full barrier, when every load has been consumed and every
MMA has completed.  These cases cover that on every input kind, at widths 32,
64, 160, 192 and 224 with one and two issuers, with K from less than one ring
to many ring cycles, TMA and row-wise stores, FP32 output, and +-1 inputs
(exact: a stage overwritten by the epilogue while still in use, or a staged
chunk overwritten by a load, would show); and that the other plans keep the
192 KB ring."""
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
DEFAULTS = {"pair": -1, "half": 0, "tile_q": 0, "splits": 0, "issuers": 0, "max_ctas": 0}


@pytest.fixture
def opts():
    ws = torch.empty(1 << 27, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0

    def set_(name, value):
        assert capi.gemm_set_option(name, value) == 0
    set_.ws = ws
    yield set_
    for name, value in DEFAULTS.items():
        capi.gemm_set_option(name, value)
    capi.gemm_set_workspace(None, 0)


def planned(kind, M, N, K, ws, flags=capi.PLAN_ALIGNED):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = capi.gemm_tn_plan(kind, M, N, K, flags=flags, workspace_bytes=ws.numel(), sms=sms)
    assert st == 0 and p["status"] == 0
    return p


def exact(kind, M, N, K, seed, ldc=None):
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=seed)
    C = run_tn(kind, ops, M, N, K, ldc=ldc)
    ref = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, ref))
    return C


PLANS = {
    # name: (options, M, N) -- pairs of halves, one unit per pair
    "halves_192": ({"half": 3, "tile_q": 192}, 190, 2000),
    "halves_160_one_issuer": ({"half": 3, "issuers": 1}, 150, 2000),
    "halves_160": ({"half": 3}, 160, 1000),
    "halves_224": ({"half": 3}, 210, 1500),
    "halves_32": ({"half": 3}, 20, 2000),
    "halves_64": ({"half": 3}, 48, 1000),
}


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("name", list(PLANS))
@pytest.mark.parametrize("K", [200, 2048, 8200])
def test_pm1_bitexact(kind, name, K, opts):
    o, M, N = PLANS[name]
    for k, v in o.items():
        opts(k, v)
    p = planned(kind, M, N, K, opts.ws)
    assert (p["pair"], p["half"], p["ring_epi"]) == (1, 1, 1), (name, p)
    exact(kind, M, N, K, seed=M + K)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("M,N,K,pair", [(16, 2048, 2048, -1), (700, 1000, 2048, 1),
                                        (300, 1500, 1000, 0)])
def test_other_plans_keep_the_short_ring(kind, M, N, K, pair, opts):
    """Split one-CTA tiles, CTA pairs 256 wide and one-CTA tiles 128 wide run
    one unit per CTA too, but measured slower with the longer ring."""
    opts("pair", pair)
    p = planned(kind, M, N, K, opts.ws)
    assert p["half"] == 0 and p["ring_epi"] == 0, p
    exact(kind, M, N, K, seed=M)


@pytest.mark.parametrize("ldc_pad", [3, 8])
def test_row_wise_and_padded_stores(ldc_pad, opts):
    """ldc = M + 3: row-wise stores through the staging buffers; ldc = M + 8:
    TMA stores (and lane stores for the halves' cut chunks); the padding keeps
    its sentinel."""
    opts("half", 3)
    M, N, K = 171, 900, 1024
    p = planned("bf16", M, N, K, opts.ws)
    assert p["ring_epi"] == 1, p
    C = exact("bf16", M, N, K, seed=ldc_pad, ldc=M + ldc_pad)
    assert torch.all(torch.isnan(C[:N, M:].float())), "C padding was written"


def test_fp8_f32_output(opts):
    from test_fp8_f32out_gpu import run, tols

    opts("half", 3)
    M, N, K = 150, 2048, 1024
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = capi.gemm_tn_plan("e4m3_f32out", M, N, K, workspace_bytes=opts.ws.numel(), sms=sms)
    assert st == 0 and (p["half"], p["tile_q"], p["ring_epi"]) == (1, 160, 1), p
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=M)
    C = run(ops, M, N, K)
    ref = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K,
                         ops["scale_a"], ops["scale_b"])
    a = ops["A"][:, :K].to(torch.float64).numpy() * ops["scale_a"]
    b = ops["B"][:, :K].to(torch.float64).numpy() * ops["scale_b"]
    contract, tight = tols(ops, K, ref, np.abs(a) @ np.abs(b).T)
    err = np.abs(C[:N, :M].double().numpy().T - ref)
    assert err.max() <= contract and np.all(err <= tight)


@pytest.mark.parametrize("kind,shape", [("bf16", (192, 8192, 8192)), ("f16", (160, 8192, 16384)),
                                        ("bf16", (224, 8192, 8192)), ("e4m3", (200, 8192, 8192))])
def test_full_size_sampled(kind, shape, opts):
    M, N, K = shape
    if kind == "e4m3":
        opts("half", 3)
    assert planned(kind, M, N, K, opts.ws)["ring_epi"] == 1
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=5, sigma=0.05)
    C = run_tn(kind, ops, M, N, K)
    check_sampled(kind, ops, M, N, K, C, seed=5)


def test_several_units_per_cta_keep_the_short_ring(opts):
    """Capping the CTAs gives them several tiles each: the ring stays clear of
    the staging area (ring_epi = 0) and the results stay exact."""
    opts("max_ctas", 8)
    M, N, K = 190, 2000, 1000
    opts("half", 3)
    p = planned("bf16", M, N, K, opts.ws)
    assert p["ring_epi"] == 0, p
    exact("bf16", M, N, K, seed=3)
