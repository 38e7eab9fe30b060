"""GPU parity of ring stages two K atoms deep (option "atoms" = 2) against
the CPU oracle, through the C ABI.

A stage then holds P atom 0, P atom 1, Q atom 0 and Q atom 1 (two 128-byte
swizzle spans of K per row), the producer issues two boxes per operand, and
the MMA warp issues eight MMAs (four per atom, for every input type) before
one commit.  These cases cover every input kind
and output type; CTA pairs, one-CTA tiles of 16 to 256 columns, pairs of
64-row halves with two issuers and one-CTA tiles with two issuers; K that
ends inside a stage's first or second atom (the second box then lies wholly
past K and is zero-filled); narrowed and K-split last waves; split-K through
the workspace; few CTAs walking many tiles (ring phases); FP16 accumulation;
the load-based producer (which keeps one atom); and +-1 inputs (exact).
Each case asserts through gemm_tn_plan that the call runs with two atoms."""
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
DEFAULTS = {"atoms": 0, "pair": -1, "half": 0, "tile_q": 0, "splits": 0, "issuers": 0,
            "tail": 0, "tail_k": 0, "max_ctas": 0}


@pytest.fixture
def atoms2():
    assert capi.gemm_set_option("atoms", 2) == 0

    def set_(name, value):
        assert capi.gemm_set_option(name, value) == 0
    yield set_
    for name, value in DEFAULTS.items():
        capi.gemm_set_option(name, value)
    capi.gemm_set_workspace(None, 0)


def planned(kind, M, N, K, ws=0, flags=capi.PLAN_ALIGNED):
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = capi.gemm_tn_plan(kind, M, N, K, flags=flags, workspace_bytes=ws, sms=sms)
    assert st == 0 and p["status"] == 0
    return p


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(1000, 1200, 700), (300, 2000, 333), (64, 900, 130),
                                   (2048, 1024, 1088), (129, 257, 2049), (1, 64, 64)])
def test_random(kind, shape, atoms2):
    M, N, K = shape
    assert planned(kind, M, N, K)["atoms"] == 2
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=M + N + K, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("K", [64, 128, 192, 200, 2048])
def test_pm1_bitexact(kind, pair, K, atoms2):
    """K ending in the first atom of a stage (64, 192, 200 for 16-bit inputs)
    or on a stage boundary (128, 2048); FP8's atom is 128 values deep."""
    atoms2("pair", pair)
    M, N = 500, 700
    p = planned(kind, M, N, K)
    assert p["atoms"] == 2 and p["pair"] == pair
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=K + pair)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("kind,M,half,issuers", [("bf16", 128, 3, 0), ("f16", 100, 3, 0),
                                                  ("bf16", 64, 0, 2), ("e4m3", 16, 0, 2),
                                                  ("bf16", 100, 0, 2)])
def test_halves_and_issuers(kind, M, half, issuers, atoms2):
    atoms2("half", half)
    atoms2("issuers", issuers)
    if half == 0:
        atoms2("pair", 0)
    N, K = 1100, 1000
    p = planned(kind, M, N, K)
    assert p["atoms"] == 2 and p["issuers"] == 2, p
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=M)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("tail,tail_k", [(2, 0), (4, 0), (0, 3)])
def test_last_wave(tail, tail_k, atoms2):
    """A narrowed last wave (2 or 4 units per tile: Q atoms stay full-width
    apart, the narrow boxes fill their start) and a K-split one."""
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    atoms2("tail", tail)
    atoms2("tail_k", tail_k)
    atoms2("max_ctas", 7)
    if tail == 4:
        atoms2("tile_q", 256)   # quarters of 64 columns
    M, N, K = 700, 1100, 1500
    p = planned("bf16", M, N, K, ws=ws.numel())
    assert p["atoms"] == 2 and p["tail_f"] > 1, p
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=tail + tail_k)
    C = run_tn("bf16", ops, M, N, K)
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("pair,splits", [(0, 0), (1, 3), (0, 5)])
def test_split_k(kind, pair, splits, atoms2):
    ws = torch.empty(1 << 27, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    atoms2("pair", pair)
    atoms2("splits", splits)
    M, N, K = 256, 1024, 4100
    p = planned(kind, M, N, K, ws=ws.numel())
    assert p["atoms"] == 2 and p["splits"] >= 2, p
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=7 + splits, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("ctas", [1, 4])
def test_few_ctas_many_tiles(ctas, atoms2):
    atoms2("max_ctas", ctas)
    M, N, K = 600, 900, 1000
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=ctas)
    C = run_tn("f16", ops, M, N, K)
    exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))


@pytest.mark.parametrize("pair", [0, 1])
def test_fp16_accumulation_pm1(pair, atoms2):
    """FP16 accumulation: +-1 sums with K <= 2048 stay integers FP16 holds."""
    from test_acc16_gpu import run

    atoms2("pair", pair)
    M, N, K = 600, 330, 2000
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=K + pair)
    C = run(ops, M, N, K)
    exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))


def test_fp8_f32_output(atoms2):
    from test_fp8_f32out_gpu import run, tols

    M, N, K = 200, 520, 640
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=M)
    C = run(ops, M, N, K)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K,
                           ops["scale_a"], ops["scale_b"])
    a = ops["A"][:, :K].to(torch.float64).numpy() * ops["scale_a"]
    b = ops["B"][:, :K].to(torch.float64).numpy() * ops["scale_b"]
    contract, tight = tols(ops, K, exact, np.abs(a) @ np.abs(b).T)
    err = np.abs(C[:N, :M].double().numpy().T - exact)
    assert err.max() <= contract and np.all(err <= tight)


def test_load_producer_keeps_one_atom(atoms2):
    """Rows TMA cannot address (lda = K + 1) without a workspace: the load-based
    producer runs, with one atom per stage."""
    M, N, K = 130, 300, 257
    flags = capi.PLAN_ALIGNED & ~(capi.PLAN_A_TMA | capi.PLAN_A_128)
    assert planned("bf16", M, N, K, flags=flags)["atoms"] == 1
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=1, lda=K + 1)
    C = run_tn("bf16", ops, M, N, K)
    check_full("bf16", ops, M, N, K, C)


@pytest.mark.parametrize("kind,shape", [("f16", (8192, 8192, 8192)), ("e4m3", (4096, 8192, 8192)),
                                        ("bf16", (128, 8192, 8192))])
def test_large_sampled(kind, shape, atoms2):
    M, N, K = shape
    assert planned(kind, M, N, K)["atoms"] == 2
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=2,
                         sigma=1.0 if kind == "e4m3" else 0.05)
    C = run_tn(kind, ops, M, N, K)
    check_sampled(kind, ops, M, N, K, C, seed=6)


@pytest.mark.parametrize("kind", ["f16", "bf16"])
def test_long_k_sub_wave_pairs_auto(kind):
    """The automatic plan for long K below a wave of tiles (M > 256, K >= 8192):
    CTA pairs 128 columns wide, two K atoms per stage, K cut into pieces through
    the workspace; +-1 inputs, exact."""
    ws = torch.empty(1 << 27, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    try:
        M, N, K = 300, 512, 8200
        p = planned(kind, M, N, K, ws=ws.numel())
        assert (p["pair"], p["tile_q"], p["atoms"]) == (1, 128, 2) and p["splits"] >= 2, p
        ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=17)
        C = run_tn(kind, ops, M, N, K)
        exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
        assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))
    finally:
        capi.gemm_set_workspace(None, 0)


def test_long_k_sub_wave_pairs_unsplit_sampled():
    """1024 x 1536 x 8192: 48 pair tiles 128 wide, one K piece each."""
    M, N, K = 1024, 1536, 8192
    p = planned("bf16", M, N, K)
    assert (p["pair"], p["tile_q"], p["splits"]) == (1, 128, 1), p
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=21, sigma=0.05)
    C = run_tn("bf16", ops, M, N, K)
    check_sampled("bf16", ops, M, N, K, C, seed=8)
