"""GPU parity of rotated K ranges (option "k_rotate" = 2) against the CPU
oracle, through the C ABI.

The TMA producer starts each unit's K range at a stage of its own (spaced by
the unit's tile row) and wraps around; the MMA warp sums whatever stage comes
next.  These cases cover every input kind, one CTA and CTA pairs, pairs of
64-row halves, two K atoms per stage, two MMA issuers, K split into pieces
(each piece rotates within its own range), few CTAs walking many tiles (the
K snake reverses every second unit as well), ragged K, and +-1 inputs (exact,
so any stage read twice or skipped shows)."""
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import assert_codes_equal, check_full, check_sampled, exact_codes, out_codes, run_tn

pytestmark = pytest.mark.gpu
KINDS = ["f16", "bf16", "e4m3"]
DEFAULTS = {"k_rotate": 0, "pair": -1, "half": 0, "splits": 0, "max_ctas": 0, "issuers": 0,
            "atoms": 0, "tile_q": 0}


@pytest.fixture
def rotate():
    assert capi.gemm_set_option("k_rotate", 2) == 0

    def set_(name, value):
        assert capi.gemm_set_option(name, value) == 0
    yield set_
    for name, value in DEFAULTS.items():
        capi.gemm_set_option(name, value)
    capi.gemm_set_workspace(None, 0)


def exact_case(kind, M, N, K, seed):
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=seed)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("K", [64, 1000, 2048, 2111])
def test_pm1_bitexact(kind, pair, K, rotate):
    rotate("pair", pair)
    exact_case(kind, 600, 1100, K, seed=K + pair)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("M", [16, 128, 192, 256])
def test_skinny_auto_plans(kind, M, rotate):
    """The automatic skinny plans: one-CTA tiles with two issuers and two
    atoms, pairs of halves, split K through the workspace."""
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    exact_case(kind, M, 2048, 2048, seed=M)


@pytest.mark.parametrize("splits", [2, 3, 5])
def test_split_pieces_rotate_within_their_range(splits, rotate):
    ws = torch.empty(1 << 27, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    rotate("splits", splits)
    M, N, K = 256, 1024, 4100
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    st, p = capi.gemm_tn_plan("bf16", M, N, K, workspace_bytes=ws.numel(), sms=sms)
    assert st == 0 and p["splits"] == splits, p
    exact_case("bf16", M, N, K, seed=splits)


@pytest.mark.parametrize("ctas", [1, 6])
def test_few_ctas_many_units(ctas, rotate):
    """Each CTA runs many units: rotated and, every second one, reversed."""
    rotate("max_ctas", ctas)
    exact_case("f16", 700, 1500, 900, seed=ctas)


@pytest.mark.parametrize("kind", KINDS)
def test_random(kind, rotate):
    M, N, K = 300, 777, 1500
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=3, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


def test_skinny_full_size_sampled(rotate):
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    M, N, K = 256, 8192, 8192
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=4, sigma=0.05)
    C = run_tn("bf16", ops, M, N, K)
    check_sampled("bf16", ops, M, N, K, C, seed=4)


def _debug_line(capfd, kind, M, N, K):
    import os
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=1)
    os.environ["GEMM_DEBUG"] = "1"
    try:
        capfd.readouterr()
        C = run_tn(kind, ops, M, N, K)
        err = capfd.readouterr().err
    finally:
        del os.environ["GEMM_DEBUG"]
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))
    return [ln for ln in err.splitlines() if ln.startswith("[gemm] tn")][-1]


def test_automatic_choice(capfd):
    """Rotation runs by itself for unsplit plans with two MMA issuers (the
    skinny shapes), not for split or one-issuer plans."""
    ws = torch.empty(1 << 26, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    try:
        line = _debug_line(capfd, "bf16", 128, 8192, 1024)        # pairs of halves
        assert "issuers=2" in line and "k_rotate=1" in line, line
        line = _debug_line(capfd, "bf16", 64, 14336, 512)         # one-CTA, two issuers
        assert "issuers=2" in line and "k_rotate=1" in line, line
        line = _debug_line(capfd, "bf16", 16, 8192, 1024)         # split K
        assert "splits=2" in line and "k_rotate=0" in line, line
        line = _debug_line(capfd, "f16", 2048, 2048, 512)         # CTA pairs
        assert "issuers=1" in line and "k_rotate=0" in line, line
        assert capi.gemm_set_option("k_rotate", 1) == 0
        line = _debug_line(capfd, "bf16", 128, 8192, 1024)
        assert "k_rotate=0" in line, line
    finally:
        capi.gemm_set_option("k_rotate", 0)
        capi.gemm_set_workspace(None, 0)
