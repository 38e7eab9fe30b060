"""K-snake and band-snake, the tensor-core kernel's L2-friendly orders (both on
by default).  K-snake: every second unit a persistent CTA runs reads its K
range backwards, so that the K slices one wave of tiles ends on are still in
L2 when the next wave starts on them; only the order in which K stages reach
the accumulator changes.  Band-snake: odd rasteriser bands walk the tile
columns backwards.  These cases pin both against the oracle with few CTAs
(most units then run reversed), several bands, a ragged last K stage, CTA
pairs and single CTAs, split-K pieces and a narrowed last wave, with the
options on and off."""
import pytest

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import assert_codes_equal, check_full, exact_codes, out_codes, run_tn

pytestmark = pytest.mark.gpu


@pytest.fixture
def opts():
    touched = []

    def set_(name, value):
        assert capi.gemm_set_option(name, value) == 0
        touched.append(name)
    yield set_
    defaults = {"pair": -1, "k_snake": 1, "band_snake": 1}
    for name in touched:
        capi.gemm_set_option(name, defaults.get(name, 0))


@pytest.mark.parametrize("snake", [0, 1])
@pytest.mark.parametrize("pair,ctas", [(1, 4), (1, 6), (0, 3), (0, 5)])
@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_reversed_k_ranges_random(kind, pair, ctas, snake, opts):
    M, N, K = 700, 1100, 1000        # ragged in every dimension and in the last K stage
    opts("k_snake", snake)
    opts("band_snake", snake)
    opts("group", 2)                 # several bands, so that some walk backwards
    opts("pair", pair)
    opts("max_ctas", ctas)
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=17 + ctas, sigma=1.0 if kind == "e4m3"
                         else 0.3)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("splits", [2, 3])
def test_reversed_k_ranges_with_split_pieces(splits, opts):
    """K pieces of split tiles, each read backwards by some CTAs; the fix-up
    still sums the pieces in piece order."""
    import torch

    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    try:
        opts("splits", splits)
        opts("max_ctas", 3)
        M, N, K = 300, 520, 2000
        ops = si.tn_operands("f16", M, N, K, dist="normal", seed=splits, sigma=0.3)
        C = run_tn("f16", ops, M, N, K)
        check_full("f16", ops, M, N, K, C)
        ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=splits)
        C = run_tn("f16", ops, M, N, K)
        exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
        assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))
    finally:
        assert capi.gemm_set_workspace(None, 0) == 0


def test_reversed_k_ranges_narrowed_tail_pm1(opts):
    """Pair tiles with a narrowed last wave (tail 2), +-1 inputs: exact."""
    opts("pair", 1)
    opts("max_ctas", 6)
    opts("tail", 2)
    M, N, K = 1024, 1536, 704
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=5)
    C = run_tn("bf16", ops, M, N, K)
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))
