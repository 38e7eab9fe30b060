"""GPU parity of the TN entry points (gemm_f16_tn, gemm_bf16_tn, gemm_fp8_tn)
against the CPU oracle, through the C ABI.

Small and mid-size shapes (several tiles, ragged tails in M, N and K) are
compared element by element; the full-size workloads are compared on 4096
seeded samples plus corners and edges.  +-1 and identity inputs must match
bit for bit.
"""
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


@pytest.fixture(autouse=True, scope="module")
def _gpu():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    capi.lib()
    yield


@pytest.fixture(params=[0, 1], ids=["cta1", "pair"])
def pair_mode(request):
    assert capi.gemm_set_option("pair", request.param) == 0
    yield request.param
    capi.gemm_set_option("pair", -1)


# ------------------------------------------------------------ exact checks

def test_pm1_256_f16_bitexact(pair_mode):
    """FP16 TN 256^3, +-1 entries (seed 0): bit-exact against the oracle."""
    M = N = K = 256
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=0)
    C = run_tn("f16", ops, M, N, K)
    exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(256, 128, 64), (300, 200, 136), (513, 257, 1000)])
def test_pm1_bitexact(kind, shape, pair_mode):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=11)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("kind", KINDS)
def test_pm1_long_k_bitexact(kind, pair_mode):
    """K = 65536 (1024 K stages of 64, or 512 of 128 for FP8) with +-1 entries:
    every partial sum is an integer of magnitude <= 65536 < 2^24, exact in the
    FP32 accumulator, so the rounded outputs must match the oracle bit for bit
    (with FP16 output, |sums| above 2048 round, identically on both sides).
    A K this long also runs the ring's slot/phase counters through many
    wrap-arounds."""
    M, N, K = 200, 136, 65536
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=13)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("kind", ["bf16", "e4m3"])
def test_max_k_sparse_exact(kind):
    """K = 2^31 - 1, the largest K the ABI accepts.  A (1 x K) and B (2 x K)
    are zero except at five k spread over the whole range (0, 1, 2^30, K - 2
    and K - 1, the last two in the final, ragged K stage), so each output is a
    sum of at most five products of powers of two, exact in every format.  The
    element just past K (inside the padded rows) holds a large value that must
    not be read.  The call splits K over a workspace (16 pieces of 2^21 K
    stages, 2^20 for FP8), with the device wait limit raised for the pieces'
    long K loops; every K coordinate stays below 2^31."""
    K = (1 << 31) - 1
    M, N, ld, ldc = 1, 2, 1 << 31, 8
    dt = torch.bfloat16 if kind == "bf16" else torch.float8_e4m3fn
    A = torch.zeros((M, ld), dtype=dt, device="cuda")
    B = torch.zeros((N, ld), dtype=dt, device="cuda")
    for k, v in zip([0, 1, 1 << 30, K - 2, K - 1], [1.0, 2.0, 4.0, 8.0, 16.0]):
        A[0, k] = v
        B[0, k] = 1.0
    B[1, K - 1] = 0.5
    B[1, 0] = 0.25
    A[0, K] = 64.0          # past K: outside the matrix
    B[0, K] = 1.0
    B[1, K] = 1.0
    C = torch.full((N, ldc), float("nan"), dtype=torch.bfloat16, device="cuda")
    ws = torch.empty(64 << 20, dtype=torch.uint8, device="cuda")
    st, plan = capi.gemm_tn_plan(kind, M, N, K, workspace_bytes=ws.numel())
    assert st == 0 and plan["splits"] == 16
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    assert capi.gemm_set_option("timeout_ns", 30_000_000_000) == 0
    try:
        if kind == "bf16":
            st = capi.gemm_bf16_tn(M, N, K, A.data_ptr(), ld, B.data_ptr(), ld, C.data_ptr(),
                                   ldc, None)
        else:
            st = capi.gemm_fp8_tn(M, N, K, A.data_ptr(), ld, B.data_ptr(), ld, 1.0, 1.0,
                                  C.data_ptr(), ldc, None)
        assert st == 0
        torch.cuda.synchronize()
        assert capi.gemm_read_watchdog(1) == capi.GEMM_OK
    finally:
        capi.gemm_set_option("timeout_ns", 2_000_000_000)
        capi.gemm_set_workspace(None, 0)
    assert C[0, 0].item() == 31.0           # 1 + 2 + 4 + 8 + 16
    assert C[1, 0].item() == 8.25           # 16 x 0.5 + 1 x 0.25
    assert torch.isnan(C[:, 1:].float()).all()   # C's padding past M untouched


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("n", [64, 384, 640])
def test_identity_bitexact(kind, n, pair_mode):
    """B = I  =>  C = A exactly (A's values are exact in the output type)."""
    # e4m3 codes are cast directly (scale 1, |x| <= 448): exact in bf16 output
    ops = si.tn_operands(kind, n, n, n, dist="normal", seed=5, dist_b="identity",
                         quantise=False, sigma=4.0 if kind == "e4m3" else 1.0)
    C = run_tn(kind, ops, n, n, n)
    exact = oracle.gemm_tn(kind, n, n, n, si.codes(ops["A"]), n, si.codes(ops["B"]), n,
                           ops["scale_a"], ops["scale_b"])
    # the oracle's exact result is A itself
    np.testing.assert_array_equal(exact, ops["A"].to(torch.float64).numpy() * ops["scale_a"])
    assert_codes_equal(out_codes(C, n, n), exact_codes(kind, exact))


def test_fp8_power_of_two_scales_bitexact(pair_mode):
    M, N, K = 384, 320, 512
    ops = si.tn_operands("e4m3", M, N, K, dist="pm1", seed=12)
    ops["scale_a"], ops["scale_b"] = 2.0 ** -3, 2.0 ** 5
    C = run_tn("e4m3", ops, M, N, K)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K,
                           ops["scale_a"], ops["scale_b"])
    assert_codes_equal(out_codes(C, M, N), exact_codes("e4m3", exact))


# --------------------------------------------------- random, full compare

@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 5, 3), (600, 330, 200), (257, 129, 65),
                                   (1024, 512, 777), (130, 700, 64)])
def test_random_full(kind, shape, pair_mode):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=sum(shape), sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("kind", KINDS)
def test_padded_ld_and_guards(kind, pair_mode):
    """Leading dimensions larger than the extents (TMA-aligned); the NaN-coded
    padding of A and B must never be read, and C's padding rows m in [M, ldc)
    must stay untouched."""
    M, N, K = 333, 190, 300
    lda = ldb = 320 if kind != "e4m3" else 336
    ldc = 344
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=21, lda=lda, ldb=ldb)
    C = run_tn(kind, ops, M, N, K, ldc=ldc)
    check_full(kind, ops, M, N, K, C)
    pad = C[:N, M:ldc].contiguous().view(torch.int16)
    sentinel = 0x7E00 if kind == "f16" else 0x7FC0
    assert torch.all(pad == sentinel), "C padding was written"


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("lds", [(129, 130, 301), (136, 129, 304), (131, 133, 305), (144, 144, 301)])
def test_unaligned_rows(kind, lds):
    """Rows that are not 16-byte aligned (odd leading dimensions, a C pitch that
    is not a multiple of 8) take the load-based producer and/or the row-wise
    epilogue stores; C's padding must stay untouched."""
    M, N, K = 301, 213, 129
    lda, ldb, ldc = lds
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=31, lda=lda, ldb=ldb)
    C = run_tn(kind, ops, M, N, K, ldc=ldc)
    check_full(kind, ops, M, N, K, C)
    if ldc > M:
        pad = C[:N, M:ldc].contiguous().view(torch.int16)
        assert torch.all(pad == (0x7E00 if kind == "f16" else 0x7FC0)), "C padding was written"


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("offset", [1, 2, 6, 8, 14])
def test_misaligned_base_pointers(kind, offset):
    """Base pointers off the 16-byte grid by `offset` elements of A, B and C."""
    M, N, K = 260, 140, 300
    es = 1 if kind == "e4m3" else 2
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=offset, lda=K + 16, ldb=K + 16)
    dt = ops["A"].dtype
    # shift each matrix by `offset` elements inside a larger buffer
    fa = torch.zeros(ops["A"].numel() + offset, dtype=dt)
    fa.view(torch.uint8 if es == 1 else torch.int16)[offset:] = ops["A"].reshape(-1).view(
        torch.uint8 if es == 1 else torch.int16)
    fb = torch.zeros(ops["B"].numel() + offset, dtype=dt)
    fb.view(torch.uint8 if es == 1 else torch.int16)[offset:] = ops["B"].reshape(-1).view(
        torch.uint8 if es == 1 else torch.int16)
    A = fa.cuda()
    B = fb.cuda()
    out_dt = torch.float16 if kind == "f16" else torch.bfloat16
    coff = offset % 8 or 1
    Cbuf = torch.full((N * M + coff,), float("nan"), dtype=out_dt, device="cuda")
    pa = A.data_ptr() + offset * es
    pb = B.data_ptr() + offset * es
    pc = Cbuf.data_ptr() + coff * 2
    s = torch.cuda.current_stream().cuda_stream
    if kind == "e4m3":
        st = capi.gemm_fp8_tn(M, N, K, pa, ops["lda"], pb, ops["ldb"], ops["scale_a"],
                              ops["scale_b"], pc, M, s)
    else:
        fn = capi.gemm_f16_tn if kind == "f16" else capi.gemm_bf16_tn
        st = fn(M, N, K, pa, ops["lda"], pb, ops["ldb"], pc, M, s)
    assert st == 0, capi.status_text(st)
    C = Cbuf.cpu()
    assert torch.all(torch.isnan(C[:coff].float())), "written before C"
    check_full(kind, ops, M, N, K, C[coff:].reshape(N, M))


@pytest.mark.parametrize("kind", KINDS)
def test_forced_load_producer_matches(kind):
    """The load-based producer on TMA-aligned operands, several K tails."""
    assert capi.gemm_set_option("path", 2) == 0
    try:
        for (M, N, K) in [(256, 128, 64), (513, 300, 1000), (129, 257, 77)]:
            ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=K)
            C = run_tn(kind, ops, M, N, K)
            exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
            assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))
    finally:
        capi.gemm_set_option("path", 0)


@pytest.mark.parametrize("kind", KINDS)
def test_forced_fallback_matches(kind):
    M, N, K = 200, 150, 96
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=41)
    assert capi.gemm_set_option("path", 1) == 0
    try:
        C = run_tn(kind, ops, M, N, K)
    finally:
        capi.gemm_set_option("path", 0)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("kind", KINDS)
def test_k_zero_writes_zeros_and_empty_noop(kind):
    M, N = 70, 40
    ops = si.tn_operands(kind, M, N, 1, dist="pm1", seed=1)
    C = run_tn(kind, ops, M, N, 0)
    assert torch.all(C[:N, :M].to(torch.float32) == 0)
    init = torch.full((N, M), 3.0, dtype=torch.bfloat16 if kind != "f16" else torch.float16)
    C = run_tn(kind, ops, 0, N, 1, c_init=init, ldc=M)
    assert torch.all(C == init)
    C = run_tn(kind, ops, M, 0, 1, c_init=init, ldc=M)
    assert torch.all(C == init)


@pytest.mark.parametrize("group", [1, 3, 8, 64])
def test_group_sizes(group):
    M, N, K = 1300, 900, 128
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=group)
    assert capi.gemm_set_option("group", group) == 0
    try:
        C = run_tn("bf16", ops, M, N, K)
    finally:
        capi.gemm_set_option("group", 0)
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))


@pytest.mark.parametrize("ctas", [1, 3, 37])
def test_few_persistent_ctas(ctas):
    """Few CTAs each walk many tiles: exercises the ring and accumulator phases."""
    M, N, K = 1100, 700, 200
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=ctas)
    assert capi.gemm_set_option("max_ctas", ctas) == 0
    try:
        C = run_tn("f16", ops, M, N, K)
    finally:
        capi.gemm_set_option("max_ctas", 0)
    exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))
    assert capi.gemm_read_watchdog(0) == capi.GEMM_OK


# ----------------------------------------------------- full-size workloads

def test_f16_8192_normal_sampled(pair_mode):
    """FP16 TN 8192^3, N(0,1)*0.1 (seed 2): 4096 samples + edges."""
    M = N = K = 8192
    ops = si.tn_operands("f16", M, N, K, dist="normal", seed=2, sigma=0.1)
    C = run_tn("f16", ops, M, N, K)
    check_sampled("f16", ops, M, N, K, C, seed=2)


def test_f16_8192_pm1_k2048_bitexact(pair_mode):
    M, N, K = 8192, 8192, 2048
    ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=2)
    C = run_tn("f16", ops, M, N, K)
    ms, ns = si.sample_positions(M, N, 4096, seed=2)
    exact = oracle.gemm_tn_sampled("f16", K, si.codes(ops["A"]), K, si.codes(ops["B"]), K, ms, ns)
    got = C[torch.from_numpy(ns), torch.from_numpy(ms)].contiguous().view(torch.int16).numpy()
    assert_codes_equal(got.view(np.uint16), exact_codes("f16", exact))


BF16_SHAPES = [(4096, 4096, 4096), (4096, 14336, 4096), (4096, 4096, 14336), (2047, 3001, 1023),
               (8191, 8191, 8191)]


@pytest.mark.parametrize("shape", BF16_SHAPES)
def test_bf16_sweep_sampled(shape, pair_mode):
    """BF16 TN sweep, N(0,1)*0.05 (seed 3), tight leading dimensions."""
    M, N, K = shape
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=3, sigma=0.05)
    C = run_tn("bf16", ops, M, N, K)
    check_sampled("bf16", ops, M, N, K, C, seed=3)


def test_bf16_ragged_tight_ld_full():
    """The ragged shape with tight leading dimensions (rows not 16-byte
    aligned: load-based producer and row-wise stores), compared in full."""
    M, N, K = 2047, 3001, 1023
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=3, sigma=0.05)
    C = run_tn("bf16", ops, M, N, K)
    check_full("bf16", ops, M, N, K, C)


def test_bf16_ragged_padded_ld_and_full():
    """The ragged shape with leading dimensions padded to 16-byte rows (TMA
    path), compared in full."""
    M, N, K = 2047, 3001, 1023
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=3, sigma=0.05, lda=1024, ldb=1024)
    C = run_tn("bf16", ops, M, N, K, ldc=2048)
    check_full("bf16", ops, M, N, K, C)


FP8_SHAPES = [(8192, 8192, 8192), (4096, 14336, 4096), (16384, 4096, 4096)]


@pytest.mark.parametrize("shape", FP8_SHAPES)
def test_fp8_sampled(shape, pair_mode):
    """FP8 E4M3 with per-tensor scales amax/448 (seed 4), bf16 output."""
    M, N, K = shape
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=4)
    C = run_tn("e4m3", ops, M, N, K)
    check_sampled("e4m3", ops, M, N, K, C, seed=4)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("tile_q", [64, 128, 192, 256])
@pytest.mark.parametrize("mode", ["cta1", "pair", "loads"])
def test_tile_q_variants(kind, tile_q, mode):
    """Every output tile width along M, with each producer / CTA grouping."""
    M, N, K = 450, 300, 333
    assert capi.gemm_set_option("tile_q", tile_q) == 0
    assert capi.gemm_set_option("pair", 1 if mode == "pair" else 0) == 0
    assert capi.gemm_set_option("path", 2 if mode == "loads" else 0) == 0
    try:
        ops = si.tn_operands(kind, M, N, K, dist="normal", seed=tile_q, sigma=0.5)
        C = run_tn(kind, ops, M, N, K)
        check_full(kind, ops, M, N, K, C)
    finally:
        capi.gemm_set_option("tile_q", 0)
        capi.gemm_set_option("pair", -1)
        capi.gemm_set_option("path", 0)


@pytest.mark.parametrize("M", [1, 16, 64, 100, 128, 200, 300])
def test_skinny_m_auto_tile(M):
    """Small M picks a narrow tile; results stay bit-exact on +-1 inputs."""
    N, K = 1000, 512
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=M)
    C = run_tn("bf16", ops, M, N, K)
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes("bf16", exact))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("tail", [2, 4])
@pytest.mark.parametrize("mode", ["cta1", "pair", "loads"])
def test_tail_split_variants(kind, tail, mode):
    """The last partial wave cut into narrower units (forced), few CTAs so that
    whole tiles and tail units share the persistent loop."""
    M, N, K = 1100, 700, 300
    opts = {"tail": tail, "pair": 1 if mode == "pair" else 0, "path": 2 if mode == "loads" else 0,
            "max_ctas": 10, "tile_q": 256}
    for k, v in opts.items():
        assert capi.gemm_set_option(k, v) == 0
    try:
        ops = si.tn_operands(kind, M, N, K, dist="normal", seed=tail, sigma=0.5)
        C = run_tn(kind, ops, M, N, K)
        check_full(kind, ops, M, N, K, C)
    finally:
        for k, v in {"tail": 0, "pair": -1, "path": 0, "max_ctas": 0, "tile_q": 0}.items():
            capi.gemm_set_option(k, v)


def test_tail_split_fp32_out():
    M, N, K = 1000, 900, 200
    for k, v in {"tail": 2, "max_ctas": 12}.items():
        assert capi.gemm_set_option(k, v) == 0
    try:
        ops = si.tn_operands("e4m3", M, N, K, dist="pm1", seed=2)
        A, B = ops["A"].cuda(), ops["B"].cuda()
        C = torch.full((N, M), float("nan"), device="cuda")
        st = capi.gemm_fp8_tn_f32(M, N, K, A.data_ptr(), K, B.data_ptr(), K, 1.0, 1.0,
                                  C.data_ptr(), M, torch.cuda.current_stream().cuda_stream)
        assert st == 0
        exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
        np.testing.assert_array_equal(C.cpu().numpy().T, exact.astype(np.float32))
    finally:
        for k, v in {"tail": 0, "max_ctas": 0}.items():
            capi.gemm_set_option(k, v)

@pytest.mark.parametrize("kind", KINDS)
def test_subwave_small_tiles(kind):
    """Pair tiles fill less than a wave (8 x 4 = 32) while single-CTA tiles of
    128 x 128 fit in one (16 x 8 = 128): the automatic choice runs the small
    tiles; ragged on both edges."""
    M, N, K = 1000, 2000, 500
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=7, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


@pytest.mark.parametrize("kind,shape", [("bf16", (256, 8192, 8192)), ("e4m3", (1024, 1024, 8192))])
def test_subwave_small_tiles_sampled(kind, shape):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=8, sigma=0.05)
    C = run_tn(kind, ops, M, N, K)
    check_sampled(kind, ops, M, N, K, C, seed=8)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(1 << 20, 128, 64), (128, 1 << 20, 64)])
def test_million_row_extents_sampled(kind, shape):
    """One operand a million rows long: 4096 tiles along one dimension, TMA row
    coordinates up to 2^20, C of 2^27 elements."""
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=9, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_sampled(kind, ops, M, N, K, C, seed=9)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(1, 1, 8192), (1, 300, 1), (300, 1, 1), (257, 129, 1)])
def test_degenerate_shapes_pm1_bitexact(kind, shape):
    """M = N = 1 with a long K, and K = 1 (a single product per output)."""
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=sum(shape))
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))
