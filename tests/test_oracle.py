"""Pins of the CPU oracle against facts fixed outside it (CPU only).

Each test checks the oracle against something other than itself: hand-worked
products (tests/golden), an independent BLAS (torch float64 matmul), torch's
own dtype casts (exhaustively for the decoders), integer arithmetic for +-1
inputs, and closed forms (identity, all-ones, row sums, exact power-of-two
scales).  The planted-mistake test shows that the hand-worked cases tell the
true product from the plausible wrong ones.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from conftest import load_golden

GOLDEN = ["hand_2x2.txt", "hand_3x3.txt", "hand_2x4x3.txt"]
TN_KINDS = ["f16", "bf16", "e4m3"]


def _tn_store(kind, A, B, lda_pad=0, ldb_pad=0):
    """Logical A (M,K), B (K,N) float arrays -> TN storage codes with padded ld."""
    M, K = A.shape
    N = B.shape[1]
    ta = torch.tensor(A, dtype=torch.float32).to(si.torch_dtype(kind))
    tb = torch.tensor(B.T.copy(), dtype=torch.float32).to(si.torch_dtype(kind))
    sa = si._pad(ta, K + lda_pad, kind)
    sb = si._pad(tb, K + ldb_pad, kind)
    return si.codes(sa), K + lda_pad, si.codes(sb), K + ldb_pad


@pytest.mark.parametrize("name", GOLDEN)
@pytest.mark.parametrize("kind", TN_KINDS)
@pytest.mark.parametrize("pad", [(0, 0), (5, 3)])
def test_golden_tn(name, kind, pad):
    M, N, K, A, B, C = load_golden(name)
    a, lda, b, ldb = _tn_store(kind, A, B, *pad)
    got = oracle.gemm_tn(kind, M, N, K, a, lda, b, ldb)
    np.testing.assert_array_equal(got, C)


@pytest.mark.parametrize("name", GOLDEN)
@pytest.mark.parametrize("pad", [(0, 0), (3, 2)])
def test_golden_f32(name, pad):
    M, N, K, A, B, C = load_golden(name)
    lda, ldb = K + pad[0], N + pad[1]
    a = si._pad(torch.tensor(A, dtype=torch.float32), lda, "f32").numpy()
    b = si._pad(torch.tensor(B, dtype=torch.float32), ldb, "f32").numpy()
    got = oracle.gemm_f32(M, N, K, a, lda, b, ldb)
    np.testing.assert_array_equal(got, C)


@pytest.mark.parametrize("name", GOLDEN)
def test_golden_sampled_matches(name):
    M, N, K, A, B, C = load_golden(name)
    a, lda, b, ldb = _tn_store("bf16", A, B)
    ms, ns = np.meshgrid(np.arange(M), np.arange(N), indexing="ij")
    got = oracle.gemm_tn_sampled("bf16", K, a, lda, b, ldb, ms.ravel(), ns.ravel())
    np.testing.assert_array_equal(got.reshape(M, N), C)
    af = np.ascontiguousarray(A, dtype=np.float32)
    bf = np.ascontiguousarray(B, dtype=np.float32)
    got32 = oracle.gemm_f32_sampled(K, af, K, bf, N, ms.ravel(), ns.ravel())
    np.testing.assert_array_equal(got32.reshape(M, N), C)


def test_fp8_scales_exact():
    """Power-of-two per-tensor scales multiply the exact product exactly."""
    M, N, K, A, B, C = load_golden("hand_2x4x3.txt")
    a, lda, b, ldb = _tn_store("e4m3", A, B)
    got = oracle.gemm_tn("e4m3", M, N, K, a, lda, b, ldb, scale_a=2.0 ** -3, scale_b=2.0 ** 5)
    np.testing.assert_array_equal(got, C * 4.0)
    got = oracle.gemm_tn("e4m3", M, N, K, a, lda, b, ldb, scale_a=0.5, scale_b=0.75)
    np.testing.assert_array_equal(got, C * 0.375)


def test_planted_mistakes_are_caught():
    """The hand-worked products differ from every plausible wrong product."""
    for name in GOLDEN:
        M, N, K, A, B, C = load_golden(name)
        wrong = []
        if A.shape == B.T.shape:
            wrong.append(A @ B.T)          # B read row-major instead of column-major
        if A.shape[0] == A.shape[1]:
            wrong.append(A.T @ B)          # A read column-major
        if B.shape[1] == A.shape[0]:
            wrong.append(B @ A)            # operands swapped
        wrong.append(A[:, :-1] @ B[:-1, :])  # last k term dropped
        wrong.append(A[:, 1:] @ B[1:, :])    # first k term dropped
        wrong.append(-(A @ B))             # sign flip
        for w in wrong:
            assert w.shape != C.shape or not np.array_equal(w, C)


@pytest.mark.parametrize("kind", TN_KINDS)
@pytest.mark.parametrize("shape", [(1, 1, 1), (7, 5, 3), (33, 17, 64), (64, 48, 129), (5, 70, 31)])
def test_tn_vs_torch_float64(kind, shape):
    """Against torch's float64 matmul of torch's own decoding of the same codes."""
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=M * 131 + N * 7 + K,
                         lda=K + 3, ldb=K + 1)
    A, B = ops["A"], ops["B"]
    ref = (A[:, :K].to(torch.float64) * ops["scale_a"]) @ (B[:, :K].to(torch.float64) * ops["scale_b"]).T
    got = oracle.gemm_tn(kind, M, N, K, si.codes(A), ops["lda"], si.codes(B), ops["ldb"],
                         ops["scale_a"], ops["scale_b"])
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("shape", [(1, 1, 1), (9, 4, 6), (40, 33, 70)])
def test_f32_vs_torch_float64(shape):
    M, N, K = shape
    ops = si.f32_operands(M, N, K, seed=sum(shape), lda=K + 2, ldb=N + 5)
    A, B = ops["A"], ops["B"]
    ref = A[:, :K].double() @ B[:, :N].double()
    got = oracle.gemm_f32(M, N, K, A.numpy(), ops["lda"], B.numpy(), ops["ldb"])
    np.testing.assert_allclose(got, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_sampled_vs_torch_float64():
    M, N, K = 50, 60, 200
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=9)
    ms, ns = si.sample_positions(M, N, 300, seed=9)
    A, B = ops["A"], ops["B"]
    full = (A.to(torch.float64) * ops["scale_a"]) @ (B.to(torch.float64) * ops["scale_b"]).T
    got = oracle.gemm_tn_sampled("e4m3", K, si.codes(A), K, si.codes(B), K, ms, ns,
                                 ops["scale_a"], ops["scale_b"])
    np.testing.assert_allclose(got, full.numpy()[ms, ns], rtol=1e-12, atol=1e-12)
    fo = si.f32_operands(M, N, K, seed=10)
    got32 = oracle.gemm_f32_sampled(K, fo["A"].numpy(), K, fo["B"].numpy(), N, ms, ns)
    ref32 = (fo["A"].double() @ fo["B"].double()).numpy()[ms, ns]
    np.testing.assert_allclose(got32, ref32, rtol=1e-12, atol=1e-12)


# ------------------------------------------------------------------ decoders

def _all_codes16():
    return np.arange(65536, dtype=np.uint32).astype(np.uint16)


@pytest.mark.parametrize("kind,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_decoder_exhaustive_16bit(kind, tdt):
    codes = _all_codes16()
    ref = torch.from_numpy(codes.view(np.int16).copy()).view(tdt).to(torch.float64).numpy()
    got = oracle.decode(kind, codes)
    nan = np.isnan(ref)
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    # signed zeros decode with their sign
    np.testing.assert_array_equal(np.signbit(got[~nan]), np.signbit(ref[~nan]))


def test_decoder_exhaustive_e4m3():
    codes = np.arange(256, dtype=np.uint8)
    ref = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = oracle.decode("e4m3", codes)
    nan = np.isnan(ref)
    assert nan.sum() == 2  # 0x7F and 0xFF
    np.testing.assert_array_equal(np.isnan(got), nan)
    np.testing.assert_array_equal(got[~nan], ref[~nan])
    assert got[0x7E] == 448.0 and got[0x01] == 2.0 ** -9


# ------------------------------------------------------------------ encoders

def _float32_probe_values():
    gen = torch.Generator().manual_seed(123)
    parts = [
        torch.randn(200000, generator=gen) * 3,
        torch.randn(50000, generator=gen) * 1e-5,      # fp16 subnormal range
        torch.randn(50000, generator=gen) * 4e4,       # fp16 overflow boundary
        torch.randn(50000, generator=gen) * 1e-39,     # bf16 subnormals
        torch.randn(50000, generator=gen) * 1e38,      # bf16 overflow boundary
        torch.tensor([0.0, -0.0, 65504.0, 65519.0, 65520.0, 65536.0, 2.0 ** -24, 2.0 ** -25,
                      3 * 2.0 ** -26, 257.0, 258.0, 259.0, 3.4028234e38, float("inf"), float("-inf")]),
    ]
    return torch.cat(parts).to(torch.float32)


def _ties(tdt, count=20000):
    """Exact midpoints between neighbouring codes, as float32 (exact there)."""
    gen = torch.Generator().manual_seed(7)
    c = torch.randint(0, 0x7BFF if tdt == torch.float16 else 0x7F7F, (count,), generator=gen,
                      dtype=torch.int32).to(torch.int16)
    lo = c.view(tdt).to(torch.float64)
    hi = (c + 1).view(tdt).to(torch.float64)
    mid = (lo + hi) / 2
    return torch.cat([mid, -mid]).to(torch.float32)


@pytest.mark.parametrize("kind,tdt", [("f16", torch.float16), ("bf16", torch.bfloat16)])
def test_encoder_vs_torch_cast(kind, tdt):
    x = torch.cat([_float32_probe_values(), _ties(tdt)])
    ref = x.to(tdt).view(torch.int16).numpy().view(np.uint16)
    got = oracle.encode_rne(kind, x.to(torch.float64).numpy())
    np.testing.assert_array_equal(got, ref)


def test_encoder_ties_to_even_examples():
    # 2049 lies halfway between fp16 2048 and 2050: even significand wins (2048).
    assert oracle.encode_rne("f16", np.array([2049.0]))[0] == 0x6800
    assert oracle.encode_rne("f16", np.array([2051.0]))[0] == 0x6802  # -> 2052
    # bf16 has 8 significant bits: 257 -> 256, 259 -> 260.
    assert oracle.encode_rne("bf16", np.array([257.0]))[0] == 0x4380
    assert oracle.encode_rne("bf16", np.array([259.0]))[0] == 0x4382


# ------------------------------------------------------------ closed forms

@pytest.mark.parametrize("kind", TN_KINDS)
def test_identity_tn(kind):
    """B = I  =>  C = A, exactly (the identity-matrix test)."""
    n = 37
    ops = si.tn_operands(kind, n, n, n, dist="normal", seed=5, dist_b="identity", ldb=n + 4)
    assert ops["scale_b"] == 1.0  # identity codes are exact and unscaled
    got = oracle.gemm_tn(kind, n, n, n, si.codes(ops["A"]), ops["lda"], si.codes(ops["B"]),
                         ops["ldb"], ops["scale_a"], 1.0)
    ref = ops["A"].to(torch.float64).numpy() * ops["scale_a"]
    np.testing.assert_array_equal(got, ref)


def test_identity_f32():
    n = 45
    ops = si.f32_operands(n, n, n, seed=1, dist_b="identity")
    got = oracle.gemm_f32(n, n, n, ops["A"].numpy(), n, ops["B"].numpy(), n)
    np.testing.assert_array_equal(got, ops["A"].double().numpy())


@pytest.mark.parametrize("kind", TN_KINDS)
def test_pm1_matches_integer_arithmetic(kind):
    """+-1 inputs: every sum is an integer; compare against int64 matmul exactly."""
    M, N, K = 40, 24, 300
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=0)
    ia = ops["A"].to(torch.float32).to(torch.int64).numpy()
    ib = ops["B"].to(torch.float32).to(torch.int64).numpy()
    ref = ia @ ib.T
    got = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    np.testing.assert_array_equal(got, ref.astype(np.float64))


def test_all_ones_and_row_sums():
    M, N, K = 19, 23, 111
    ops = si.tn_operands("bf16", M, N, K, dist="ones", seed=0)
    got = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert np.all(got == K)
    ops = si.tn_operands("f16", M, N, K, dist="normal", seed=3, dist_b="ones")
    got = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    rows = ops["A"].to(torch.float64).numpy().sum(axis=1)
    np.testing.assert_allclose(got, np.repeat(rows[:, None], N, axis=1), rtol=1e-13, atol=1e-13)
    fo = si.f32_operands(M, N, K, seed=4, dist_b="ones")
    got32 = oracle.gemm_f32(M, N, K, fo["A"].numpy(), K, fo["B"].numpy(), N)
    rows32 = fo["A"].double().numpy().sum(axis=1)
    np.testing.assert_allclose(got32, np.repeat(rows32[:, None], N, axis=1), rtol=1e-13, atol=1e-13)


def test_empty_shapes():
    a = np.zeros(8, np.uint16)
    assert oracle.gemm_tn("f16", 0, 3, 2, a, 2, a, 2).shape == (0, 3)
    got = oracle.gemm_tn("f16", 2, 2, 0, a, 1, a, 1)
    assert got.shape == (2, 2) and np.all(got == 0)  # empty sum
    got = oracle.gemm_f32(2, 3, 0, np.zeros(2, np.float32), 1, np.zeros(3, np.float32), 3)
    assert np.all(got == 0)
