"""The seeded input recipe (synthetic_inputs.py), checked on the CPU: the same
seed gives the same operands, the distributions are the named ones, FP8
operands are quantised per tensor with scale = amax / 448, padding columns
past K hold NaN codes, and sample positions stay inside C and include its
corners and edges.  Every parity test and the benchmark draw from here, so a
drift in this module would change what all of them compare."""
import math

import numpy as np
import pytest
import torch

import synthetic_inputs as si


@pytest.mark.parametrize("kind", ["f16", "bf16", "e4m3"])
def test_same_seed_same_operands(kind):
    a = si.tn_operands(kind, 37, 29, 53, dist="normal", seed=7)
    b = si.tn_operands(kind, 37, 29, 53, dist="normal", seed=7)
    c = si.tn_operands(kind, 37, 29, 53, dist="normal", seed=8)
    for key in ("A", "B"):
        assert np.array_equal(si.codes(a[key]), si.codes(b[key]))
    assert not np.array_equal(si.codes(a["A"]), si.codes(c["A"]))
    assert (a["scale_a"], a["scale_b"]) == (b["scale_a"], b["scale_b"])


def test_a_is_drawn_before_b_from_one_generator():
    """A and B come from one generator, A first: B's values are the ones that
    follow A's M x K draws in the stream."""
    M, N, K = 5, 4, 6
    ops = si.tn_operands("f16", M, N, K, dist="normal", seed=3)
    gen = torch.Generator("cpu").manual_seed(3)
    xa = torch.randn((M, K), generator=gen)
    xb = torch.randn((N, K), generator=gen)
    assert torch.equal(ops["A"], xa.to(torch.float16))
    assert torch.equal(ops["B"], xb.to(torch.float16))


def test_distributions():
    pm1 = si.tn_operands("bf16", 64, 48, 80, dist="pm1", seed=0)
    vals = set(pm1["A"].float().unique().tolist()) | set(pm1["B"].float().unique().tolist())
    assert vals == {-1.0, 1.0}
    ones = si.tn_operands("f16", 8, 8, 8, dist="ones")
    assert torch.all(ones["A"].float() == 1) and torch.all(ones["B"].float() == 1)
    ident = si.tn_operands("bf16", 16, 16, 16, dist="normal", dist_b="identity", seed=1)
    assert torch.equal(ident["B"].float(), torch.eye(16))
    uni = si.f32_operands(64, 64, 64, dist="uniform", seed=1)
    assert uni["A"].min() >= -1.0 and uni["A"].max() < 1.0
    normal = si.tn_operands("f16", 256, 256, 256, dist="normal", seed=2, sigma=0.1)
    std = float(normal["A"].float().std())
    assert 0.095 < std < 0.105


def test_fp8_per_tensor_quantisation():
    """scale = amax / 448 per tensor; the largest magnitude maps to 448 exactly
    and every code is finite."""
    M, N, K = 96, 64, 128
    gen = torch.Generator("cpu").manual_seed(4)
    xa = torch.randn((M, K), generator=gen)
    xb = torch.randn((N, K), generator=gen)
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=4)
    assert ops["scale_a"] == pytest.approx(float(xa.abs().max()) / 448.0, rel=1e-7)
    assert ops["scale_b"] == pytest.approx(float(xb.abs().max()) / 448.0, rel=1e-7)
    for key in ("A", "B"):
        q = ops[key].float()
        assert torch.isfinite(q).all()
        assert float(q.abs().max()) == 448.0
    # exact-valued operands keep scale 1
    pm1 = si.tn_operands("e4m3", 8, 8, 32, dist="pm1", seed=0)
    assert (pm1["scale_a"], pm1["scale_b"]) == (1.0, 1.0)


@pytest.mark.parametrize("kind,nan_code", [("f16", 0x7E00), ("bf16", 0x7FC0), ("e4m3", 0x7F)])
def test_padding_past_k_holds_nan_codes(kind, nan_code):
    M, N, K = 6, 5, 10
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=1, lda=16, ldb=24)
    assert tuple(ops["A"].shape) == (M, 16) and tuple(ops["B"].shape) == (N, 24)
    a, b = si.codes(ops["A"]), si.codes(ops["B"])
    assert np.all(a[:, K:] == nan_code) and np.all(b[:, K:] == nan_code)
    tight = si.tn_operands(kind, M, N, K, dist="normal", seed=1)
    assert np.array_equal(a[:, :K], si.codes(tight["A"]))
    assert np.array_equal(b[:, :K], si.codes(tight["B"]))


def test_f32_padding_and_layout():
    ops = si.f32_operands(4, 6, 5, dist="uniform", seed=1, lda=8, ldb=9)
    assert tuple(ops["A"].shape) == (4, 8) and tuple(ops["B"].shape) == (5, 9)
    assert torch.isnan(ops["A"][:, 5:]).all() and torch.isnan(ops["B"][:, 6:]).all()
    assert not torch.isnan(ops["A"][:, :5]).any() and not torch.isnan(ops["B"][:, :6]).any()


def test_sample_positions():
    M, N = 37, 91
    ms, ns = si.sample_positions(M, N, 500, seed=5)
    assert len(ms) == len(ns) == 507
    assert ms.min() >= 0 and ms.max() < M and ns.min() >= 0 and ns.max() < N
    pairs = set(zip(ms.tolist(), ns.tolist()))
    for corner in [(0, 0), (M - 1, 0), (0, N - 1), (M - 1, N - 1)]:
        assert corner in pairs
    ms2, ns2 = si.sample_positions(M, N, 500, seed=5)
    assert np.array_equal(ms, ms2) and np.array_equal(ns, ns2)
    ms3, _ = si.sample_positions(M, N, 500, seed=5, edges=False)
    assert len(ms3) == 500 and np.array_equal(ms3, ms[:500])
    # roughly uniform: every row index appears about 500 / 37 times
    counts = np.bincount(ms3, minlength=M)
    assert counts.min() > 0 and counts.max() < 4 * math.ceil(500 / M)


def test_codes_views_storage():
    t = torch.tensor([[1.0, -2.0]], dtype=torch.bfloat16)
    assert si.codes(t).tolist() == [[0x3F80, 0xC000]]
    t8 = torch.tensor([[448.0, -1.0]]).to(torch.float8_e4m3fn)
    assert si.codes(t8).tolist() == [[0x7E, 0xB8]]
