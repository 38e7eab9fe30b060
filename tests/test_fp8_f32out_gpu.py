"""GPU parity of gemm_fp8_tn_f32 (E4M3 inputs, per-tensor scales, FP32
output, as the FP8 page writes C) against the CPU oracle, through the C ABI,
including the page's transformer shapes."""
import math

import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi, tn

pytestmark = pytest.mark.gpu


@pytest.fixture(params=[0, 1], ids=["cta1", "pair"])
def pair_mode(request):
    assert capi.gemm_set_option("pair", request.param) == 0
    yield request.param
    capi.gemm_set_option("pair", -1)


def run(ops, M, N, K, ldc=None):
    ldc = M if ldc is None else ldc
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C = torch.full((max(N, 1), ldc), float("nan"), dtype=torch.float32, device="cuda")
    st = capi.gemm_fp8_tn_f32(M, N, K, A.data_ptr(), ops["lda"], B.data_ptr(), ops["ldb"],
                              ops["scale_a"], ops["scale_b"], C.data_ptr(), ldc,
                              torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    torch.cuda.synchronize()
    return C.cpu()


def tols(ops, K, exact, absdot):
    ma = float(ops["A"][:, :K].float().abs().max()) * ops["scale_a"]
    mb = float(ops["B"][:, :K].float().abs().max()) * ops["scale_b"]
    contract = 1e-2 * math.sqrt(K) * ma * mb
    mag = np.maximum(np.abs(exact), 2.0 ** -60)
    tight = np.exp2(np.floor(np.log2(mag)) - 23) + 2.0 * K * 2.0 ** -24 * absdot
    return contract, tight


@pytest.mark.parametrize("shape", [(256, 256, 256), (300, 200, 136), (513, 257, 1000)])
def test_pm1_bitexact(shape, pair_mode):
    M, N, K = shape
    ops = si.tn_operands("e4m3", M, N, K, dist="pm1", seed=7)
    C = run(ops, M, N, K)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    np.testing.assert_array_equal(C[:N, :M].numpy().T, exact.astype(np.float32))


@pytest.mark.parametrize("shape,ldc", [((600, 330, 200), None), ((257, 129, 65), 260),
                                       ((301, 213, 129), 303), ((130, 700, 256), 133)])
def test_random_full(shape, ldc, pair_mode):
    M, N, K = shape
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=sum(shape))
    C = run(ops, M, N, K, ldc=ldc)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K,
                           ops["scale_a"], ops["scale_b"])
    got = C[:N, :M].double().numpy().T
    a = ops["A"].double().numpy() * ops["scale_a"]
    b = ops["B"].double().numpy() * ops["scale_b"]
    contract, tight = tols(ops, K, exact, np.abs(a) @ np.abs(b).T)
    err = np.abs(got - exact)
    assert err.max() <= contract
    assert np.all(err <= tight)
    if ldc is not None and ldc > M:
        assert torch.all(torch.isnan(C[:N, M:ldc])), "C padding was written"


def test_unaligned_operand_rows():
    M, N, K = 301, 213, 129
    ops = si.tn_operands("e4m3", M, N, K, dist="pm1", seed=3, lda=K, ldb=K + 3)
    C = run(ops, M, N, K, ldc=M + 1)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K + 3)
    np.testing.assert_array_equal(C[:N, :M].numpy().T, exact.astype(np.float32))
    assert torch.all(torch.isnan(C[:N, M:]))


def test_tensor_api_float32_out():
    M, N, K = 384, 256, 512
    ops = si.tn_operands("e4m3", M, N, K, dist="ones", seed=0)
    out = tn(ops["A"].cuda(), ops["B"].cuda(), out_dtype=torch.float32)
    torch.cuda.synchronize()
    assert out.dtype == torch.float32 and torch.all(out == K)


# The FP8 page's transformer shapes ("FP8 GEMM Optimization on AMD RDNA 4", "Results").
PAGE_SHAPES = [(8192, 8192, 8192), (8192, 28672, 8192), (8192, 10240, 8192), (3072, 4096, 8192)]


@pytest.mark.parametrize("shape", PAGE_SHAPES)
def test_page_shapes_sampled(shape):
    M, N, K = shape
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=4)
    C = run(ops, M, N, K)
    ms, ns = si.sample_positions(M, N, 4096, seed=4)
    exact = oracle.gemm_tn_sampled("e4m3", K, si.codes(ops["A"]), K, si.codes(ops["B"]), K, ms, ns,
                                   ops["scale_a"], ops["scale_b"])
    got = C[torch.from_numpy(ns), torch.from_numpy(ms)].double().numpy()
    a = ops["A"].view(torch.uint8)[torch.from_numpy(ms)].view(torch.float8_e4m3fn).double().numpy()
    b = ops["B"].view(torch.uint8)[torch.from_numpy(ns)].view(torch.float8_e4m3fn).double().numpy()
    absdot = np.sum(np.abs(a * ops["scale_a"]) * np.abs(b * ops["scale_b"]), axis=1)
    contract, tight = tols(ops, K, exact, absdot)
    err = np.abs(got - exact)
    assert err.max() <= contract
    assert np.all(err <= tight)


@pytest.mark.parametrize("shape", [(8192, 28672, 8192), (8192, 10240, 8192)])
def test_page_fp16_shapes_sampled(shape):
    """The FP16 page's wide shapes with the FP16 entry point."""
    from gpu_util import check_sampled, run_tn

    M, N, K = shape
    ops = si.tn_operands("f16", M, N, K, dist="normal", seed=2, sigma=0.1)
    C = run_tn("f16", ops, M, N, K)
    check_sampled("f16", ops, M, N, K, C, seed=2)


@pytest.mark.parametrize("tile_q", [64, 128, 192, 256])
@pytest.mark.parametrize("M", [257, 450, 385])
def test_ragged_chunk_then_more_chunks(tile_q, M):
    """A ragged last chunk (M not a multiple of the 16-byte granule) followed by
    out-of-range chunks of the same tile, with TMA-stored C (ldc multiple of 4):
    the staging buffers must not be reused while a store still reads them."""
    N, K = 129, 65
    assert capi.gemm_set_option("tile_q", tile_q) == 0
    try:
        ops = si.tn_operands("e4m3", M, N, K, dist="pm1", seed=M + tile_q)
        C = run(ops, M, N, K, ldc=M + (4 - M % 4) % 4 + 4)
        exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
        np.testing.assert_array_equal(C[:N, :M].numpy().T, exact.astype(np.float32))
    finally:
        capi.gemm_set_option("tile_q", 0)
