"""GPU parity of the tensor-core kernel with clusters of two CTA pairs that
share their P tiles through TMA multicast (option "cluster" = 4).

Each case is checked against the CPU oracle and, bit for bit, against the
pair kernel without tail splitting: the multicast kernel issues the same MMA
sequence per tile, so only the operand delivery differs."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import (assert_codes_equal, check_full, check_sampled, contract_tol, exact_codes,
                      maxabs_dequant, out_codes, run_tn)

pytestmark = pytest.mark.gpu
KINDS = ["f16", "bf16", "e4m3"]


@pytest.fixture(autouse=True)
def _reset():
    yield
    for name, value in (("cluster", 0), ("tile_q", 0), ("tail", 0), ("max_ctas", 0),
                        ("pair", -1), ("splits", 0)):
        capi.gemm_set_option(name, value)


def run_both(kind, ops, M, N, K, opts):
    """C from the multicast kernel and from the pair kernel (tail splitting
    off in both), with the extra options `opts`."""
    for name, value in opts.items():
        assert capi.gemm_set_option(name, value) == 0
    assert capi.gemm_set_option("tail", 1) == 0
    assert capi.gemm_set_option("pair", 1) == 0
    assert capi.gemm_set_option("cluster", 4) == 0
    c_mc = run_tn(kind, ops, M, N, K)
    assert capi.gemm_set_option("cluster", 2) == 0
    c_pair = run_tn(kind, ops, M, N, K)
    return c_mc, c_pair


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape,tile_q", [
    ((512, 512, 256), 256),      # 2 x 2 tiles: one cluster unit per P tile
    ((768, 512, 300), 256),      # 3 tile columns: the second pair's last tile is outside M
    ((1000, 700, 333), 192),     # ragged on every edge
    ((450, 300, 129), 128),
    ((200, 260, 64), 64),
])
def test_multicast_full(kind, shape, tile_q):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=M + K, sigma=0.5)
    c_mc, c_pair = run_both(kind, ops, M, N, K, {"tile_q": tile_q})
    check_full(kind, ops, M, N, K, c_mc)
    assert torch.equal(c_mc[:N, :M].contiguous().view(torch.int16),
                       c_pair[:N, :M].contiguous().view(torch.int16))


@pytest.mark.parametrize("kind", KINDS)
def test_multicast_pm1_bitexact_few_clusters(kind):
    """+-1 entries, bit-exact; two clusters only, so each loops over many
    cluster units (ring phases and accumulator buffers wrap many times)."""
    M, N, K = 1536, 1280, 520
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=21)
    c_mc, c_pair = run_both(kind, ops, M, N, K, {"max_ctas": 8})
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(c_mc, M, N), exact_codes(kind, exact))
    assert torch.equal(c_mc[:N, :M].contiguous().view(torch.int16),
                       c_pair[:N, :M].contiguous().view(torch.int16))


def test_multicast_fp8_f32_out():
    M, N, K = 1000, 700, 500
    ops = si.tn_operands("e4m3", M, N, K, dist="normal", seed=5, sigma=1.0)
    assert capi.gemm_set_option("tail", 1) == 0
    outs = []
    for cl in (4, 2):
        assert capi.gemm_set_option("cluster", cl) == 0
        A, B = ops["A"].cuda(), ops["B"].cuda()
        C = torch.full((N, M), float("nan"), device="cuda")
        st = capi.gemm_fp8_tn_f32(M, N, K, A.data_ptr(), K, B.data_ptr(), K, ops["scale_a"],
                                  ops["scale_b"], C.data_ptr(), M,
                                  torch.cuda.current_stream().cuda_stream)
        assert st == 0, capi.status_text(st)
        torch.cuda.synchronize()
        outs.append(C.cpu())
    assert torch.equal(outs[0], outs[1])
    ref = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K,
                         scale_a=ops["scale_a"], scale_b=ops["scale_b"])
    err = np.abs(outs[0].double().numpy().T - ref).max()
    ma, mb = maxabs_dequant(ops, "e4m3")
    assert err <= contract_tol("e4m3", K, ma, mb)


@pytest.mark.parametrize("kind,shape,tile_q", [("bf16", (4096, 4096, 4096), 192),
                                                ("f16", (8192, 8192, 2048), 256),
                                                ("e4m3", (4096, 4096, 8192), 192)])
def test_multicast_large_sampled(kind, shape, tile_q):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=6, sigma=0.1)
    c_mc, c_pair = run_both(kind, ops, M, N, K, {"tile_q": tile_q})
    check_sampled(kind, ops, M, N, K, c_mc, seed=6)
    assert torch.equal(c_mc.view(torch.int16), c_pair.view(torch.int16))
    assert capi.gemm_read_watchdog(0) == capi.GEMM_OK
