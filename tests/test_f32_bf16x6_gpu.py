"""GPU parity of gemm_f32_bf16x6 (FP32 GEMM on the tensor cores through exact
three-way BF16 splits) against the CPU oracle.

Bounds.  Each FP32 value is split exactly, x = x0 + x1 + x2, and C is the sum
of the six largest piece products, formed exactly and summed in the tensor
cores' FP32 accumulator.  The three products left out are below 2^-25 |a b|;
what remains is FP32 accumulation.  The tests hold every element to

    |C - exact| <= 2^-20 * sqrt(1 + K / 256) * sum_k |a(m,k)| |b(k,n)|,

which FP32 accumulation meets with room to spare (measured on GB300: at most
about 2^-21 of sum |a||b| up to K = 65536), while a lost or mispaired piece
product costs 2^-18 (a1 b1) to 2^-9 (a1 b0, a0 b1) relative and fails it at
small K.  Inputs whose products and sums are exact in FP32 (small integers, +-1,
permutation operands) must come out exact.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import contract_tol

pytestmark = pytest.mark.gpu


def stream():
    return torch.cuda.current_stream().cuda_stream


class Workspace:
    """Registers a device workspace of `nbytes` for the test and removes it after."""

    def __init__(self, nbytes):
        self.buf = torch.empty(max(nbytes, 256), dtype=torch.uint8, device="cuda")
        self.nbytes = nbytes

    def __enter__(self):
        ptr = self.buf.data_ptr() if self.nbytes else None
        assert capi.gemm_set_workspace(ptr, self.nbytes) == 0
        return self

    def __exit__(self, *exc):
        torch.cuda.synchronize()
        capi.gemm_set_workspace(None, 0)


def run_x6(ops, M, N, K, ldc=None, c_init=None, extra=0, expect=capi.GEMM_OK, ws=None):
    ldc = N if ldc is None else ldc
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C = (torch.full((max(M, 1), ldc), float("nan"), device="cuda") if c_init is None
         else c_init.cuda())
    nbytes = capi.gemm_f32_bf16x6_workspace_bytes(M, N, K) + extra if ws is None else ws
    with Workspace(nbytes):
        st = capi.gemm_f32_bf16x6(M, N, K, A.data_ptr(), ops["lda"], B.data_ptr(), ops["ldb"],
                                  C.data_ptr(), ldc, stream())
        assert st == expect, capi.status_text(st)
        torch.cuda.synchronize()
    return C.cpu()


def x6_bound(a, b, K):
    return 2.0 ** -20 * np.sqrt(1.0 + K / 256.0) * (np.abs(a) @ np.abs(b))


def check_full(ops, M, N, K, C):
    got = C[:M, :N].double().numpy()
    exact = oracle.gemm_f32(M, N, K, ops["A"].numpy(), ops["lda"], ops["B"].numpy(), ops["ldb"])
    a, b = ops["A"][:, :K].double().numpy(), ops["B"][:, :N].double().numpy()
    err = np.abs(got - exact)
    assert err.max() <= contract_tol("f32", K, float(np.abs(a).max()), float(np.abs(b).max()))
    assert np.all(err <= x6_bound(a, b, K)), float((err / x6_bound(a, b, K)).max())


@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 3, 7), (64, 64, 1), (64, 64, 2),
                                   (128, 128, 16), (300, 260, 129), (513, 1030, 77),
                                   (129, 4, 1000), (4, 129, 1000), (256, 512, 4096)])
@pytest.mark.parametrize("dist", ["uniform", "normal"])
def test_random_full(shape, dist):
    M, N, K = shape
    ops = si.f32_operands(M, N, K, dist=dist, seed=sum(shape) + len(dist))
    check_full(ops, M, N, K, run_x6(ops, M, N, K))


def test_unaligned_and_padded_ld():
    """lda = K + 1 takes the split's scalar loads; C's padding stays untouched."""
    M, N, K = 257, 130, 70
    ops = si.f32_operands(M, N, K, dist="uniform", seed=3, lda=K + 1, ldb=N + 3)
    C = run_x6(ops, M, N, K, ldc=N + 5)
    check_full(ops, M, N, K, C)
    assert torch.all(torch.isnan(C[:M, N:])), "C padding was written"


def test_wide_exponents():
    """Values spread over 2^-40 .. 2^40: the splits stay exact, so the relative
    bound holds at every scale."""
    M, N, K = 96, 80, 48
    gen = torch.Generator("cpu").manual_seed(11)
    a = torch.rand((M, K), generator=gen) * 2 - 1
    b = torch.rand((K, N), generator=gen) * 2 - 1
    a *= torch.exp2(torch.randint(-40, 41, (M, K), generator=gen).float())
    b *= torch.exp2(torch.randint(-40, 41, (K, N), generator=gen).float())
    ops = {"A": a.contiguous(), "B": b.contiguous(), "lda": K, "ldb": N}
    check_full(ops, M, N, K, run_x6(ops, M, N, K))


def _perm(n, seed):
    gen = torch.Generator("cpu").manual_seed(seed)
    p = torch.randperm(n, generator=gen)
    P = torch.zeros((n, n))
    P[torch.arange(n), p] = 1.0
    return P, p


@pytest.mark.parametrize("M,n", [(300, 257), (1024, 1024)])
def test_right_permutation_exact(M, n):
    """C = A P with P a permutation (not symmetric): every element of C is one
    element of A, exactly, so a wrong layout of B's split shows."""
    gen = torch.Generator("cpu").manual_seed(M)
    A = torch.randn((M, n), generator=gen)
    P, p = _perm(n, M + 1)
    ops = {"A": A, "B": P, "lda": n, "ldb": n}
    C = run_x6(ops, M, n, n)
    expect = torch.empty_like(A)
    expect[:, p] = A          # (A P)[m, p[i]] = A[m, i]
    assert torch.equal(C[:M, :n], expect)


@pytest.mark.parametrize("n,N", [(257, 300), (1024, 1024)])
def test_left_permutation_exact(n, N):
    """C = P B: every row of C is a row of B, exactly (A's split layout)."""
    gen = torch.Generator("cpu").manual_seed(N)
    B = torch.randn((n, N), generator=gen)
    P, p = _perm(n, N + 1)
    ops = {"A": P, "B": B, "lda": n, "ldb": N}
    C = run_x6(ops, n, N, n)
    assert torch.equal(C[:n, :N], B[p])   # (P B)[i] = B[p[i]]


def test_identity_2048_exact():
    n = 2048
    ops = si.f32_operands(n, n, n, dist="uniform", seed=1, dist_b="identity")
    assert torch.equal(run_x6(ops, n, n, n), ops["A"])


def test_pm1_long_k_exact():
    """+-1 entries, K = 16384: integer partial sums below 2^24, exact."""
    M, N, K = 130, 140, 16384
    ops = si.f32_operands(M, N, K, dist="pm1", seed=5)
    C = run_x6(ops, M, N, K)[:M, :N].double().numpy()
    exact = oracle.gemm_f32(M, N, K, ops["A"].numpy(), K, ops["B"].numpy(), N)
    assert np.array_equal(C, exact)


def test_small_integers_exact():
    """Integers in [-64, 64] with K = 1000: products and sums exact in FP32."""
    M, N, K = 200, 190, 1000
    gen = torch.Generator("cpu").manual_seed(21)
    A = torch.randint(-64, 65, (M, K), generator=gen).float()
    B = torch.randint(-64, 65, (K, N), generator=gen).float()
    ops = {"A": A, "B": B, "lda": K, "ldb": N}
    C = run_x6(ops, M, N, K)[:M, :N].double().numpy()
    exact = oracle.gemm_f32(M, N, K, A.numpy(), K, B.numpy(), N)
    assert np.array_equal(C, exact)


def test_split_k_with_extra_workspace():
    """Few output tiles and long K: with room beyond the splits the GEMM splits
    K (as the TN calls do), without it it runs unsplit; both meet the bound."""
    M, N, K = 128, 256, 8192
    ops = si.f32_operands(M, N, K, dist="normal", seed=9)
    extra = capi.gemm_workspace_bytes(N, M, 6 * K)
    split = run_x6(ops, M, N, K, extra=extra)
    plain = run_x6(ops, M, N, K, extra=0)
    check_full(ops, M, N, K, split)
    check_full(ops, M, N, K, plain)


def test_cuda_core_fallback_path():
    """Option "path" = 1 runs the split operands through the CUDA-core TN kernel
    (BF16 in, FP32 out): same bound."""
    M, N, K = 200, 150, 300
    ops = si.f32_operands(M, N, K, dist="uniform", seed=13)
    try:
        assert capi.gemm_set_option("path", 1) == 0
        C = run_x6(ops, M, N, K)
    finally:
        capi.gemm_set_option("path", 0)
    check_full(ops, M, N, K, C)


def test_4096_uniform_sampled():
    """The bench workload, FP32 4096^3 U[-1,1] (seed 1): 4096 samples + edges."""
    n = 4096
    ops = si.f32_operands(n, n, n, dist="uniform", seed=1)
    C = run_x6(ops, n, n, n)
    ms, ns = si.sample_positions(n, n, 4096, seed=1)
    exact = oracle.gemm_f32_sampled(n, ops["A"].numpy(), n, ops["B"].numpy(), n, ms, ns)
    got = C[torch.from_numpy(ms), torch.from_numpy(ns)].double().numpy()
    err = np.abs(got - exact)
    assert err.max() <= contract_tol("f32", n, 1.0, 1.0)
    a = ops["A"][torch.from_numpy(ms)].double().numpy()
    b = ops["B"][:, torch.from_numpy(ns)].double().numpy().T
    bound = 2.0 ** -20 * np.sqrt(1.0 + n / 256.0) * np.sum(np.abs(a) * np.abs(b), axis=1)
    assert np.all(err <= bound)


def test_workspace_required():
    """Without a workspace, or one byte short of gemm_f32_bf16x6_workspace_bytes,
    the call fails with GEMM_ERR_WORKSPACE and writes nothing."""
    M, N, K = 64, 48, 100
    ops = si.f32_operands(M, N, K, seed=2)
    need = capi.gemm_f32_bf16x6_workspace_bytes(M, N, K)
    init = torch.full((M, N), 7.0)
    for nbytes in (0, need - 1):
        C = run_x6(ops, M, N, K, c_init=init, ws=nbytes, expect=capi.GEMM_ERR_WORKSPACE)
        assert torch.equal(C, init)
    check_full(ops, M, N, K, run_x6(ops, M, N, K, ws=need))


def test_k_zero_and_empty():
    M, N = 33, 17
    ops = si.f32_operands(M, N, 1, seed=0)
    C = run_x6(ops, M, N, 0, ws=0)
    assert torch.all(C[:M, :N] == 0)
    init = torch.full((M, N), 5.0)
    assert torch.equal(run_x6(ops, 0, N, 1, c_init=init, ws=0), init)
