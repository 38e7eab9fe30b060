"""GPU parity of gemm_f32 (SIMT FFMA, all row-major) against the CPU oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import contract_tol

pytestmark = pytest.mark.gpu


def run_f32(ops, M, N, K, ldc=None, c_init=None):
    ldc = N if ldc is None else ldc
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C = (torch.full((max(M, 1), ldc), float("nan"), device="cuda") if c_init is None
         else c_init.cuda())
    st = capi.gemm_f32(M, N, K, A.data_ptr(), ops["lda"], B.data_ptr(), ops["ldb"],
                       C.data_ptr(), ldc, torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    torch.cuda.synchronize()
    return C.cpu()


def tight_f32(a, b, K):
    """FP32 FMA chain: |err| <= K * 2^-24 * sum |a||b| (plus slack factor 2)."""
    return 2.0 * K * 2.0 ** -24 * (np.abs(a) @ np.abs(b)) + 1e-30


@pytest.mark.parametrize("shape", [(1, 1, 1), (5, 3, 7), (128, 128, 8), (300, 260, 129),
                                   (513, 1030, 77), (129, 4, 1000)])
def test_random_full(shape):
    M, N, K = shape
    ops = si.f32_operands(M, N, K, dist="uniform", seed=sum(shape))
    C = run_f32(ops, M, N, K)[:M, :N].double().numpy()
    exact = oracle.gemm_f32(M, N, K, ops["A"].numpy(), K, ops["B"].numpy(), N)
    err = np.abs(C - exact)
    assert err.max() <= contract_tol("f32", K, 1.0, 1.0)
    a, b = ops["A"][:, :K].double().numpy(), ops["B"][:, :N].double().numpy()
    assert np.all(err <= tight_f32(a, b, K))


def test_unaligned_and_padded_ld():
    M, N, K = 257, 130, 70
    ops = si.f32_operands(M, N, K, dist="uniform", seed=3, lda=K + 1, ldb=N + 3)
    C = run_f32(ops, M, N, K, ldc=N + 5)
    exact = oracle.gemm_f32(M, N, K, ops["A"].numpy(), ops["lda"], ops["B"].numpy(), ops["ldb"])
    got = C[:M, :N].double().numpy()
    a, b = ops["A"][:, :K].double().numpy(), ops["B"][:, :N].double().numpy()
    assert np.all(np.abs(got - exact) <= tight_f32(a, b, K))
    assert torch.all(torch.isnan(C[:M, N:])), "C padding was written"


@pytest.mark.parametrize("shape", [(2304, 2300, 40), (2304, 2204, 19), (2048, 3580, 24),
                                   (2560, 3000, 33), (1000, 130, 300), (2304, 2304, 48),
                                   (2048, 3584, 16)])
def test_half_width_tail(shape):
    """On 152 SMs with two blocks each: 324 tiles run as 304 whole + 20 halved
    (with N = 2204 the right halves of the last tile column hold no columns at
    all); 448 tiles all whole (remainder 144); 480 as 304 whole + 176 halved;
    16 tiles all halved; the last two
    shapes are multiples of the tile and of the K slice, so they take the
    variant without bounds checks (whole and half tiles).  Every tail mode
    ("f32_tail" 0 = halves behind a dependent launch, 1 = whole tiles, 2 = halves
    in a plain second launch, 3 = halves for any last partial wave) must give
    bit-identical C, since each output is the same chain of FMAs in k order;
    C's padding columns stay untouched."""
    M, N, K = shape
    ops = si.f32_operands(M, N, K, dist="uniform", seed=M + K)
    outs = []
    try:
        for mode in (0, 1, 2, 3):
            assert capi.gemm_set_option("f32_tail", mode) == 0
            outs.append(run_f32(ops, M, N, K, ldc=N + 7))
    finally:
        capi.gemm_set_option("f32_tail", 0)
    C = outs[0]
    exact = oracle.gemm_f32(M, N, K, ops["A"].numpy(), K, ops["B"].numpy(), N)
    got = C[:M, :N].double().numpy()
    a, b = ops["A"][:, :K].double().numpy(), ops["B"][:, :N].double().numpy()
    assert np.all(np.abs(got - exact) <= tight_f32(a, b, K))
    assert torch.all(torch.isnan(C[:M, N:])), "C padding was written"
    for other in outs[1:]:
        assert torch.equal(other[:M, :N], C[:M, :N])
        assert torch.all(torch.isnan(other[:M, N:]))


@pytest.mark.parametrize("case", ["ragged_chunk", "odd_lda_unchecked", "a_offset"])
def test_copy_paths(case):
    """The copies into shared memory: B's 16-byte copies with a last chunk of
    N only partly inside (N = 130, ldb = 132: 8 of its 16 bytes are read, the
    rest zero-filled); A, which always moves in 4-byte copies, with an odd lda
    on a shape that takes the variant without bounds checks (M, N multiples of
    128, K of 16); and A starting 4 bytes past a 16-byte boundary."""
    if case == "ragged_chunk":
        M, N, K, lda, ldb, ldc = 257, 130, 70, 70, 132, 132
    elif case == "odd_lda_unchecked":
        M, N, K, lda, ldb, ldc = 256, 384, 64, 65, 384, 384
    else:
        M, N, K, lda, ldb, ldc = 300, 256, 48, 48, 256, 256
    ops = si.f32_operands(M, N, K, dist="uniform", seed=M + N + lda, lda=lda, ldb=ldb)
    if case == "a_offset":
        flat = torch.empty(M * lda + 1, dtype=torch.float32)
        flat[1:] = ops["A"].reshape(-1)
        A = flat.cuda()[1:]
        assert A.data_ptr() % 16 == 4
    else:
        A = ops["A"].cuda()
    B = ops["B"].cuda()
    C = torch.full((M, ldc), float("nan"), device="cuda")
    st = capi.gemm_f32(M, N, K, A.data_ptr(), lda, B.data_ptr(), ldb, C.data_ptr(), ldc,
                       torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    torch.cuda.synchronize()
    C = C.cpu()
    exact = oracle.gemm_f32(M, N, K, ops["A"].numpy(), lda, ops["B"].numpy(), ldb)
    got = C[:M, :N].double().numpy()
    a, b = ops["A"][:, :K].double().numpy(), ops["B"][:K, :N].double().numpy()
    assert np.all(np.abs(got - exact) <= tight_f32(a, b, K))
    if ldc > N:
        assert torch.all(torch.isnan(C[:M, N:])), "C padding was written"


def test_pm1_long_k_exact():
    """FP32 with +-1 entries and K = 65536: every partial sum is an integer below
    2^24, so each FMA chain is exact and C equals the oracle exactly."""
    M, N, K = 130, 140, 65536
    ops = si.f32_operands(M, N, K, dist="pm1", seed=5)
    C = run_f32(ops, M, N, K)[:M, :N].double().numpy()
    exact = oracle.gemm_f32(M, N, K, ops["A"].numpy(), K, ops["B"].numpy(), N)
    assert np.array_equal(C, exact)


def test_identity_4096_exact():
    """B = I  =>  C = A exactly ("Optimizing GEMM in HIP": the identity test)."""
    n = 4096
    ops = si.f32_operands(n, n, n, dist="uniform", seed=1, dist_b="identity")
    C = run_f32(ops, n, n, n)
    assert torch.equal(C, ops["A"])


def test_4096_uniform_sampled():
    """FP32 4096^3, U[-1,1] (seed 1): 4096 samples + edges within 2e-5*K."""
    n = 4096
    ops = si.f32_operands(n, n, n, dist="uniform", seed=1)
    C = run_f32(ops, n, n, n)
    ms, ns = si.sample_positions(n, n, 4096, seed=1)
    exact = oracle.gemm_f32_sampled(n, ops["A"].numpy(), n, ops["B"].numpy(), n, ms, ns)
    got = C[torch.from_numpy(ms), torch.from_numpy(ns)].double().numpy()
    err = np.abs(got - exact)
    assert err.max() <= contract_tol("f32", n, 1.0, 1.0)
    a = ops["A"][torch.from_numpy(ms)].double().numpy()
    b = ops["B"][:, torch.from_numpy(ns)].double().numpy().T
    assert np.all(err <= 2.0 * n * 2.0 ** -24 * np.sum(np.abs(a) * np.abs(b), axis=1))


def test_k_zero_and_empty():
    M, N = 33, 17
    ops = si.f32_operands(M, N, 1, seed=0)
    C = run_f32(ops, M, N, 0)
    assert torch.all(C[:M, :N] == 0)
    init = torch.full((M, N), 5.0)
    assert torch.equal(run_f32(ops, 0, N, 1, c_init=init), init)


@pytest.mark.parametrize("ktail", [1, 3, 7, 15])
@pytest.mark.parametrize("shape,lds", [((300, 260, 129), None), ((129, 4, 1000), None),
                                       ((257, 130, 70), (75, 133, 131)), ((1, 1, 17), None),
                                       ((2048, 3584, None), None)])
def test_k_tail_continues_the_chain(ktail, shape, lds):
    """K above 2^31 - 16 runs its last terms (at most 15) in a second kernel
    that continues each output's FMA chain from the value the tile kernel
    stored.  Option "f32_ktail" moves the last 1, 3, 7 or 15 terms there at
    any K: C must be bit-identical to the one-kernel result (the same chain of
    FMAs in k order), and match the oracle; with padded leading dimensions too,
    and with the tile kernel's unchecked variant (the last shape, K = 16 +
    ktail, so the tile kernel's 16 terms are one whole slice)."""
    M, N, K = shape
    if K is None:
        K = 16 + ktail
    lda, ldb, ldc = lds if lds else (K, N, N)
    ops = si.f32_operands(M, N, K, dist="uniform", seed=M + N + K, lda=lda, ldb=ldb)
    whole = run_f32(ops, M, N, K, ldc=ldc)
    assert capi.gemm_set_option("f32_ktail", ktail) == 0
    try:
        split = run_f32(ops, M, N, K, ldc=ldc)
    finally:
        assert capi.gemm_set_option("f32_ktail", 0) == 0
    assert torch.equal(whole[:M, :N], split[:M, :N])
    if ldc > N:
        assert torch.all(torch.isnan(split[:M, N:])), "C padding was written"
    exact = oracle.gemm_f32(M, N, K, ops["A"].numpy(), lda, ops["B"].numpy(), ldb)
    err = np.abs(split[:M, :N].double().numpy() - exact)
    a, b = ops["A"][:, :K].double().numpy(), ops["B"][:K, :N].double().numpy()
    assert np.all(err <= tight_f32(a, b, K))
