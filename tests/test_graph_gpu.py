"""Calls captured into a CUDA graph and replayed.

A captured call keeps what the host chose at capture time: its tensor maps,
its grid, and for split-K the counter set it counts in (the launch zeroes
the other set, and the last piece of every slice resets its own counter, so
the set is clean again for the next replay).  Programmatic dependent launch
becomes a programmatic edge between the captured kernels.  Each case refills
the captured input buffers between replays and checks every replay bit for
bit against the oracle."""
import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import assert_codes_equal, exact_codes, out_codes

pytestmark = pytest.mark.gpu


@pytest.fixture(params=["auto", "split3"])
def mode(request):
    """A registered workspace; "auto" splits K where the automatic rule does,
    "split3" forces three K pieces on every call."""
    ws = torch.empty(1 << 27, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    if request.param == "split3":
        assert capi.gemm_set_option("splits", 3) == 0
    yield request.param
    capi.gemm_set_option("splits", 0)
    assert capi.gemm_set_workspace(None, 0) == 0


def test_replayed_chain(mode):
    """Captured: C1 = A B, then C2 = C1' D (C1's storage as the next A).
    Replayed four times with new A, B, D each time."""
    M, N, K, N2 = 128, 384, 1024, 256
    A = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    D = torch.empty((N2, M), dtype=torch.bfloat16, device="cuda")
    C1 = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
    C2 = torch.empty((N2, N), dtype=torch.bfloat16, device="cuda")

    def calls(st):
        assert capi.gemm_bf16_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C1.data_ptr(), M,
                                 st) == 0
        assert capi.gemm_bf16_tn(N, N2, M, C1.data_ptr(), M, D.data_ptr(), M, C2.data_ptr(), N,
                                 st) == 0

    def fill(seed):
        ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=seed)
        d = si.tn_operands("bf16", N, N2, M, dist="pm1", seed=seed + 1)["B"]
        A.copy_(ops["A"])
        B.copy_(ops["B"])
        D.copy_(d)
        return ops["A"], ops["B"], d

    fill(60)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        calls(side.cuda_stream)          # first calls outside capture (attributes, addresses)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        calls(torch.cuda.current_stream().cuda_stream)
    for rep in range(4):
        a, b, d = fill(61 + 10 * rep)
        C1.fill_(float("nan"))
        C2.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        c1 = exact_codes("bf16", oracle.gemm_tn("bf16", M, N, K, si.codes(a), K, si.codes(b), K))
        c2 = exact_codes("bf16", oracle.gemm_tn("bf16", N, N2, M, c1.T.copy(), M, si.codes(d), M))
        assert_codes_equal(out_codes(C1.cpu(), M, N), c1)
        assert_codes_equal(out_codes(C2.cpu(), N, N2), c2)


def test_replay_after_eager_calls(mode):
    """Eager split calls between replays move the host's choice of counter
    set; the captured launch keeps its own and must stay exact."""
    M, N, K = 64, 2048, 2048
    A = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=70)
    A.copy_(ops["A"])
    B.copy_(ops["B"])

    def call(st, out):
        assert capi.gemm_bf16_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, out.data_ptr(), M,
                                 st) == 0

    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        call(side.cuda_stream, C)
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        call(torch.cuda.current_stream().cuda_stream, C)
    exact = exact_codes("bf16", oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K,
                                               si.codes(ops["B"]), K))
    other = torch.empty_like(C)
    st = torch.cuda.current_stream().cuda_stream
    for eager in (0, 1, 2, 3):
        for _ in range(eager):
            call(st, other)
        C.fill_(float("nan"))
        graph.replay()
        torch.cuda.synchronize()
        assert_codes_equal(out_codes(C.cpu(), M, N), exact)
        if eager:
            assert_codes_equal(out_codes(other.cpu(), M, N), exact)
