"""GPU parity of split-K (tiles cut along K when one wave of output tiles
cannot fill the GPU; partials in a caller-registered workspace, summed by the
last piece in piece order) against the CPU oracle, through the C ABI."""
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


@pytest.fixture
def workspace():
    ws = torch.empty(1 << 28, dtype=torch.uint8, device="cuda")  # 256 MiB
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    yield ws
    assert capi.gemm_set_workspace(None, 0) == 0
    capi.gemm_set_option("splits", 0)
    capi.gemm_set_option("pair", -1)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("shape", [(256, 512, 4096), (300, 200, 1000), (64, 2048, 2048)])
def test_auto_split_pm1_bitexact(kind, shape, workspace):
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=M + N)
    C = run_tn(kind, ops, M, N, K)
    exact = oracle.gemm_tn(kind, M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    assert_codes_equal(out_codes(C, M, N), exact_codes(kind, exact))


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("pair", [0, 1])
@pytest.mark.parametrize("splits", [2, 3, 7])
def test_forced_split_random(kind, pair, splits, workspace):
    M, N, K = 600, 330, 1000
    assert capi.gemm_set_option("pair", pair) == 0
    assert capi.gemm_set_option("splits", splits) == 0
    ops = si.tn_operands(kind, M, N, K, dist="normal", seed=splits, sigma=0.5)
    C = run_tn(kind, ops, M, N, K)
    check_full(kind, ops, M, N, K, C)


def test_split_is_deterministic(workspace):
    M, N, K = 512, 256, 8192
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=5)
    runs = [run_tn("bf16", ops, M, N, K) for _ in range(3)]
    for r in runs[1:]:
        assert torch.equal(r.view(torch.int16), runs[0].view(torch.int16))
    check_full("bf16", ops, M, N, K, runs[0])


def test_split_with_unaligned_rows_and_fp32_out(workspace):
    M, N, K = 301, 213, 1001
    assert capi.gemm_set_option("splits", 4) == 0
    ops = si.tn_operands("e4m3", M, N, K, dist="pm1", seed=9, lda=K, ldb=K + 2)
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C = torch.full((N, M + 3), float("nan"), device="cuda")
    st = capi.gemm_fp8_tn_f32(M, N, K, A.data_ptr(), K, B.data_ptr(), K + 2, 1.0, 1.0,
                              C.data_ptr(), M + 3, torch.cuda.current_stream().cuda_stream)
    assert st == 0, capi.status_text(st)
    exact = oracle.gemm_tn("e4m3", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K + 2)
    got = C.cpu()
    np.testing.assert_array_equal(got[:, :M].numpy().T, exact.astype(np.float32))
    assert torch.all(torch.isnan(got[:, M:]))


def test_small_workspace_does_not_split_and_stays_correct():
    ws = torch.empty(4096, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    try:
        M, N, K = 256, 512, 4096
        ops = si.tn_operands("f16", M, N, K, dist="pm1", seed=1)
        C = run_tn("f16", ops, M, N, K)
        exact = oracle.gemm_tn("f16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
        assert_codes_equal(out_codes(C, M, N), exact_codes("f16", exact))
    finally:
        capi.gemm_set_workspace(None, 0)


@pytest.mark.parametrize("shape", [(128, 8192, 8192), (64, 14336, 4096), (1024, 1024, 8192),
                                   (16, 8192, 8192), (100, 8192, 2048)])
def test_skinny_sampled(shape, workspace):
    M, N, K = shape
    ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=3, sigma=0.05)
    C = run_tn("bf16", ops, M, N, K)
    check_sampled("bf16", ops, M, N, K, C, seed=3)
    assert capi.gemm_read_watchdog(0) == capi.GEMM_OK


def test_workspace_api_checks():
    assert capi.gemm_set_workspace(None, 10) == capi.GEMM_ERR_INVALID_DIM
    ws = torch.empty(1024, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr() + 8, 512) == capi.GEMM_ERR_MISALIGNED
    assert capi.gemm_workspace_bytes(1024, 1024, 8192) > 0


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("pair", [0, 1])
def test_tail_k_pieces_full(kind, pair, workspace):
    """A partial last wave with a workspace: its tiles are cut into K pieces
    (few CTAs force several waves and a partial last one)."""
    M, N, K = 1100, 700, 1000
    for k, v in {"pair": pair, "max_ctas": 10, "tail_k": 3}.items():
        assert capi.gemm_set_option(k, v) == 0
    try:
        ops = si.tn_operands(kind, M, N, K, dist="normal", seed=pair + 11, sigma=0.5)
        C1 = run_tn(kind, ops, M, N, K)
        check_full(kind, ops, M, N, K, C1)
        C2 = run_tn(kind, ops, M, N, K)
        assert torch.equal(C1.view(torch.int16), C2.view(torch.int16)), "not deterministic"
    finally:
        capi.gemm_set_option("max_ctas", 0)
        capi.gemm_set_option("tail_k", 0)


@pytest.mark.parametrize("shape,tail_k", [((4096, 4096, 4096), 2), ((3072, 4096, 8192), 5)])
def test_tail_k_pieces_large_sampled(shape, tail_k, workspace):
    M, N, K = shape
    assert capi.gemm_set_option("tail_k", tail_k) == 0
    try:
        ops = si.tn_operands("bf16", M, N, K, dist="normal", seed=3, sigma=0.05)
        C = run_tn("bf16", ops, M, N, K)
        check_sampled("bf16", ops, M, N, K, C, seed=3)
    finally:
        capi.gemm_set_option("tail_k", 0)


def _issue(kind, shape, seed, opts, st):
    """Copies seeded +-1 operands to the GPU and issues one call (no sync)."""
    M, N, K = shape
    ops = si.tn_operands(kind, M, N, K, dist="pm1", seed=seed)
    A, B = ops["A"].cuda(), ops["B"].cuda()
    C = torch.full((N, M), float("nan"), dtype=torch.bfloat16, device="cuda")
    try:
        for k, v in opts.items():
            if k != "noalloc":
                assert capi.gemm_set_option(k, v) == 0
        if opts.get("noalloc"):
            rc = capi.gemm_bf16_tn_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), K,
                                           C.data_ptr(), M, 0, st)
        else:
            rc = capi.gemm_bf16_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C.data_ptr(), M, st)
        assert rc == 0, capi.status_text(rc)
    finally:
        for k in opts:
            if k != "noalloc":
                capi.gemm_set_option(k, 0)
    return ops, shape, (A, B, C)


def _check_exact(ops, shape, bufs, what=""):
    M, N, K = shape
    exact = oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K, si.codes(ops["B"]), K)
    got, want = out_codes(bufs[2].cpu(), M, N), exact_codes("bf16", exact)
    bad = int(np.count_nonzero((got != want) & ((got | want) != 0x8000)))
    assert bad == 0, "%s %s: %d of %d outputs differ" % (what, shape, bad, M * N)
    assert_codes_equal(got, want)


def test_counter_sets_back_to_back(workspace):
    """Split launches count in one of the workspace's two counter sets and
    zero the other for the next; the last piece of each slice resets its own
    counter.  A run of split calls of several shapes and kinds (automatic
    split-K, forced pieces, a K-split tail, the no-allocation array's own
    sets in between), issued back to back on one stream with no host sync,
    must each match the oracle bit for bit."""
    st = torch.cuda.current_stream().cuda_stream
    plan = [((256, 512, 4096), {}), ((600, 330, 1000), {"splits": 3}),
            ((300, 200, 1000), {}), ((2048, 2048, 2048), {"tail_k": 2}),
            ((64, 2048, 2048), {"noalloc": 1}), ((64, 2048, 2048), {}),
            ((600, 330, 1000), {"splits": 7}), ((1024, 1024, 8192), {})] * 2
    pending = [_issue("bf16", shape, 200 + i, opts, st) for i, (shape, opts) in enumerate(plan)]
    torch.cuda.synchronize()
    bad = []
    for i, item in enumerate(pending):
        try:
            _check_exact(*item, what="call %d %s" % (i, plan[i][1]))
        except AssertionError as exc:
            bad.append(str(exc).splitlines()[0])
    assert not bad, "; ".join(bad)


def test_registration_zeroes_the_counter_sets():
    """The counter sets at the start of a workspace are zeroed when it is
    registered: fill them with garbage, register, and split calls must still be
    exact (a counter that did not start at zero would let a piece combine the
    slice before the other pieces wrote their partial sums)."""
    ws = torch.empty(1 << 27, dtype=torch.uint8, device="cuda")
    ws[: 2 * 16384 * 4].fill_(0xFF)
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    try:
        st = torch.cuda.current_stream().cuda_stream
        pending = [_issue("bf16", (256, 512, 4096), 300 + i, {}, st) for i in range(3)]
        torch.cuda.synchronize()
        for item in pending:
            _check_exact(*item)
    finally:
        assert capi.gemm_set_workspace(None, 0) == 0


def test_more_counters_than_a_set_holds():
    """Forced pieces over more than 16384 32-row slices (4128 tiles of 128 x
    256) do not fit a fixed counter set: those counters go to the scratch and
    are zeroed on the stream instead.  Fixed-set split calls before and after
    stay exact."""
    ws = torch.empty(1200 << 20, dtype=torch.uint8, device="cuda")
    assert capi.gemm_set_workspace(ws.data_ptr(), ws.numel()) == 0
    try:
        st = torch.cuda.current_stream().cuda_stream
        before = _issue("bf16", (256, 512, 4096), 400, {}, st)
        M, N, K = 8192, 16512, 128
        ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=401)
        A, B = ops["A"].cuda(), ops["B"].cuda()
        C = torch.full((N, M), float("nan"), dtype=torch.bfloat16, device="cuda")
        assert capi.gemm_set_option("pair", 0) == 0
        assert capi.gemm_set_option("splits", 2) == 0
        try:
            rc = capi.gemm_bf16_tn(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C.data_ptr(), M, st)
            assert rc == 0, capi.status_text(rc)
        finally:
            capi.gemm_set_option("pair", -1)
            capi.gemm_set_option("splits", 0)
        after = _issue("bf16", (256, 512, 4096), 402, {}, st)
        torch.cuda.synchronize()
        check_sampled("bf16", ops, M, N, K, C.cpu(), seed=401)
        for item in (before, after):
            _check_exact(*item)
    finally:
        assert capi.gemm_set_workspace(None, 0) == 0


def test_automatic_k_split_tail(workspace, capfd):
    """96 pair tiles of 256 x 256 with 192 K stages each (BF16, K = 12288): one
    wave of 76 and a last wave of 20, which the automatic rule cuts into two K
    pieces per tile (20 x 2 units still fit in one wave).  With "tail" = 2 the
    last wave is narrowed instead; both exact."""
    import os
    M, N, K = 2048, 3072, 12288
    ops = si.tn_operands("bf16", M, N, K, dist="pm1", seed=81)
    exact = exact_codes("bf16", oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), K,
                                               si.codes(ops["B"]), K))
    lines = {}
    os.environ["GEMM_DEBUG"] = "1"
    try:
        for tail in (0, 2):
            assert capi.gemm_set_option("tail", tail) == 0
            capfd.readouterr()
            C = run_tn("bf16", ops, M, N, K)
            lines[tail] = [ln for ln in capfd.readouterr().err.splitlines()
                           if ln.startswith("[gemm] tn")][-1]
            assert_codes_equal(out_codes(C, M, N), exact)
    finally:
        del os.environ["GEMM_DEBUG"]
        capi.gemm_set_option("tail", 0)
    assert "ktail=1" in lines[0] and "tail=2" in lines[0], lines[0]
    assert "ktail=0" in lines[2] and "tail=2" in lines[2], lines[2]
