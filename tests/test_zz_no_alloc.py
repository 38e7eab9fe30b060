"""gemm_bf16_tn_noalloc -- BF16 TN GEMM whose split-K scratch is a fixed array
inside the library, for callers that may not allocate device memory (code
whose memory belongs to a pooled allocator it must not bypass, plugins whose
host forbids device allocation, loops where an allocation would synchronise
the device).

Each case calls the entry point twice in a row through the C ABI.  Both
outputs are checked against the CPU oracle (bit for bit on +-1 inputs, whose
sums are exact integers; otherwise the contract tolerance
1e-2 * sqrt(K) * max|a| * max|b| plus the tighter per-element bound the other
parity tests use) and against gemm_bf16_tn's output within the contract
tolerance.  gemm_tn_plan, planning as the no-allocation call does, shows that
each case really splits K, so a call that silently ran unsplit, or a wrong
fix-up of the pieces, fails here.  This file sorts last so that a run stopping
at its first failure has run every other test first."""
import math

import pytest
import torch

import oracle
import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi
from gpu_util import check_full, check_sampled, out_codes, assert_codes_equal, exact_codes

pytestmark = pytest.mark.gpu

ALIGNED = capi.PLAN_ALIGNED


def _stream():
    return torch.cuda.current_stream().cuda_stream


def _planned_splits(M, N, K, flags, splits):
    """K pieces the no-allocation call takes for this shape (host planner)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert capi.gemm_set_option("splits", splits) == capi.GEMM_OK
    try:
        st, plan = capi.gemm_tn_plan("bf16", M, N, K, flags=flags | capi.PLAN_NOALLOC,
                                     workspace_bytes=capi.GEMM_NOALLOC_SCRATCH_BYTES, sms=sms)
    finally:
        assert capi.gemm_set_option("splits", 0) == capi.GEMM_OK
    assert st == capi.GEMM_OK and plan["status"] == capi.GEMM_OK
    return plan


# (M, N, K), splits argument, input distribution, ldb (None: tight), how the
# output is checked, and whether the plan must copy B into the array.
CASES = [
    ((256, 512, 4096), 0, "pm1", None, "exact", 0),
    ((300, 200, 1000), 3, "normal", None, "full", 0),
    ((64, 2048, 2048), 0, "normal", None, "full", 0),
    ((1024, 1024, 8192), 0, "normal", None, "sampled", 0),
    # B's rows not 16-byte aligned: its copy shares the array with the split,
    # which shrinks to fit beside it
    ((64, 2048, 4096), 0, "normal", 4097, "full", 1),
    # a forced split that does not fit beside the copy runs without it
    ((64, 2048, 4096), 8, "normal", 4097, "full", 0),
]


@pytest.mark.parametrize("shape,splits,dist,ldb,check,copy_b", CASES)
def test_noalloc_matches_oracle_and_gemm_bf16_tn_on_two_calls(shape, splits, dist, ldb, check,
                                                               copy_b):
    M, N, K = shape
    flags = ALIGNED
    if ldb is not None and (ldb * 2) % 16:
        flags &= ~(capi.PLAN_B_TMA | capi.PLAN_B_128)
    plan = _planned_splits(M, N, K, flags, splits)
    assert plan["splits"] >= 2, plan
    if splits:
        assert plan["splits"] == splits
    assert plan["copy_b"] == copy_b, plan

    assert capi.gemm_set_workspace(None, 0) == capi.GEMM_OK  # reference call: no split
    ops = si.tn_operands("bf16", M, N, K, dist=dist, seed=M + K, sigma=0.5, ldb=ldb)
    A, B = ops["A"].cuda(), ops["B"].cuda()
    ref = torch.empty((N, M), dtype=torch.bfloat16, device="cuda")
    st = capi.gemm_bf16_tn(M, N, K, A.data_ptr(), ops["lda"], B.data_ptr(), ops["ldb"],
                           ref.data_ptr(), M, _stream())
    assert st == capi.GEMM_OK, capi.status_text(st)
    torch.cuda.synchronize()
    ref_cpu = ref.cpu()
    ma = float(ops["A"][:, :K].float().abs().max())
    mb = float(ops["B"][:, :K].float().abs().max())
    tol = 1e-2 * math.sqrt(K) * ma * mb
    want = None
    if check == "exact":
        want = exact_codes("bf16", oracle.gemm_tn("bf16", M, N, K, si.codes(ops["A"]), ops["lda"],
                                                  si.codes(ops["B"]), ops["ldb"]))
    for call in range(2):
        out = torch.full((N, M), float("nan"), dtype=torch.bfloat16, device="cuda")
        st = capi.gemm_bf16_tn_noalloc(M, N, K, A.data_ptr(), ops["lda"], B.data_ptr(),
                                       ops["ldb"], out.data_ptr(), M, splits, _stream())
        assert st == capi.GEMM_OK, capi.status_text(st)
        torch.cuda.synchronize()
        got = out.cpu()
        if check == "exact":
            assert_codes_equal(out_codes(got, M, N), want)
        elif check == "full":
            check_full("bf16", ops, M, N, K, got)
        else:
            check_sampled("bf16", ops, M, N, K, got, seed=call)
        diff = (got.double() - ref_cpu.double()).abs()
        assert bool(torch.isfinite(diff).all()), "non-finite output"
        assert float(diff.max()) <= tol


def test_noalloc_rejects_a_split_beyond_the_scratch():
    """16 forced pieces of a 4096^2 output need far more than the array holds:
    the call must refuse before launching and leave C untouched."""
    M = N = K = 4096
    A = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    B = torch.zeros((N, K), dtype=torch.bfloat16, device="cuda")
    C = torch.full((N, M), 3.0, dtype=torch.bfloat16, device="cuda")
    st = capi.gemm_bf16_tn_noalloc(M, N, K, A.data_ptr(), K, B.data_ptr(), K, C.data_ptr(), M,
                                   16, _stream())
    assert st == capi.GEMM_ERR_SCRATCH
    assert "scratch" in capi.status_text(st)
    torch.cuda.synchronize()
    assert bool((C == 3.0).all())
