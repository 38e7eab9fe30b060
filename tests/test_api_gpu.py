"""C-ABI behaviour on the GPU: argument errors launch nothing, the watchdog
reports a wait that ran out and leaves the context usable, calls on a
non-default stream."""
import pytest
import torch

import synthetic_inputs as si
from dense_gemm_tcgen05_gb300 import capi, f32, f32_bf16x6, tn
from gpu_util import run_tn

pytestmark = pytest.mark.gpu


def test_device_is_supported():
    assert torch.cuda.get_device_capability() == (10, 3)


def test_errors_do_not_write():
    C = torch.full((16, 16), 7.0, dtype=torch.bfloat16, device="cuda")
    A = torch.zeros((16, 16), dtype=torch.bfloat16, device="cuda")
    s = torch.cuda.current_stream().cuda_stream
    assert capi.gemm_bf16_tn(16, 16, 16, A.data_ptr(), 8, A.data_ptr(), 16, C.data_ptr(), 16,
                             s) == capi.GEMM_ERR_INVALID_LD
    assert capi.gemm_bf16_tn(16, 16, 16, A.data_ptr() + 1, 16, A.data_ptr(), 16, C.data_ptr(),
                             16, s) == capi.GEMM_ERR_MISALIGNED
    torch.cuda.synchronize()
    assert torch.all(C == 7.0)


def test_watchdog_reports_timeout_and_context_survives():
    assert capi.gemm_read_watchdog(1) == capi.GEMM_OK
    assert capi.gemm_watchdog_selftest(2_000_000) == capi.GEMM_OK  # 2 ms limit
    assert capi.gemm_read_watchdog(0) == capi.GEMM_ERR_TIMEOUT
    assert capi.gemm_read_watchdog(1) == capi.GEMM_ERR_TIMEOUT
    assert capi.gemm_read_watchdog(0) == capi.GEMM_OK
    # the context is still usable
    M, N, K = 256, 256, 128
    ops = si.tn_operands("bf16", M, N, K, dist="ones", seed=0)
    C = run_tn("bf16", ops, M, N, K)
    assert torch.all(C.to(torch.float32) == K)
    assert capi.gemm_read_watchdog(0) == capi.GEMM_OK


def test_side_stream_and_tensor_api():
    M, N, K = 512, 384, 256
    ops = si.tn_operands("f16", M, N, K, dist="ones", seed=0)
    a, b = ops["A"].cuda(), ops["B"].cuda()
    s = torch.cuda.Stream()
    with torch.cuda.stream(s):
        out = tn(a, b)
    s.synchronize()
    assert out.shape == (N, M)
    assert torch.all(out.float() == K)


def test_tensor_helpers_reject_mismatched_out():
    """An `out` of the wrong shape or dtype is refused before any launch (the
    library writes the whole product, so a smaller `out` would overflow)."""
    a = torch.ones((64, 32), dtype=torch.float32, device="cuda")
    b = torch.ones((32, 48), dtype=torch.float32, device="cuda")
    for fn in (f32, f32_bf16x6):
        short = torch.full((63, 48), 7.0, device="cuda")
        with pytest.raises(ValueError):
            fn(a, b, out=short)
        with pytest.raises(ValueError):
            fn(a, b, out=torch.empty((64, 48), dtype=torch.float16, device="cuda"))
        assert torch.all(short == 7.0)
    ah = torch.ones((64, 32), dtype=torch.float16, device="cuda")
    bh = torch.ones((48, 32), dtype=torch.float16, device="cuda")
    with pytest.raises(ValueError):
        tn(ah, bh, out=torch.empty((47, 64), dtype=torch.float16, device="cuda"))
    out = f32(a, b, out=torch.empty((64, 48), device="cuda"))
    torch.cuda.synchronize()
    assert torch.all(out == 32.0)


def test_tuner_runs_and_restores_defaults():
    from dense_gemm_tcgen05_gb300 import tune

    res = tune.tune_shape("bf16:512x384x256", iters=2, quick=True)
    assert res["best"]["tflops"] > 0 and res["auto_tflops"] > 0
    assert len(res["configs"]) == 2 * 1 * 3 * 2
    # options are back to their defaults: a normal call still works
    M, N, K = 256, 256, 128
    ops = si.tn_operands("bf16", M, N, K, dist="ones", seed=0)
    C = run_tn("bf16", ops, M, N, K)
    assert torch.all(C.to(torch.float32) == K)
