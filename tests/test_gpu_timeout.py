"""Failure detection on the GPU without a fault: every wait in the GEMM
kernel is bounded.  The test hook makes the producer never fill one pipeline
stage, so the MMA warp's wait on it runs out; the kernel must record the
time-out in the workspace status word, free its tensor memory and return, and
the CUDA context must stay usable for a correct GEMM afterwards."""
import ctypes

import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import check_y, oracle_layer

pytestmark = pytest.mark.gpu

TIMEOUT_DEVICE = 7


def _stall(xq, xs, wq, ws, y, M, N, K, work, skip_unit, timeout_ns):
    L = fb.lib()
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.fp8bs_testhook_gemm_stall(
        ctypes.c_void_p(xq.data_ptr()), ctypes.c_void_p(xs.data_ptr()), ctypes.c_void_p(wq.data_ptr()),
        ctypes.c_void_p(ws.data_ptr()), ctypes.c_void_p(y.data_ptr()), M, N, K,
        ctypes.c_void_p(work.data_ptr()), work.numel(), skip_unit, timeout_ns, stream)


# 16-token tile (decode), and the wider tiles whose epilogue forms its scale
# products per warp with no barrier across the epilogue warps: after the
# time-out every epilogue warp must still run through its units and meet the
# exchange's barriers, and the CTA must still free its tensor memory.
@pytest.mark.parametrize("M,N,K,skip", [(8, 256, 512, 0), (8, 5120, 5120, 3), (33, 5120, 5120, 2),
                                        (128, 5120, 5120, 5), (512, 384, 512, 1)])
def test_bounded_wait_reports_timeout_and_context_survives(M, N, K, skip):
    # the skipped unit index is per CTA: every CTA must have more units than that
    sched = fb.gemm_schedule(M, N, K)
    assert sched["units"] // sched["ctas"] > skip
    x = synth.activations(M, K, seed=5)
    w = synth.weights(N, K, seed=6)
    xd, wd = x.cuda(), w.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(wd)
    xq, xs = fb.fp8_quant_act(xd)
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K))
    rc = _stall(xq, xs, wq, ws, y, M, N, K, work, skip, 100_000_000)   # 0.1 s limit
    assert rc == 0, fb.status_string(rc)
    code = fb.workspace_status(work)                                     # synchronises
    assert code != 0, "the stalled kernel did not report its time-out"
    L = fb.lib()
    c = ctypes.c_int(0)
    assert L.fp8bs_workspace_status(ctypes.c_void_p(work.data_ptr()), 1, ctypes.byref(c)) == TIMEOUT_DEVICE
    assert fb.workspace_status(work) == 0                                # cleared
    # the context is still usable: a normal call on a fresh workspace is correct
    ref = oracle_layer(x, w)
    y2 = fb.fp8_blockscaled_gemm(xq, xs, wq, ws)
    torch.cuda.synchronize()
    check_y(y2, ref["y"], ref["bound"], "after time-out")


def test_stall_hook_rejects_bad_arguments():
    """No skip unit, a zero or too-long limit: rejected on the host before
    anything is enqueued (real buffers of the stated sizes, so nothing could
    fault even if a check were missing)."""
    M, N, K = 8, 256, 512
    xq = torch.zeros((M, K), dtype=torch.uint8, device="cuda")
    xs = torch.ones((M, K // 128), dtype=torch.float32, device="cuda")
    wq = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    ws = torch.ones((N // 128, K // 128), dtype=torch.float32, device="cuda")
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K))
    for skip, limit in ((-1, 1000), (0, 0), (0, 20_000_000_000)):
        assert _stall(xq, xs, wq, ws, y, M, N, K, work, skip, limit) == 1
    torch.cuda.synchronize()
    assert not y.any() and not work.any(), "a rejected call must not launch"
