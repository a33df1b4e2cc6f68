"""fp8_blockscaled_gemm_fused_noalloc: the fused layer for callers that cannot
allocate device memory (code running under a graph capture that must not
allocate, allocator-less embedded runtimes, hooks running while a framework
holds its memory pool).  They cannot hand the GEMM a workspace, so the library
uses a scratch array of its own.

Called through the C ABI and compared with the existing entry point,
fp8_blockscaled_gemm_fused with a caller-provided workspace: both run the same
kernels on the same schedule, so the results must be bitwise equal, on two
calls in a row (the second call finds the scratch as the first left it); the
result is also checked against the oracle.  Nothing here depends on test
order: run alone in a fresh process, its first call does the per-device
set-up of the scratch array.
"""
import ctypes

import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import check_y, oracle_layer

pytestmark = pytest.mark.gpu

SHAPE = 2  # FP8BS_ERR_UNSUPPORTED_SHAPE


def _noalloc(x, wq, ws, y, M, N, K, flags):
    f = fb.lib().fp8_blockscaled_gemm_fused_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint, ctypes.c_void_p]
    return f(x.data_ptr(), x.stride(0), wq.data_ptr(), ws.data_ptr(), y.data_ptr(), M, N, K, flags,
             torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("M,N,K,tiled", [(8, 5120, 5120, False), (3, 300, 1280, True), (64, 1000, 2048, False),
                                         (8, 256, 512, True)])
def test_noalloc_matches_workspace_entry_point(M, N, K, tiled):
    x_cpu = synth.activations(M, K, seed=M + 300, outlier_p=0.001)
    w_cpu = synth.weights(N, K, seed=M + 301, outlier_p=0.01)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=tiled)
    flags = fb.FLAG_WEIGHTS_TILED if tiled else 0
    ref_y = fb.fp8_blockscaled_gemm_fused(x, wq, ws, n=N)
    ref = oracle_layer(x_cpu, w_cpu)
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = _noalloc(x, wq, ws, y, M, N, K, flags)
        assert rc == 0, fb.status_string(rc)
        torch.cuda.synchronize()
        assert torch.equal(y.view(torch.int16), ref_y.view(torch.int16)), "call %d differs" % call
        check_y(y, ref["y"], ref["bound"], "noalloc call %d" % call)


def test_noalloc_rejects_oversized_shapes():
    # 64 tokens x K = 65,536: the activation area alone (4 MiB) plus the
    # split-K slots need more scratch than the library's 12 MiB; rejected on
    # the host before anything is enqueued.  Real buffers of the stated sizes.
    M, N, K = 64, 128, 65536
    assert fb.fp8_blockscaled_gemm_workspace_size(M, N, K) > 12 << 20
    x = torch.zeros((M, K), dtype=torch.bfloat16, device="cuda")
    wq = torch.zeros((N, K), dtype=torch.uint8, device="cuda")
    ws = torch.ones((1, K // 128), dtype=torch.float32, device="cuda")
    y = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(x, wq, ws, y, M, N, K, 0) == SHAPE
    # and more than 64 tokens (the fused layer without a workspace stops there)
    x65 = torch.zeros((65, 512), dtype=torch.bfloat16, device="cuda")
    wq2 = torch.zeros((N, 512), dtype=torch.uint8, device="cuda")
    ws2 = torch.ones((1, 4), dtype=torch.float32, device="cuda")
    y2 = torch.zeros((65, N), dtype=torch.bfloat16, device="cuda")
    assert _noalloc(x65, wq2, ws2, y2, 65, N, 512, 0) == SHAPE
    torch.cuda.synchronize()
    assert not y.any() and not y2.any(), "a rejected call must not write"
