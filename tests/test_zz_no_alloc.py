"""fp8_blockscaled_gemm_fused_noalloc: the fused layer for callers that cannot
allocate device memory (they cannot hand the GEMM a workspace, so the library
uses a scratch array of its own).  Called through the C ABI and checked
against the existing entry point, fp8_blockscaled_gemm_fused with a
caller-provided workspace, on two calls in a row (the second call finds the
scratch as the first left it).  Collected last on purpose; it also passes on
its own in a fresh process, where its first call does the per-device set-up.
"""
import ctypes

import numpy as np
import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import REL_TOL, ABS_TOL, oracle_layer, y_values

pytestmark = pytest.mark.gpu


def _noalloc(x, wq, ws, y, M, N, K, flags):
    f = fb.lib().fp8_blockscaled_gemm_fused_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint, ctypes.c_void_p]
    return f(x.data_ptr(), x.stride(0), wq.data_ptr(), ws.data_ptr(), y.data_ptr(), M, N, K, flags,
             torch.cuda.current_stream().cuda_stream)


@pytest.mark.parametrize("M,N,K,tiled", [(8, 5120, 5120, False), (3, 300, 1280, True), (64, 1000, 2048, False)])
def test_noalloc_matches_workspace_entry_point(M, N, K, tiled):
    x_cpu = synth.activations(M, K, seed=M + 300, outlier_p=0.001)
    w_cpu = synth.weights(N, K, seed=M + 301, outlier_p=0.01)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=tiled)
    flags = fb.FLAG_WEIGHTS_TILED if tiled else 0
    ref_y = fb.fp8_blockscaled_gemm_fused(x, wq, ws, n=N)
    bound = oracle_layer(x_cpu, w_cpu)["bound"]
    lim = REL_TOL * bound + ABS_TOL
    for call in range(2):
        y = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
        rc = _noalloc(x, wq, ws, y, M, N, K, flags)
        assert rc == 0, fb.status_string(rc)
        torch.cuda.synchronize()
        diff = np.abs(y_values(y) - y_values(ref_y))
        assert np.all(diff <= lim), "call %d: %d elements outside tolerance" % (call, int((diff > lim).sum()))


def test_noalloc_rejects_oversized_shapes():
    # 64 tokens x K = 2^20 needs 64 MiB of activation scratch, more than the
    # library holds: rejected on the host, nothing launched
    p = ctypes.c_void_p(0x10000)
    f = fb.lib().fp8_blockscaled_gemm_fused_noalloc
    f.restype = ctypes.c_int
    f.argtypes = [ctypes.c_void_p, ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                  ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_uint, ctypes.c_void_p]
    assert f(p, 1 << 20, p, p, p, 64, 128, 1 << 20, 0, None) == 2
