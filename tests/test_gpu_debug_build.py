"""The FP8BS_DEBUG build (libfp8bs_debug.so): every tensor-load coordinate,
ring stage, activation-cache slot, scale index, split-K slot and counter
index of the GEMM kernel is checked on the device, and a failed check is
recorded in the workspace status word (bit 0x20) instead of trapping.  It is
the stand-in for a device memory checker.

Clean runs: small shapes covering every schedule and both fused routes leave
the status word at zero and give bitwise the normal build's results.  A
planted coordinate one weight tile past the end (a test hook of the debug
build; such a load would only read zero-filled rows, so it is safe even if a
check missed it) must be caught, and the context must stay usable.
"""
import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import Ran, check_y, oracle_layer

pytestmark = pytest.mark.gpu

ERR_BOUNDS = 0x20

CASES = [  # (M, N, K): both fused routes, ragged N, every token-tile width, larger-M schedules
    (8, 256, 512), (1, 5120, 5120), (8, 5120, 5120), (13, 300, 1280), (33, 1000, 3072), (64, 1024, 2048),
    (100, 640, 1024), (256, 5120, 1024), (512, 384, 512),
]


@pytest.fixture(scope="module", autouse=True)
def debug_lib_built():
    from fp8_block_scaled_token_gb300 import build as fbuild
    fbuild.build(variants=("release", "debug"))
    with fb.debug_library() as L:
        assert L.fp8bs_testhook_debug_build() == 1
    assert fb.lib().fp8bs_testhook_debug_build() == 0


def _layer(x, wq, ws, N, work):
    # the fused entry point on its prologue-cast route where that fits (the
    # separate cast elsewhere), and the two-kernel path
    y = fb.fp8_blockscaled_gemm_fused(x, wq, ws, workspace=work, n=N, flags=fb.FLAG_PROLOGUE_CAST)
    xq, xs = fb.fp8_quant_act(x)
    y2 = fb.fp8_blockscaled_gemm(xq, xs, wq, ws, workspace=work, n=N)
    return y, y2


@pytest.mark.parametrize("M,N,K", CASES)
def test_debug_build_clean_and_bitwise_equal(M, N, K):
    x_cpu = synth.activations(M, K, seed=M + 1100, outlier_p=0.001)
    w_cpu = synth.weights(N, K, seed=M + 1101, outlier_p=0.01)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=True)
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K))
    y_rel, y2_rel = _layer(x, wq, ws, N, work)
    with fb.debug_library():
        work_d = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K))
        with Ran() as r:
            y_dbg, y2_dbg = _layer(x, wq, ws, N, work_d)
        assert sum(r.launched().values()) >= 3, "the debug build's kernels must be the ones that ran"
        assert fb.workspace_status(work_d) == 0, "a device-side check fired"
        if M <= 64:
            tok, lg, y3 = fb.fp8_blockscaled_gemm_fused_greedy(x, wq, ws, workspace=work_d, n=N)
            assert fb.workspace_status(work_d) == 0
    torch.cuda.synchronize()
    for a, b in ((y_rel, y_dbg), (y2_rel, y2_dbg), (y_rel, y2_rel)):
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    if M <= 64:
        assert torch.equal(y3.view(torch.int16), y_rel.view(torch.int16))
    ref = oracle_layer(x_cpu, w_cpu)
    check_y(y_dbg, ref["y"], ref["bound"], "debug build M=%d N=%d K=%d" % (M, N, K))


def test_debug_build_bf16_clean():
    M, N, K = 8, 1000, 1024
    x = synth.activations(M, K, seed=5).cuda()
    w = synth.weights(N, K, seed=6).to(torch.bfloat16).cuda()
    y = fb.bf16_gemm_ref(x, w)
    with fb.debug_library():
        work = fb.make_workspace(fb.bf16_gemm_ref_workspace_size(M, N, K))
        yd = fb.bf16_gemm_ref(x, w, workspace=work)
        assert fb.workspace_status(work) == 0
    torch.cuda.synchronize()
    assert torch.equal(y.view(torch.int16), yd.view(torch.int16))


def test_planted_bad_coordinate_is_caught():
    M, N, K = 8, 1024, 2048
    x = synth.activations(M, K, seed=7).cuda()
    wq, ws = fb.fp8_quant_weight_blocks(synth.weights(N, K, seed=8).cuda())
    xq, xs = fb.fp8_quant_act(x)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    need = fb.fp8_blockscaled_gemm_workspace_size(M, N, K)
    # the normal build refuses the hook: it has no checks to exercise
    assert fb.lib().fp8bs_testhook_debug_bad_tile(xq.data_ptr(), xs.data_ptr(), wq.data_ptr(), ws.data_ptr(),
                                                  y.data_ptr(), M, N, K, 0, need, 0, 100_000_000, None) == 1
    with fb.debug_library() as L:
        work = fb.make_workspace(need)
        rc = L.fp8bs_testhook_debug_bad_tile(xq.data_ptr(), xs.data_ptr(), wq.data_ptr(), ws.data_ptr(),
                                             y.data_ptr(), M, N, K, work.data_ptr(), need, 0, 100_000_000,
                                             torch.cuda.current_stream().cuda_stream)
        assert rc == 0, fb.status_string(rc)
        code = fb.workspace_status(work, clear=True)
        assert code & ERR_BOUNDS, "status word %#x: the bad coordinate was not caught" % code
        # the context is still usable: a correct layer on a fresh workspace
        work2 = fb.make_workspace(need)
        y_ok = fb.fp8_blockscaled_gemm(xq, xs, wq, ws, workspace=work2)
        assert fb.workspace_status(work2) == 0
    y_rel = fb.fp8_blockscaled_gemm(xq, xs, wq, ws)
    torch.cuda.synchronize()
    assert torch.equal(y_ok.view(torch.int16), y_rel.view(torch.int16))
