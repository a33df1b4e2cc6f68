"""The activation-scale layout follows the token count: token-major
[M][K/128] up to 16 tokens, K-block-major [K/128][M] above (where the GEMM's
epilogue forms its scale products per warp from one coalesced load).

fp8_quant_act must write the layout for its M (checked against the oracle's
token-major scales), the GEMM must read it (results within the layer's
tolerance at both sides of the boundary), and the fused entry point, which
casts into its workspace the same way, must equal the two-kernel path
bitwise above 16 tokens.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
import oracle
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import bits16, check_y, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [1, 2, 16, 17, 40, 65, 512])
def test_scale_layout_follows_token_count(M):
    K = 640
    x_cpu = synth.activations(M, K, seed=M + 70, outlier_p=0.001)
    xq, xs = fb.fp8_quant_act(x_cpu.cuda())
    kg = K // 128
    assert tuple(xs.shape) == ((M, kg) if M <= 16 else (kg, M))
    _, os_ = oracle.default().quant_act(bits16(x_cpu))
    flat = xs.cpu().numpy().reshape(-1)
    # element (m, g) at m*kg + g up to 16 tokens, at g*M + m above
    for m in range(M):
        for g in range(kg):
            idx = m * kg + g if M <= 16 else g * M + m
            assert flat[idx].view(np.uint32) == os_[m, g].view(np.uint32), (m, g)


@pytest.mark.parametrize("M,N,K", [(16, 1000, 2048), (17, 1000, 2048), (33, 384, 1280), (129, 640, 1024)])
def test_gemm_reads_the_layout_of_its_token_count(M, N, K):
    x_cpu = synth.activations(M, K, seed=M + 80, outlier_p=0.001)
    w_cpu = synth.weights(N, K, seed=M + 81, outlier_p=0.01)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=True)
    xq, xs = fb.fp8_quant_act(x)
    y = fb.fp8_blockscaled_gemm(xq, xs, wq, ws, n=N)
    y_f = fb.fp8_blockscaled_gemm_fused(x, wq, ws, n=N)
    torch.cuda.synchronize()
    ref = oracle_layer(x_cpu, w_cpu)
    check_y(y, ref["y"], ref["bound"], "M=%d N=%d K=%d" % (M, N, K))
    assert torch.equal(y.view(torch.int16), y_f.view(torch.int16))


def test_binding_checks_the_layout_shape():
    M, N, K = 17, 256, 512
    x = synth.activations(M, K, seed=3, device="cuda")
    wq, ws = fb.fp8_quant_weight_blocks(synth.weights(N, K, seed=4, device="cuda"))
    xq, xs = fb.fp8_quant_act(x)
    with pytest.raises(ValueError):
        fb.fp8_blockscaled_gemm(xq, xs.t().contiguous(), wq, ws)  # token-major shape at M = 17
