"""GPU parity of the quantisation kernels: bytes and scales bit-exact against
the oracle on the same seeded inputs."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
import oracle
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import bits16

pytestmark = pytest.mark.gpu


def _act_case(x_cpu, K=None):
    o = oracle.default()
    x = x_cpu.cuda()
    if K is not None and K != x.shape[1]:
        x = x[:, :K]
    xq, xs = fb.fp8_quant_act(x)
    torch.cuda.synchronize()
    oq, os_ = o.quant_act(bits16(x_cpu), K=K)
    assert np.array_equal(xq.cpu().numpy(), oq)
    # the library's scales are K-block-major above 16 tokens; the oracle's token-major
    M = x.shape[0]
    assert tuple(xs.shape) == fb.scales_shape(M, x.shape[1])
    xs_tm = xs.cpu().numpy() if M <= 16 else xs.cpu().numpy().T
    assert np.array_equal(xs_tm.view(np.uint32), os_.view(np.uint32))


@pytest.mark.parametrize("M,K,seed", [(8, 512, 0), (8, 5120, 1), (1, 5120, 1), (64, 5120, 5), (13, 17408, 3),
                                      (3, 128, 9), (16, 1280, 6), (17, 1280, 7), (300, 1024, 8)])
def test_quant_act_matches_oracle(M, K, seed):
    _act_case(synth.activations(M, K, seed=seed))


def test_quant_act_outliers_and_row_stride():
    x = synth.activations(8, 5120 + 256, seed=2, outlier_p=0.001)
    _act_case(x, K=5120)


def test_quant_act_edge_values():
    # zero groups, negative zeros, tiny values (fp32 subnormal quotients), ties
    M, K = 4, 512
    x = torch.zeros((M, K), dtype=torch.float32)
    x[1, :128] = -0.0
    x[1, 128:256] = torch.tensor([2.0 ** -130] * 64 + [-(2.0 ** -133)] * 64)
    x[2] = torch.linspace(-3.0, 3.0, K)
    x[3, ::2] = 448.0
    x[3, 1::2] = 1.0 / 1024.0
    _act_case(x.to(torch.bfloat16))


@pytest.mark.parametrize("N,K,dtype,seed", [(256, 512, torch.float32, 0), (5120, 5120, torch.float32, 1),
                                            (200, 384, torch.float32, 7), (300, 1024, torch.bfloat16, 8),
                                            (34816, 512, torch.float32, 2)])
def test_quant_weight_matches_oracle(N, K, dtype, seed):
    w_cpu = synth.weights(N, K, seed=seed, outlier_p=0.01)
    if dtype == torch.bfloat16:
        w_cpu = w_cpu.to(torch.bfloat16)
        ref_in = bits16(w_cpu)
    else:
        ref_in = w_cpu.numpy()
    wq, ws = fb.fp8_quant_weight_blocks(w_cpu.cuda())
    torch.cuda.synchronize()
    oq, os_ = oracle.default().quant_weight(ref_in)
    assert np.array_equal(wq.cpu().numpy(), oq)
    assert np.array_equal(ws.cpu().numpy().view(np.uint32), os_.view(np.uint32))


def test_quant_weight_zero_block_and_ties():
    w = torch.zeros((256, 256), dtype=torch.float32)
    w[0:128, 128:256] = torch.linspace(-448.0, 448.0, 128 * 128).reshape(128, 128)
    w[128:256, 0:128] = -0.0
    wq, ws = fb.fp8_quant_weight_blocks(w.cuda())
    torch.cuda.synchronize()
    oq, os_ = oracle.default().quant_weight(w.numpy())
    assert np.array_equal(wq.cpu().numpy(), oq)
    assert np.array_equal(ws.cpu().numpy(), os_)


def untile(wt, N, K, block_cols):
    """Tiled [tiles, 128, block_cols] -> row-major [N, K] (test-side reshaping only)."""
    kg = K // block_cols
    nt = wt.shape[0] // kg
    return wt.view(nt, kg, 128, block_cols).permute(0, 2, 1, 3).reshape(nt * 128, K)[:N]


@pytest.mark.parametrize("N,K,dtype", [(256, 512, torch.float32), (300, 1024, torch.float32),
                                       (200, 384, torch.bfloat16)])
def test_quant_weight_tiled_layout(N, K, dtype):
    w = synth.weights(N, K, seed=41, outlier_p=0.01).to(dtype).cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w)
    wt, wst = fb.fp8_quant_weight_blocks(w, tiled=True)
    torch.cuda.synchronize()
    assert torch.equal(untile(wt, N, K, 128), wq)
    assert torch.equal(ws, wst)
    nt = (N + 127) // 128
    pad = wt.view(nt, K // 128, 128, 128)[-1, :, N - (nt - 1) * 128:, :]
    assert not pad.any(), "rows past N must be zero in the tiled layout"


def test_bf16_pack_tiled_layout():
    N, K = 300, 640
    w = synth.weights(N, K, seed=42).to(torch.bfloat16).cuda()
    wt = fb.bf16_pack_weights_tiled(w)
    torch.cuda.synchronize()
    assert torch.equal(untile(wt, N, K, 64).view(torch.int16), w.view(torch.int16))
    nt = (N + 127) // 128
    pad = wt.view(nt, K // 64, 128, 64)[-1, :, N - (nt - 1) * 128:, :]
    assert not pad.view(torch.int16).any()
