"""The larger-M regime (65..512 tokens, chunked-prefill-like): token tiles of
up to 128, one CTA per (token tile, weight tile) pair or stream-K over the
pairs.  Same numeric contract and oracle as the decode path: codes and scales
bit-exact, Y within the layer's tolerance, bitwise reproducible."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
import oracle
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import bits16, check_y, oracle_layer

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M", [65, 100, 128, 129, 200, 256, 257, 300, 512])
def test_token_counts_match_oracle(M):
    N, K = 640, 1024
    x_cpu = synth.activations(M, K, seed=M + 700, outlier_p=0.001)
    w_cpu = synth.weights(N, K, seed=M + 701, outlier_p=0.01)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w)
    xq, xs = fb.fp8_quant_act(x)
    y = fb.fp8_blockscaled_gemm(xq, xs, wq, ws)
    yf = fb.fp8_blockscaled_gemm_fused(x, wq, ws)
    torch.cuda.synchronize()
    ref = oracle_layer(x_cpu, w_cpu)
    assert np.array_equal(xq.cpu().numpy(), ref["xq"])
    check_y(y, ref["y"], ref["bound"], "M=%d" % M)
    assert torch.equal(yf.view(torch.int16), y.view(torch.int16)), "fused differs from two-kernel"


@pytest.mark.parametrize("M,N", [(150, 300), (384, 129), (512, 1)])
def test_ragged_n(M, N):
    K = 640
    x_cpu = synth.activations(M, K, seed=M + 710)
    w_cpu = synth.weights(N, K, seed=M + 711)
    y = fb.fp8_blockscaled_gemm_fused(x_cpu.cuda(), *fb.fp8_quant_weight_blocks(w_cpu.cuda()))
    torch.cuda.synchronize()
    ref = oracle_layer(x_cpu, w_cpu)
    check_y(y, ref["y"], ref["bound"], "M=%d N=%d" % (M, N))


@pytest.mark.parametrize("M", [256, 512])
def test_square_layer(M):
    """The 5,120 x 5,120 layer in the benchmark's launch configuration (tiled
    weights, fused entry point, programmatic dependent launch); at M = 512
    the oracle checks 1,024 sampled columns."""
    x_cpu, w_cpu = synth.workload_inputs("square_decode", M=M)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    N, K = w.shape
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=True)
    y = fb.fp8_blockscaled_gemm_fused(x, wq, ws, flags=fb.FLAG_OVERLAP_PREV, n=N)
    torch.cuda.synchronize()
    cols = None if M == 256 else np.sort(np.random.default_rng(M).choice(N, 1024, replace=False))
    ref = oracle_layer(x_cpu, w_cpu, cols=cols)
    yv = y.cpu() if cols is None else y.cpu()[:, torch.from_numpy(cols)]
    check_y(yv, ref["y"], ref["bound"], "square M=%d" % M)


@pytest.mark.parametrize("M,N,K", [(512, 5120, 1024), (256, 7168, 1024), (300, 1024, 1024), (33, 640, 1024),
                                   (64, 5120, 512)])
def test_y_tma_store_matches_row_stores(M, N, K):
    """From 32 tokens up the plain layer writes Y through a shared-memory tile
    and one TMA store when Y is 16-byte aligned and N a multiple of 8, else
    row by row.  Both routes give the same bits; the TMA store writes no row
    past M (the 48- and 64-token tiles are taller than 33 tokens); the result
    matches the oracle.  Schedules: stream-K with whole and split tiles, one
    pair per CTA, every tile split, K split across every SM."""
    x_cpu = synth.activations(M, K, seed=M + 740, outlier_p=0.001)
    w_cpu = synth.weights(N, K, seed=M + 741, outlier_p=0.01)
    wq, ws = fb.fp8_quant_weight_blocks(w_cpu.cuda())
    xq, xs = fb.fp8_quant_act(x_cpu.cuda())
    guard = torch.full((M + 1, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_tma = guard[:M]                                   # 16-byte aligned: TMA store
    flat = torch.full((M * N + 1,), float("nan"), dtype=torch.bfloat16, device="cuda")
    y_rows = flat[1:].view(M, N)                        # 2-byte aligned only: row stores
    assert y_tma.data_ptr() % 16 == 0 and y_rows.data_ptr() % 16 == 2
    fb.fp8_blockscaled_gemm(xq, xs, wq, ws, y=y_tma)
    fb.fp8_blockscaled_gemm(xq, xs, wq, ws, y=y_rows)
    torch.cuda.synchronize()
    assert torch.isnan(guard[M]).all(), "a row past M was written"
    assert torch.isnan(flat[0]), "the element before Y was written"
    assert torch.equal(y_tma.view(torch.int16), y_rows.view(torch.int16)), "TMA store and row stores differ"
    ref = oracle_layer(x_cpu, w_cpu)
    check_y(y_tma, ref["y"], ref["bound"], "M=%d N=%d" % (M, N))


def test_deterministic_tiled_and_counters():
    M, N, K = 300, 1000, 2048
    x = synth.activations(M, K, seed=720, device="cuda")
    w = synth.weights(N, K, seed=721, device="cuda")
    wq, ws = fb.fp8_quant_weight_blocks(w)
    wt, _ = fb.fp8_quant_weight_blocks(w, tiled=True)
    xq, xs = fb.fp8_quant_act(x)
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K))
    first = fb.fp8_blockscaled_gemm(xq, xs, wq, ws, workspace=work)
    for _ in range(9):
        again = fb.fp8_blockscaled_gemm(xq, xs, wt, ws, workspace=work, n=N, flags=fb.FLAG_OVERLAP_PREV)
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
    torch.cuda.synchronize()
    assert not work[:1024].any(), "status word and greedy area must stay clear"


def test_bf16_gemm_large_m():
    M, N, K = 200, 384, 640
    x = synth.activations(M, K, seed=730)
    w = synth.weights(N, K, seed=731).to(torch.bfloat16)
    y = fb.bf16_gemm_ref(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    yr, bound = oracle.default().gemm_bf16(bits16(x), bits16(w))
    check_y(y, yr, bound, "bf16 M=%d" % M)


def test_limits():
    x = synth.activations(65, 512, seed=740, device="cuda")
    wq, ws = fb.fp8_quant_weight_blocks(synth.weights(256, 512, seed=741, device="cuda"))
    with pytest.raises(fb.Fp8bsError):
        fb.fp8_blockscaled_gemm_fused_greedy(x, wq, ws)          # greedy: at most 64 tokens
    x513 = synth.activations(513, 512, seed=742, device="cuda")
    with pytest.raises(fb.Fp8bsError):
        fb.fp8_blockscaled_gemm_fused(x513, wq, ws)              # at most 512 tokens


def test_pair_stream_k_every_pair_split():
    """152 (token tile, weight tile) pairs of two K blocks each: stream-K over
    the pairs gives every CTA two units, so every pair is shared by two CTAs
    and goes through the exchange."""
    M, N, K = 512, 128 * 38, 256
    x_cpu = synth.activations(M, K, seed=750, outlier_p=0.001)
    w_cpu = synth.weights(N, K, seed=751, outlier_p=0.01)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=True)
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K))
    y = fb.fp8_blockscaled_gemm_fused(x, wq, ws, workspace=work, n=N)
    torch.cuda.synchronize()
    ref = oracle_layer(x_cpu, w_cpu)
    check_y(y, ref["y"], ref["bound"], "pairs M=%d N=%d K=%d" % (M, N, K))
    again = fb.fp8_blockscaled_gemm_fused(x, wq, ws, workspace=work, n=N, flags=fb.FLAG_OVERLAP_PREV)
    torch.cuda.synchronize()
    assert torch.equal(again.view(torch.int16), y.view(torch.int16))
    ntiles, ttiles = N // 128, (M + 127) // 128
    assert not work[:1024 + ntiles * ttiles * 4].any(), "status, greedy area and counters back at zero"


def test_square_m512_bitwise_over_10_runs():
    x = synth.activations(512, 5120, seed=760, device="cuda")
    wq, ws = fb.fp8_quant_weight_blocks(synth.weights(5120, 5120, seed=761, device="cuda"), tiled=True)
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(512, 5120, 5120))
    first = fb.fp8_blockscaled_gemm_fused(x, wq, ws, workspace=work, n=5120)
    for _ in range(9):
        again = fb.fp8_blockscaled_gemm_fused(x, wq, ws, workspace=work, n=5120, flags=fb.FLAG_OVERLAP_PREV)
        assert torch.equal(again.view(torch.int16), first.view(torch.int16))
