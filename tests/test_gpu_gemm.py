"""GPU parity of the block-scaled GEMM (pre-quantised and fused) and of the
bf16 comparison GEMM against the oracle, plus determinism, guard bands and
host-reported errors."""
import numpy as np
import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
import oracle
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import (MODE_BF16, MODE_FP8, MODE_FUSED, RUNS_QUANT_ACT, RUNS_QUANT_WEIGHT, Ran, bits16,
                               check_y, oracle_layer, runs_gemm)

pytestmark = pytest.mark.gpu


def gpu_layer(x, w, fused=False, flags=0, workspace=None):
    wq, ws = fb.fp8_quant_weight_blocks(w)
    if fused:
        y = fb.fp8_blockscaled_gemm_fused(x, wq, ws, workspace=workspace, flags=flags)
    else:
        xq, xs = fb.fp8_quant_act(x)
        y = fb.fp8_blockscaled_gemm(xq, xs, wq, ws, workspace=workspace, flags=flags)
    torch.cuda.synchronize()
    return y


def _full_case(M, N, K, seed, fused=False, w_out=0.0, x_out=0.0):
    x = synth.activations(M, K, seed=seed, outlier_p=x_out)
    w = synth.weights(N, K, seed=seed + 1000, outlier_p=w_out)
    ref = oracle_layer(x, w)
    y = gpu_layer(x.cuda(), w.cuda(), fused=fused)
    check_y(y, ref["y"], ref["bound"], "M=%d N=%d K=%d fused=%s" % (M, N, K, fused))
    return y, ref


def test_tiny_workload():
    _full_case(8, 256, 512, 0)


@pytest.mark.parametrize("M", [1, 8])
def test_square_decode_layer(M):
    _full_case(M, 5120, 5120, 1)


@pytest.mark.parametrize("M", [1, 2, 3, 7, 16, 17, 31, 32, 33, 47, 48, 49, 63, 64])
def test_token_counts(M):
    _full_case(M, 384, 1024, 40 + M)


@pytest.mark.parametrize("M", [1, 5, 16, 29, 64])
def test_fused_matches_oracle(M):
    _full_case(M, 640, 2048, 60 + M, fused=True)


@pytest.mark.parametrize("M", [1, 5, 16])
def test_fused_prologue_cast_matches_oracle(M):
    """The prologue-cast route (FP8BS_FLAG_PROLOGUE_CAST) against the oracle."""
    assert fb.fused_route(M, 640, 2048, flags=fb.FLAG_PROLOGUE_CAST) == "prologue"
    x = synth.activations(M, 2048, seed=70 + M)
    w = synth.weights(640, 2048, seed=71 + M)
    ref = oracle_layer(x, w)
    y = gpu_layer(x.cuda(), w.cuda(), fused=True, flags=fb.FLAG_PROLOGUE_CAST)
    check_y(y, ref["y"], ref["bound"], "prologue cast M=%d" % M)


def test_ragged_n_and_outliers():
    _full_case(8, 300, 1280, 11, w_out=0.01, x_out=0.001)
    _full_case(5, 129, 384, 12)
    _full_case(8, 1, 128, 13)


def test_long_k():
    _full_case(8, 512, 17408, 3, w_out=0.01, x_out=0.001)


def test_closed_form_constant():
    # X == 1, W == 0.5: every code 448, y = 128(1+d)^2 -> bf16 128 exactly
    M, N, K = 2, 128, 256
    x = torch.ones((M, K), dtype=torch.bfloat16, device="cuda")
    w = torch.full((N, K), 0.5, dtype=torch.float32, device="cuda")
    y = gpu_layer(x, w)
    assert torch.all(y.float() == 128.0)


def test_fused_is_bitwise_the_two_kernel_path():
    # by default through the separate cast kernel; with the prologue-cast flag
    # the first three cast in the kernel prologue (at most 16 rows per CTA)
    for M, N, K, seed in ((1, 5120, 5120, 27), (2, 2048, 1024, 28), (16, 640, 2048, 29), (8, 5120, 5120, 1),
                          (33, 1000, 3072, 21), (64, 256, 512, 22), (64, 5120, 5120, 25), (16, 2048, 17408, 26)):
        x = synth.activations(M, K, seed=seed, outlier_p=0.001).cuda()
        w = synth.weights(N, K, seed=seed + 1).cuda()
        a = gpu_layer(x, w, fused=False)
        b = gpu_layer(x, w, fused=True)
        c = gpu_layer(x, w, fused=True, flags=fb.FLAG_PROLOGUE_CAST)
        assert torch.equal(a.view(torch.int16), b.view(torch.int16)), (M, N, K)
        assert torch.equal(a.view(torch.int16), c.view(torch.int16)), (M, N, K, "prologue flag")


def _tpad(M):
    return 16 if M <= 16 else 32 if M <= 32 else 48 if M <= 48 else 64


@pytest.mark.parametrize("prologue", [False, True])
@pytest.mark.parametrize("M,N,K,route", [(8, 256, 512, "prologue"), (1, 5120, 5120, "prologue"),
                                         (2, 2048, 1024, "prologue"), (16, 640, 2048, "prologue"),
                                         (8, 5120, 5120, "separate"), (33, 1000, 3072, "separate"),
                                         (64, 256, 512, "separate"), (16, 2048, 17408, "separate")])
def test_fused_route_runs_the_intended_kernels(M, N, K, route, prologue):
    """Looks inside the process: the fused entry point launches exactly the
    kernels of the route its query names -- one prologue-cast GEMM, or the
    cast kernel followed by the pre-quantised GEMM -- and nothing else.
    `route` is the route with FP8BS_FLAG_PROLOGUE_CAST; without it the route
    is always the separate cast."""
    flags = fb.FLAG_PROLOGUE_CAST if prologue else 0
    if not prologue:
        route = "separate"
    assert fb.fused_route(M, N, K, flags=flags) == route
    x = synth.activations(M, K, seed=M + 5).cuda()
    wq, ws = fb.fp8_quant_weight_blocks(synth.weights(N, K, seed=M + 6).cuda())
    torch.cuda.synchronize()
    with Ran() as r:
        fb.fp8_blockscaled_gemm_fused(x, wq, ws, flags=flags)
    if route == "prologue":
        assert r.launched() == {runs_gemm(MODE_FUSED, _tpad(M)): 1}
    else:
        assert r.launched() == {RUNS_QUANT_ACT: 1, runs_gemm(MODE_FP8, _tpad(M)): 1}


def test_entry_points_run_their_kernels():
    M, N, K = 8, 384, 1024
    x = synth.activations(M, K, seed=3).cuda()
    w = synth.weights(N, K, seed=4).cuda()
    with Ran() as r:
        wq, ws = fb.fp8_quant_weight_blocks(w)
    assert r.launched() == {RUNS_QUANT_WEIGHT: 1}
    with Ran() as r:
        xq, xs = fb.fp8_quant_act(x)
    assert r.launched() == {RUNS_QUANT_ACT: 1}
    with Ran() as r:
        fb.fp8_blockscaled_gemm(xq, xs, wq, ws)
    assert r.launched() == {runs_gemm(MODE_FP8, 16): 1}
    with Ran() as r:
        fb.bf16_gemm_ref(x, w.to(torch.bfloat16))
    assert r.launched() == {runs_gemm(MODE_BF16, 16): 1}
    with Ran() as r:
        fb.fp8_blockscaled_gemm(fb.fp8_quant_act(synth.activations(200, K, seed=5).cuda())[0],
                                fb.fp8_quant_act(synth.activations(200, K, seed=5).cuda())[1], wq, ws)
    assert r.count(runs_gemm(MODE_FP8, fb.gemm_schedule(200, N, K)["npad"])) == 1


def test_fused_row_stride():
    x_full = synth.activations(8, 1024 + 64, seed=23).cuda()
    x = x_full[:, :1024]
    w = synth.weights(384, 1024, seed=24).cuda()
    a = gpu_layer(x.contiguous(), w, fused=True)
    b = gpu_layer(x, w, fused=True)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


@pytest.mark.parametrize("fused", [False, True])
def test_bitwise_deterministic_over_10_runs(fused):
    M, N, K = 8, 5120, 5120
    x = synth.activations(M, K, seed=1).cuda()
    w = synth.weights(N, K, seed=1001).cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w)
    xq, xs = fb.fp8_quant_act(x)
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K))
    outs = []
    for _ in range(10):
        if fused:
            outs.append(fb.fp8_blockscaled_gemm_fused(x, wq, ws, workspace=work))
        else:
            outs.append(fb.fp8_blockscaled_gemm(xq, xs, wq, ws, workspace=work))
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert fb.workspace_status(work) == 0
    # the counters are back at zero after every call
    assert not work[1024:1024 + 4 * ((N + 127) // 128)].any()


def test_overlap_flag_same_result():
    M, N, K = 8, 5120, 5120
    x = synth.activations(M, K, seed=1).cuda()
    w = synth.weights(N, K, seed=1001).cuda()
    a = gpu_layer(x, w, fused=False, flags=0)
    b = gpu_layer(x, w, fused=False, flags=fb.FLAG_OVERLAP_PREV)
    c = gpu_layer(x, w, fused=True, flags=fb.FLAG_OVERLAP_PREV)
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))
    assert torch.equal(a.view(torch.int16), c.view(torch.int16))


def test_guard_bands_untouched():
    M, N, K = 8, 300, 1024
    x = synth.activations(M, K, seed=31).cuda()
    w = synth.weights(N, K, seed=32).cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w)
    xq, xs = fb.fp8_quant_act(x)
    pad = 4096
    sentinel = -12345
    buf = torch.full((M * N + 2 * pad,), sentinel, dtype=torch.int16, device="cuda")
    y = buf[pad:pad + M * N].view(torch.bfloat16).view(M, N)
    wsize = fb.fp8_blockscaled_gemm_workspace_size(M, N, K)
    wbuf = torch.zeros(wsize + 2 * 4096, dtype=torch.uint8, device="cuda")
    wbuf[:4096] = 0xA5
    wbuf[-4096:] = 0x5A
    work = wbuf[4096:4096 + wsize]
    fb.fp8_blockscaled_gemm(xq, xs, wq, ws, y=y, workspace=work)
    fb.fp8_blockscaled_gemm_fused(x, wq, ws, y=y, workspace=work)
    torch.cuda.synchronize()
    assert torch.all(buf[:pad] == sentinel) and torch.all(buf[-pad:] == sentinel)
    assert not torch.any(buf[pad:pad + M * N] == sentinel)
    assert torch.all(wbuf[:4096] == 0xA5) and torch.all(wbuf[-4096:] == 0x5A)


def test_host_errors_on_gpu():
    M, N, K = 8, 256, 512
    x = synth.activations(M, K, seed=0).cuda()
    w = synth.weights(N, K, seed=1).cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w)
    xq, xs = fb.fp8_quant_act(x)
    need = fb.fp8_blockscaled_gemm_workspace_size(M, N, K)
    small = fb.make_workspace(need - 256)
    with pytest.raises(fb.Fp8bsError) as e:
        fb.fp8_blockscaled_gemm(xq, xs, wq, ws, workspace=small)
    assert e.value.code == 4
    buf = torch.zeros(N * K + 16, dtype=torch.uint8, device="cuda")
    wq_mis = buf[1:1 + N * K].view(N, K)
    wq_mis.copy_(wq)
    with pytest.raises(fb.Fp8bsError) as e:
        fb.fp8_blockscaled_gemm(xq, xs, wq_mis, ws)
    assert e.value.code == 3


# ------------------------------------------------------------- bf16 baseline
def _bf16_case(M, N, K, seed):
    x = synth.activations(M, K, seed=seed)
    w = synth.weights(N, K, seed=seed + 1).to(torch.bfloat16)
    y = fb.bf16_gemm_ref(x.cuda(), w.cuda())
    torch.cuda.synchronize()
    yr, bound = oracle.default().gemm_bf16(bits16(x), bits16(w))
    check_y(y, yr, bound, "bf16 M=%d N=%d K=%d" % (M, N, K))
    return y


@pytest.mark.parametrize("M,N,K", [(8, 256, 512), (1, 5120, 5120), (8, 5120, 5120), (64, 300, 640),
                                   (17, 1000, 192)])
def test_bf16_gemm_matches_oracle(M, N, K):
    _bf16_case(M, N, K, 70 + M)


def test_bf16_gemm_deterministic():
    M, N, K = 8, 5120, 5120
    x = synth.activations(M, K, seed=1).cuda()
    w = synth.weights(N, K, seed=2).to(torch.bfloat16).cuda()
    work = fb.make_workspace(fb.bf16_gemm_ref_workspace_size(M, N, K))
    outs = [fb.bf16_gemm_ref(x, w, workspace=work) for _ in range(10)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))


@pytest.mark.parametrize("M,N,K", [(8, 5120, 5120), (3, 300, 1280), (64, 640, 2048), (17, 129, 384)])
def test_tiled_weights_bitwise_equal(M, N, K):
    x = synth.activations(M, K, seed=M + 7, outlier_p=0.001).cuda()
    w = synth.weights(N, K, seed=M + 8, outlier_p=0.01).cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w)
    wt, _ = fb.fp8_quant_weight_blocks(w, tiled=True)
    xq, xs = fb.fp8_quant_act(x)
    for flags in (0, fb.FLAG_OVERLAP_PREV):
        a = fb.fp8_blockscaled_gemm(xq, xs, wq, ws, flags=flags)
        b = fb.fp8_blockscaled_gemm(xq, xs, wt, ws, n=N, flags=flags)
        c = fb.fp8_blockscaled_gemm_fused(x, wt, ws, n=N, flags=flags)
        torch.cuda.synchronize()
        assert torch.equal(a.view(torch.int16), b.view(torch.int16))
        assert torch.equal(a.view(torch.int16), c.view(torch.int16))
    ref = oracle_layer(x.cpu(), w.cpu())
    check_y(b, ref["y"], ref["bound"], "tiled M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K", [(8, 5120, 5120), (5, 300, 640)])
def test_bf16_tiled_bitwise_equal(M, N, K):
    x = synth.activations(M, K, seed=90).cuda()
    w = synth.weights(N, K, seed=91).to(torch.bfloat16).cuda()
    wt = fb.bf16_pack_weights_tiled(w)
    a = fb.bf16_gemm_ref(x, w)
    b = fb.bf16_gemm_ref(x, wt, n=N)
    torch.cuda.synchronize()
    assert torch.equal(a.view(torch.int16), b.view(torch.int16))


def test_column_shards_match_the_whole_layer():
    """Column sharding (each GPU would hold a 128-row-aligned slice of W and
    compute its own columns of Y, with no reduction between GPUs): slices
    quantised on their own give the same codes and scales as the slice of the
    whole matrix, and the concatenated outputs meet the same tolerance."""
    M, N, K = 8, 5120, 5120
    x_cpu, w_cpu = synth.activations(M, K, seed=61), synth.weights(N, K, seed=62, outlier_p=0.01)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w)
    cuts = [0, 1280, 2688, 4096, 5120]
    parts = []
    for a, b in zip(cuts[:-1], cuts[1:]):
        sq, ss = fb.fp8_quant_weight_blocks(w[a:b].contiguous())
        assert torch.equal(sq, wq[a:b]) and torch.equal(ss, ws[a // 128:b // 128])
        parts.append(fb.fp8_blockscaled_gemm_fused(x, sq, ss))
    torch.cuda.synchronize()
    ref = oracle_layer(x_cpu, w_cpu)
    check_y(torch.cat(parts, dim=1), ref["y"], ref["bound"], "column shards")
