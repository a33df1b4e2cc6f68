"""The greedy next-token choice fused into the output layer's epilogue.

The choice is an integer decided by floating point, so both sides take it on
the same numbers: the GPU's own bf16 logits (which must be bitwise those of
the plain fused layer) go through the oracle's greedy rule, and the token and
logit must match exactly.  Against the oracle's fp64 product the choice must
be valid: no other column can be larger by more than the two elements'
tolerances.  Exact ties (values every summation order reproduces) check the
lowest-column rule across whole and K-split tiles.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
import oracle
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import ABS_TOL, MODE_FP8, MODE_FUSED, REL_TOL, RUNS_QUANT_ACT, Ran, bits16, oracle_layer, runs_gemm

pytestmark = pytest.mark.gpu


def check_against_own_logits(token, logit, y):
    tok_o, logit_o = oracle.default().greedy(bits16(y))
    assert np.array_equal(token.cpu().numpy(), tok_o)
    assert np.array_equal(logit.cpu().numpy().view(np.uint32), logit_o.view(np.uint32))


def check_valid_choice(token, ref, cols=None):
    """token[m] is within tolerance of the oracle's best column (over `cols`)."""
    y, lim = ref["y"], REL_TOL * ref["bound"] + ABS_TOL
    tok = token.cpu().numpy()
    for m in range(y.shape[0]):
        j = int(tok[m]) if cols is None else int(np.where(cols == tok[m])[0][0])
        assert y[m, j] + lim[m, j] >= np.max(y[m] - lim[m]), "token row %d" % m


@pytest.mark.parametrize("prologue", [False, True])
@pytest.mark.parametrize("M,N,K,tiled", [(8, 5120, 5120, True), (1, 2000, 1280, False), (3, 300, 512, True),
                                         (16, 4096, 1024, True), (33, 1000, 640, False), (64, 3000, 2048, True)])
def test_greedy_matches_own_logits_and_oracle(M, N, K, tiled, prologue):
    flags = fb.FLAG_PROLOGUE_CAST if prologue else 0
    x_cpu = synth.activations(M, K, seed=M + 500)
    w_cpu = synth.weights(N, K, seed=M + 501, outlier_p=0.01)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=tiled)
    y_ref = fb.fp8_blockscaled_gemm_fused(x, wq, ws, n=N)
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K))
    with Ran() as r:
        token, logit, y = fb.fp8_blockscaled_gemm_fused_greedy(x, wq, ws, workspace=work, n=N, flags=flags)
    # the greedy instantiation of the route's GEMM is the kernel that ran
    npad = fb.gemm_schedule(M, N, K)["npad"]
    if fb.fused_route(M, N, K, flags=flags) == "prologue":
        assert r.launched() == {runs_gemm(MODE_FUSED, npad, greedy=True): 1}
    else:
        assert r.launched() == {RUNS_QUANT_ACT: 1, runs_gemm(MODE_FP8, npad, greedy=True): 1}
    assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), "logits differ from the plain layer"
    check_against_own_logits(token, logit, y)
    check_valid_choice(token, oracle_layer(x_cpu, w_cpu))
    # again, without storing the logits, on the same workspace (keys cleared)
    t2, l2, none = fb.fp8_blockscaled_gemm_fused_greedy(x, wq, ws, store_y=False, workspace=work,
                                                        flags=flags | fb.FLAG_OVERLAP_PREV, n=N)
    torch.cuda.synchronize()
    assert none is None
    assert torch.equal(t2, token) and torch.equal(l2.view(torch.int32), logit.view(torch.int32))
    assert not work[:4].any(), "status word must stay clear"
    assert not work[256:1024].any(), "greedy keys and counter must be left at zero"


def _tie_inputs(N, K, tied, sign):
    """X = 0.875 (code 448, scale 2^-9 exactly); the tied weight rows are
    sign*0.4375 (code 448, scale 2^-10), the others small, so every product,
    partial and sum on the tied rows is exact: their logits are equal in any
    summation order.  Row 1 of X is negated."""
    x = torch.full((2, K), 0.875, dtype=torch.float32)
    x[1] = -0.875
    w = synth.weights(N, K, seed=77, std=0.002)
    for n in tied:
        w[n] = sign * 0.4375
    return x.to(torch.bfloat16), w


@pytest.mark.parametrize("tiled", [False, True])
def test_exact_ties_take_the_lowest_column(tiled):
    N, K = 5120, 5120           # ~10 units per CTA: whole tiles and K-split tiles
    tied = [37, 100, 300, 1000, 2500, 5119]
    x_cpu, w_cpu = _tie_inputs(N, K, tied, +1.0)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=tiled)
    token, logit, y = fb.fp8_blockscaled_gemm_fused_greedy(x, wq, ws, n=N)
    torch.cuda.synchronize()
    yv = y.float().cpu()
    assert torch.all(yv[0, tied] == 1960.0), "tied logits must be exact"
    assert int(token[0]) == 37 and float(logit[0]) == 1960.0
    check_against_own_logits(token, logit, y)
    check_valid_choice(token, oracle_layer(x_cpu, w_cpu))


def test_all_equal_negative_logits():
    # every logit of row 0 is exactly -1960: the choice is column 0
    N, K = 3000, 5120
    x_cpu, w_cpu = _tie_inputs(N, K, range(N), -1.0)
    x, w = x_cpu.cuda(), w_cpu.cuda()
    wq, ws = fb.fp8_quant_weight_blocks(w, tiled=True)
    token, logit, y = fb.fp8_blockscaled_gemm_fused_greedy(x, wq, ws, n=N)
    torch.cuda.synchronize()
    assert int(token[0]) == 0 and float(logit[0]) == -1960.0
    assert int(token[1]) == 0 and float(logit[1]) == 1960.0
    check_against_own_logits(token, logit, y)


def test_bitwise_deterministic_and_host_errors():
    M, N, K = 8, 7000, 1536
    x = synth.activations(M, K, seed=9, device="cuda")
    wq, ws = fb.fp8_quant_weight_blocks(synth.weights(N, K, seed=10, device="cuda"), tiled=True)
    work = fb.make_workspace(fb.fp8_blockscaled_gemm_workspace_size(M, N, K))
    first = fb.fp8_blockscaled_gemm_fused_greedy(x, wq, ws, store_y=False, workspace=work, n=N)
    for _ in range(9):
        again = fb.fp8_blockscaled_gemm_fused_greedy(x, wq, ws, store_y=False, workspace=work, n=N)
        assert torch.equal(again[0], first[0]) and torch.equal(again[1].view(torch.int32), first[1].view(torch.int32))
    L = fb.lib()
    p = x.data_ptr()
    S = torch.cuda.current_stream().cuda_stream
    # token is required; a misaligned logit is refused; nothing is launched
    assert L.fp8_blockscaled_gemm_fused_greedy(p, K, wq.data_ptr(), ws.data_ptr(), None, M, N, K, None, None,
                                               work.data_ptr(), work.numel(), 0, S) == 1
    assert L.fp8_blockscaled_gemm_fused_greedy(p, K, wq.data_ptr(), ws.data_ptr(), None, M, N, K,
                                               first[0].data_ptr(), first[1].data_ptr() + 2,
                                               work.data_ptr(), work.numel(), 0, S) == 3
