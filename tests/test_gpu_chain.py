"""Chains of layers as the benchmark and a decode step run them: different
shapes back to back on one stream, one shared workspace, programmatic
dependent launch between them (the next layer streams its weights while the
previous one finishes), eagerly and captured in a CUDA graph.  Every output
must be bitwise the one a standalone call with its own workspace gives, and
the workspace must come back clean."""
import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
from fp8_block_scaled_token_gb300 import synth

pytestmark = pytest.mark.gpu

# (M, N, K, tiled): split-K decode tiles of every width, a two-CTA-per-SM
# shape, the larger-M 2-D schedule and a ragged N
SHAPES = [(8, 1280, 5120, True), (8, 4352, 1280, True), (1, 1280, 4352, False), (33, 640, 1024, True),
          (64, 2560, 1280, True), (200, 5120, 640, True), (3, 300, 640, False), (16, 5120, 5120, True)]


def _layers(seed):
    out = []
    for i, (M, N, K, tiled) in enumerate(SHAPES):
        x = synth.activations(M, K, seed=seed + i, device="cuda")
        wq, ws = fb.fp8_quant_weight_blocks(synth.weights(N, K, seed=seed + 50 + i, device="cuda"), tiled=tiled)
        out.append(dict(M=M, N=N, K=K, x=x, wq=wq, ws=ws, y=torch.empty((M, N), dtype=torch.bfloat16, device="cuda")))
    return out


def _reference(layers):
    refs = []
    for L in layers:
        refs.append(fb.fp8_blockscaled_gemm_fused(L["x"], L["wq"], L["ws"], n=L["N"]))
    torch.cuda.synchronize()
    return refs


def _shared_workspace(layers):
    size = max(fb.fp8_blockscaled_gemm_workspace_size(L["M"], L["N"], L["K"]) for L in layers)
    return fb.make_workspace(size)


def _run_chain(layers, work, token=None, logit=None, greedy_at=None):
    for i, L in enumerate(layers):
        if i == greedy_at:
            fb.fp8_blockscaled_gemm_fused_greedy(L["x"], L["wq"], L["ws"], y=L["y"], token=token, logit=logit,
                                                 workspace=work, flags=fb.FLAG_OVERLAP_PREV, n=L["N"])
        else:
            fb.fp8_blockscaled_gemm_fused(L["x"], L["wq"], L["ws"], y=L["y"], workspace=work,
                                          flags=fb.FLAG_OVERLAP_PREV, n=L["N"])


def _check(layers, refs, work):
    for L, r in zip(layers, refs):
        assert torch.equal(L["y"].view(torch.int16), r.view(torch.int16)), "M=%d N=%d K=%d" % (L["M"], L["N"], L["K"])
    assert not work[:256].any(), "status word"
    assert not work[256:1024].any(), "greedy keys and counter"


def test_eager_chain_shared_workspace():
    layers = _layers(900)
    refs = _reference(layers)
    work = _shared_workspace(layers)
    for _ in range(3):
        for L in layers:
            L["y"].fill_(float("nan"))
        _run_chain(layers, work)
        torch.cuda.synchronize()
        _check(layers, refs, work)


def test_graph_chain_with_greedy():
    layers = _layers(930)
    refs = _reference(layers)
    g_at = 0  # an M <= 64 layer carries the greedy choice
    tok_ref, logit_ref, _ = fb.fp8_blockscaled_gemm_fused_greedy(layers[g_at]["x"], layers[g_at]["wq"],
                                                                 layers[g_at]["ws"], n=layers[g_at]["N"])
    work = _shared_workspace(layers)
    token = torch.empty((64,), dtype=torch.int32, device="cuda")
    logit = torch.empty((64,), dtype=torch.float32, device="cuda")
    _run_chain(layers, work, token, logit, greedy_at=g_at)  # warm-up: per-device set-up before capture
    torch.cuda.synchronize()
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        _run_chain(layers, work, token, logit, greedy_at=g_at)
    for _ in range(3):
        for L in layers:
            L["y"].fill_(float("nan"))
        token.fill_(-1)
        torch.cuda.synchronize()
        graph.replay()
        torch.cuda.synchronize()
        _check(layers, refs, work)
        M = layers[g_at]["M"]
        assert torch.equal(token[:M], tok_ref) and torch.equal(logit[:M].view(torch.int32), logit_ref.view(torch.int32))
