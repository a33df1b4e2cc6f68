"""GPU parity of the native block-scaled (MX) variant against the oracle's MX
mode: one power-of-two (UE8M0) scale per 32 consecutive K per row, E4M3
codes, the scales applied by the tensor core (kind::mxf8f6f4 block_scale).

Codes and scale bytes must be bit-exact with oracle_mx_quant (the library
writes codes tiled and scale bytes in 512-byte tensor-memory atoms; the
helpers below only rearrange bytes).  Y must meet the layer's tolerance
|y - y_oracle| <= 4e-3 * sum|a w| + 1e-6 against oracle_mx_gemm's fp64
product, and repeat bit for bit.
"""
import numpy as np
import pytest
import torch

import fp8_block_scaled_token_gb300 as fb
import oracle
from fp8_block_scaled_token_gb300 import synth
from tests.gpu_helpers import Ran, bits16, check_y, runs_gemm

pytestmark = pytest.mark.gpu

MODE_MX = 3
RUNS_MX_QUANT_WEIGHT, RUNS_MX_QUANT_ACT = 3, 4

# byte offset of (row r, 32-wide K block j) inside a 512-byte scale atom
_R = np.arange(128)
ATOM_OFF = 16 * (_R % 32)[:, None] + 4 * (_R // 32)[:, None] + np.arange(4)[None, :]  # [128, 4]


def untile_codes(wq, N, K):
    """[tiles, 128, 128] tiled codes -> [N, K]."""
    nbr, kg = (N + 127) // 128, K // 128
    t = wq.cpu().numpy().reshape(nbr, kg, 128, 128).transpose(0, 2, 1, 3).reshape(nbr * 128, K)
    return t[:N]


def atoms_to_bytes(atoms, rows, K):
    """[row blocks * K/128, 512] scale atoms -> scale bytes [rows, K/32]."""
    nbr, kg = (rows + 127) // 128, K // 128
    a = atoms.cpu().numpy().reshape(nbr, kg, 512)
    out = a[:, :, ATOM_OFF]                               # [nbr, kg, 128, 4]
    return out.transpose(0, 2, 1, 3).reshape(nbr * 128, kg * 4)[:rows]


def _weights_case(N, K, seed, dtype=torch.float32, outlier_p=0.01):
    w = synth.weights(N, K, seed=seed, outlier_p=outlier_p)
    if dtype == torch.bfloat16:
        w = w.to(torch.bfloat16)
    return w


def _oracle_quant(t):
    """The oracle's MX quantisation of a CPU tensor (fp32 or bf16)."""
    o = oracle.default()
    return o.mx_quant(bits16(t) if t.dtype == torch.bfloat16 else t.numpy())


@pytest.mark.parametrize("N,K,dtype", [(256, 512, torch.float32), (300, 1280, torch.float32),
                                       (128, 256, torch.bfloat16), (1, 128, torch.float32),
                                       (5120, 5120, torch.float32)])
def test_mx_quant_weights_bit_exact(N, K, dtype):
    w = _weights_case(N, K, seed=N + 11, dtype=dtype)
    with Ran() as r:
        wq, wa = fb.fp8_mx_quant_weights(w.cuda())
    assert r.launched() == {RUNS_MX_QUANT_WEIGHT: 1}
    codes, sb = _oracle_quant(w)
    assert np.array_equal(untile_codes(wq, N, K), codes)
    assert np.array_equal(atoms_to_bytes(wa, N, K), sb)
    # rows past N: zero codes and zero scale bytes
    nbr = (N + 127) // 128
    full = wq.cpu().numpy().reshape(nbr, K // 128, 128, 128).transpose(0, 2, 1, 3).reshape(nbr * 128, K)
    assert not full[N:].any()
    assert not atoms_to_bytes(wa, nbr * 128, K)[N:].any()


def test_mx_quant_edge_values():
    """Zero blocks (e = 0), subnormal block maxima (e clamped to -127),
    blocks whose top values saturate at 448 (between 448 and 512 after
    scaling), exact powers of two, signed zeros and ties."""
    K = 256
    rows = []
    rows.append(np.zeros(K, np.float32))
    rows.append(np.full(K, 2.0 ** -130, np.float32))                      # subnormal amax
    rows.append(np.linspace(-2.0 ** -128, 2.0 ** -128, K).astype(np.float32))
    r = np.full(K, 1.0, np.float32)
    r[::32] = 1.99                                                         # 1.99 * 2^8 = 509 -> saturates
    rows.append(r)
    rows.append(np.array([2.0 ** (j % 40 - 20) for j in range(K)], np.float32))
    z = np.zeros(K, np.float32)
    z[1::2] = -0.0
    z[::64] = 3.0
    rows.append(z)
    t = np.array([(1.0 + (j % 16) / 16.0) * 2.0 ** (j % 7) for j in range(K)], np.float32)
    t[::2] *= -1
    rows.append(t)
    w = torch.from_numpy(np.stack(rows))
    wq, wa = fb.fp8_mx_quant_weights(w.cuda())
    codes, sb = oracle.default().mx_quant(w.numpy())
    N = w.shape[0]
    assert np.array_equal(untile_codes(wq, N, K), codes)
    assert np.array_equal(atoms_to_bytes(wa, N, K), sb)
    assert sb[0, 0] == 127 and sb[1, 0] == 0 and (codes[3, ::32] == 0x7E).all()
    # the same rows as activations (bf16 copies)
    xb = w.to(torch.bfloat16)
    xq, xa = fb.fp8_mx_quant_act(xb.cuda())
    c2, s2 = oracle.default().mx_quant(bits16(xb))
    assert np.array_equal(xq.cpu().numpy(), c2)
    assert np.array_equal(atoms_to_bytes(xa, N, K), s2)


@pytest.mark.parametrize("M,K", [(1, 128), (8, 5120), (13, 1280), (64, 2048), (129, 256), (300, 1024), (512, 512)])
def test_mx_quant_act_bit_exact(M, K):
    x = synth.activations(M, K, seed=M + 21, outlier_p=0.001)
    with Ran() as r:
        xq, xa = fb.fp8_mx_quant_act(x.cuda())
    assert r.launched() == {RUNS_MX_QUANT_ACT: 1}
    codes, sb = _oracle_quant(x)
    assert np.array_equal(xq.cpu().numpy(), codes)
    assert np.array_equal(atoms_to_bytes(xa, M, K), sb)
    padded = (M + 127) // 128 * 128                       # one atom per 128-token tile and K block
    assert xa.shape[0] == padded // 128 * (K // 128)
    assert not atoms_to_bytes(xa, padded, K)[M:].any(), "token rows past M must be zero"


def _mx_layer(M, N, K, seed, x_out=0.0, w_out=0.0):
    x = synth.activations(M, K, seed=seed, outlier_p=x_out)
    w = synth.weights(N, K, seed=seed + 1000, outlier_p=w_out)
    xq, xa = fb.fp8_mx_quant_act(x.cuda())
    wq, wa = fb.fp8_mx_quant_weights(w.cuda())
    o = oracle.default()
    ca, sa = _oracle_quant(x)
    cw, sw = _oracle_quant(w)
    y_ref, bound = o.mx_gemm(ca, sa, cw, sw)
    return xq, xa, wq, wa, y_ref, bound


def test_mx_gemm_smallest():
    """One 128 x 128 tile, one K block: a single CTA, one unit."""
    M, N, K = 8, 128, 128
    xq, xa, wq, wa, y_ref, bound = _mx_layer(M, N, K, seed=5)
    work = fb.make_workspace(fb.fp8_mx_gemm_workspace_size(M, N, K))
    with Ran() as r:
        y = fb.fp8_mx_gemm(xq, xa, wq, wa, N, workspace=work)
    assert r.launched() == {runs_gemm(MODE_MX, 16): 1}
    assert fb.workspace_status(work) == 0
    check_y(y, y_ref, bound, "MX M=%d N=%d K=%d" % (M, N, K))


@pytest.mark.parametrize("M,N,K", [(8, 256, 512), (1, 640, 1024), (13, 300, 1280), (33, 1000, 2048),
                                   (64, 384, 1024), (8, 5120, 5120), (1, 5120, 5120), (8, 512, 17408),
                                   (65, 640, 1024), (128, 1000, 2048), (300, 5120, 1024), (512, 640, 512),
                                   (256, 7168, 1024)])
def test_mx_gemm_matches_oracle(M, N, K):
    """Above 64 tokens the 128-token tile (stream-K over token-tile pairs, or
    one pair per CTA), its token scale atoms one per 128-token tile."""
    xq, xa, wq, wa, y_ref, bound = _mx_layer(M, N, K, seed=M + N, x_out=0.001, w_out=0.01)
    work = fb.make_workspace(fb.fp8_mx_gemm_workspace_size(M, N, K))
    npad = 16 if M <= 16 else 32 if M <= 32 else 48 if M <= 48 else 64 if M <= 64 else 128
    with Ran() as r:
        y = fb.fp8_mx_gemm(xq, xa, wq, wa, N, workspace=work)
    assert r.launched() == {runs_gemm(MODE_MX, npad): 1}
    assert fb.workspace_status(work) == 0
    check_y(y, y_ref, bound, "MX M=%d N=%d K=%d" % (M, N, K))


def test_mx_gemm_deterministic_and_overlap_flag():
    M, N, K = 8, 5120, 5120
    xq, xa, wq, wa, _, _ = _mx_layer(M, N, K, seed=3)
    work = fb.make_workspace(fb.fp8_mx_gemm_workspace_size(M, N, K))
    outs = [fb.fp8_mx_gemm(xq, xa, wq, wa, N, workspace=work, flags=(fb.FLAG_OVERLAP_PREV if i % 2 else 0))
            for i in range(10)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert fb.workspace_status(work) == 0
    assert not work[1024:1024 + 4 * (N // 128)].any(), "arrival counters back at zero"


def test_mx_host_errors():
    x = synth.activations(513, 256, seed=1).cuda()
    with pytest.raises(fb.Fp8bsError) as e:
        fb.fp8_mx_quant_act(x)
    assert e.value.code == 2
    with pytest.raises(fb.Fp8bsError) as e:
        fb.fp8_mx_gemm_workspace_size(513, 256, 256)
    assert e.value.code == 2


def test_mx_large_m_reruns_bitwise():
    """128-token tiles with K split across CTAs: ten reruns give the same bits."""
    M, N, K = 300, 1024, 4096
    xq, xa, wq, wa, _, _ = _mx_layer(M, N, K, seed=11)
    work = fb.make_workspace(fb.fp8_mx_gemm_workspace_size(M, N, K))
    outs = [fb.fp8_mx_gemm(xq, xa, wq, wa, N, workspace=work) for _ in range(10)]
    torch.cuda.synchronize()
    for o in outs[1:]:
        assert torch.equal(o.view(torch.int16), outs[0].view(torch.int16))
    assert fb.workspace_status(work) == 0
