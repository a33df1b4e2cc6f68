"""Pins for the CPU oracle: checks against facts that do not come from the
oracle itself (hand-worked values, the format definition, closed forms,
invariants, brute force, and independent library routines such as torch's
float8_e4m3fn and bfloat16 casts).

Each ``pin_*`` takes an ``oracle.Oracle`` and raises AssertionError when the
oracle disagrees.  ``tests/test_oracle_pins.py`` runs them on the oracle;
``tests/test_oracle_mutants.py`` runs them on copies of the oracle with a
deliberate mistake planted and requires that some pin rejects every copy.
"""
import math
import os
import struct

import numpy as np
import torch

from fp8_block_scaled_token_gb300 import synth

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


# ---------------------------------------------------------------------------
# fixture readers
# ---------------------------------------------------------------------------
def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            yield line.split()


def _f32_from_bits(h):
    return struct.unpack("<f", struct.pack("<I", int(h, 16)))[0]


def _f32_bits(v):
    return struct.unpack("<I", struct.pack("<f", float(v)))[0]


def _keyvals(name):
    return {r[0]: r[1] for r in _rows(name)}


# Independent decode through torch's float8_e4m3fn dtype (a library routine).
def torch_decode(codes):
    c = torch.from_numpy(np.ascontiguousarray(codes, dtype=np.uint8))
    return c.view(torch.float8_e4m3fn).to(torch.float64).numpy()


def _bf16_values(bits):
    return (np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)


# ---------------------------------------------------------------------------
# E4M3 decode
# ---------------------------------------------------------------------------
def pin_decode_hand_values(o):
    t = o.e4m3_decode_table()
    for code, val, *_ in _rows("e4m3_codes.txt"):
        c = int(code, 16)
        if val == "nan":
            assert math.isnan(t[c]), code
        else:
            v = float(val)
            assert t[c] == v, (code, t[c], v)
            assert math.copysign(1.0, t[c]) == math.copysign(1.0, v), code


def pin_decode_vs_torch(o):
    t = o.e4m3_decode_table()
    ref = torch_decode(np.arange(256))
    nan_o = np.isnan(t)
    assert np.array_equal(nan_o, np.isnan(ref))
    assert np.array_equal(t[~nan_o], ref[~nan_o])
    assert np.array_equal(np.signbit(t[~nan_o]), np.signbit(ref[~nan_o]))


def pin_decode_order(o):
    t = o.e4m3_decode_table()
    pos = t[:0x7F]
    assert np.all(np.diff(pos) > 0), "positive codes must increase"
    assert np.array_equal(t[0x80:0xFF], -pos), "negative codes mirror"
    assert int(np.isnan(t).sum()) == 2


# ---------------------------------------------------------------------------
# E4M3 encode
# ---------------------------------------------------------------------------
def pin_encode_hand_values(o):
    for val, code, *_ in _rows("e4m3_encode.txt"):
        v = np.float32(float.fromhex(val))
        got = int(o.e4m3_encode([v])[0])
        assert got == int(code, 16), (val, hex(got), code)


def pin_encode_roundtrip(o):
    t = o.e4m3_decode_table()
    codes = np.array([c for c in range(256) if not math.isnan(t[c])], dtype=np.uint8)
    vals = torch_decode(codes).astype(np.float32)
    assert np.array_equal(o.e4m3_encode(vals), codes)


def pin_encode_midpoints(o):
    # brute force over every neighbouring pair of positive finite codes
    vals = torch_decode(np.arange(0x7F))
    lo, hi = vals[:-1], vals[1:]
    mids = ((lo + hi) / 2).astype(np.float32)           # exact in fp32
    assert np.array_equal(mids.astype(np.float64), (lo + hi) / 2)
    even = np.where(np.arange(0x7E) % 2 == 0, np.arange(0x7E), np.arange(1, 0x7F))
    assert np.array_equal(o.e4m3_encode(mids), even.astype(np.uint8))
    up = np.nextafter(mids, np.float32(np.inf))
    down = np.nextafter(mids, np.float32(0))
    assert np.array_equal(o.e4m3_encode(up), np.arange(1, 0x7F, dtype=np.uint8))
    assert np.array_equal(o.e4m3_encode(down), np.arange(0, 0x7E, dtype=np.uint8))
    assert np.array_equal(o.e4m3_encode(-up), (np.arange(1, 0x7F) | 0x80).astype(np.uint8))


def pin_encode_vs_torch(o):
    rng = np.random.default_rng(12345)
    a = rng.standard_normal(20000).astype(np.float32) * np.float32(60.0)
    b = (rng.uniform(-1, 1, 20000) * 2.0 ** rng.integers(-14, 0, 20000)).astype(np.float32)
    v = np.concatenate([a, b])
    v = v[np.abs(v) <= 448.0]
    ref = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(o.e4m3_encode(v), ref)


def pin_encode_saturates(o):
    v = np.array([448.0, 448.5, 463.99, 464.0, 500.0, 1e6, 3.0e38], dtype=np.float32)
    assert np.all(o.e4m3_encode(v) == 0x7E)
    assert np.all(o.e4m3_encode(-v) == 0xFE)


# ---------------------------------------------------------------------------
# bf16 rounding
# ---------------------------------------------------------------------------
def pin_bf16_hand_values(o):
    for val, bits, *_ in _rows("bf16_round.txt"):
        got = int(o.round_bf16([float.fromhex(val)])[0])
        assert got == int(bits, 16), (val, hex(got), bits)


def pin_bf16_vs_torch(o):
    rng = np.random.default_rng(7)
    v = (rng.standard_normal(20000) * 2.0 ** rng.integers(-130, 120, 20000)).astype(np.float32)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.round_bf16(v.astype(np.float64)), ref)


def pin_bf16_nearest_bruteforce(o):
    # fp64 inputs that fp32 cannot hold: the result must be the nearer of the
    # two bf16 neighbours (ties are covered by the hand values).
    rng = np.random.default_rng(8)
    v = rng.standard_normal(4000) * 2.0 ** rng.integers(-20, 20, 4000)
    bits = o.round_bf16(v)
    r = _bf16_values(bits)
    for delta in (1, -1):
        nb = _bf16_values((bits.astype(np.int32) + delta).astype(np.uint16))
        assert np.all(np.abs(v - r) <= np.abs(v - nb))


# ---------------------------------------------------------------------------
# activation / weight quantisation
# ---------------------------------------------------------------------------
def pin_quant_act_hand_group(o):
    rows = list(_rows("quant_group.txt"))
    x = np.zeros((1, 256), dtype=np.float64)
    want = np.zeros(256, dtype=np.uint8)
    scales = {}
    for r in rows:
        if r[0].startswith("scale"):
            scales[r[0]] = int(r[1], 16)
        else:
            i = int(r[0])
            x[0, i] = float.fromhex(r[1])
            want[i] = int(r[3], 16)
    xb = torch.from_numpy(x).to(torch.bfloat16)
    assert torch.equal(xb.to(torch.float64), torch.from_numpy(x)), "fixture values are bf16-exact"
    xq, xs = o.quant_act(xb.view(torch.int16).numpy().view(np.uint16))
    assert np.array_equal(xq[0], want)
    assert _f32_bits(xs[0, 0]) == scales["scale0"]
    assert _f32_bits(xs[0, 1]) == scales["scale1"]


def _torch_group_quant(v2d):
    """Independent restatement with torch CPU ops: rows of 128 values (fp32)."""
    t = torch.from_numpy(v2d.astype(np.float32))
    amax = t.abs().amax(dim=1, keepdim=True)
    s = torch.where(amax == 0, torch.ones_like(amax), amax / torch.tensor(448.0, dtype=torch.float32))
    q = (t / s).to(torch.float8_e4m3fn).view(torch.uint8)
    return q.numpy(), s[:, 0].numpy()


def pin_quant_act_vs_torch(o):
    x = synth.activations(5, 1024, seed=21, outlier_p=0.01)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    xq, xs = o.quant_act(bits)
    v = x.to(torch.float32).numpy().reshape(-1, 128)
    q, s = _torch_group_quant(v)
    assert np.array_equal(xq.reshape(-1, 128), q)
    assert np.array_equal(xs.reshape(-1), s)


def pin_quant_act_row_stride(o):
    x = synth.activations(3, 640, seed=22)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    xq_full, xs_full = o.quant_act(bits[:, :512])
    xq, xs = o.quant_act(bits, K=512)     # row stride 640, first 512 used
    assert np.array_equal(xq, xq_full) and np.array_equal(xs, xs_full)


def pin_quant_weight_vs_torch(o):
    for N in (256, 200):          # 200: ragged last block
        w = synth.weights(N, 384, seed=23, outlier_p=0.01).numpy()
        wq, ws = o.quant_weight(w)
        nb = (N + 127) // 128
        for b in range(nb):
            rows = w[b * 128:min(N, b * 128 + 128)]
            for kb in range(3):
                blk = rows[:, kb * 128:(kb + 1) * 128]
                q, s = _torch_group_quant(blk.reshape(1, -1))
                assert np.array_equal(wq[b * 128:b * 128 + rows.shape[0], kb * 128:(kb + 1) * 128].reshape(-1), q[0])
                assert ws[b, kb] == s[0]


def pin_quant_weight_bf16_input(o):
    w = synth.weights(128, 256, seed=24)
    wb = w.to(torch.bfloat16)
    bits = wb.view(torch.int16).numpy().view(np.uint16)
    q1, s1 = o.quant_weight(bits)
    q2, s2 = o.quant_weight(wb.to(torch.float32).numpy())
    assert np.array_equal(q1, q2) and np.array_equal(s1, s2)


def pin_quant_single_entry_block(o):
    kv = _keyvals("gemm_closed_form.txt")
    w = np.zeros((128, 128), dtype=np.float32)
    w[37, 91] = 2.0
    wq, ws = o.quant_weight(w)
    assert _f32_bits(ws[0, 0]) == int(kv["single.s_w"], 16)
    assert wq[37, 91] == int(kv["single.code"], 16)
    wq[37, 91] = 0
    assert not wq.any()


def pin_quant_halfulp(o):
    x = synth.activations(4, 2048, seed=25, outlier_p=0.01)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    xq, xs = o.quant_act(bits)
    v = x.to(torch.float32).numpy()
    s = np.repeat(xs, 128, axis=1)
    t = (v / s).astype(np.float64)                    # the fp32 quotient
    d = torch_decode(xq)
    mag = np.abs(t)
    e = np.floor(np.log2(np.maximum(mag, 2.0 ** -6)))
    ulp = 2.0 ** (e - 3)                              # e4m3 spacing in that binade
    sat = mag >= 448.0
    assert np.all(np.abs(t - d)[~sat] <= 0.5 * ulp[~sat])
    assert np.all(np.abs(d[sat]) == 448.0)


def pin_quant_amax_is_448(o):
    x = synth.activations(6, 1024, seed=26, outlier_p=0.01)
    bits = x.view(torch.int16).numpy().view(np.uint16)
    xq, _ = o.quant_act(bits)
    v = x.to(torch.float32).numpy().reshape(-1, 128)
    idx = np.abs(v).argmax(axis=1)
    codes = xq.reshape(-1, 128)[np.arange(v.shape[0]), idx]
    assert np.all((codes & 0x7F) == 0x7E)


def pin_quant_pow2_equivariance(o):
    w = synth.weights(256, 256, seed=27).numpy()
    q0, s0 = o.quant_weight(w)
    for j in (-5, 3):
        q, s = o.quant_weight((w * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(q, q0)
        assert np.array_equal(s, s0 * np.float32(2.0 ** j))


def pin_quant_zero_group(o):
    x = np.zeros((2, 256), dtype=np.uint16)
    x[1, 128:] = 0x3F80                        # second row, second group = 1.0
    xq, xs = o.quant_act(x)
    assert np.all(xs[0] == 1.0) and xs[1, 0] == 1.0
    assert not xq[0].any() and not xq[1, :128].any()
    assert np.all(xq[1, 128:] == 0x7E)
    w = np.zeros((128, 128), dtype=np.float32)
    wq, ws = o.quant_weight(w)
    assert ws[0, 0] == 1.0 and not wq.any()


def pin_quant_sign_symmetry(o):
    w = synth.weights(128, 256, seed=28).numpy()
    q, s = o.quant_weight(w)
    qn, sn = o.quant_weight(-w)
    assert np.array_equal(s, sn)
    assert np.array_equal(qn, q ^ 0x80)


# ---------------------------------------------------------------------------
# block-scaled product
# ---------------------------------------------------------------------------
def _dense_reference(xq, xs, wq, ws):
    """Brute force: dequantise both operands to dense fp64 and multiply."""
    A = torch_decode(xq) * np.repeat(xs.astype(np.float64), 128, axis=1)
    N = wq.shape[0]
    sw = np.repeat(np.repeat(ws.astype(np.float64), 128, axis=0)[:N], 128, axis=1)
    W = torch_decode(wq) * sw
    return A @ W.T, np.abs(A) @ np.abs(W).T


def pin_gemm_bruteforce(o):
    for (M, N, K, seed) in ((8, 256, 512, 30), (3, 200, 256, 31), (1, 128, 128, 32)):
        x = synth.activations(M, K, seed=seed, outlier_p=0.01)
        w = synth.weights(N, K, seed=seed + 100, outlier_p=0.01).numpy()
        xq, xs = o.quant_act(x.view(torch.int16).numpy().view(np.uint16))
        wq, ws = o.quant_weight(w)
        y, bound = o.gemm_fp8(xq, xs, wq, ws)
        yr, br = _dense_reference(xq, xs, wq, ws)
        assert np.all(np.abs(y - yr) <= 1e-12 * br + 1e-300), (M, N, K)
        assert np.allclose(bound, br, rtol=1e-12, atol=0)
        # the dequantised product approximates the fp64 product of the raw inputs
        raw = x.to(torch.float64).numpy() @ w.astype(np.float64).T
        rawb = np.abs(x.to(torch.float64).numpy()) @ np.abs(w.astype(np.float64)).T
        assert np.all(np.abs(y - raw) <= 0.13 * rawb)


def pin_gemm_constant_closed_form(o):
    kv = _keyvals("gemm_closed_form.txt")
    M, N, K = int(kv["constant.M"]), int(kv["constant.N"]), int(kv["constant.K"])
    x = torch.full((M, K), float(kv["constant.x"]), dtype=torch.bfloat16)
    w = np.full((N, K), float(kv["constant.w"]), dtype=np.float32)
    xq, xs = o.quant_act(x.view(torch.int16).numpy().view(np.uint16))
    wq, ws = o.quant_weight(w)
    sa, sw = _f32_from_bits(kv["constant.s_a"]), _f32_from_bits(kv["constant.s_w"])
    assert np.all(xs == np.float32(sa)) and np.all(ws == np.float32(sw))
    code = int(kv["constant.code"], 16)
    assert np.all(xq == code) and np.all(wq == code)
    y, bound = o.gemm_fp8(xq, xs, wq, ws)
    expected = (K // 128) * (sa * sw * float(kv["constant.P_block"]))
    assert np.all(np.abs(y - expected) <= 1e-15 * expected)
    assert np.allclose(bound, y, rtol=1e-15)
    assert np.all(o.round_bf16(y) == int(kv["constant.y_bf16"], 16))


def pin_gemm_identity_blocks(o):
    K = 256
    w = np.eye(K, dtype=np.float32)
    x = synth.activations(4, K, seed=33)
    xq, xs = o.quant_act(x.view(torch.int16).numpy().view(np.uint16))
    wq, ws = o.quant_weight(w)
    kv = _keyvals("gemm_closed_form.txt")
    s_diag = np.float32(_f32_from_bits(kv["constant.s_a"]))   # fl32(1/448)
    assert ws[0, 0] == s_diag and ws[1, 1] == s_diag and ws[0, 1] == 1.0 and ws[1, 0] == 1.0
    assert np.array_equal(wq, np.eye(K, dtype=np.uint8) * 0x7E)
    y, _ = o.gemm_fp8(xq, xs, wq, ws)
    dec = torch_decode(xq)
    sa = np.repeat(xs.astype(np.float64), 128, axis=1)
    expected = (sa * float(s_diag)) * (dec * 448.0)
    assert np.array_equal(y, expected)


def pin_gemm_sign_and_pow2(o):
    x = synth.activations(4, 384, seed=34)
    w = synth.weights(256, 384, seed=35).numpy()
    xb = x.view(torch.int16).numpy().view(np.uint16)
    xq, xs = o.quant_act(xb)
    wq, ws = o.quant_weight(w)
    y, _ = o.gemm_fp8(xq, xs, wq, ws)
    wqn, wsn = o.quant_weight(-w)
    yn, _ = o.gemm_fp8(xq, xs, wqn, wsn)
    assert np.array_equal(yn, -y)
    x8 = (x.to(torch.float32) * 8.0).to(torch.bfloat16)
    xq8, xs8 = o.quant_act(x8.view(torch.int16).numpy().view(np.uint16))
    wq4, ws4 = o.quant_weight((w * np.float32(0.25)).astype(np.float32))
    y2, _ = o.gemm_fp8(xq8, xs8, wq4, ws4)
    assert np.array_equal(y2, 2.0 * y)


def pin_gemm_columns_and_threads(o):
    x = synth.activations(5, 256, seed=36)
    w = synth.weights(384, 256, seed=37).numpy()
    xq, xs = o.quant_act(x.view(torch.int16).numpy().view(np.uint16))
    wq, ws = o.quant_weight(w)
    y1, b1 = o.gemm_fp8(xq, xs, wq, ws, nthreads=1)
    y4, b4 = o.gemm_fp8(xq, xs, wq, ws, nthreads=4)
    assert np.array_equal(y1, y4) and np.array_equal(b1, b4)
    cols = [383, 0, 129, 7]
    yc, bc = o.gemm_fp8(xq, xs, wq, ws, cols=cols)
    assert np.array_equal(yc, y1[:, cols]) and np.array_equal(bc, b1[:, cols])


def pin_gemm_bf16_bruteforce(o):
    x = synth.activations(3, 320, seed=38)
    w = synth.weights(130, 320, seed=39)
    wb = w.to(torch.bfloat16)                       # torch's RNE cast
    wbits = wb.view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(o.f32_to_bf16_bits(w.numpy()), wbits)
    y, bound = o.gemm_bf16(x.view(torch.int16).numpy().view(np.uint16), wbits)
    X = x.to(torch.float64).numpy()
    W = wb.to(torch.float64).numpy()
    assert np.all(np.abs(y - X @ W.T) <= 1e-12 * (np.abs(X) @ np.abs(W).T))
    assert np.allclose(bound, np.abs(X) @ np.abs(W).T, rtol=1e-12)


# ---------------------------------------------------------------- greedy choice
def _bf16_bits_of(values):
    t = torch.tensor(np.asarray(values, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def pin_greedy_vs_numpy_argmax(o):
    # numpy's argmax returns the first of equal maxima and compares -0 == +0:
    # the same rule, computed by a library routine.  Small integers make ties
    # (and signed zeros) frequent.
    rng = np.random.default_rng(51)
    vals = rng.integers(-6, 7, size=(9, 700)).astype(np.float32)
    vals[rng.random(vals.shape) < 0.2] *= -0.0   # zeros of both signs, negatives flipped
    vals[3] = -vals[3] - 1.0                     # an all-negative row
    bits = _bf16_bits_of(vals)
    tok, logit = o.greedy(bits)
    ref = np.argmax(vals.astype(np.float64), axis=1)
    assert np.array_equal(tok, ref)
    assert np.array_equal(logit, vals.max(axis=1) + np.float32(0.0))


def pin_greedy_hand_cases(o):
    rows = [
        ([1.0, 3.0, 3.0, 2.0], 1, 3.0),
        ([-0.0, 0.0, -1.0], 0, 0.0),            # -0 equals +0: the lower column
        ([-5.0, -1.0, -1.0], 1, -1.0),
        ([2.0, 2.0, 2.0, 2.0], 0, 2.0),
        ([0.5, 0.25, 448.0, 1e30], 3, 1e30),
    ]
    for vals, want, wlogit in rows:
        tok, logit = o.greedy(_bf16_bits_of([vals]))
        assert tok[0] == want, vals
        assert float(logit[0]) == float(torch.tensor(wlogit).to(torch.bfloat16).float())
        assert not np.signbit(logit[0]) or logit[0] != 0


def pin_greedy_first_n_columns(o):
    # columns at or past N are not candidates
    bits = _bf16_bits_of([[1.0, 2.0, 9.0, 9.0], [4.0, 4.0, 9.0, 0.0]])
    tok, _ = o.greedy(bits, N=2)
    assert list(tok) == [1, 0]


# ---------------------------------------------------------------- MX (microscaling) mode
def pin_mx_hand_values(o):
    # amax 1.0: e = floor(log2 1) - 8 = -8 (byte 119), 1.0 -> 256 = code 0x78,
    # 0.5 -> 128 = 0x70; amax 448: e = 0 (byte 127), 448 -> 0x7E; amax 1.9:
    # e = -8, 1.9 * 256 = 486.4 saturates to 448 (0x7E); -0.25 * 256 = -64 =
    # sign | exponent field 13 (2^(13-7)) = 0xE8
    x = np.array([[1.0, 0.5] + [0.0] * 30, [448.0] + [1.0] * 31, [1.9, -0.25] + [0.1] * 30], dtype=np.float32)
    codes, sb = o.mx_quant(x)
    assert list(sb[:, 0]) == [119, 127, 119]
    assert list(codes[:, 0]) == [0x78, 0x7E, 0x7E]
    assert codes[0, 1] == 0x70 and codes[2, 1] == 0xE8 and codes[0, 2] == 0x00


def _mx_reference(v2d):
    """Independent restatement with numpy (exponent) and torch (E4M3 cast)."""
    rows, K = v2d.shape
    blocks = v2d.reshape(rows, K // 32, 32).astype(np.float64)
    amax = np.abs(blocks).max(axis=2)
    e = np.where(amax > 0, np.floor(np.log2(np.where(amax > 0, amax, 1.0))) - 8, 0).clip(-127, 127)
    q = np.clip(blocks * np.exp2(-e)[..., None], -448.0, 448.0)
    codes = torch.tensor(q.reshape(rows, K).astype(np.float32)).to(torch.float8_e4m3fn)
    return codes.view(torch.uint8).numpy(), (e + 127).astype(np.uint8)


def pin_mx_vs_numpy_torch(o):
    g = torch.Generator().manual_seed(61)
    w = (torch.randn(40, 256, generator=g) * 0.02)
    w[torch.rand(40, 256, generator=g) < 0.02] *= 30.0
    x = torch.randn(6, 256, generator=g).to(torch.bfloat16)
    for v, inp in ((w.numpy(), w.numpy()), (x.float().numpy(), x.view(torch.int16).numpy().view(np.uint16))):
        codes, sb = o.mx_quant(inp)
        rc, rs = _mx_reference(v)
        assert np.array_equal(sb, rs)
        assert np.array_equal(codes, rc)


def pin_mx_pow2_equivariance(o):
    g = torch.Generator().manual_seed(62)
    v = (torch.randn(4, 128, generator=g)).numpy()
    c0, s0 = o.mx_quant(v)
    for j in (-20, -3, 5, 40):
        c1, s1 = o.mx_quant((v * np.float32(2.0 ** j)).astype(np.float32))
        assert np.array_equal(c1, c0) and np.array_equal(s1.astype(int), s0.astype(int) + j)


def pin_mx_zero_block(o):
    v = np.zeros((2, 64), dtype=np.float32)
    v[1, :32] = -0.0
    v[1, 32:] = 3.0
    codes, sb = o.mx_quant(v)
    assert list(sb.ravel()) == [127, 127, 127, 120]   # amax 3: floor(log2 3) - 8 = -7
    assert not codes[0].any() and np.all(codes[1, :32] == 0x80)


def pin_mx_gemm_bruteforce(o):
    g = torch.Generator().manual_seed(63)
    a = torch.randn(5, 192, generator=g).numpy()
    w = (torch.randn(70, 192, generator=g) * 0.05).numpy()
    aq, asb = o.mx_quant(a)
    wq, wsb = o.mx_quant(w)
    table = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    A = table[aq] * np.repeat(np.exp2(asb.astype(np.float64) - 127), 32, axis=1)
    W = table[wq] * np.repeat(np.exp2(wsb.astype(np.float64) - 127), 32, axis=1)
    y, bound = o.mx_gemm(aq, asb, wq, wsb)
    assert np.array_equal(y, A @ W.T) or np.allclose(y, A @ W.T, rtol=1e-15, atol=0)
    assert np.allclose(bound, np.abs(A) @ np.abs(W).T, rtol=1e-15)
    # a power of two on the weight scales scales Y exactly
    y2, _ = o.mx_gemm(aq, asb, wq, (wsb.astype(int) + 3).astype(np.uint8))
    assert np.array_equal(y2, y * 8.0)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
