"""The C-ABI library on the CPU: it builds, loads, exports every symbol the
headers declare, and rejects bad arguments on the host before anything would
reach a GPU.  Nothing here launches a kernel."""
import ctypes
import glob
import os
import re

import pytest

import fp8_block_scaled_token_gb300 as fb
from fp8_block_scaled_token_gb300 import build as fbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

OK, INVALID, SHAPE, MISALIGNED, WS_SMALL, DEVICE, CUDA, TIMEOUT = range(8)


@pytest.fixture(scope="module")
def L():
    fbuild.build()
    return fb.lib()


def declared_symbols():
    names = []
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        text = open(h).read()
        names += re.findall(r"FP8BS_API\s+[A-Za-z_][A-Za-z0-9_ ]*?\**\s*\b([a-z0-9_]+)\s*\(", text)
    return sorted(set(names))


def test_headers_declare_the_boundary():
    names = declared_symbols()
    for n in ("fp8_quant_act", "fp8_quant_weight_blocks", "fp8_blockscaled_gemm",
              "fp8_blockscaled_gemm_fused", "fp8_blockscaled_gemm_workspace_size",
              "bf16_gemm_ref", "bf16_gemm_ref_workspace_size", "fp8bs_status_string",
              "fp8bs_workspace_status", "fp8bs_split_plan", "fp8bs_gemm_schedule", "fp8bs_fused_route",
              "fp8_blockscaled_gemm_fused_greedy", "fp8_blockscaled_gemm_fused_noalloc",
              "fp8bs_testhook_kernel_runs", "fp8bs_testhook_gemm_fused_sms", "fp8bs_testhook_gemm_stall",
              "fp8_mx_quant_weights", "fp8_mx_quant_act", "fp8_mx_gemm", "fp8_mx_gemm_workspace_size"):
        assert n in names


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert names
    raw = ctypes.CDLL(fb.LIB_PATH)
    for n in names:
        assert hasattr(raw, n), n


def test_status_strings(L):
    seen = set()
    for code in range(8):
        s = fb.status_string(code)
        assert s and s not in seen
        seen.add(s)
    assert fb.status_string(99) == "unknown status"


P = ctypes.c_void_p
A16 = P(0x10000)      # 16-byte aligned fake address: never dereferenced
A1 = P(0x10001)       # misaligned fake address
NUL = P(0)
S = P(0)              # default stream


def test_quant_act_validation(L):
    assert L.fp8_quant_act(NUL, 8, 512, 512, A16, A16, 0, S) == INVALID
    assert L.fp8_quant_act(A16, 0, 512, 512, A16, A16, 0, S) == INVALID
    assert L.fp8_quant_act(A16, 8, 512, 256, A16, A16, 0, S) == INVALID        # ldx < K
    assert L.fp8_quant_act(A16, 8, 512, 512, A16, A16, 2, S) == INVALID        # unknown flag
    assert L.fp8_quant_act(A16, 8, 500, 512, A16, A16, 0, S) == SHAPE          # K % 128
    assert L.fp8_quant_act(A1, 8, 512, 512, A16, A16, 0, S) == MISALIGNED
    assert L.fp8_quant_act(A16, 8, 512, 516, A16, A16, 0, S) == MISALIGNED     # ldx % 8


def test_quant_weight_validation(L):
    assert L.fp8_quant_weight_blocks(NUL, 0, 256, 512, A16, A16, S) == INVALID
    assert L.fp8_quant_weight_blocks(A16, 7, 256, 512, A16, A16, S) == INVALID
    assert L.fp8_quant_weight_blocks(A16, 0, 0, 512, A16, A16, S) == INVALID
    assert L.fp8_quant_weight_blocks(A16, 0, 256, 200, A16, A16, S) == SHAPE
    assert L.fp8_quant_weight_blocks(A16, 0, 256, 512, A1, A16, S) == MISALIGNED


def test_gemm_validation(L):
    g = L.fp8_blockscaled_gemm
    assert g(NUL, A16, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, S) == INVALID
    assert g(A16, A16, A16, A16, A16, 0, 256, 512, A16, 1 << 20, 0, S) == INVALID
    assert g(A16, A16, A16, A16, A16, 513, 256, 512, A16, 1 << 20, 0, S) == SHAPE     # M above 512
    assert g(A16, A16, A16, A16, A16, 8, 256, 520, A16, 1 << 20, 0, S) == SHAPE
    assert g(A16, A16, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 4, S) == INVALID
    assert g(A1, A16, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, S) == MISALIGNED
    assert g(A16, A16, A16, A16, A16, 8, 256, 512, P(0x10010), 1 << 20, 0, S) == MISALIGNED  # workspace % 256
    f = L.fp8_blockscaled_gemm_fused
    assert f(A16, 100, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, S) == INVALID           # ldx < K
    assert f(A16, 516, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, S) == MISALIGNED        # ldx % 8
    gr = L.fp8_blockscaled_gemm_fused_greedy
    assert gr(A16, 512, A16, A16, A16, 65, 256, 512, A16, NUL, A16, 1 << 20, 0, S) == SHAPE  # greedy: M <= 64
    assert gr(A16, 512, A16, A16, A16, 8, 256, 512, NUL, NUL, A16, 1 << 20, 0, S) == INVALID  # token required
    b = L.bf16_gemm_ref
    assert b(A16, A16, A16, 8, 256, 96, A16, 1 << 20, 0, S) == SHAPE                         # K % 64
    assert b(A16, A16, A16, 64, 256, 128, A16, 1 << 20, 0, S) != SHAPE
    sz = ctypes.c_size_t(5)
    assert L.fp8_blockscaled_gemm_workspace_size(8, 256, 100, ctypes.byref(sz)) == SHAPE and sz.value == 0


def test_mx_validation(L):
    q = L.fp8_mx_quant_weights
    assert q(NUL, 0, 256, 512, A16, A16, S) == INVALID
    assert q(A16, 3, 256, 512, A16, A16, S) == INVALID
    assert q(A16, 0, 256, 160, A16, A16, S) == SHAPE                      # K % 128
    assert q(A16, 0, 256, 512, A16, P(0x10008), S) == MISALIGNED          # atoms 16-byte aligned
    a = L.fp8_mx_quant_act
    assert a(A16, 513, 512, 512, A16, A16, 0, S) == SHAPE                 # at most 512 tokens
    assert a(A16, 8, 512, 256, A16, A16, 0, S) == INVALID                 # ldx < K
    assert a(A16, 8, 512, 512, A16, A16, 2, S) == INVALID                 # unknown flag
    assert a(A16, 8, 512, 512, A1, A16, 0, S) == MISALIGNED
    g = L.fp8_mx_gemm
    assert g(A16, A16, A16, A16, A16, 513, 256, 512, A16, 1 << 20, 0, S) == SHAPE
    assert g(A16, A16, A16, A16, A16, 8, 256, 384 + 64, A16, 1 << 20, 0, S) == SHAPE
    assert g(A16, A16, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 2, S) == INVALID  # tiled is implied
    assert g(A16, P(0x10004), A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, S) == MISALIGNED
    assert g(NUL, A16, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, S) == INVALID
    sz = ctypes.c_size_t(3)
    assert L.fp8_mx_gemm_workspace_size(513, 256, 512, ctypes.byref(sz)) == SHAPE and sz.value == 0


def test_split_plan_partitions_units(L):
    for (N, K, bf16, sms) in ((256, 512, 0, 152), (5120, 5120, 0, 152), (248320, 5120, 0, 152),
                              (34816, 5120, 0, 148), (5120, 17408, 0, 160), (300, 640, 1, 152), (128, 128, 0, 1)):
        ctas, units, _, _ = fb.split_plan(N, K, bool(bf16), sms)
        kg = K // (64 if bf16 else 128)
        assert units == ((N + 127) // 128) * kg
        assert ctas == min(units, sms)
        prev_end, sizes = 0, []
        partial_tiles = {}
        for c in range(ctas):
            _, _, b, e = fb.split_plan(N, K, bool(bf16), sms, c)
            assert b == prev_end and e > b
            sizes.append(e - b)
            prev_end = e
            tiles = set(range(b // kg, (e - 1) // kg + 1))
            owned = [t for t in tiles if b <= t * kg and (t + 1) * kg <= e]
            partial_tiles[c] = sorted(tiles - set(owned))
        assert prev_end == units
        assert max(sizes) - min(sizes) <= 1
        # the reduction gives every CTA two partial slots: it may never need more
        assert all(len(v) <= 2 for v in partial_tiles.values())
        # each split tile is shared by CTAs with consecutive indices
        for t in range((N + 127) // 128):
            contrib = [c for c, v in partial_tiles.items() if t in v]
            if contrib:
                assert contrib == list(range(contrib[0], contrib[-1] + 1))


def test_gemm_schedule_policy(L):
    """The schedule for M tokens: up to 64 tokens one token tile and K split
    over every SM; above, whole (token tile, weight tile) pairs per CTA when
    they fit in one wave and leave at most a 16/kg fraction of the SMs idle,
    stream-K over 128-token pairs otherwise (always when the 128-token pairs
    cover every SM)."""
    def tpad(M):
        return 16 if M <= 16 else 32 if M <= 32 else 48 if M <= 48 else 64
    for sms in (152, 148, 160):
        for M in (1, 8, 16, 17, 33, 64, 65, 100, 128, 129, 256, 300, 384, 512):
            for N, K in ((5120, 5120), (7168, 5120), (34816, 5120), (5120, 17408), (640, 1024), (300, 256),
                         (128, 128)):
                s = fb.gemm_schedule(M, N, K, sms)
                ntiles, kg = (N + 127) // 128, K // 128
                assert s["units"] == s["token_tiles"] * ntiles * kg
                assert s["token_tiles"] == (M + s["npad"] - 1) // s["npad"]
                if M <= 64:
                    assert (s["npad"], s["token_tiles"], s["split"]) == (tpad(M), 1, True)
                    assert s["ctas"] == min(s["units"], sms)
                elif not s["split"]:
                    pairs = s["ctas"]
                    assert s["npad"] in (32, 64, 128)
                    assert pairs == s["token_tiles"] * ntiles and pairs <= sms
                    assert pairs * (kg + 16) >= sms * kg, "too many idle SMs for an unsplit K"
                    assert ntiles * ((M + 127) // 128) < sms, "pairs cover the SMs: stream-K expected"
                    # the widest token tile that qualifies
                    for wider in (128, 64):
                        if wider > s["npad"]:
                            p2 = ntiles * ((M + wider - 1) // wider)
                            assert not (p2 <= sms and p2 * (kg + 16) >= sms * kg)
                else:
                    assert s["npad"] == 128 and s["ctas"] == min(s["units"], sms)
    sched = lambda M, N, K: fb.gemm_schedule(M, N, K, 152)
    assert sched(512, 5120, 5120) == dict(npad=128, token_tiles=4, ctas=152, units=6400, split=True)
    # 80 pairs of a short K, 80 of a long K: both stream-K
    assert sched(256, 5120, 5120) == dict(npad=128, token_tiles=2, ctas=152, units=3200, split=True)
    assert sched(128, 5120, 17408) == dict(npad=128, token_tiles=1, ctas=152, units=5440, split=True)
    # 112 pairs of a 40-block K: one CTA per pair
    assert sched(256, 7168, 5120) == dict(npad=128, token_tiles=2, ctas=112, units=4480, split=False)
    assert sched(128, 7168, 5120) == dict(npad=64, token_tiles=2, ctas=112, units=4480, split=False)
    assert sched(8, 5120, 5120) == dict(npad=16, token_tiles=1, ctas=152, units=1600, split=True)
    with pytest.raises(fb.Fp8bsError):
        fb.gemm_schedule(513, 5120, 5120, 152)


def test_fused_route_policy(L):
    """By default the fused entry point runs the cast kernel first; with
    FP8BS_FLAG_PROLOGUE_CAST it casts in the GEMM prologue when every CTA has
    at most 16 (K block, token) rows to cast.  The decision is a pure
    function of (M, N, K, SM count, flags)."""
    PRO = fb.FLAG_PROLOGUE_CAST
    for M, N, K in ((8, 256, 512), (1, 5120, 5120), (2, 2048, 1024), (16, 640, 2048), (64, 5120, 5120)):
        assert fb.fused_route(M, N, K, 152) == "separate"
        assert fb.fused_route(M, N, K, 152, flags=fb.FLAG_OVERLAP_PREV | fb.FLAG_WEIGHTS_TILED) == "separate"
    with pytest.raises(fb.Fp8bsError):
        fb.fused_route(8, 256, 512, 152, flags=8)          # not a flag of the fused entry points
    r = lambda M, N, K, sms=152: fb.fused_route(M, N, K, sms, flags=PRO)
    # the tiny workload: 8 units on 8 CTAs, one K block of 8 rows each
    assert r(8, 256, 512) == "prologue"
    # square layer: ~11 K blocks per CTA; 11 rows at M = 1, 88 at M = 8
    assert r(1, 5120, 5120) == "prologue"
    assert r(8, 5120, 5120) == "separate"
    assert r(2, 2048, 1024) == "prologue" and r(16, 640, 2048) == "prologue"
    for M, N, K in ((33, 1000, 3072), (64, 256, 512), (64, 5120, 5120), (16, 2048, 17408), (8, 248320, 5120),
                    (65, 5120, 5120), (512, 5120, 5120)):
        assert r(M, N, K) == "separate", (M, N, K)
    # the rule itself, over shapes and SM counts
    for sms in (37, 76, 148, 152):
        for M in (1, 2, 3, 8, 16, 17, 64):
            for N, K in ((256, 512), (640, 2048), (5120, 5120), (1000, 3072), (128, 128)):
                s = fb.gemm_schedule(M, N, K, sms)
                kg = K // 128
                per_cta = -(-s["units"] // s["ctas"])
                rows = min(per_cta, kg) * M
                cache = min(per_cta, kg) * (s["npad"] * 128 + s["npad"] * 4)
                want = "prologue" if rows <= 16 and cache <= 96 * 1024 else "separate"
                assert r(M, N, K, sms) == want, (M, N, K, sms)
    with pytest.raises(fb.Fp8bsError):
        fb.fused_route(8, 256, 500, 152)


def test_testing_hooks_validate_on_host(L):
    out = (ctypes.c_ulonglong * 4)()
    assert L.fp8bs_testhook_kernel_runs(-1, 4, out) == INVALID
    assert L.fp8bs_testhook_kernel_runs(126, 4, out) == INVALID
    assert L.fp8bs_testhook_kernel_runs(0, 4, None) == INVALID
    sz = ctypes.c_size_t(7)
    assert L.fp8bs_testhook_workspace_size_sms(8, 256, 512, 0, ctypes.byref(sz)) == INVALID
    assert L.fp8bs_testhook_workspace_size_sms(8, 256, 500, 37, ctypes.byref(sz)) == SHAPE and sz.value == 0
    assert L.fp8bs_testhook_workspace_size_sms(8, 5120, 5120, 37, ctypes.byref(sz)) == OK
    assert sz.value > L_ws(8, 5120, 5120, 1) and sz.value < L_ws(8, 5120, 5120, 152)
    f = L.fp8bs_testhook_gemm_fused_sms
    assert f(A16, 512, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, 0, S) == INVALID       # SM count
    assert f(A16, 512, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, 5000, S) == INVALID    # SM count
    assert f(A1, 512, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, 37, S) == MISALIGNED


def test_debug_library_builds_and_exports_everything(L):
    """The FP8BS_DEBUG build links, reports itself as such, and exports the
    same symbols; the normal build refuses the debug-only hook."""
    fbuild.build(variants=("release", "debug"))
    D = fb._load(fb.DEBUG_LIB_PATH)
    assert D.fp8bs_testhook_debug_build() == 1 and L.fp8bs_testhook_debug_build() == 0
    raw = ctypes.CDLL(fb.DEBUG_LIB_PATH)
    for n in declared_symbols():
        assert hasattr(raw, n), n
    assert L.fp8bs_testhook_debug_bad_tile(A16, A16, A16, A16, A16, 8, 256, 512, A16, 1 << 20, 0, 1000, S) == INVALID
    assert D.fp8bs_testhook_debug_bad_tile(A16, A16, A16, A16, A16, 8, 256, 512, A16, 1 << 20, -1, 1000, S) == INVALID


def L_ws(M, N, K, sms):
    sz = ctypes.c_size_t(0)
    assert fb.lib().fp8bs_testhook_workspace_size_sms(M, N, K, sms, ctypes.byref(sz)) == OK
    return sz.value


def test_c_caller_compiles_and_runs(L, tmp_path):
    """A plain C program, compiled with the system C compiler against the
    header and linked with the library, runs the host-side calls."""
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    exe = str(tmp_path / "abi_from_c")
    libdir = os.path.dirname(fb.LIB_PATH)
    src = os.path.join(ROOT, "tests", "c", "abi_from_c.c")
    r = subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"), src, "-o", exe,
                        "-L", libdir, "-lfp8bs", "-Wl,-rpath," + libdir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    r = subprocess.run([exe], capture_output=True, text=True, timeout=60)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stdout + r.stderr
