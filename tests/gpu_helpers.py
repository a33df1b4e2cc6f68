"""Shared helpers for the GPU parity tests: move seeded inputs between torch
and the oracle's numpy views, and the element-wise acceptance check.

Acceptance for Y (per output element), the bound stated for the layer:
    |y_gpu - y_oracle| <= 4e-3 * sum_k |a_k * w_k| + 1e-6
where y_oracle is the oracle's fp64 value and the sum is over the dequantised
operands.  The bound covers the one bf16 rounding of the output (at most
2^-8 relative to |y| <= sum|a w|) plus fp32 accumulation.
"""
import ctypes

import numpy as np
import torch

import fp8_block_scaled_token_gb300 as fb
import oracle

REL_TOL = 4e-3
ABS_TOL = 1e-6


def bits16(t):
    """bf16 tensor (any device) -> uint16 numpy bit patterns."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


def y_values(y):
    """bf16 Y tensor -> float64 numpy."""
    return y.detach().cpu().to(torch.float64).numpy()


def check_y(y_gpu, y_ref, bound, what=""):
    yg = y_values(y_gpu) if isinstance(y_gpu, torch.Tensor) else np.asarray(y_gpu, dtype=np.float64)
    err = np.abs(yg - y_ref)
    lim = REL_TOL * bound + ABS_TOL
    bad = err > lim
    assert not bad.any(), "%s: %d of %d outside tolerance; worst excess %g at %s" % (
        what, int(bad.sum()), bad.size, float((err - lim).max()), np.unravel_index(np.argmax(err - lim), err.shape))
    assert np.all(np.isfinite(yg))


def oracle_layer(x_bf16, w_f32, cols=None):
    """The oracle's full layer from raw torch inputs (CPU copies)."""
    return oracle.default().linear_fp8(bits16(x_bf16), w_f32.detach().cpu().numpy(), cols=cols)


# ------------------------------------------------------------ "did it run"
RUNS_SLOTS = 128
RUNS_QUANT_ACT, RUNS_QUANT_WEIGHT, RUNS_PACK_BF16 = 0, 1, 2
MODE_FP8, MODE_FUSED, MODE_BF16 = 0, 1, 2


def runs_gemm(mode, npad, greedy=False):
    """Launch-counter slot of a GEMM kernel instantiation (the slot rule of
    include/fp8bs_testing.h)."""
    idx = npad // 16 - 1 if npad <= 64 else (4 if npad == 128 else 5)
    return 8 + mode * 16 + idx * 2 + (1 if greedy else 0)


def kernel_runs():
    """The library's per-device launch counters (synchronises the device)."""
    out = (ctypes.c_ulonglong * RUNS_SLOTS)()
    rc = fb.lib().fp8bs_testhook_kernel_runs(0, RUNS_SLOTS, out)
    assert rc == 0, fb.status_string(rc)
    return np.array(list(out), dtype=np.int64)


class Ran:
    """Counts the library's kernel launches inside a `with` block:
    ``with Ran() as r: ...`` then ``r.count(slot)``, ``r.launched()``."""

    def __enter__(self):
        self.before = kernel_runs()
        return self

    def __exit__(self, *exc):
        self.after = kernel_runs()
        return False

    def count(self, slot):
        return int(self.after[slot] - self.before[slot])

    def launched(self):
        d = self.after - self.before
        return {int(i): int(d[i]) for i in np.nonzero(d)[0]}
