"""Shared helpers for the GPU parity tests: move seeded inputs between torch
and the oracle's numpy views, and the element-wise acceptance check.

Acceptance for Y (per output element), the bound stated for the layer:
    |y_gpu - y_oracle| <= 4e-3 * sum_k |a_k * w_k| + 1e-6
where y_oracle is the oracle's fp64 value and the sum is over the dequantised
operands.  The bound covers the one bf16 rounding of the output (at most
2^-8 relative to |y| <= sum|a w|) plus fp32 accumulation.
"""
import numpy as np
import torch

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
