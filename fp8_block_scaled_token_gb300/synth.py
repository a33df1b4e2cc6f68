"""Seeded synthetic inputs shaped like the decode-time FP8 linear layers.

This module holds only random-number recipes.  It contains none of the
layer's arithmetic (no scaling, no FP8 encoding, no product), so both the CUDA
library's tests and the CPU oracle can draw the same raw inputs from it
without sharing any of the method.

Recipe (the pages measure on real Qwen weights and live decode traffic, which
these stand in for):

* activations X: fp32 N(0, 1), rounded to bf16 (round-to-nearest-even by
  torch's cast), shape [M, K];
* weights W: fp32 N(0, 0.02^2), shape [N, K];
* optional outliers: an independent Bernoulli(p) mask drawn from its own
  generator (seed + 7919) multiplies the selected entries by a constant,
  keeping the sign (1% x8 for weights, 0.1% x20 for activations in the
  MLP-shaped workload).

Generators are torch's (CPU: Mersenne Twister; CUDA: Philox).  The same
(seed, shape, device) always gives the same tensor; CPU and CUDA draws differ
from each other, so a test that compares the two sides draws once and copies.
"""
import torch

OUTLIER_SEED_OFFSET = 7919


def _gen(device, seed):
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _outliers(t, seed, p, mult):
    if p <= 0.0:
        return t
    g = _gen(t.device, seed + OUTLIER_SEED_OFFSET)
    mask = torch.rand(t.shape, generator=g, device=t.device) < p
    return torch.where(mask, t * mult, t)


def activations(M, K, seed, outlier_p=0.0, outlier_mult=20.0, device="cpu"):
    """bf16 [M, K]: N(0,1) draws rounded to bf16, optional outliers."""
    g = _gen(device, seed)
    x = torch.randn((M, K), generator=g, device=device, dtype=torch.float32)
    x = _outliers(x, seed, outlier_p, outlier_mult)
    return x.to(torch.bfloat16)


def weights(N, K, seed, std=0.02, outlier_p=0.0, outlier_mult=8.0, device="cpu"):
    """fp32 [N, K]: N(0, std^2) draws, optional outliers."""
    g = _gen(device, seed)
    w = torch.randn((N, K), generator=g, device=device, dtype=torch.float32)
    w.mul_(std)
    return _outliers(w, seed, outlier_p, outlier_mult)


# The workloads (shapes and distributions) the tests and the benchmark use.
WORKLOADS = {
    "tiny": dict(M=8, N=256, K=512, seed=0),
    "square_decode": dict(M=8, N=5120, K=5120, seed=1),
    "mlp_up": dict(M=8, N=34816, K=5120, seed=2, w_outlier_p=0.01, x_outlier_p=0.001),
    "mlp_down": dict(M=8, N=5120, K=17408, seed=3, w_outlier_p=0.01, x_outlier_p=0.001),
    "vocab": dict(M=8, N=248320, K=5120, seed=4),
    "attn_7168": dict(M=8, N=7168, K=5120, seed=5),
}


def workload_inputs(name, device="cpu", M=None):
    """(X bf16 [M,K], W fp32 [N,K]) for a named workload."""
    cfg = dict(WORKLOADS[name])
    m = cfg["M"] if M is None else M
    x = activations(m, cfg["K"], cfg["seed"], outlier_p=cfg.get("x_outlier_p", 0.0),
                    device=device)
    w = weights(cfg["N"], cfg["K"], cfg["seed"] + 1000, outlier_p=cfg.get("w_outlier_p", 0.0),
                device=device)
    return x, w
