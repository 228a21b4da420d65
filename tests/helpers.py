"""Shared helpers for the GPU parity tests: seeded inputs (from the package's
input module, which holds no attention arithmetic), tolerance checks, and
row sampling for full-size shapes."""
import math

import numpy as np
import torch

from tiled_attention_02_gb300.inputs import make_bias, make_chain, make_qkv, to_oracle

# Tolerances for bf16 O, fp32 LSE, the backward gradients and the emitted
# fp32 logits.
O_MAX_ABS = 1.6e-2
O_MEAN_ABS = 2e-3
LSE_ABS = 1e-3
GRAD_MAX_ABS = 3e-2
LOGIT_ABS = 1e-3


def sample_rows(B, H, N, n, seed=0, block=128):
    """Flat row indices (b*H + h)*N + i: tile edges, the first and last row
    of each sampled head, and random rows."""
    rng = np.random.default_rng(seed)
    total = B * H * N
    picks = {0, total - 1}
    for _ in range(max(1, n // 8)):
        bh = int(rng.integers(0, B * H))
        t = int(rng.integers(0, max(1, (N + block - 1) // block)))
        for i in (t * block, t * block + block - 1, t * block + block // 2):
            if i < N:
                picks.add(bh * N + i)
        picks.add(bh * N)
        picks.add(bh * N + N - 1)
    while len(picks) < min(n, total):
        picks.add(int(rng.integers(0, total)))
    return np.array(sorted(picks), dtype=np.int64)


def check_o(o_gpu, o_ref, what=""):
    """o_gpu: bf16 tensor (any shape matching o_ref's size); o_ref: fp64 array."""
    got = o_gpu.detach().float().cpu().numpy().reshape(o_ref.shape).astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite output"
    err = np.abs(got - o_ref)
    mx, mean = float(err.max()), float(err.mean())
    assert mx <= O_MAX_ABS, f"{what}: O max-abs {mx:.3e} > {O_MAX_ABS}"
    assert mean <= O_MEAN_ABS, f"{what}: O mean-abs {mean:.3e} > {O_MEAN_ABS}"
    return mx, mean


def check_lse(lse_gpu, lse_ref, what=""):
    got = lse_gpu.detach().cpu().numpy().reshape(lse_ref.shape).astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite LSE"
    mx = float(np.abs(got - lse_ref).max())
    assert mx <= LSE_ABS, f"{what}: LSE max-abs {mx:.3e} > {LSE_ABS}"
    return mx


def check_logits(lg_gpu, lg_ref, what=""):
    """Compare emitted logits where the reference is defined (not NaN)."""
    got = lg_gpu.detach().cpu().numpy().reshape(lg_ref.shape).astype(np.float64)
    keep = ~np.isnan(lg_ref)
    assert np.isfinite(got[keep]).all(), f"{what}: non-finite emitted logits"
    mx = float(np.abs(got[keep] - lg_ref[keep]).max())
    assert mx <= LOGIT_ABS, f"{what}: logits max-abs {mx:.3e} > {LOGIT_ABS}"
    return mx


def check_grad(g_gpu, g_ref, what=""):
    got = g_gpu.detach().float().cpu().numpy().reshape(g_ref.shape).astype(np.float64)
    assert np.isfinite(got).all(), f"{what}: non-finite gradient"
    mx = float(np.abs(got - g_ref).max())
    assert mx <= GRAD_MAX_ABS, f"{what}: max-abs {mx:.3e} > {GRAD_MAX_ABS} (max |ref| {np.abs(g_ref).max():.3g})"
    return mx


__all__ = ["make_bias", "make_chain", "make_qkv", "to_oracle", "sample_rows", "check_o",
           "check_lse", "check_logits", "check_grad", "math", "torch", "np"]
