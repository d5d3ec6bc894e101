"""Parity comparison between the CUDA path and the float64 oracle.

Tolerances (bf16 inputs, fp32 accumulation), element by element:
  * fp32 output: |gpu - oracle| <= 1e-2 everywhere and mean |gpu - oracle| <= 1e-3;
  * bf16 output: the output itself is rounded to bf16, whose spacing exceeds
    1e-2 for |x| >= 2; each element may therefore differ by max(1e-2, one bf16
    spacing at the oracle value), and the mean bound 1e-3 still holds.
Where the oracle output is -inf/inf (lse of an empty row), the GPU must agree
exactly.
"""
import math

import numpy as np
import torch

MAX_ABS = 1e-2
MEAN_ABS = 1e-3


def to_f64(x) -> np.ndarray:
    if isinstance(x, torch.Tensor):
        return x.detach().float().cpu().numpy().astype(np.float64)
    return np.asarray(x, dtype=np.float64)


def bf16_spacing(x: np.ndarray) -> np.ndarray:
    ax = np.abs(x)
    e = np.floor(np.log2(np.where(ax > 0, ax, 1.0)))
    return np.where(ax > 0, np.exp2(e - 7), 0.0)


def errors(got, want):
    g, w = to_f64(got), to_f64(want)
    assert g.shape == w.shape, (g.shape, w.shape)
    return np.abs(g - w), g, w


def assert_parity(got, want, bf16_output: bool = False, what: str = "out"):
    g, w = to_f64(got), to_f64(want)
    assert g.shape == w.shape, (what, g.shape, w.shape)
    inf_w = ~np.isfinite(w)
    if inf_w.any():
        assert np.array_equal(g[inf_w], w[inf_w]), f"{what}: non-finite oracle entries differ"
    fin = ~inf_w
    assert np.all(np.isfinite(g[fin])), f"{what}: GPU produced non-finite values"
    err = np.abs(g[fin] - w[fin])
    if err.size == 0:
        return 0.0, 0.0
    allowed = np.full_like(err, MAX_ABS)
    if bf16_output:
        allowed = np.maximum(allowed, bf16_spacing(w[fin]))
    worst = int(np.argmax(err - allowed))
    assert np.all(err <= allowed), (
        f"{what}: max abs err {err.max():.3e} (worst over budget: got {g[fin].ravel()[worst]:.6f} "
        f"want {w[fin].ravel()[worst]:.6f})")
    assert err.mean() <= MEAN_ABS, f"{what}: mean abs err {err.mean():.3e}"
    return float(err.max()), float(err.mean())


# The kernels normalise by the sum of the bf16-rounded softmax weights that
# the value product uses (so out and lse stay mutually consistent).  Each
# weight carries a relative rounding error of at most 2^-8, hence so does the
# sum, and |lse - lse_exact| <= log(1 + 2^-8) < 2^-8; fp32 adds ~1e-6.
LSE_ATOL = 2.0 ** -8 + 1e-5


def lse_close(got, want, atol=LSE_ATOL):
    """lse (natural log of the normaliser, sink included) within LSE_ATOL."""
    g, w = to_f64(got), to_f64(want)
    inf_w = ~np.isfinite(w)
    assert np.array_equal(np.isfinite(g), ~inf_w)
    if (~inf_w).any():
        err = np.abs(g[~inf_w] - w[~inf_w])
        assert err.max() <= atol, f"lse max abs err {err.max():.3e}"
