"""Float64 oracle for the QKV bias and YaRN rotary position encoding applied to
q, k and v before sink attention.

TEST INFRASTRUCTURE ONLY, like the rest of ``oracle/``: only ``tests/``,
``__graft_entry__.smoke()`` and the CPU legs of ``bench.py`` call it; it
shares no code with the CUDA library.

Source: Perplexity, "GPT-OSS on day 0", model overview: the attention uses
YaRN positional encoding (as DeepSeek-V3 does) and the QKV projections carry
biases (as in Qwen 2).  The pages give no formula for either, so this module
follows the published definitions:

  * Rotary position encoding (RoFormer, Su et al.): the head dimension is
    split into D/2 planes, plane i rotated by the angle  position * theta_i.
    Reading taken: plane i pairs dims i and i + D/2 (the half-split layout).
  * YaRN (Peng et al., "YaRN: Efficient Context Window Extension of Large
    Language Models", the "NTK-by-parts" interpolation and the attention
    temperature): with base frequencies theta_i = base^(-2i/D), wavelength
    lambda_i = 2 pi / theta_i, ratio r_i = L_orig / lambda_i, ramp
    gamma(r) = 0 for r < alpha, 1 for r > beta, (r - alpha) / (beta - alpha)
    between, the frequency becomes
        theta'_i = (1 - gamma(r_i)) * theta_i / s + gamma(r_i) * theta_i
    (s = the context extension factor), and the logits are scaled through
    q and k each multiplied by  0.1 ln(s) + 1  (1 when s <= 1).
    alpha = beta_slow, beta = beta_fast.  Reading taken: the ramp is linear
    in r as the paper writes it (some implementations ramp linearly over the
    dimension index between the same two boundary planes instead).
  * The biases are added to the projections' outputs before the rotation;
    v gets its bias and no rotation.

Pins (tests/test_oracle_rope_pins.py): identity at position 0, norm
preservation, relative-position invariance of q.k, composition of rotations,
the plane pairing on one-hot inputs, YaRN's closed-form limits (unchanged
high-frequency planes, planes divided by s at low frequency, the exact
midpoint of the ramp), the temperature formula, and linearity (which fixes
the order bias-then-rotate).
"""
from __future__ import annotations

import math

import numpy as np

from .sink_attention import _as_f64, _as_int

__all__ = ["yarn_inv_freq", "rope", "qkv_bias_rope"]


def yarn_inv_freq(head_dim: int, base: float, factor: float, original_max_position: int,
                  beta_fast: float, beta_slow: float):
    """YaRN per-plane frequencies theta'_i (float64 [D/2]) and the factor that
    multiplies q and k (0.1 ln s + 1).  factor <= 1 gives plain RoPE."""
    half = head_dim // 2
    i = np.arange(half, dtype=np.float64)
    theta = base ** (-2.0 * i / head_dim)
    if factor <= 1.0:
        return theta, 1.0
    r = original_max_position * theta / (2.0 * math.pi)  # L_orig / wavelength
    gamma = np.clip((r - beta_slow) / (beta_fast - beta_slow), 0.0, 1.0)
    theta_new = (1.0 - gamma) * theta / factor + gamma * theta
    return theta_new, 0.1 * math.log(factor) + 1.0


def rope(x, positions, inv_freq, attn_factor: float = 1.0):
    """Rotate each head vector of x [T, H, D] (float64) by its token's
    position: plane i = (dim i, dim i + D/2), angle positions[t] * inv_freq[i];
    the result is multiplied by attn_factor."""
    x = _as_f64(x)
    pos = _as_int(positions).astype(np.float64)
    f = _as_f64(inv_freq)
    half = x.shape[-1] // 2
    ang = pos[:, None] * f[None, :]  # [T, D/2]
    c = np.cos(ang)[:, None, :]
    s = np.sin(ang)[:, None, :]
    x1, x2 = x[..., :half], x[..., half:]
    out = np.concatenate([x1 * c - x2 * s, x2 * c + x1 * s], axis=-1)
    return out * attn_factor


def qkv_bias_rope(q, k, v, q_bias, k_bias, v_bias, positions, inv_freq, attn_factor: float = 1.0):
    """(rope(q + q_bias), rope(k + k_bias), v + v_bias) in float64; a bias of
    None is zero.  q [T, Hq, D], k and v [T, Hkv, D], biases [H, D]."""
    q, k, v = _as_f64(q), _as_f64(k), _as_f64(v)
    if q_bias is not None:
        q = q + _as_f64(q_bias)[None]
    if k_bias is not None:
        k = k + _as_f64(k_bias)[None]
    if v_bias is not None:
        v = v + _as_f64(v_bias)[None]
    return rope(q, positions, inv_freq, attn_factor), rope(k, positions, inv_freq, attn_factor), v
