"""Reference rotary position embedding (fp64), for the fused RoPE entry points.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``).  Written from the TensorSharp
"Mistral 3" page, section 3 "Forward graph" and section 4.2 "RoPE - GPT-J style with YaRN":

* the frequency table has one entry per rotated pair, ``base^(-2i / rope_dim)`` (the standard
  RoPE schedule, built once at load time), YaRN-corrected when a scaling is set: with
  ``r = orig_ctx / (2 pi / f)`` (turns over the original context), pairs with
  ``r > beta_fast`` keep f, pairs with ``r < beta_slow`` take ``f / scale``, and in between
  f mixes linearly in r (the page elides this ramp; the reading is the linear ramp of the
  YaRN method, weight of ``f / scale`` = ``(beta_fast - r) / (beta_fast - beta_slow)``);
  the table is stored in fp32 (reading: the model's table is fp32);
* GPT-J pairing: elements ``(x[2i], x[2i+1])`` rotate together by ``pos * f_i``;
* the query is then scaled by ``1 + beta * ln(1 + floor(pos / orig_ctx))`` when
  ``orig_ctx > 0``.
"""
from __future__ import annotations

import math

import numpy as np


def yarn_freqs(rope_dim: int, base: float, scale: float = 1.0, orig_ctx: int = 0,
               beta_fast: float = 32.0, beta_slow: float = 1.0) -> np.ndarray:
    out = np.empty(rope_dim // 2, dtype=np.float32)
    yarn = scale != 1.0 and orig_ctx > 0
    for i in range(rope_dim // 2):
        f = float(base) ** (-2.0 * i / rope_dim)
        if yarn:
            r = orig_ctx * f / (2.0 * math.pi)
            if r < beta_slow:
                f = f / scale
            elif r <= beta_fast:
                g = (beta_fast - r) / (beta_fast - beta_slow)
                f = f * (1.0 - g) + (f / scale) * g
        out[i] = f
    return out


def apply_rope(x: np.ndarray, positions, freqs: np.ndarray, rope_dim: int) -> np.ndarray:
    """Rotate rows ``x[t][h][:]`` (any float dtype, returned in fp64) at ``positions[t]``."""
    y = np.array(x, dtype=np.float64, copy=True)
    pos = np.asarray(positions, dtype=np.float64)
    for i in range(rope_dim // 2):
        ang = pos * float(freqs[i])
        c, s = np.cos(ang)[:, None], np.sin(ang)[:, None]
        a, b = y[:, :, 2 * i].copy(), y[:, :, 2 * i + 1].copy()
        y[:, :, 2 * i] = a * c - b * s
        y[:, :, 2 * i + 1] = a * s + b * c
    return y


def q_scale(positions, beta: float, orig_ctx: int) -> np.ndarray:
    pos = np.asarray(positions, dtype=np.int64)
    if orig_ctx <= 0:
        return np.ones(pos.shape, dtype=np.float64)
    return 1.0 + beta * np.log1p((pos // orig_ctx).astype(np.float64))
