"""CPU fp64 oracle of the fused in-place QK-norm + RoPE step.

TEST INFRASTRUCTURE.  Only the tests, the package smoke check and the
benchmark's CPU-baseline leg may import this module; the library's own code
never does, and it shares no code with the CUDA path.

What it computes (sources, by page and section):

* Sarvam blog = NVIDIA technical blog "How NVIDIA extreme hardware-software
  co-design delivered a large inference boost for Sarvam AI's sovereign
  models", Table 1 row "QK Norm + RoPE" (414 -> 54 us per layer) and the
  paragraph on fused positional embedding: the query-key normalisation and
  the rotary position embedding run as one in-place kernel, one pass over
  the data instead of two reads and writes.
* Sarvam summary = peacm.com news/791474, section 3.1: the fused kernel's
  outline takes q, k and a precomputed frequency table (freq_cis) and does
  the normalisation and the rotary embedding in one memory pass.

Readings where the pages are silent (the plainest reading in each case):
  QK-norm is an RMSNorm over each head's vector (the summary's "L2
  normalisation" up to the learnt per-channel weight gamma, which absorbs
  the sqrt(head_dim) factor), separate gammas for q and k, eps = 1e-6 inside
  the root; RoPE rotates the two halves of the normalised vector ("rotate
  half"): for i < D/2, (a, b) = (y_i, y_{i+D/2}) becomes
  (a cos - b sin, b cos + a sin) with cos, sin taken from the table row of
  the token's position; outputs are rounded to bf16 in place.

Every function computes in float64.
"""
from __future__ import annotations

import numpy as np


def rms_norm(x: np.ndarray, gamma: np.ndarray, eps: float) -> np.ndarray:
    """y = x / sqrt(mean(x^2) + eps) * gamma over the last axis."""
    x = np.asarray(x, dtype=np.float64)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps) * np.asarray(gamma, dtype=np.float64)


def rope_rotate_half(y: np.ndarray, cos: np.ndarray, sin: np.ndarray) -> np.ndarray:
    """Rotate-half RoPE: y [..., D], cos / sin [..., D/2] (broadcast over the
    leading axes the caller aligns)."""
    y = np.asarray(y, dtype=np.float64)
    h = y.shape[-1] // 2
    a, b = y[..., :h], y[..., h:]
    return np.concatenate([a * cos - b * sin, b * cos + a * sin], axis=-1)


def rope_table(n_pos: int, head_dim: int, theta: float = 10000.0) -> np.ndarray:
    """The frequency table [n_pos][D/2][2] = (cos, sin) of pos * theta^(-2i/D),
    in float64 (the library consumes its float32 rounding)."""
    i = np.arange(head_dim // 2, dtype=np.float64)
    inv = theta ** (-2.0 * i / head_dim)
    ang = np.arange(n_pos, dtype=np.float64)[:, None] * inv[None, :]
    return np.stack([np.cos(ang), np.sin(ang)], axis=-1)


def qk_norm_rope(q, k, gamma_q, gamma_k, cos_sin, positions, eps=1e-6):
    """q [T][Hq][D], k [T][Hkv][D] (values), gamma_* [D], cos_sin
    [n_pos][D/2][2], positions [T] -> (q', k') in float64 (before the bf16
    rounding of the stored outputs)."""
    cs = np.asarray(cos_sin, dtype=np.float64)[np.asarray(positions, dtype=np.int64)]   # [T][D/2][2]
    cos, sin = cs[:, None, :, 0], cs[:, None, :, 1]
    qo = rope_rotate_half(rms_norm(q, gamma_q, eps), cos, sin)
    ko = rope_rotate_half(rms_norm(k, gamma_k, eps), cos, sin)
    return qo, ko
