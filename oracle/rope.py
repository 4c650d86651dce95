"""Rotary position embedding in float64 (oracle; test infrastructure only).

The MiniPIC summary (gist.science 2606.13126, section 2.1) writes the rotation
of a vector at position p as the matrix R_p and states that the kernel applies
it with a cosine/sine table lookup and multiply-adds per key element.  The
pages do not fix the rotary variant; this oracle takes the half-rotation form
(element i pairs with element i + d/2) with theta_i = base^(-2i/d):

    x'_i       = x_i       cos(p theta_i) - x_{i+d/2} sin(p theta_i)
    x'_{i+d/2} = x_{i+d/2} cos(p theta_i) + x_i       sin(p theta_i)

Angles p * theta_i are formed in numpy's extended precision (80-bit on x86-64,
128-bit on aarch64) so that positions up to ~131k keep ~1e-14 absolute angle
accuracy; cosines and sines are then rounded to float64.
"""

from __future__ import annotations

import numpy as np

_LD = np.longdouble


def inv_freq(d: int, base: float) -> np.ndarray:
    """theta_i = base^(-2 i / d) for i = 0 .. d/2 - 1, in extended precision."""
    if d % 2:
        raise ValueError("head_dim must be even")
    i = np.arange(d // 2, dtype=_LD)
    return np.power(_LD(base), -(_LD(2) * i) / _LD(d))


def rope_angles(pos, d: int, base: float) -> np.ndarray:
    """Angles p * theta_i, shape [n, d/2], extended precision."""
    p = np.asarray(pos, dtype=np.int64).astype(_LD).reshape(-1, 1)
    return p * inv_freq(d, base).reshape(1, -1)


def rope_cos_sin(pos, d: int, base: float):
    """(cos, sin) of p * theta_i as float64 arrays of shape [n, d/2]."""
    a = rope_angles(pos, d, base)
    return np.cos(a).astype(np.float64), np.sin(a).astype(np.float64)


def rope_table(max_pos: int, d: int, base: float) -> np.ndarray:
    """Table [max_pos, d] float64: cos(p theta_i) in columns [0, d/2) and
    sin(p theta_i) in columns [d/2, d) -- the layout the library's table uses."""
    c, s = rope_cos_sin(np.arange(max_pos), d, base)
    return np.concatenate([c, s], axis=1)


def rope_rotate(x, pos, base: float) -> np.ndarray:
    """Rotate rows of x (shape [..., n, d]) by R_{pos[k]} for row k."""
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    h = d // 2
    c, s = rope_cos_sin(pos, d, base)          # [n, d/2]
    a, b = x[..., :h], x[..., h:]
    out = np.empty_like(x)
    out[..., :h] = a * c - b * s
    out[..., h:] = b * c + a * s
    return out
