"""Partial RoPE (oracle side).  TEST INFRASTRUCTURE ONLY.

"DeepSeek-V4 deep dive", §3.3 "Partial RoPE and the inverse rotation on the
output": only the last 64 of the 512 dims are rotated; the 64 dims are viewed
as 32 adjacent pairs (2k, 2k+1), pair k turning by position * theta^(-2k/64);
compressed layers use base theta = 160,000 (§2.2, §9.1).  The output of
attention is turned back by minus the query's position.

The rotation of a pair by angle a is  (y0, y1) -> (y0 cos a - y1 sin a,
y0 sin a + y1 cos a);  the inverse uses -a.
"""

import numpy as np

ROPE_DIM = 64
THETA_COMPRESSED = 160000.0


def inv_freq(theta=THETA_COMPRESSED, rope_dim=ROPE_DIM):
    k = np.arange(rope_dim // 2, dtype=np.float64)
    return theta ** (-2.0 * k / rope_dim)


def angles(positions, theta=THETA_COMPRESSED, rope_dim=ROPE_DIM):
    """[n] positions -> [n, 32] rotation angles in radians (fp64)."""
    pos = np.asarray(positions, dtype=np.float64)
    return pos[..., None] * inv_freq(theta, rope_dim)


def table(positions, theta=THETA_COMPRESSED, rope_dim=ROPE_DIM):
    """[n] positions -> float32 [n, 32, 2] of (cos, sin), computed in fp64, rounded once."""
    a = angles(positions, theta, rope_dim)
    return np.stack([np.cos(a), np.sin(a)], axis=-1).astype(np.float32)


def rotate_fp64(x, ang, inverse=False):
    """Rotate the last 64 dims of x [..., D] (fp64) by angles ang [..., 32] (fp64)."""
    x = np.array(x, dtype=np.float64, copy=True)
    c, s = np.cos(ang), np.sin(ang)
    if inverse:
        s = -s
    y0 = x[..., -ROPE_DIM::2].copy()
    y1 = x[..., -ROPE_DIM + 1::2].copy()
    x[..., -ROPE_DIM::2] = y0 * c - y1 * s
    x[..., -ROPE_DIM + 1::2] = y0 * s + y1 * c
    return x


def rotate_table_fp32(y, cs):
    """Contract-order rotation of fp32 rows y [..., D] with an fp32 (cos, sin) table [..., 32, 2].

    y0' = y0*c - y1*s ;  y1' = y0*s + y1*c ; every product and sum rounded to fp32.
    """
    y = np.array(y, dtype=np.float32, copy=True)
    c = cs[..., 0].astype(np.float32)
    s = cs[..., 1].astype(np.float32)
    y0 = y[..., -ROPE_DIM::2].copy()
    y1 = y[..., -ROPE_DIM + 1::2].copy()
    y[..., -ROPE_DIM::2] = ((y0 * c).astype(np.float32) - (y1 * s).astype(np.float32)).astype(np.float32)
    y[..., -ROPE_DIM + 1::2] = ((y0 * s).astype(np.float32) + (y1 * c).astype(np.float32)).astype(np.float32)
    return y
