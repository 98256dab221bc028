"""Partial RoPE (oracle side).  TEST INFRASTRUCTURE ONLY.

"DeepSeek-V4 deep dive", §3.3 "Partial RoPE and the inverse rotation on the
output": only the last 64 of the 512 dims are rotated; the 64 dims are viewed
as 32 adjacent pairs (2k, 2k+1), pair k turning by position * theta^(-2k/64);
compressed layers use base theta = 160,000 (§2.2, §9.1), optionally with YaRN
(§9.1 "Positions to 1M"; the frequency blend of the YaRN method, Peng et al.
2023, over the pair range the settings give).  The output of attention is turned
back by minus the query's position.

The rotation of a pair by angle a is  (y0, y1) -> (y0 cos a - y1 sin a,
y0 sin a + y1 cos a);  the inverse uses -a.
"""

import numpy as np

ROPE_DIM = 64
THETA_COMPRESSED = 160000.0


# YaRN as the compressed layers configure it (§9.1 "Positions to 1M"): the
# original 65,536 positions stretched 16-fold; betas 32 (fast) and 1 (slow).
YARN_V4 = dict(factor=16.0, original=65536, beta_fast=32.0, beta_slow=1.0)


def yarn_pair_range(theta, rope_dim, original, beta_fast, beta_slow):
    """(low, high): the pair indices between which YaRN blends, by the YaRN method's
    correction range.  Pair k turns once every 2*pi*theta^(2k/rope_dim) positions; the
    pair that turns `beta` times over the original length sits at
    k(beta) = rope_dim * ln(original / (2*pi*beta)) / (2 ln theta); low = floor of
    k(beta_fast), high = ceil of k(beta_slow), kept inside [0, rope_dim/2 - 1]."""
    def k_of(beta):
        return rope_dim * np.log(original / (2.0 * np.pi * beta)) / (2.0 * np.log(theta))
    low = max(int(np.floor(k_of(beta_fast))), 0)
    high = min(int(np.ceil(k_of(beta_slow))), rope_dim // 2 - 1)
    return low, high


def inv_freq(theta=THETA_COMPRESSED, rope_dim=ROPE_DIM, yarn=None):
    """Per-pair angular speed theta^(-2k/rope_dim); with yarn (a dict like YARN_V4) the
    speeds of pairs above the correction range are divided by the factor, those below
    it kept, and those inside it blended along a linear ramp over the pair index:
    f_k = f_k / factor * ramp_k + f_k * (1 - ramp_k), ramp_k = clip((k - low)/(high - low), 0, 1)."""
    k = np.arange(rope_dim // 2, dtype=np.float64)
    f = theta ** (-2.0 * k / rope_dim)
    if yarn is None:
        return f
    low, high = yarn_pair_range(theta, rope_dim, yarn["original"], yarn["beta_fast"], yarn["beta_slow"])
    ramp = np.clip((k - low) / max(high - low, 1e-3), 0.0, 1.0)
    return f / yarn["factor"] * ramp + f * (1.0 - ramp)


def angles(positions, theta=THETA_COMPRESSED, rope_dim=ROPE_DIM, yarn=None):
    """[n] positions -> [n, 32] rotation angles in radians (fp64)."""
    pos = np.asarray(positions, dtype=np.float64)
    return pos[..., None] * inv_freq(theta, rope_dim, yarn)


def table(positions, theta=THETA_COMPRESSED, rope_dim=ROPE_DIM, yarn=None):
    """[n] positions -> float32 [n, 32, 2] of (cos, sin), computed in fp64, rounded once."""
    a = angles(positions, theta, rope_dim, yarn)
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
