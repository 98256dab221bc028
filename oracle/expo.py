"""exp_own: the exponential of the compressor's bit-exact fp32 contract (oracle side).

TEST INFRASTRUCTURE ONLY.

The compressor's softmax over slots must give the same fp32 bits on the CPU
and on the GPU, so it cannot use either platform's libm.  Both sides implement
the same textbook method, each from this description:

  Cody & Waite additive range reduction (W. J. Cody and W. Waite, "Software
  Manual for the Elementary Functions", 1980):
      t   = x * LOG2E                         (fp32)
      if not (t >= -126): return 0            (covers -inf; result < 2^-126)
      n   = rint(t)                           (round half to even)
      r   = (x - n*LN2_HI) - n*LN2_LO         (each product and difference rounded)
  then the degree-7 Taylor polynomial of e^r in Horner form
      p = C7; p = p*r + C6; ...; p = p*r + C0        (C_k = fp32(1/k!), mul then add)
  and the result p * 2^n (exact power-of-two scaling).

Constants are derived here from ln 2, not copied from any library:
LN2_HI is ln 2 rounded to 16 significant bits (so n*LN2_HI is exact for
|n| <= 127), LN2_LO the fp32 rounding of the remainder.  No fused multiply-add
is used anywhere: every step is a separately rounded fp32 operation.
The truncation error of the polynomial on |r| <= ln2/2 is below 6e-9 relative.
"""

import math

import numpy as np

F32 = np.float32

LOG2E = F32(1.0 / math.log(2.0))
LN2_HI = F32(round(math.log(2.0) * 65536.0) / 65536.0)
LN2_LO = F32(math.log(2.0) - float(LN2_HI))
COEFFS = [F32(1.0 / math.factorial(k)) for k in range(8)]   # C0..C7


def exp_own(x):
    """Elementwise e^x in the contract order; x float32 array (x <= 88)."""
    x = np.asarray(x, dtype=F32)
    t = (x * LOG2E).astype(F32)
    live = t >= F32(-126.0)                       # False for -inf and NaN
    n = np.rint(np.where(live, t, F32(0.0))).astype(F32)
    xs = np.where(live, x, F32(0.0)).astype(F32)
    r = ((xs - (n * LN2_HI).astype(F32)).astype(F32) - (n * LN2_LO).astype(F32)).astype(F32)
    p = COEFFS[7]
    for k in range(6, -1, -1):
        p = ((p * r).astype(F32) + COEFFS[k]).astype(F32)
    scale = np.ldexp(F32(1.0), n.astype(np.int64)).astype(F32)
    return np.where(live, (p * scale).astype(F32), F32(0.0)).astype(F32)
