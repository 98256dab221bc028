"""KV compressor: learned gated per-channel pooling (oracle side).

TEST INFRASTRUCTURE ONLY.

What it computes ("DeepSeek-V4 deep dive", §4.1 "Idea: average, but let the
model choose the weights per channel", and §4.2 "Ratio 4 (CSA) overlaps; ratio
128 (HCA) does not"):

  For entry i and channel c, over the slots j of the entry's window,
      s_j = gate_j + B[slot position of j]           (slot bias "ape")
      C_{i,c} = sum_j softmax_j(s_{j,c}) * v_{j,c}   (softmax over slots, per channel)

  * ratio r without overlap: the slots are the r tokens r*i .. r*i + r-1, one
    projection half (coff = 1).
  * ratio 4 with overlap (coff = 2): an 8-slot window; slots 0-3 are the
    previous block's 4 tokens read through channel half 0, slots 4-7 the
    entry's own 4 tokens through half 1.  The slot bias is added before this
    transform, so slots 0-3 carry ape[:, :D] and slots 4-7 ape[:, D:].  The
    first entry of a sequence has no previous block: value 0, score -inf.
  * the V4.1 compressor ("DeepSeek-V4.1 Flash", section 1.1; the deep dive's
    implementation notes to section 4) is the no-overlap case with ratio 2
    (encoder) or 1 (decoder) and no slot bias, i.e. a zero B.
  * then RMSNorm over the D channels with a learned weight, and RoPE on the
    last 64 dims at the position of the first token of the entry's own block
    (i * r).

Two renderings:

``compress_fp64``      the definition, in fp64 (softmax with np.exp).
``compress_contract``  the fp32 operation order the GPU kernel follows
                       bit for bit:
   1. s_j  = fp32(gate_j) + ape[...]                     (one fp32 add)
   2. m    = max_j s_j
   3. e_j  = exp_own(s_j - m)                            (see expo.py)
      num  = (...((0 + e_0*v_0) + e_1*v_1) ...)          slot order, mul then add
      den  = (...((0 + e_0) + e_1) ...)                  slot order
      C    = num / den                                   (IEEE division)
   4. ss   = pairwise sum of C_c*C_c over channel index (recursive halves:
             sum(v) = sum(v[:n/2]) + sum(v[n/2:]), i.e. adjacent pairs first)
      rr   = 1 / sqrt(ss / D + eps)                      (IEEE div, sqrt, div)
      y_c  = (C_c * rr) * w_c
   5. RoPE on pairs (2k, 2k+1) of the last 64 dims with the fp32 table
      (cos, sin):  y0' = y0*cos - y1*sin,  y1' = y0*sin + y1*cos
   Every step is a separately rounded fp32 operation (no fused multiply-add).
"""

import numpy as np

from . import codecs, rope
from .expo import exp_own

F32 = np.float32


def _windows(kv, gate, ape, ratio, overlap, prev_kv, prev_gate, dtype):
    """Slot values V [n, S, D] and scores Sc [n, S, D] (bias included) of every entry."""
    kv = np.asarray(kv, dtype=dtype)
    gate = np.asarray(gate, dtype=dtype)
    T, coff, D = kv.shape
    assert T % ratio == 0 and coff == (2 if overlap else 1)
    n = T // ratio
    apeb = np.asarray(ape, dtype=dtype).reshape(ratio, coff, D)
    cur_v = kv.reshape(n, ratio, coff, D)
    cur_s = (gate.reshape(n, ratio, coff, D) + apeb[None]).astype(dtype)
    if not overlap:
        return cur_v[:, :, 0], cur_s[:, :, 0]
    prev_v = np.empty((n, ratio, D), dtype=dtype)
    prev_s = np.empty((n, ratio, D), dtype=dtype)
    prev_v[1:] = cur_v[:-1, :, 0]
    prev_s[1:] = cur_s[:-1, :, 0]
    if prev_kv is None:
        prev_v[0] = 0.0
        prev_s[0] = -np.inf
    else:
        pk = np.asarray(prev_kv, dtype=dtype).reshape(ratio, coff, D)
        pg = np.asarray(prev_gate, dtype=dtype).reshape(ratio, coff, D)
        prev_v[0] = pk[:, 0]
        prev_s[0] = (pg[:, 0] + apeb[:, 0]).astype(dtype)
    V = np.concatenate([prev_v, cur_v[:, :, 1]], axis=1)
    Sc = np.concatenate([prev_s, cur_s[:, :, 1]], axis=1)
    return V, Sc


def compress_fp64(kv, gate, ape, ratio, overlap, prev_kv=None, prev_gate=None,
                  norm_w=None, eps=1e-6, positions=None, theta=rope.THETA_COMPRESSED):
    """Definition of the compressor in fp64 -> entries [n, D] float64.

    positions: [n] RoPE positions of the entries (normally i*r), or None for no RoPE.
    """
    V, Sc = _windows(kv, gate, ape, ratio, overlap, prev_kv, prev_gate, np.float64)
    m = np.max(Sc, axis=1, keepdims=True)
    wgt = np.exp(Sc - m)
    wgt = wgt / np.sum(wgt, axis=1, keepdims=True)
    C = np.sum(wgt * V, axis=1)
    if norm_w is not None:
        C = C / np.sqrt(np.mean(C * C, axis=-1, keepdims=True) + eps) * np.asarray(norm_w, np.float64)
    if positions is not None:
        C = rope.rotate_fp64(C, rope.angles(positions, theta))
    return C


def pairwise_sum_f32(v):
    """Recursive-halves fp32 sum over the last axis (length a power of two)."""
    v = np.asarray(v, dtype=F32)
    while v.shape[-1] > 1:
        v = (v[..., 0::2] + v[..., 1::2]).astype(F32)
    return v[..., 0]


def compress_contract(kv, gate, ape, ratio, overlap, prev_kv=None, prev_gate=None,
                      norm_w=None, eps=1e-6, rope_cs=None):
    """fp32 contract rendering -> entries [n, D] float32 (bit-exact target of the GPU)."""
    V, Sc = _windows(kv, gate, ape, ratio, overlap, prev_kv, prev_gate, F32)
    n, S, D = V.shape
    m = np.max(Sc, axis=1)
    num = np.zeros((n, D), dtype=F32)
    den = np.zeros((n, D), dtype=F32)
    for j in range(S):
        e = exp_own((Sc[:, j] - m).astype(F32))
        num = (num + (e * V[:, j]).astype(F32)).astype(F32)
        den = (den + e).astype(F32)
    C = (num / den).astype(F32)
    if norm_w is not None:
        ss = pairwise_sum_f32((C * C).astype(F32))
        mean = (ss / F32(D)).astype(F32)
        rr = (F32(1.0) / np.sqrt((mean + F32(eps)).astype(F32))).astype(F32)
        C = (((C * rr[:, None]).astype(F32)) * np.asarray(norm_w, F32)).astype(F32)
    if rope_cs is not None:
        C = rope.rotate_table_fp32(C, np.asarray(rope_cs, F32))
    return C


def entries_to_bytes(entries, fmt):
    """Contract entries [n, D] float32 -> stored bytes (inline rows, or pages for page-split)."""
    if fmt == codecs.FMT_FP8_PAGESPLIT:
        return codecs.encode_pagesplit(entries)
    if fmt == codecs.FMT_FP4H_PAGESPLIT:
        return codecs.encode_fp4h_pagesplit(entries)   # rotated, then coded
    return codecs.encode_rows(entries, fmt)
