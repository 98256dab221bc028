"""Decode-step state update (oracle side).  TEST INFRASTRUCTURE ONLY.

What it follows ("DeepSeek-V4 deep dive", §4.3 "What is cached" and the
implementation notes to §4): during decode each compressor keeps a fixed-size
per-request state of projected tokens that have no entry yet, together with
the block before them when the compressor overlaps:

  * the state has coff*r slots of kv and of scores (r = ratio); a fresh request's
    slots hold kv 0 and score -inf;
  * the token at position p goes into slot r + (p mod r) with overlap (the
    current block; slots 0 .. r-1 hold the previous block), else slot p mod r;
  * when (p + 1) mod r == 0 the block is complete: entry (p + 1)/r - 1 is pooled
    from the previous block's channel half 0 and the current block's half 1
    (overlap) or from the current block alone, normalised, rotated to the
    position of the block's first token, p + 1 - r, and written; with overlap
    the current block then moves into the previous-block slots;
  * the window keeps the last 128 tokens as a ring: the token at position p goes
    to slot p mod 128, normalised and rotated to its own position (the same
    per-row steps as an entry of ratio 1).

The pooling itself is the compressor contract of compress.py, called on the
block's own tokens with the previous block passed as its preceding block; the
state keeps the raw gate scores, to which the contract adds the slot bias.
"""

import numpy as np

from . import compress, rope

WINDOW = 128


class CompressorState:
    """One request's state for one compressor (ratio r, overlap or not, width D)."""

    def __init__(self, ratio, overlap, dim):
        self.r, self.overlap, self.dim = ratio, bool(overlap), dim
        coff = 2 if overlap else 1
        nslot = 2 * ratio if overlap else ratio
        self.kv = np.zeros((nslot, coff, dim), np.float32)
        self.gate = np.full((nslot, coff, dim), -np.inf, np.float32)

    def push(self, p, kv_tok, gate_tok, ape, norm_w=None, eps=1e-6, theta=rope.THETA_COMPRESSED, yarn=None):
        """Token at position p ([coff, D] kv and gate, fp32 values) -> (entry index, entry [D]
        float32) when it completes a block, else None."""
        r = self.r
        slot = (r if self.overlap else 0) + p % r
        self.kv[slot] = kv_tok
        self.gate[slot] = gate_tok
        if (p + 1) % r:
            return None
        cur = slice(r, 2 * r) if self.overlap else slice(0, r)
        prev = dict(prev_kv=self.kv[:r], prev_gate=self.gate[:r]) if self.overlap else {}
        first = p + 1 - r
        cs = rope.table([first], theta=theta, yarn=yarn)
        e = compress.compress_contract(self.kv[cur], self.gate[cur], ape, r, self.overlap, norm_w=norm_w,
                                       eps=eps, rope_cs=cs, **prev)
        if self.overlap:
            self.kv[:r] = self.kv[r:]
            self.gate[:r] = self.gate[r:]
        return (p + 1) // r - 1, e[0]


def window_row(kv_tok, p, norm_w=None, eps=1e-6, theta=rope.THETA_COMPRESSED, yarn=None):
    """The window ring's row for the token at position p: (slot p mod 128, row [D] float32)."""
    kv = np.asarray(kv_tok, np.float32).reshape(1, 1, -1)
    cs = rope.table([p], theta=theta, yarn=yarn)
    row = compress.compress_contract(kv, np.zeros_like(kv), np.zeros((1, kv.shape[-1]), np.float32), 1, False,
                                     norm_w=norm_w, eps=eps, rope_cs=cs)
    return p % WINDOW, row[0]
