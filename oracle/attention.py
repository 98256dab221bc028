"""Shared-KV sparse decode attention with a sliding window and a sink (oracle side).

TEST INFRASTRUCTURE ONLY.

"DeepSeek-V4 deep dive":
* §3.1 "Idea first: K = V, one head": one 512-d entry is the key and the value
  of every query head; no up-projection.
* §3.3 "Partial RoPE and the inverse rotation on the output": the query's last
  64 dims are rotated by its position t; the output's last 64 dims are turned
  back by -t.  Stored entries are already rotated (at i*r for compressed ones).
* §3.4 "One softmax, a sink, and the window" (Eq. 27):
      s_{h,j} = exp(z_{h,j}) / (sum_k exp(z_{h,k}) + exp(z'_h)),
      z_{h,j} = (q_h . c_j) * 512^-1/2,   o_h = sum_j s_{h,j} c_j.
* §2.1 and §5.3: the key list is the window (positions max(0, t-127) .. t, the
  query's own token included; the ring slot of position p is p mod 128),
  followed by the compressed part: the indexer's selection (CSA) or every
  visible entry j < floor((t+1)/r) (HCA, §6.1).  -1 ids are skipped and
  duplicates are kept (a key listed twice counts twice).
"""

import numpy as np

from . import rope

WINDOW = 128


def window_positions(t, window=WINDOW):
    return np.arange(max(0, t - window + 1), t + 1, dtype=np.int64)


def compressed_ids(ctx_len, ratio, topk=None):
    """Entry ids of the compressed part of the key list, in list order."""
    if topk is None:
        return np.arange(ctx_len // ratio, dtype=np.int64)
    topk = np.asarray(topk, dtype=np.int64)
    return topk[topk >= 0]


def key_count(ctx_len, ratio, k=None, window=WINDOW):
    """Keys in one query's softmax: window part + min(k, n) (CSA) or n (HCA)."""
    t = ctx_len - 1
    n = ctx_len // ratio
    w = min(window, t + 1)
    return w + (n if k is None else min(k, n))


def decode_attention_fp64(q, t, window_rows, entry_rows, sink, scale,
                          theta=rope.THETA_COMPRESSED):
    """One request.

    q            [H, 512] query (pre-RoPE)
    t            query position
    window_rows  [nw, 512] decoded window keys in list order (already rotated)
    entry_rows   [nc, 512] decoded compressed keys in list order (already rotated)
    sink         [H] sink logits or None
    Returns o [H, 512] float64 after the inverse rotation.
    """
    keys = np.concatenate([np.asarray(window_rows, np.float64).reshape(-1, 512),
                           np.asarray(entry_rows, np.float64).reshape(-1, 512)], axis=0)
    ang = rope.angles(np.array([t]))[0]
    qr = rope.rotate_fp64(np.asarray(q, np.float64), ang[None, :])
    z = (qr @ keys.T) * scale                                   # [H, nk]
    zs = np.full(z.shape[0], -np.inf) if sink is None else np.asarray(sink, np.float64)
    M = np.maximum(np.max(z, axis=1), zs)
    p = np.exp(z - M[:, None])
    den = np.sum(p, axis=1) + np.exp(zs - M)
    o = (p @ keys) / den[:, None]
    return rope.rotate_fp64(o, ang[None, :], inverse=True)


def request_attention(q, ctx_len, ratio, swa_decoded, entries_decoded, topk, sink, scale):
    """Build one request's key list and attend.

    swa_decoded     [128, 512] decoded ring (slot = position mod 128)
    entries_decoded callable ids -> [len(ids), 512] decoded compressed rows, or an
                    array indexed by entry id
    topk            [k] selected ids (CSA) or None (HCA: all visible entries)
    """
    t = ctx_len - 1
    wpos = window_positions(t)
    wrows = np.asarray(swa_decoded)[wpos % WINDOW]
    ids = compressed_ids(ctx_len, ratio, topk)
    if callable(entries_decoded):
        erows = entries_decoded(ids)
    else:
        erows = np.asarray(entries_decoded)[ids]
    return decode_attention_fp64(q, t, wrows, erows, sink, scale)
