"""Lightning indexer and top-k selection (oracle side).  TEST INFRASTRUCTURE ONLY.

"DeepSeek-V4 deep dive", §5.2 "What is different from V3.2's indexer" (the
score formula I_{s,t} and the visibility rule) and §5.3 "Selection and the
window in one softmax":

    I_j = sum_h w_h * ReLU(q_h . k_j)           for visible entries j < n
    n   = floor((t + 1) / r) = floor(L / r)     (query at position t = L - 1)

k_j is one 128-d key shared by all indexer heads.  The selector keeps
min(k, n) entries; missing slots are -1.

Readings: larger score first, ties to the smaller
entry index; the output is a set, returned here in ascending entry order.
With FP8 keys the queries are coded e4m3 with one e8m0 scale per head, and
the exact values of the coded operands enter the fp64 score.  With FP4 index
keys ("DeepSeek-V4 deep dive", section 5.2) the queries are rotated and coded
like the keys (e2m1, e8m0 per 32), and the scores are stored in BF16 before the
selection ("DeepSeek-V4.1 Flash", section 10.4), so that ties between equal
bf16 scores go to the smaller entry.
"""

import numpy as np

from . import codecs


def visible_entries(ctx_len, ratio):
    """Entries a query at position ctx_len - 1 may read: floor(ctx_len / ratio)."""
    return np.asarray(ctx_len, dtype=np.int64) // ratio


def scores_fp64(q_hat, w, k_hat):
    """q_hat [Hi, Di], w [Hi], k_hat [n, Di] (exact operand values) -> I [n] float64."""
    dots = np.asarray(k_hat, np.float64) @ np.asarray(q_hat, np.float64).T     # [n, Hi]
    return np.maximum(dots, 0.0) @ np.asarray(w, np.float64)


def select_topk(scores, k):
    """Indices of the min(k, n) largest scores (ties -> smaller index), ascending, -1 padded to k."""
    scores = np.asarray(scores, np.float64)
    n = scores.shape[0]
    order = np.lexsort((np.arange(n), -scores))        # primary: score desc, secondary: index asc
    keep = np.sort(order[:min(k, n)])
    out = np.full(k, -1, dtype=np.int64)
    out[:keep.shape[0]] = keep
    return out


def quantize_queries(q):
    """Indexer queries [Hi, 128] (bf16 values) -> exact values of their FP8 per-head coding."""
    q32 = np.asarray(q, np.float32)
    c, s = codecs.encode_q_perhead(q32)
    return codecs.e4m3_decode(c) * codecs.e8m0_decode(s)[..., None]


def quantize_queries_fp4(q):
    """Indexer queries [Hi, 128] (bf16 values) -> exact values of their rotated FP4 coding."""
    c, s = codecs.encode_q_fp4h(np.asarray(q, np.float32))
    return codecs.fp4b32_decode(c, s)


def bf16_scores(I):
    """Index scores stored in BF16 ("DeepSeek-V4.1 Flash", section 10.4): the score,
    rounded to fp32 (the precision it is computed in), then to bf16, RNE both times."""
    return codecs.bf16_decode(codecs.bf16_encode(np.asarray(I, np.float64).astype(np.float32)))


def index_topk_fp4(q, w, k_hat, ctx_len, ratio, k):
    """One request with FP4 index keys: the rotated FP4 queries against the rotated
    FP4 keys (exact values, fp64 score), the scores rounded to bf16, top-k on those.

    k_hat  [>= n, 128] exact (rotated) key values in entry order
    Returns (topk [k] int64, bf16 scores [n] float64, fp64 scores [n]).
    """
    n = int(visible_entries(ctx_len, ratio))
    I = scores_fp64(quantize_queries_fp4(q), w, np.asarray(k_hat)[:n])
    Ib = bf16_scores(I)
    return select_topk(Ib, k), Ib, I


def index_topk(q, w, k_hat, ctx_len, ratio, k, fp8_keys):
    """One request: scores of the visible entries and the selected set.

    q      [Hi, 128] indexer queries (post-RoPE, bf16 values)
    w      [Hi] head weights (already scaled)
    k_hat  [>= n, 128] exact key values in entry order
    Returns (topk [k] int64, scores [n] float64).
    """
    n = int(visible_entries(ctx_len, ratio))
    q_hat = quantize_queries(q) if fp8_keys else np.asarray(q, np.float64)
    I = scores_fp64(q_hat, w, np.asarray(k_hat)[:n])
    return select_topk(I, k), I


def accumulation_bound(q_hat, w, k_hat):
    """Per-entry bound on fp32 accumulation error of I_j: 128 u * sum_h |w_h| sum_d |q_hd k_jd|.

    u = 2^-24.  128 covers the 128-term dot product, the 4-term scale merge,
    the weight product and the 64-term head sum with room to spare.
    """
    a = np.abs(np.asarray(k_hat, np.float64)) @ np.abs(np.asarray(q_hat, np.float64)).T
    return 128.0 * 2.0 ** -24 * (a @ np.abs(np.asarray(w, np.float64)))
