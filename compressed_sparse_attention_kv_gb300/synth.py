"""Seeded synthetic decode workloads.

This module only draws random numbers and builds structure (context lengths,
shuffled page tables); it holds none of the method's arithmetic (no coding,
no pooling, no scoring, no rotation).  Every array comes from its own numpy
PCG64 stream keyed by (seed, tag, indices...), so any page of any request can
be regenerated on its own and x86 and Arm hosts draw identical values.

Workloads (seed n - 1 for workload n):

1. tiny_csa      batch 1, 4,096 tokens, ratio 4 (1,024 entries), top-512,
                 16 query heads, 4 indexer heads, bf16 everywhere; the caches
                 are produced by compressing N(0,1) kv / gate inputs.
2. hca_128k      batch 32, 131,072 tokens, ratio 128 (1,024 entries, all read),
                 64 heads, FP8-528 entries and window, values N(0,1).
3. csa_1m        batch 8, 1,048,576 tokens, ratio 4 (262,144 entries), 64
                 indexer heads x 128 FP8 keys, w ~ U(0,1), top-512, 64 heads,
                 FP8-528 entries and window.
4. compressor    65,536-token chunk, 512-d bf16 kv / gate, ratio 4 (overlap)
                 and ratio 128, out FP8-528 / FP4-288 / bf16.
5. mixed_mxfp4   batch 64, contexts ~ U{32,768 .. 524,288}, FP4-288 entries,
                 FP8 window, FP8-132 index keys, top-512, 64 heads.
6. csa_fp4       csa_1m with FP4 index keys (rotated, e2m1 + e8m0 per 32,
                 68 bytes per key); the same seed and values as csa_1m.

The pages measure on model layers over real text and name no dataset for this
path; these seeded inputs stand in with the shapes the pages give.  Value
distributions the pages leave open: slot bias ~ 0.5 N(0,1), RMSNorm weight
~ U(0.5, 1.5), sink logits ~ N(0,1), queries and keys N(0,1).
"""

from dataclasses import dataclass, field
from typing import Optional

import numpy as np

PAGE_ROWS = 64
WINDOW = 128
D_MAIN = 512
D_INDEX = 128

# format ids (same numbering as the C header)
FMT_BF16 = 0
FMT_FP8 = 1
FMT_FP4 = 2
FMT_FP8_PAGESPLIT = 3
FMT_FP4H_PAGESPLIT = 4

# stream tags
T_CTX, T_PAGES, T_MAIN, T_INDEX, T_SWA, T_Q, T_QIDX, T_W, T_SINK = range(1, 10)
T_KV, T_GATE, T_APE, T_NORM, T_PREV_KV, T_PREV_GATE = range(10, 16)
T_IKV, T_IGATE, T_IAPE, T_INORM, T_IPREV_KV, T_IPREV_GATE = range(16, 22)


def rng(seed, *tags):
    return np.random.default_rng([int(seed)] + [int(t) for t in tags])


def normal(seed, tags, shape, scale=1.0):
    x = rng(seed, *tags).standard_normal(shape, dtype=np.float32)
    return x if scale == 1.0 else (x * np.float32(scale)).astype(np.float32)


def uniform(seed, tags, shape, lo, hi):
    return rng(seed, *tags).uniform(lo, hi, size=shape).astype(np.float32)


@dataclass
class DecodeWorkload:
    name: str
    seed: int
    B: int
    ratio: int
    k: Optional[int]               # None -> HCA (read every visible entry)
    H: int
    Hi: int
    main_fmt: int
    swa_fmt: int
    key_fmt: int
    ctx_len: np.ndarray = field(repr=False)
    sink: bool = True

    @property
    def n_entries(self):
        return self.ctx_len // self.ratio

    @property
    def max_ctx(self):
        return int(self.ctx_len.max())

    def pages_per_req(self):
        return (self.n_entries + PAGE_ROWS - 1) // PAGE_ROWS


def workload(name, batch=None):
    """The named decode workload (optionally with a smaller batch for tests)."""
    if name == "tiny_csa":
        w = DecodeWorkload(name, 0, 1, 4, 512, 16, 4, FMT_BF16, FMT_BF16, FMT_BF16,
                           np.array([4096], dtype=np.int64))
    elif name == "hca_128k":
        w = DecodeWorkload(name, 1, 32, 128, None, 64, 0, FMT_FP8, FMT_FP8, FMT_FP8,
                           np.full(32, 131072, dtype=np.int64))
    elif name == "csa_1m":
        w = DecodeWorkload(name, 2, 8, 4, 512, 64, 64, FMT_FP8, FMT_FP8, FMT_FP8_PAGESPLIT,
                           np.full(8, 1 << 20, dtype=np.int64))
    elif name == "csa_fp4":
        w = DecodeWorkload(name, 2, 8, 4, 512, 64, 64, FMT_FP8, FMT_FP8, FMT_FP4H_PAGESPLIT,
                           np.full(8, 1 << 20, dtype=np.int64))
    elif name == "mixed_mxfp4":
        L = rng(4, T_CTX).integers(32768, 524288, size=64, endpoint=True).astype(np.int64)
        w = DecodeWorkload(name, 4, 64, 4, 512, 64, 64, FMT_FP4, FMT_FP8, FMT_FP8_PAGESPLIT, L)
    else:
        raise KeyError(name)
    if batch is not None and batch != w.B:
        w.ctx_len = w.ctx_len[:batch].copy()
        w.B = batch
    return w


def custom_workload(name, seed, ctx_len, ratio, k, H, Hi, main_fmt, swa_fmt, key_fmt, sink=True):
    ctx = np.asarray(ctx_len, dtype=np.int64)
    return DecodeWorkload(name, seed, int(ctx.shape[0]), ratio, k, H, Hi, main_fmt, swa_fmt,
                          key_fmt, ctx, sink)


# ----------------------------------------------------------------------------
# structure
# ----------------------------------------------------------------------------

def page_tables(w, lane):
    """Shuffled page pool for one cache lane ('main' or 'index').

    Returns (block_table int32 [B, max_pages], num_pages).  Request b owns
    ceil(n_b / 64) pages; all pages of all requests are one pool in random order.
    """
    tag = T_MAIN if lane == "main" else T_INDEX
    ppr = w.pages_per_req()
    total = int(ppr.sum())
    perm = rng(w.seed, T_PAGES, tag).permutation(total).astype(np.int32)
    max_pages = int(max(1, ppr.max()))
    bt = np.full((w.B, max_pages), -1, dtype=np.int32)
    off = 0
    for b in range(w.B):
        bt[b, :ppr[b]] = perm[off:off + ppr[b]]
        off += ppr[b]
    return bt, total


# ----------------------------------------------------------------------------
# values (float32; the caller rounds to bf16 or codes them as it needs)
# ----------------------------------------------------------------------------

def main_page_values(w, b, page, dim=D_MAIN):
    """N(0,1) values of logical page `page` of request b's compressed entries: [64, dim]."""
    return normal(w.seed, (T_MAIN, b, page), (PAGE_ROWS, dim))


def index_page_values(w, b, page, dim=D_INDEX):
    """N(0,1) values of logical page `page` of request b's index keys: [64, dim]."""
    return normal(w.seed, (T_INDEX, b, page), (PAGE_ROWS, dim))


def request_values(w, b, lane, rows=None):
    """All pages of one request's lane concatenated: [pages*64, dim]."""
    n_pages = int(w.pages_per_req()[b])
    f = main_page_values if lane == "main" else index_page_values
    if rows is None:
        return np.concatenate([f(w, b, p) for p in range(n_pages)], axis=0)
    pages = sorted(set(int(r) // PAGE_ROWS for r in rows))
    return {p: f(w, b, p) for p in pages}


def swa_values(w, b):
    """N(0,1) window ring values as stored (already rotated): [128, 512]."""
    return normal(w.seed, (T_SWA, b), (WINDOW, D_MAIN))


def queries(w):
    """Attention queries [B, H, 512], indexer queries [B, Hi, 128], weights [B, Hi], sink [H]."""
    q = normal(w.seed, (T_Q,), (w.B, w.H, D_MAIN))
    qi = normal(w.seed, (T_QIDX,), (w.B, max(w.Hi, 1), D_INDEX))[:, :w.Hi]
    wt = uniform(w.seed, (T_W,), (w.B, max(w.Hi, 1)), 0.0, 1.0)[:, :w.Hi]
    sink = normal(w.seed, (T_SINK,), (w.H,)) if w.sink else None
    return q, np.ascontiguousarray(qi), np.ascontiguousarray(wt), sink


def compressor_params(seed, ratio, overlap, dim, index_lane=False):
    """Slot bias ape [ratio, coff*dim] ~ 0.5 N(0,1) and RMSNorm weight [dim] ~ U(0.5, 1.5)."""
    coff = 2 if overlap else 1
    ta, tn = (T_IAPE, T_INORM) if index_lane else (T_APE, T_NORM)
    ape = normal(seed, (ta, ratio, dim), (ratio, coff * dim), scale=0.5)
    nw = uniform(seed, (tn, ratio, dim), (dim,), 0.5, 1.5)
    return ape, nw


def compressor_tokens(seed, T, ratio, overlap, dim, index_lane=False, seq=0):
    """kv, gate [T, coff, dim] ~ N(0,1) for one sequence chunk."""
    coff = 2 if overlap else 1
    tk, tg = (T_IKV, T_IGATE) if index_lane else (T_KV, T_GATE)
    kv = normal(seed, (tk, seq, ratio, dim), (T, coff, dim))
    gate = normal(seed, (tg, seq, ratio, dim), (T, coff, dim))
    return kv, gate


def compressor_prev(seed, ratio, dim, index_lane=False, seq=0):
    """kv, gate [ratio, 2, dim] of the block before a chunk (continuation inputs)."""
    tk, tg = (T_IPREV_KV, T_IPREV_GATE) if index_lane else (T_PREV_KV, T_PREV_GATE)
    return (normal(seed, (tk, seq, ratio, dim), (ratio, 2, dim)),
            normal(seed, (tg, seq, ratio, dim), (ratio, 2, dim)))


def integer_index_inputs(seed, B, Hi, n_rows):
    """Integer-valued indexer inputs (q, k in {-3..3}, w in {0..7}/8): every fp32 partial
    sum of a score is exact in any order, so GPU and oracle scores agree exactly."""
    r = rng(seed, 99)
    q = r.integers(-3, 4, size=(B, Hi, D_INDEX)).astype(np.float32)
    k = r.integers(-3, 4, size=(n_rows, D_INDEX)).astype(np.float32)
    wt = (r.integers(0, 8, size=(B, Hi)) / 8.0).astype(np.float32)
    return q, k, wt
