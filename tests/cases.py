"""Shared builders for the GPU parity tests.

Inputs come from the seeded generator (compressed_sparse_attention_kv_gb300.synth);
cache bytes are coded on the host by the oracle's codecs, so the CUDA path and the
oracle read the very same bytes.  Expected values are always computed by the
oracle, never by the CUDA path.
"""

import numpy as np
import torch

import compressed_sparse_attention_kv_gb300 as cskv
from compressed_sparse_attention_kv_gb300 import synth
from oracle import attention as o_attn
from oracle import codecs, indexer

PAGE = 64


def bf16_values(x):
    """float32 array -> (torch bf16 tensor on CPU, float32 numpy of its exact values)."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t, t.float().numpy()


def cuda(x, dtype=None):
    if isinstance(x, np.ndarray):
        x = torch.from_numpy(np.ascontiguousarray(x))
    if dtype is not None:
        x = x.to(dtype)
    return x.contiguous().cuda()


def page_bytes_of(fmt, dim):
    return (PAGE * codecs.row_bytes(fmt, dim) + 15) // 16 * 16


class HostPaged:
    """A paged cache assembled on the host: logical rows of each request coded by the
    oracle and placed in shuffled physical pages."""

    def __init__(self, fmt, dim, rows_per_req, seed, extra_pages=3):
        self.fmt, self.dim = fmt, dim
        self.rows_per_req = list(rows_per_req)
        ppr = [(n + PAGE - 1) // PAGE for n in self.rows_per_req]
        total = sum(ppr) + extra_pages
        perm = np.random.default_rng(seed).permutation(total).astype(np.int32)
        self.max_pages = max(1, max(ppr))
        self.block_table = np.full((len(ppr), self.max_pages), -1, np.int32)
        off = 0
        for b, p in enumerate(ppr):
            self.block_table[b, :p] = perm[off:off + p]
            off += p
        self.num_pages = total
        self.page_bytes = page_bytes_of(fmt, dim)
        self.pool = np.zeros((total, self.page_bytes), np.uint8)
        self.decoded = [None] * len(ppr)

    def fill(self, b, values):
        """Code the rows `values` [n_b, dim] float32 of request b (n_b padded to pages with zeros)."""
        n = self.rows_per_req[b]
        v = np.zeros(((n + PAGE - 1) // PAGE * PAGE, self.dim), np.float32)
        v[:n] = values[:n]
        if self.fmt == codecs.FMT_FP8_PAGESPLIT:
            pages = codecs.encode_pagesplit(v)
            rb = codecs.row_bytes(self.fmt, self.dim)
            for p in range(pages.shape[0]):
                self.pool[self.block_table[b, p], :pages.shape[1]] = pages[p]
            self.decoded[b] = codecs.decode_pagesplit(pages, self.dim)[:n]
        elif self.fmt == codecs.FMT_FP4H_PAGESPLIT:
            pages = codecs.encode_fp4h_pagesplit(v)
            for p in range(pages.shape[0]):
                self.pool[self.block_table[b, p], :pages.shape[1]] = pages[p]
            self.decoded[b] = codecs.decode_fp4h_pagesplit(pages, self.dim)[:n]   # rotated values
        else:
            rows = codecs.encode_rows(v, self.fmt)
            rb = rows.shape[1]
            for p in range(v.shape[0] // PAGE):
                self.pool[self.block_table[b, p], :PAGE * rb] = rows[p * PAGE:(p + 1) * PAGE].reshape(-1)
            self.decoded[b] = codecs.decode_rows(rows, self.fmt, self.dim)[:n]

    def to_device(self):
        return cskv.PagedCache(cuda(self.pool), cuda(self.block_table), self.fmt, self.dim)

    def read_rows(self, pool_bytes, b):
        """Raw bytes of request b's rows from a pool image (for byte-exact comparisons)."""
        n = self.rows_per_req[b]
        out = []
        rb = codecs.row_bytes(self.fmt, self.dim)
        for p in range((n + PAGE - 1) // PAGE):
            pg = pool_bytes[self.block_table[b, p]]
            if self.fmt in (codecs.FMT_FP8_PAGESPLIT, codecs.FMT_FP4H_PAGESPLIT):
                out.append(pg[:PAGE * rb])
            else:
                out.append(pg[:PAGE * rb].reshape(PAGE, rb))
        return out


def swa_ring(values, fmt):
    """[B, 128, 512] float32 -> (uint8 [B, 128, row] bytes, decoded float64 [B, 128, 512])."""
    B = values.shape[0]
    rows = codecs.encode_rows(values.reshape(B * 128, 512), fmt)
    dec = codecs.decode_rows(rows, fmt, 512).reshape(B, 128, 512)
    return rows.reshape(B, 128, -1), dec


def check_attention(got, ref, fp4=False):
    """Parity bar for attention outputs: max |d| <= 2e-2 (3e-2 with FP4 KV) and
    ||d||_2 / ||ref||_2 <= 1e-2, d = gpu - oracle on the same coded bytes."""
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    d = got - ref
    max_abs = float(np.max(np.abs(d)))
    rel = float(np.linalg.norm(d) / max(np.linalg.norm(ref), 1e-30))
    lim = 3e-2 if fp4 else 2e-2
    assert max_abs <= lim and rel <= 1e-2, "max|d|=%.3g rel=%.3g" % (max_abs, rel)
    return max_abs, rel


def check_topk(got_idx, got_score, q_hat, w, k_hat, n, k):
    """Top-k parity against the fp64 definition.

    Exact where the scores decide it: every entry in the symmetric difference of the
    GPU set and the oracle set must have an oracle score within the fp32 accumulation
    bound of the k-th score (a near-tie).  Returns the number of such near-tie swaps.
    """
    I = indexer.scores_fp64(q_hat, w, k_hat[:n])
    ref = indexer.select_topk(I, k)
    got = np.asarray(got_idx, np.int64)
    m = min(k, n)
    assert np.all(got[m:] == -1)
    gs = got[:m]
    assert np.all(np.diff(gs) > 0), "indices not ascending/unique"
    assert np.all((gs >= 0) & (gs < n))
    rs = ref[:m]
    diff = set(gs.tolist()) ^ set(rs.tolist())
    if diff:
        bound = indexer.accumulation_bound(q_hat, w, k_hat[:n])
        kth = np.sort(I)[::-1][m - 1]
        for j in diff:
            assert abs(I[j] - kth) <= bound[j] + bound.max(), (j, I[j], kth)
    if got_score is not None:
        sc = np.asarray(got_score, np.float64)[:m]
        bound = indexer.accumulation_bound(q_hat, w, k_hat[:n])
        assert np.all(np.abs(sc - I[gs]) <= bound[gs] + 1e-30)
    return len(diff) // 2


def check_topk_fp4(got_idx, got_score, q, w, k_hat, n, k):
    """Top-k parity for FP4 index keys (rotated FP4 queries and keys, BF16 scores).

    The GPU's fp32 score of entry j lies within the accumulation bound e_j of the fp64
    score I_j, and bf16 rounding is monotone, so its bf16 score lies in
    [lo_j, hi_j] = [bf16(I_j - e_j), bf16(I_j + e_j)].  The returned set must be the top
    min(k, n) of some scores in those intervals with ties to the smaller entry: its
    weakest member (smallest hi, then largest index) must beat the strongest entry left
    out (largest lo, then smallest index).  Returned scores lie in their intervals.
    Returns the number of entries that differ from the oracle's own selection.
    """
    q_hat = indexer.quantize_queries_fp4(q)
    I = indexer.scores_fp64(q_hat, w, k_hat[:n])
    ref = indexer.select_topk(indexer.bf16_scores(I), k)
    bound = indexer.accumulation_bound(q_hat, w, k_hat[:n])
    lo = indexer.bf16_scores(I - bound)
    hi = indexer.bf16_scores(I + bound)
    got = np.asarray(got_idx, np.int64)
    m = min(k, n)
    assert np.all(got[m:] == -1)
    gs = got[:m]
    assert np.all(np.diff(gs) > 0), "indices not ascending/unique"
    assert np.all((gs >= 0) & (gs < n))
    if m < n:
        inset = np.zeros(n, bool)
        inset[gs] = True
        g_hi, g_idx = hi[inset], np.flatnonzero(inset)
        weakest = np.lexsort((-g_idx, g_hi))[0]          # smallest hi, then largest index
        o_lo, o_idx = lo[~inset], np.flatnonzero(~inset)
        strongest = np.lexsort((o_idx, -o_lo))[0]        # largest lo, then smallest index
        a_s, a_j = g_hi[weakest], g_idx[weakest]
        b_s, b_j = o_lo[strongest], o_idx[strongest]
        assert a_s > b_s or (a_s == b_s and a_j < b_j), (a_j, a_s, b_j, b_s)
    if got_score is not None:
        sc = np.asarray(got_score, np.float64)[:m]
        assert np.all((sc >= lo[gs]) & (sc <= hi[gs]))
        assert np.array_equal(sc, indexer.bf16_scores(sc))   # bf16 values
    return len(set(gs.tolist()) ^ set(ref[:m].tolist()))
