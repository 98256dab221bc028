"""Quantisation error of the stored formats against unquantised data (reported, not graded).

Uses only the oracle and the seeded generator.  For the 1M-context workload (batch 8,
262,144 N(0,1) index keys per request, 64 indexer heads, top-512):

* indexer recall: the selection from the FP8 index keys (128 e4m3 codes, one power-of-two
  scale per key) and FP8 queries (one scale per head), and from the FP4 index keys
  (rotated, e2m1 + e8m0 per 32, BF16 scores), against the selection from the same keys
  and queries unquantised (fp32 values, fp64 scores); recall = |both| / k;
* attention error: the attention output of a request over FP8-528 or MXFP4-288 main
  entries (and an FP8 window) against the same entries unquantised: max |d| and
  ||d||_2 / ||ref||_2.

    python tests/quant_report.py [requests]
"""

import os
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from compressed_sparse_attention_kv_gb300 import synth  # noqa: E402
from oracle import attention, codecs, indexer  # noqa: E402


def bf(x):
    return codecs.bf16_decode(codecs.bf16_encode(x))


def index_recall(wl, b, q_idx, w):
    """Recall of the FP8 selection of request b against the unquantised one."""
    n = int(wl.n_entries[b])
    keys = synth.request_values(wl, b, "index")[:n]
    q = bf(q_idx[b])
    exact = indexer.select_topk(indexer.scores_fp64(q, w[b], keys.astype(np.float64)), wl.k)
    k_hat = codecs.decode_pagesplit(codecs.encode_pagesplit(synth.request_values(wl, b, "index")), 128)[:n]
    quant = indexer.select_topk(indexer.scores_fp64(indexer.quantize_queries(q), w[b], k_hat), wl.k)
    m = min(wl.k, n)
    return len(set(exact[:m].tolist()) & set(quant[:m].tolist())) / m


def index_recall_fp4(wl, b, q_idx, w):
    """Recall of the FP4 selection (rotated keys and queries, e2m1 + e8m0 per 32, BF16
    scores) of request b against the unquantised one."""
    n = int(wl.n_entries[b])
    keys = synth.request_values(wl, b, "index")
    q = bf(q_idx[b])
    exact = indexer.select_topk(indexer.scores_fp64(q, w[b], keys[:n].astype(np.float64)), wl.k)
    k_hat = codecs.decode_fp4h_pagesplit(codecs.encode_fp4h_pagesplit(keys), 128)
    quant = indexer.index_topk_fp4(q, w[b], k_hat, int(wl.ctx_len[b]), wl.ratio, wl.k)[0]
    m = min(wl.k, n)
    return len(set(exact[:m].tolist()) & set(quant[:m].tolist())) / m


def attention_error(wl, b, q, sink, fmt, topk):
    """max |d| and relative L2 of request b's output over `fmt` entries against fp32 entries."""
    sel = topk[topk >= 0]
    rows = sorted(set(int(j) for j in sel))
    pages = synth.request_values(wl, b, "main", rows=rows)
    n = int(wl.n_entries[b])
    exact = np.zeros((n, 512))
    coded = np.zeros((n, 512))
    for p, v in pages.items():
        lo, hi = p * 64, min(n, p * 64 + 64)
        exact[lo:hi] = v[:hi - lo]
        coded[lo:hi] = codecs.decode_rows(codecs.encode_rows(v, fmt), fmt, 512)[:hi - lo]
    swa = synth.swa_values(wl, b)
    swa_c = codecs.decode_rows(codecs.encode_rows(swa, codecs.FMT_FP8), codecs.FMT_FP8, 512)
    qb = bf(q[b])
    ctx = int(wl.ctx_len[b])
    ref = attention.request_attention(qb, ctx, wl.ratio, swa.astype(np.float64), exact, topk, sink, 512 ** -0.5)
    got = attention.request_attention(qb, ctx, wl.ratio, swa_c, coded, topk, sink, 512 ** -0.5)
    d = got - ref
    return float(np.abs(d).max()), float(np.linalg.norm(d) / np.linalg.norm(ref))


def report(requests):
    wl = synth.workload("csa_1m")
    q, q_idx, w, sink = synth.queries(wl)
    rows = []
    for b in requests:
        rec = index_recall(wl, b, q_idx, w)
        rec4 = index_recall_fp4(wl, b, q_idx, w)
        n = int(wl.n_entries[b])
        keys = synth.request_values(wl, b, "index")[:n]
        topk = indexer.select_topk(indexer.scores_fp64(bf(q_idx[b]), w[b], keys.astype(np.float64)), wl.k)
        e8 = attention_error(wl, b, q, sink, codecs.FMT_FP8, topk)
        e4 = attention_error(wl, b, q, sink, codecs.FMT_FP4, topk)
        rows.append((b, rec, e8, e4, rec4))
        print("request %d: index recall FP8 %.4f FP4 %.4f | FP8-528 attention max|d| %.2e rel %.2e | "
              "MXFP4-288 max|d| %.2e rel %.2e" % (b, rec, rec4, e8[0], e8[1], e4[0], e4[1]))
    return rows


if __name__ == "__main__":
    req = [int(x) for x in sys.argv[1:]] or list(range(8))
    rows = report(req)
    print("mean recall FP8 %.4f FP4 %.4f" % (np.mean([r[1] for r in rows]), np.mean([r[4] for r in rows])))
