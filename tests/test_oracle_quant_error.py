"""The quantisation error of the stored formats, reported (tests/quant_report.py prints it
for the whole 1M-context batch); checked here on one full-size request against loose
sanity bounds only - the pages' own quality bar is the 99.7% recall of their FP4 indexer
("DeepSeek-V4 deep dive", section 5.2), which the FP8 keys here are not held to."""

import numpy as np

from compressed_sparse_attention_kv_gb300 import synth
from oracle import codecs, indexer

import quant_report  # noqa: E402  (tests/ is on sys.path)


def test_fp8_index_recall_and_attention_error_one_full_size_request():
    wl = synth.workload("csa_1m")
    q, q_idx, w, sink = synth.queries(wl)
    rec = quant_report.index_recall(wl, 0, q_idx, w)
    assert 0.9 <= rec <= 1.0, rec
    n = int(wl.n_entries[0])
    keys = synth.request_values(wl, 0, "index")[:n].astype(np.float64)
    topk = indexer.select_topk(indexer.scores_fp64(quant_report.bf(q_idx[0]), w[0], keys), wl.k)
    e8 = quant_report.attention_error(wl, 0, q, sink, codecs.FMT_FP8, topk)
    e4 = quant_report.attention_error(wl, 0, q, sink, codecs.FMT_FP4, topk)
    assert e8[1] < 0.05 and e4[1] < 0.2 and e8[1] < e4[1], (e8, e4)
